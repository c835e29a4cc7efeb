// ds_warp_common.cuh -- pieces shared by the one-warp-per-cell sampling kernels.
//
// The cp.async helpers, the geometry of a cell, the walk from a cell to its
// request, the copies of a cell's logits into shared memory, and the Gumbel race
// over a balanced candidate list with its exact fallback.
#pragma once

#include <cfloat>
#include <climits>

#include "ds_launch.h"
#include "ds_sample_common.cuh"

namespace ds {

constexpr int kDenseCap = 256;  // candidates gathered into one balanced list

__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// (z, id) pair stored at a 32-bit shared-memory address.
__device__ __forceinline__ void st_pair(uint32_t addr, float z, int id) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(z), "f"(__int_as_float(id)) : "memory");
}

// Everything a warp needs to know about one cell before touching its logits.
struct CellGeo {
  int c, t;
  float g, tau;
  uint32_t rid;
  uint32_t err;       // DS_DEV_ERR_* for this cell, 0 if fine
  const uint16_t* crow;
  const uint16_t* urow;
  int h, nfc, ns, sid;
  bool u_vec;         // u row aligned like the c row: vector loads
  int k;              // the request's kept count
  float q_lo;         // and its lower threshold quantile
  uint32_t iter_hi;   // and its iteration << 8
};


// Walks a warp's cells in order, keeping the request that owns the current
// position (O(1) per cell for contiguous ranges; `fresh` looks a cell up from
// scratch, for cells visited out of order).
struct CellWalker {
  ReqCursor cur;
  int c, p;
  long long P_u;

  __device__ __forceinline__ void begin(const SampleArgs& a, long long cell0, long long p_u, int lane) {
    P_u = p_u;
    c = (int)(cell0 / a.P);
    p = (int)(cell0 - (long long)c * a.P);
    warp_find_request(a, p, lane, cur);
  }

  __device__ __forceinline__ CellGeo geo(const SampleArgs& a, long long cell, bool fresh, int lane) {
    const int P = a.P, V = a.V;
    if (fresh) {
      c = (int)(cell / P);
      p = (int)(cell - (long long)c * P);
      warp_find_request(a, p, lane, cur);
    }
    if (p == P) {
      p = 0;
      ++c;
      warp_find_request(a, 0, lane, cur);
    }
    while (p >= cur.off + cur.T) {
      cur.off += cur.T;
      if (cur.g != 0.f) cur.off_u += cur.T;
      ++cur.r;
      cur.T = max(a.seq_lens[cur.r], 0);
      cur.g = a.guidance[cur.r];
      cur.tau = a.temperature[cur.r];
      cur.rid = (uint32_t)a.request_ids[cur.r];
      req_params(a, cur.r, cur);
    }
    CellGeo G;
    G.c = c;
    G.t = p - cur.off;
    ++p;
    G.g = cur.g;
    G.tau = cur.tau;
    G.rid = cur.rid;
    G.err = (!(G.tau >= 0.f) || isnan(G.g) || cur.perr) ? DS_DEV_ERR_PARAM
                                                        : ((G.g != 0.f && a.u == nullptr) ? DS_DEV_ERR_NO_UNCOND : 0u);
    G.k = cur.k;
    G.q_lo = cur.q_w;
    G.iter_hi = cur.iter_hi;
    G.crow = a.c + cell * (long long)V;
    const uintptr_t ca = reinterpret_cast<uintptr_t>(G.crow);
    G.h = min((int)(((16u - (unsigned)(ca & 15)) & 15u) >> 1), V);
    G.nfc = (V - G.h) >> 3;
    G.ns = V - 8 * G.nfc;
    G.sid = (lane < G.h) ? lane : lane + 8 * G.nfc;
    G.urow = nullptr;
    G.u_vec = true;
    if (G.err == 0u && G.g != 0.f) {
      G.urow = a.u + ((long long)c * P_u + cur.off_u + G.t) * (long long)V;
      G.u_vec = (reinterpret_cast<uintptr_t>(G.urow) & 15) == (ca & 15);
    }
    return G;
  }
};

// Starts the copies of a cell's logits into the warp's shared buffers: each
// lane copies its own chunks (lane + 32 j) to cdst(j) and udst(j), so it later
// reads only what it copied. The scalar head or tail element goes to registers.
// The kernel for NCH chunks per lane runs V >= 256 (NCH - 1) + 8, so a row
// holds at least 32 (NCH - 1) full chunks at any alignment: chunks 0..NCH-2 of
// every lane are always full and only the last is predicated.
template <int NCH, typename CDst, typename UDst>
__device__ __forceinline__ void prefetch_cell(const CellGeo& G, int lane, CDst cdst, UDst udst, uint32_t& sc,
                                              uint32_t& su) {
  const uint4* cb = reinterpret_cast<const uint4*>(G.crow + G.h);
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int q = lane + 32 * j;
    if (j < NCH - 1)
      cp_async16(cdst(j), cb + q, 16u);
    else
      cp_async16(cdst(j), (q < G.nfc) ? cb + q : cb, (q < G.nfc) ? 16u : 0u);
  }
  sc = (lane < G.ns) ? (uint32_t)__ldg(G.crow + G.sid) : 0u;
  su = 0u;
  if (G.g != 0.f) {
    if (G.u_vec) {
      const uint4* ub = reinterpret_cast<const uint4*>(G.urow + G.h);
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int q = lane + 32 * j;
        if (j < NCH - 1)
          cp_async16(udst(j), ub + q, 16u);
        else
          cp_async16(udst(j), (q < G.nfc) ? ub + q : ub, (q < G.nfc) ? 16u : 0u);
      }
    } else {
      // u row aligned differently from the c row: gather element by element.
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int q = lane + 32 * j;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (q < G.nfc) {
          const uint16_t* src = G.urow + G.h + 8 * q;
#pragma unroll
          for (int hh = 0; hh < 4; ++hh)
            w[hh] = (uint32_t)__ldg(src + 2 * hh) | ((uint32_t)__ldg(src + 2 * hh + 1) << 16);
        }
        *udst(j) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    su = (lane < G.ns) ? (uint32_t)__ldg(G.urow + G.sid) : 0u;
  }
  cp_async_commit();
}

// k-th largest composite key (z desc, id asc) among n candidates read through
// get(i), by an 8-bit radix select over a shared-memory histogram (keys are
// distinct, so exactly one candidate holds it).
template <typename Get>
__device__ __forceinline__ unsigned long long kth_key(Get get, int n_it, int k, int lane, int* hist) {
  unsigned long long kth = 0ull;
  int need = k;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = lane; b < 256; b += 32) hist[b] = 0;
    __syncwarp();
    for (int it = 0; it < n_it; ++it) {
      float2 v;
      if (!get(it, v)) continue;
      const unsigned long long key = rank_key(v.x, __float_as_int(v.y));
      const bool match = (shift == 56) || ((key >> (shift + 8)) == (kth >> (shift + 8)));
      if (match) atomicAdd(&hist[(int)((key >> shift) & 255ull)], 1);
    }
    __syncwarp();
    // bins in descending digit order: lane l holds digits 255-8l .. 248-8l
    int cl[8], tot = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      cl[e] = hist[255 - 8 * lane - e];
      tot += cl[e];
    }
    const int above_lane = warp_excl_scan(tot, lane);
    const bool here = above_lane < need && need <= above_lane + tot;
    const int src = __ffs(__ballot_sync(0xffffffffu, here)) - 1;
    int digit = 0, above = 0;
    if (lane == src) {
      int run = above_lane;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (run + cl[e] >= need) {
          digit = 255 - 8 * lane - e;
          above = run;
          break;
        }
        run += cl[e];
      }
    }
    digit = __shfl_sync(0xffffffffu, digit, src);
    above = __shfl_sync(0xffffffffu, above, src);
    kth |= (unsigned long long)digit << shift;
    need -= above;
    __syncwarp();
  }
  return kth;
}

// Exact race over the candidates at or above key kth: G evaluated exactly for every one.
template <typename Get>
__device__ __forceinline__ float2 race_exact(const SampleArgs& a, Get get, int n_it, unsigned long long kth, float tau,
                                          uint32_t t32, uint32_t rid, uint32_t ctr3) {
  float bs = -kInf, bz = 0.f;
  int bid = INT_MAX;
  for (int it = 0; it < n_it; ++it) {
    float2 v;
    if (!get(it, v)) continue;
    const int id = __float_as_int(v.y);
    if (member_key(rank_key(v.x, id), a.keep_ties) >= member_key(kth, a.keep_ties)) {
      const uint32_t x = noise_word((uint32_t)id, t32, rid, ctr3, a.rk0, a.rk1);
      const float scr = __fmaf_rn(tau, gumbel_accurate(x), v.x);
      if (bid == INT_MAX || scr > bs || (scr == bs && id < bid)) {
        bs = scr;
        bid = id;
        bz = v.x;
      }
    }
  }
  const int wl = warp_argmax_lane(bs, bid);
  return make_float2(__shfl_sync(0xffffffffu, bz, wl), __int_as_float(__shfl_sync(0xffffffffu, bid, wl)));
}

// Exact G for the candidates whose upper bound reaches thr, then the argmax.
template <typename Get>
__device__ __forceinline__ float2 race_resolve(const SampleArgs& a, Get get, int n_it, float thr, float tau,
                                            uint32_t t32, uint32_t rid, uint32_t ctr3) {
  float bs = -kInf, bz = 0.f;
  int bid = INT_MAX;
  for (int it = 0; it < n_it; ++it) {
    float2 v;
    if (!get(it, v)) continue;
    const int id = __float_as_int(v.y);
    const uint32_t x = noise_word((uint32_t)id, t32, rid, ctr3, a.rk0, a.rk1);
    if (__fmaf_rn(tau, gumbel_bounds(x).y, v.x) >= thr) {
      const float scr = __fmaf_rn(tau, gumbel_accurate(x), v.x);
      if (bid == INT_MAX || scr > bs || (scr == bs && id < bid)) {
        bs = scr;
        bid = id;
        bz = v.x;
      }
    }
  }
  const int wl = warp_argmax_lane(bs, bid);
  return make_float2(__shfl_sync(0xffffffffu, bz, wl), __int_as_float(__shfl_sync(0xffffffffu, bid, wl)));
}

// Rank of (zw, idw) among the candidates: how many precede it in (z desc, id asc).
template <typename Get>
__device__ __forceinline__ int rank_of(Get get, int n_it, float zw, int idw) {
  int rr = 0;
  for (int it = 0; it < n_it; ++it) {
    float2 v;
    if (!get(it, v)) continue;
    rr += (v.x > zw || (v.x == zw && __float_as_int(v.y) < idw)) ? 1 : 0;
  }
  return warp_sum_i(rr);
}

// Exact race over a balanced candidate list whose bounded race was won by a
// candidate outside the top k: every candidate gets its exact score (written
// over the upper scores), then the best candidate by (score desc, id asc) is
// taken while it ranks outside the top k (its rank counted among the
// candidates, which hold the whole kept set), and dropped. Members have finite
// scores, so a member is reached after at most ctot - k drops. Ranks come from
// counting, so no shared-memory histogram (whose atomics serialise when the
// keys share their top bytes) is needed.
__device__ __noinline__ float2 race_exact_by_rank(const SampleArgs& a, const float2* dense, float* score, int ctot,
                                                     int k, float tau, uint32_t t32, uint32_t rid, uint32_t ctr3,
                                                     int lane) {
  const int n_it = (ctot + 31) >> 5;
  __syncwarp();
  for (int it = 0; it < n_it; ++it) {
    const int i = lane + 32 * it;
    if (i < ctot) {
      const float2 v = dense[i];
      const uint32_t x = noise_word(__float_as_uint(v.y), t32, rid, ctr3, a.rk0, a.rk1);
      score[i] = __fmaf_rn(tau, gumbel_accurate(x), v.x);
    }
  }
  __syncwarp();
  float2 w = make_float2(0.f, 0.f);
  for (int drop = 0; drop <= ctot - k; ++drop) {
    float bs = -kInf;
    int bid = INT_MAX, bi = 0;
    for (int it = 0; it < n_it; ++it) {
      const int i = lane + 32 * it;
      if (i < ctot) {
        const float sc = score[i];
        const int id = __float_as_int(dense[i].y);
        if (sc > bs || (sc == bs && id < bid)) {
          bs = sc;
          bid = id;
          bi = i;
        }
      }
    }
    const int wl = warp_argmax_lane(bs, bid);
    const int iw = __shfl_sync(0xffffffffu, bi, wl);
    w = dense[iw];
    const int idw = __float_as_int(w.y);
    int c = 0;
    for (int it = 0; it < n_it; ++it) {
      const int i = lane + 32 * it;
      if (i < ctot) {
        const float2 v = dense[i];
        c += (v.x > w.x || (!a.keep_ties && v.x == w.x && __float_as_int(v.y) < idw)) ? 1 : 0;
      }
    }
    if (warp_sum_i(c) < k) break;
    if (lane == 0) score[iw] = -kInf;
    __syncwarp();
  }
  return w;
}

// Exact G for the listed candidates of the balanced list (their indices in
// list[0..n)), then the argmax by (score desc, id asc). Out of line: it runs
// when the table bounds leave more than one candidate in reach.
__device__ __noinline__ float2 race_listed(const SampleArgs& a, const float2* dense, const int* list, int n, float tau,
                                          uint32_t t32, uint32_t rid, uint32_t ctr3, int lane) {
  float bs = -kInf, bz = 0.f;
  int bid = INT_MAX;
  for (int o = lane; o < n; o += 32) {
    const float2 v = dense[list[o]];
    const int id = __float_as_int(v.y);
    const uint32_t x = noise_word((uint32_t)id, t32, rid, ctr3, a.rk0, a.rk1);
    const float scr = __fmaf_rn(tau, gumbel_accurate(x), v.x);
    if (bid == INT_MAX || scr > bs || (scr == bs && id < bid)) {
      bs = scr;
      bid = id;
      bz = v.x;
    }
  }
  const int wl = warp_argmax_lane(bs, bid);
  return make_float2(__shfl_sync(0xffffffffu, bz, wl), __int_as_float(__shfl_sync(0xffffffffu, bid, wl)));
}

// The race over a balanced candidate list of at most 32 NS candidates, with
// the candidates lane + 32 q (q < NS) of each lane held in registers: every
// draw, table bound and upper score stays in registers and the NS noise chains
// run side by side. The winner is the one candidate whose upper score reaches
// the best lower score S (less a margin); otherwise the candidates in reach get
// exact G. A winner that ranks outside the top k takes the exact race.
template <int NS>
__device__ __forceinline__ float2 race_slots(const SampleArgs& a, const float2* dense, float* hs, int* list, int ctot,
                                             int k, float tau, uint32_t t32, uint32_t rid, uint32_t ctr3, int lane) {
  float2 v[NS];
  uint32_t x[NS];
  float lo[NS], hi[NS];
#pragma unroll
  for (int q = 0; q < NS; ++q) {
    const int i = lane + 32 * q;
    v[q] = dense[i];  // i < 256 = list capacity; entries past ctot are masked below
    x[q] = noise_word(__float_as_uint(v[q].y), t32, rid, ctr3, a.rk0, a.rk1);
  }
  float lm = -kInf;
#pragma unroll
  for (int q = 0; q < NS; ++q) {
    const bool ok = lane + 32 * q < ctot;
    const float2 b = gumbel_bounds(x[q]);
    lo[q] = ok ? __fmaf_rn(tau, b.x, v[q].x) : -kInf;
    hi[q] = ok ? __fmaf_rn(tau, b.y, v[q].x) : -kInf;
    lm = fmaxf(lm, lo[q]);
  }
  const float S = warp_max_r(lm);
  const float thr = S - (fabsf(S) + 1.f) * 0x1p-20f;
  int nin = 0;
  float2 wv = make_float2(0.f, 0.f);
#pragma unroll
  for (int q = 0; q < NS; ++q) {
    const bool in = hi[q] >= thr;
    nin += in ? 1 : 0;
    wv = in ? v[q] : wv;
  }
  float2 w;
  if (warp_sum_i(nin) == 1) {
    const int src = __ffs(__ballot_sync(0xffffffffu, nin != 0)) - 1;
    w = make_float2(__shfl_sync(0xffffffffu, wv.x, src), __shfl_sync(0xffffffffu, wv.y, src));
  } else {
    // exact G for the candidates still in reach (usually two or three), listed
    // by their place in the balanced list
    int n = 0;
    __syncwarp();
#pragma unroll
    for (int q = 0; q < NS; ++q) {
      const bool in = hi[q] >= thr;
      const unsigned b = __ballot_sync(0xffffffffu, in);
      if (in) list[n + __popc(b & ((1u << lane) - 1u))] = lane + 32 * q;
      n += __popc(b);
    }
    __syncwarp();
    w = race_listed(a, dense, list, n, tau, t32, rid, ctr3, lane);
  }
  // membership of the winner in the exact top k: its rank among the candidates
  if (ctot > k) {
    const int idw = __float_as_int(w.y);
    int c = 0;
#pragma unroll
    for (int q = 0; q < NS; ++q) {
      const bool ok = lane + 32 * q < ctot;
      c += (ok && (v[q].x > w.x || (!a.keep_ties && v[q].x == w.x && __float_as_int(v[q].y) < idw))) ? 1 : 0;
    }
    if (warp_sum_i(c) >= k) w = race_exact_by_rank(a, dense, hs, ctot, k, tau, t32, rid, ctr3, lane);
  }
  return w;
}

// The race over a balanced candidate list (the common case): table bounds for
// two candidates per lane and iteration, branch-free top-2 by upper bound, and
// each upper score kept in shared memory. When the bounds do not settle the
// winner, the candidates whose upper score reaches the best lower score are
// gathered by ballot (usually two or three) and only they get exact G.
template <bool FULL>
__device__ __forceinline__ float2 race_dense(const SampleArgs& a, const float2* dense, float* hs, int ctot, int k,
                                             float tau, uint32_t t32, uint32_t rid, uint32_t ctr3, int lane,
                                             int* hist, bool& unsettled) {
  const float2 tau2 = make_float2(tau, tau);
  float loMax = -kInf, hA = -kInf, hB = -kInf;
  int iA = 0;
  // the first 128 candidates stay in registers for the rank check below
  float2 keep[4] = {make_float2(-kInf, 0.f), make_float2(-kInf, 0.f), make_float2(-kInf, 0.f),
                    make_float2(-kInf, 0.f)};
#pragma unroll 1
  for (int base = 0; base < ctot; base += 64) {
    const int i0 = base + lane, i1 = i0 + 32;
    const bool ok0 = i0 < ctot, ok1 = i1 < ctot;
    const float2 v0 = dense[ok0 ? i0 : 0];
    const float2 v1 = dense[ok1 ? i1 : 0];
    if (base == 0) {
      keep[0] = ok0 ? v0 : make_float2(-kInf, __int_as_float(INT_MAX));
      keep[1] = ok1 ? v1 : make_float2(-kInf, __int_as_float(INT_MAX));
    } else if (base == 64) {
      keep[2] = ok0 ? v0 : make_float2(-kInf, __int_as_float(INT_MAX));
      keep[3] = ok1 ? v1 : make_float2(-kInf, __int_as_float(INT_MAX));
    }
    const uint32_t x0 = noise_word(__float_as_uint(v0.y), t32, rid, ctr3, a.rk0, a.rk1);
    const uint32_t x1 = noise_word(__float_as_uint(v1.y), t32, rid, ctr3, a.rk0, a.rk1);
    float2 s0 = __ffma2_rn(tau2, gumbel_bounds(x0), make_float2(v0.x, v0.x));  // (lower, upper) score
    float2 s1 = __ffma2_rn(tau2, gumbel_bounds(x1), make_float2(v1.x, v1.x));
    s0 = ok0 ? s0 : make_float2(-kInf, -kInf);
    s1 = ok1 ? s1 : make_float2(-kInf, -kInf);
    if (ok0) hs[i0] = s0.y;
    if (ok1) hs[i1] = s1.y;
    loMax = fmaxf(loMax, fmaxf(s0.x, s1.x));
    bool gt = s0.y > hA;
    hB = gt ? hA : fmaxf(hB, s0.y);
    iA = gt ? i0 : iA;
    hA = fmaxf(hA, s0.y);
    gt = s1.y > hA;
    hB = gt ? hA : fmaxf(hB, s1.y);
    iA = gt ? i1 : iA;
    hA = fmaxf(hA, s1.y);
  }
  auto get = [&](int it, float2& v) {
    const int i = lane + 32 * it;
    if (i >= ctot) return false;
    v = dense[i];
    return true;
  };
  const int n_it = (ctot + 31) >> 5;
  const float S = warp_max_r(loMax);
  float2 w;
  bool exact = !(S > -kInf);
  if (!exact) {
    const float thr = S - (fabsf(S) + 1.f) * 0x1p-20f;
    const unsigned bc = __ballot_sync(0xffffffffu, hA >= thr);
    const bool cplx = __any_sync(0xffffffffu, hB >= thr);
    if (__popc(bc) == 1 && !cplx) {
      w = dense[__shfl_sync(0xffffffffu, iA, __ffs(bc) - 1)];
    } else {
      // gather the candidates still in reach, then exact G for each
      __syncwarp();
      int nov = 0;
      for (int it = 0; it < n_it; ++it) {
        const int i = lane + 32 * it;
        const bool in = i < ctot && hs[i] >= thr;
        const unsigned b = __ballot_sync(0xffffffffu, in);
        if (in && nov + __popc(b & ((1u << lane) - 1u)) < 256) hist[nov + __popc(b & ((1u << lane) - 1u))] = i;
        nov += __popc(b);
      }
      __syncwarp();
      nov = min(nov, 256);
      float bs = -kInf, bz = 0.f;
      int bid = INT_MAX;
      for (int o = lane; o < nov; o += 32) {
        const float2 v = dense[hist[o]];
        const int id = __float_as_int(v.y);
        const uint32_t x = noise_word((uint32_t)id, t32, rid, ctr3, a.rk0, a.rk1);
        const float scr = __fmaf_rn(tau, gumbel_accurate(x), v.x);
        if (bid == INT_MAX || scr > bs || (scr == bs && id < bid)) {
          bs = scr;
          bid = id;
          bz = v.x;
        }
      }
      const int wl = warp_argmax_lane(bs, bid);
      w = make_float2(__shfl_sync(0xffffffffu, bz, wl), __int_as_float(__shfl_sync(0xffffffffu, bid, wl)));
      __syncwarp();
    }
    // membership of the winner in the exact top-k
    if (ctot > k) {
      int rr;
      if (ctot <= 128) {  // from registers: the candidates this lane held in the race
        const int idw = __float_as_int(w.y);
        int c = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          c += (keep[u].x > w.x || (!a.keep_ties && keep[u].x == w.x && __float_as_int(keep[u].y) < idw)) ? 1 : 0;
        rr = warp_sum_i(c);
      } else {
        rr = rank_of(get, n_it, w.x, a.keep_ties ? INT_MIN : __float_as_int(w.y));
      }
      if (rr >= k) exact = true;
    }
  }
  unsettled = false;
  if (exact) {
    if (FULL)
      w = race_exact_by_rank(a, dense, hs, ctot, k, tau, t32, rid, ctr3, lane);
    else
      unsettled = true;  // left to the exact pass
  }
  return w;
}

}  // namespace ds
