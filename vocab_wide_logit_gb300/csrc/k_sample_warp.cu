// k_sample_warp.cu -- sampling pass for small vocabularies: one warp per cell.
//
// A cell's row (V <= 2055) is read once from HBM: cp.async copies it, in
// 16-byte chunks, into the warp's shared memory while the previous cell races,
// and the cell keeps it in registers as fp32 z. Each lane owns NCH aligned
// 16-byte chunks (8 elements each) plus at most one scalar element from the
// unaligned head or tail of the row. Every later step (max, logsumexp, the
// top-ratio cut, the Gumbel race) runs on-chip. Warps own contiguous cell
// ranges, so the position -> request walk advances in O(1) per cell.
//
// Steps per cell ("Sampler support for discrete diffusion", Hert4's first
// comment; "Add a sampler resource for discrete diffusion", Contract):
//   1. z = c + g (c - u)                 (u skipped for g == 0), row max,
//                                        moments of a subsample
//   2. lse = m + log sum exp(z - m) and, in the same sweep, every element with
//      z >= t_lo is written to a per-lane column of shared memory (the store
//      is unconditional, the column pointer advances only for kept elements),
//      t_lo being a threshold guessed from the moments
//   3. the guess is verified exactly: count(z >= t_lo) >= k, so the kept set
//      (the k largest z, ties to the smallest id) lies inside the candidates
//   4. Gumbel race over the candidates: table bounds on G settle the winner
//      unless they overlap, in which case G is evaluated exactly for the few
//      that overlap; the winner's membership in the exact top-k is checked by
//      its rank, and a rare miss falls back to an exact 64-bit radix select
//   5. (token, logprob = z_tok - lse)
#include <cfloat>
#include <climits>

#include "ds_launch.h"
#include "ds_sample_common.cuh"

namespace ds {

constexpr int kDenseCap = 256;  // candidates gathered into one balanced list

// The candidate columns are dead once the balanced list is built. From then on
// the same bytes hold the race's upper scores and histogram and the next cell's
// logits, which cp.async copies in while the race runs.
template <int NCH>
struct WarpSmem {
  union {
    float2 col[NCH * 8 + 1][32];  // per-lane candidate columns: (z, id as int bits)
    struct {
      float hs[kDenseCap];        // upper-bound score of each dense candidate
      int hist[256];              // radix histogram of the exact fallback; overlap list of the race
      uint4 rawc[NCH][32];        // the next cell's c chunks (chunk lane + 32 j)
      uint4 rawu[NCH][32];        // and its u chunks
    } r;
  };
  float2 dense[kDenseCap];  // balanced candidate list (the histogram while the columns race)
};

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

// Iterates over this lane's share of the candidates: a balanced slice of the
// dense list, or (when it overflowed) the lane's own column.
struct Items {
  bool dense;
  int n;      // dense: candidate count; column: this lane's count
  int n_it;   // iterations the warp runs
  __device__ __forceinline__ bool get(const float2 (*col)[32], const float2* dl, int it, int lane,
                                      float2& v) const {
    if (dense) {
      const int i = lane + 32 * it;
      if (i >= n) return false;
      v = dl[i];
      return true;
    }
    if (it >= n) return false;
    v = col[it][lane];
    return true;
  }
};

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

// The race over a balanced candidate list (the common case): table bounds for
// two candidates per lane and iteration, branch-free top-2 by upper bound, and
// each upper score kept in shared memory. When the bounds do not settle the
// winner, the candidates whose upper score reaches the best lower score are
// gathered by ballot (usually two or three) and only they get exact G.
__device__ __forceinline__ float2 race_dense(const SampleArgs& a, const float2* dense, float* hs, int ctot, int k,
                                             float tau, uint32_t t32, uint32_t rid, uint32_t ctr3, int lane,
                                             int* hist) {
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
  if (exact) {
    const unsigned long long kth = (ctot > k) ? kth_key(get, n_it, k, lane, hist) : 0ull;
    w = race_exact(a, get, n_it, kth, tau, t32, rid, ctr3);
  }
  return w;
}

// The race over per-lane candidate columns (when too many candidates for the
// balanced list): every step walks the lane's own column.
template <int NCH>
__device__ __forceinline__ float2 race_generic(const SampleArgs& a, WarpSmem<NCH>& sm, const Items& items, int ctot,
                                            int k, float tau, uint32_t t32, uint32_t rid, uint32_t ctr3, int lane) {
  auto get = [&](int it, float2& v) { return items.get(sm.col, sm.dense, it, lane, v); };
  float loMax = -kInf, hA = -kInf, hB = -kInf;
  for (int it = 0; it < items.n_it; ++it) {
    float2 v;
    if (!get(it, v)) continue;
    const uint32_t x = noise_word(__float_as_uint(v.y), t32, rid, ctr3, a.rk0, a.rk1);
    const float2 sc = __ffma2_rn(make_float2(tau, tau), gumbel_bounds(x), make_float2(v.x, v.x));
    loMax = fmaxf(loMax, sc.x);
    hB = (sc.y > hA) ? hA : fmaxf(hB, sc.y);
    hA = fmaxf(hA, sc.y);
  }
  const float S = warp_max(loMax);
  float2 w = make_float2(0.f, 0.f);
  bool exact = !(S > -kInf);
  if (!exact) {
    const float thr = S - (fabsf(S) + 1.f) * 0x1p-20f;
    w = race_resolve(a, get, items.n_it, thr, tau, t32, rid, ctr3);
    if (ctot > k && rank_of(get, items.n_it, w.x, a.keep_ties ? INT_MIN : __float_as_int(w.y)) >= k) exact = true;
  }
  if (exact) {
    const unsigned long long kth =
        (ctot > k) ? kth_key(get, items.n_it, k, lane, reinterpret_cast<int*>(sm.dense)) : 0ull;
    w = race_exact(a, get, items.n_it, kth, tau, t32, rid, ctr3);
  }
  return w;
}

// Starts the copies of a cell's logits into this warp's shared buffers: each
// lane copies its own chunks (lane + 32 j), so it later reads only what it
// copied. The scalar head or tail element goes to registers.
template <int NCH>
__device__ __forceinline__ void prefetch_cell(const CellGeo& G, int lane, WarpSmem<NCH>& sm, uint32_t& sc,
                                              uint32_t& su) {
  const uint4* cb = reinterpret_cast<const uint4*>(G.crow + G.h);
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int q = lane + 32 * j;
    cp_async16(&sm.r.rawc[j][lane], (q < G.nfc) ? cb + q : cb, (q < G.nfc) ? 16u : 0u);
  }
  sc = (lane < G.ns) ? (uint32_t)__ldg(G.crow + G.sid) : 0u;
  su = 0u;
  if (G.g != 0.f) {
    if (G.u_vec) {
      const uint4* ub = reinterpret_cast<const uint4*>(G.urow + G.h);
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int q = lane + 32 * j;
        cp_async16(&sm.r.rawu[j][lane], (q < G.nfc) ? ub + q : ub, (q < G.nfc) ? 16u : 0u);
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
        sm.r.rawu[j][lane] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    su = (lane < G.ns) ? (uint32_t)__ldg(G.urow + G.sid) : 0u;
  }
  cp_async_commit();
}

// Occupancy: with the next cell's logits in shared memory rather than
// registers, 4 CTAs of 4 warps fit per SM.
#ifndef DS_WARP_MINB
#define DS_WARP_MINB 4
#endif

template <int NCH>
__global__ void __launch_bounds__(kWarpKernelThreads, (NCH <= 4) ? DS_WARP_MINB : ((NCH <= 6) ? 3 : 2))
    k_sample_warp(const SampleArgs a) {
  pdl_release();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  WarpSmem<NCH>& sm = reinterpret_cast<WarpSmem<NCH>*>(smem_raw)[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;

  const long long n_cells = (long long)a.C * a.P;
  const long long nw = (long long)gridDim.x * (kWarpKernelThreads / 32);
  const long long gw = (long long)blockIdx.x * (kWarpKernelThreads / 32) + (threadIdx.x >> 5);
  const long long cbeg = gw * n_cells / nw;
  const long long cend = (gw + 1) * n_cells / nw;
  if (cbeg >= cend) return;

  const int P = a.P, V = a.V;
  const BatchTotals bt = warp_batch_totals(a, lane);
  if (bt.bad || bt.tot != (long long)P) {
    for (long long cell = cbeg + lane; cell < cend; cell += 32) {
      a.out_tokens[cell] = -1;
      a.out_logprobs[cell] = __int_as_float(0x7fc00000);
    }
    if (lane == 0) report(a.d_status, DS_DEV_ERR_LAYOUT);
    return;
  }
  const long long P_u = bt.tot_u;
  const float2 neg1 = make_float2(-1.f, -1.f);
  const float2 l2e = make_float2(kLog2e, kLog2e);

  // position -> request cursor over the warp's contiguous cell range
  ReqCursor cur;
  int c = (int)(cbeg / P);
  int p = (int)(cbeg - (long long)c * P);
  warp_find_request(a, p, lane, cur);
  auto next_geo = [&](long long cell) {
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
    G.q_lo = cur.q_lo;
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
  };

  uint32_t sc = 0u, su = 0u;
  CellGeo nxt = next_geo(cbeg);
  if (nxt.err == 0u) prefetch_cell<NCH>(nxt, lane, sm, sc, su);

  for (long long cell = cbeg; cell < cend; ++cell) {
    cp_async_wait_all();  // this lane's chunks of the cell have landed
    const CellGeo G = nxt;
    const bool has_next = cell + 1 < cend;
    auto prefetch_next = [&]() {
      if (has_next) {
        nxt = next_geo(cell + 1);
        if (nxt.err == 0u) prefetch_cell<NCH>(nxt, lane, sm, sc, su);
      }
    };
    if (G.err != 0u) {
      if (lane == 0) {
        a.out_tokens[cell] = -1;
        a.out_logprobs[cell] = __int_as_float(0x7fc00000);
        report(a.d_status, G.err);
      }
      prefetch_next();
      continue;
    }
    const float g = G.g, tau = G.tau;
    const int k = G.k;
    const bool guided = g != 0.f;
    const int ns = G.ns, sid = G.sid;

    // ---- step 1: z, row max, moments of chunks 0..NCH-2 (always full)
    float2 z[NCH][4];
    const float2 g2 = make_float2(g, g);
    float m0 = -kInf, m1 = -kInf;
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const uint4 vc = sm.r.rawc[j][lane];
      const uint4 vu = guided ? sm.r.rawu[j][lane] : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t wc[4] = {vc.x, vc.y, vc.z, vc.w};
      const uint32_t wu[4] = {vu.x, vu.y, vu.z, vu.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 cp = make_float2(bf_lo(wc[i]), bf_hi(wc[i]));
        if (guided) {
          const float2 up = make_float2(bf_lo(wu[i]), bf_hi(wu[i]));
          z[j][i] = __ffma2_rn(g2, __ffma2_rn(up, neg1, cp), cp);  // fl(c - u), then one fma
        } else {
          z[j][i] = cp;
        }
      }
      if (j == NCH - 1 && !(lane + 32 * j < G.nfc)) {
#pragma unroll
        for (int i = 0; i < 4; ++i) z[j][i] = make_float2(-kInf, -kInf);
      }
      m0 = max3(m0, z[j][0].x, z[j][0].y);
      m1 = max3(m1, z[j][1].x, z[j][1].y);
      m0 = max3(m0, z[j][2].x, z[j][2].y);
      m1 = max3(m1, z[j][3].x, z[j][3].y);
      if (j < NCH - 1) {
        s1 = __fadd2_rn(s1, __fadd2_rn(z[j][0], z[j][1]));
        s1 = __fadd2_rn(s1, __fadd2_rn(z[j][2], z[j][3]));
        s2 = __ffma2_rn(z[j][0], z[j][0], s2);
        s2 = __ffma2_rn(z[j][1], z[j][1], s2);
        s2 = __ffma2_rn(z[j][2], z[j][2], s2);
        s2 = __ffma2_rn(z[j][3], z[j][3], s2);
      }
    }
    __syncwarp();  // every lane has read its chunks: the columns may overwrite them
    float zs1;
    {
      const float cf = __uint_as_float(sc << 16);
      zs1 = (lane < ns) ? (guided ? cfg_combine(cf, __uint_as_float(su << 16), g) : cf) : -kInf;
    }
    const float m = warp_max_r(max3(m0, m1, zs1));
    if (m == -kInf) {  // every logit is -inf: token 0, logprob NaN
      prefetch_next();
      if (lane == 0) {
        a.out_tokens[cell] = 0;
        a.out_logprobs[cell] = __int_as_float(0x7fc00000);
      }
      continue;
    }
    const float2 nml = make_float2(-m * kLog2e, -m * kLog2e);
    const int idb = G.h + 8 * lane;  // id of element (j, 0) is idb + 256 j

    // ---- tau == 0: logsumexp and the smallest id attaining the max
    if (!(tau > 0.f)) {
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      int am = INT_MAX;
#pragma unroll
      for (int j = NCH - 1; j >= 0; --j) {
#pragma unroll
        for (int i = 3; i >= 0; --i) {
          const float2 tt = __ffma2_rn(z[j][i], l2e, nml);
          if (i & 1)
            acc1 = __fadd2_rn(acc1, make_float2(ex2_approx(tt.x), ex2_approx(tt.y)));
          else
            acc0 = __fadd2_rn(acc0, make_float2(ex2_approx(tt.x), ex2_approx(tt.y)));
          if (z[j][i].y == m) am = idb + 256 * j + 2 * i + 1;
          if (z[j][i].x == m) am = idb + 256 * j + 2 * i;
        }
      }
      float ssum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
      if (lane < ns) {
        ssum += ex2_approx((zs1 - m) * kLog2e);
        if (zs1 == m) am = min(am, sid);
      }
      prefetch_next();
      const float lse = m + logf(warp_sum(ssum));
      am = warp_min_i(am);
      if (lane == 0) {
        a.out_tokens[cell] = am;
        a.out_logprobs[cell] = m - lse;
      }
      continue;
    }

    // ---- threshold guess from the subsample moments
    float tlo = -FLT_MAX;  // -FLT_MAX: keep every finite element
    bool guessed = false;
    float sd = 0.f;
    if (NCH >= 2 && G.q_lo > -kInf) {
      const float inv_n = 1.0f / (float)(32 * 8 * (NCH > 1 ? NCH - 1 : 1));  // power of two: exact
      const float S1 = warp_sum(s1.x + s1.y), S2 = warp_sum(s2.x + s2.y);
      const float mu = S1 * inv_n;
      sd = sqrtf(fmaxf(fmaf(S2, inv_n, -mu * mu), 0.f));
      const float guess = fmaf(sd, G.q_lo, mu);
      if (isfinite(guess)) {
        tlo = fminf(guess, m);
        guessed = true;
      }
    }

    // ---- step 2: logsumexp and speculative compaction of z >= t_lo into this lane's column
    // (the store is unconditional; the column address advances by one row only
    // for kept elements, so the lane's last store lands in an unused row)
    const uint32_t col0 = (uint32_t)__cvta_generic_to_shared(&sm.col[0][lane]);
    uint32_t ca = col0;
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 zz = z[j][i];
        const float2 tt = __ffma2_rn(zz, l2e, nml);
        if (i & 1)
          acc1 = __fadd2_rn(acc1, make_float2(ex2_approx(tt.x), ex2_approx(tt.y)));
        else
          acc0 = __fadd2_rn(acc0, make_float2(ex2_approx(tt.x), ex2_approx(tt.y)));
        const int id0 = idb + 256 * j + 2 * i;
        st_pair(ca, zz.x, id0);
        ca += (zz.x >= tlo) ? 256u : 0u;
        st_pair(ca, zz.y, id0 + 1);
        ca += (zz.y >= tlo) ? 256u : 0u;
      }
    }
    float ssum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
    ssum += (lane < ns) ? ex2_approx((zs1 - m) * kLog2e) : 0.f;
    st_pair(ca, zs1, sid);
    ca += (zs1 >= tlo) ? 256u : 0u;  // zs1 is -inf for lanes without a scalar element
    int cnt = (int)((ca - col0) >> 8);
    int ctot = warp_sum_i(cnt);

    // ---- step 3: the guess must cover the top k. Otherwise lower it once by
    // 0.3 sd (a few dozen more candidates near the usual quantiles), and if that
    // still falls short keep every finite element: a short count is usually a
    // near miss, and keeping all V elements costs several cells' work.
#pragma unroll 1
    for (int retry = 0; guessed && ctot < k && retry < 2; ++retry) {
      const float lower = tlo - 0.3f * sd;
      tlo = (retry == 0 && lower < tlo && lower > -FLT_MAX) ? lower : -FLT_MAX;
      ca = col0;
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int id0 = idb + 256 * j + 2 * i;
          st_pair(ca, z[j][i].x, id0);
          ca += (z[j][i].x >= tlo) ? 256u : 0u;
          st_pair(ca, z[j][i].y, id0 + 1);
          ca += (z[j][i].y >= tlo) ? 256u : 0u;
        }
      }
      st_pair(ca, zs1, sid);
      ca += (zs1 >= tlo) ? 256u : 0u;
      cnt = (int)((ca - col0) >> 8);
      ctot = warp_sum_i(cnt);
    }
    const float lse = m + logf(warp_sum(ssum));
    __syncwarp();
    Items items;
    items.dense = ctot <= kDenseCap;
    if (items.dense) {
      const int base = warp_excl_scan(cnt, lane);
      for (int j = 0; j < cnt; ++j) sm.dense[base + j] = sm.col[j][lane];
      __syncwarp();
      // the columns are dead: the next cell's logits load while this one races
      prefetch_next();
      items.n = ctot;
      items.n_it = (ctot + 31) >> 5;
    } else {
      items.n = cnt;
      items.n_it = -warp_min_i(-cnt);
    }

    // ---- step 4: Gumbel race
    const uint32_t t32 = (uint32_t)G.t;
    const uint32_t ctr3 = G.iter_hi | (uint32_t)G.c;
    const uint32_t rid = G.rid;
    float2 w;
    if (items.dense) {
      w = race_dense(a, sm.dense, sm.r.hs, ctot, k, tau, t32, rid, ctr3, lane, sm.r.hist);
    } else {
      w = race_generic<NCH>(a, sm, items, ctot, k, tau, t32, rid, ctr3, lane);
      __syncwarp();
      prefetch_next();
    }
    // ---- step 5: output
    if (lane == 0) {
      a.out_tokens[cell] = __float_as_int(w.y);
      a.out_logprobs[cell] = w.x - lse;
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- launcher
template <int NCH>
static cudaError_t launch_nch(const SampleArgs& a, cudaStream_t st, int num_sms) {
  const size_t smem = (size_t)(kWarpKernelThreads / 32) * sizeof(WarpSmem<NCH>);
  cudaError_t e = cudaFuncSetAttribute(k_sample_warp<NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_sample_warp<NCH>, kWarpKernelThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const long long n_cells = (long long)a.C * a.P;
  long long blocks = (long long)num_sms * per_sm;
  const long long max_useful = (n_cells + (kWarpKernelThreads / 32) - 1) / (kWarpKernelThreads / 32);
  if (blocks > max_useful) blocks = max_useful;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(kWarpKernelThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_sample_warp<NCH>, a);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

int warp_kernel_max_vocab() { return 8 * 256 + 7; }

cudaError_t launch_sample_warp(const SampleArgs& a, cudaStream_t st, int num_sms) {
  const int nch = ((a.V >> 3) + 31) / 32;
  switch (nch < 1 ? 1 : nch) {
    case 1: return launch_nch<1>(a, st, num_sms);
    case 2: return launch_nch<2>(a, st, num_sms);
    case 3: return launch_nch<3>(a, st, num_sms);
    case 4: return launch_nch<4>(a, st, num_sms);
    case 5: return launch_nch<5>(a, st, num_sms);
    case 6: return launch_nch<6>(a, st, num_sms);
    case 7: return launch_nch<7>(a, st, num_sms);
    case 8: return launch_nch<8>(a, st, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ds
