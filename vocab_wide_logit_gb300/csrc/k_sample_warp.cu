// k_sample_warp.cu -- sampling pass for small vocabularies: one warp per cell.
//
// A cell's row (V <= 2055) is read once from HBM with 16-byte streaming loads
// and kept in registers as fp32 z: each lane owns NCH aligned 16-byte chunks
// (8 elements each) plus at most one scalar element from the unaligned head or
// tail of the row. Every later step (max, logsumexp, the top-ratio cut, the
// Gumbel race) runs on-chip. Warps own contiguous cell ranges, so the position
// -> request walk advances in O(1) per cell.
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

template <int NCH>
struct WarpSmem {
  float2 col[NCH * 8 + 1][32];  // per-lane candidate columns: (z, id as int bits)
  float2 dense[kDenseCap];      // balanced candidate list
  int hist[256];                // radix histogram of the exact fallback
};

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
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
};

// Per-lane top-2 of the race by upper score bound, plus the largest bound of the rest.
struct LaneTop2 {
  float hA, hB, h3;
  float2 vA, vB;  // (z, id bits)
  uint32_t xA, xB;
  __device__ __forceinline__ void init() {
    hA = hB = h3 = -kInf;
    vA = vB = make_float2(0.f, __int_as_float(-1));
    xA = xB = 0u;
  }
  __device__ __forceinline__ void insert(float h, float2 v, uint32_t x) {
    if (__float_as_int(vA.y) < 0 || h > hA) {
      h3 = fmaxf(h3, hB);
      hB = hA; vB = vA; xB = xA;
      hA = h; vA = v; xA = x;
    } else if (__float_as_int(vB.y) < 0 || h > hB) {
      h3 = fmaxf(h3, hB);
      hB = h; vB = v; xB = x;
    } else {
      h3 = fmaxf(h3, h);
    }
  }
};

template <int NCH>
__device__ __forceinline__ void load_cell(const CellGeo& G, int lane, uint4 (&rc)[NCH], uint4 (&ru)[NCH],
                                          uint32_t& sc, uint32_t& su) {
  const uint4* cb = reinterpret_cast<const uint4*>(G.crow + G.h);
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int q = lane + 32 * j;
    rc[j] = (q < G.nfc) ? ld_stream16(cb + q) : make_uint4(0u, 0u, 0u, 0u);
  }
  sc = (lane < G.ns) ? (uint32_t)__ldg(G.crow + G.sid) : 0u;
  su = 0u;
  if (G.g != 0.f) {
    if (G.u_vec) {
      const uint4* ub = reinterpret_cast<const uint4*>(G.urow + G.h);
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int q = lane + 32 * j;
        ru[j] = (q < G.nfc) ? ld_stream16(ub + q) : make_uint4(0u, 0u, 0u, 0u);
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
        ru[j] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    su = (lane < G.ns) ? (uint32_t)__ldg(G.urow + G.sid) : 0u;
  }
}

template <int NCH>
__global__ void __launch_bounds__(kWarpKernelThreads, (NCH <= 4) ? 4 : ((NCH <= 6) ? 3 : 2))
    k_sample_warp(const SampleArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  WarpSmem<NCH>& sm = reinterpret_cast<WarpSmem<NCH>*>(smem_raw)[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;

  const long long n_cells = (long long)a.C * a.P;
  const long long nw = (long long)gridDim.x * (kWarpKernelThreads / 32);
  const long long gw = (long long)blockIdx.x * (kWarpKernelThreads / 32) + (threadIdx.x >> 5);
  const long long cbeg = gw * n_cells / nw;
  const long long cend = (gw + 1) * n_cells / nw;
  if (cbeg >= cend) return;

  const int P = a.P, V = a.V, k = a.k;
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
    }
    CellGeo G;
    G.c = c;
    G.t = p - cur.off;
    ++p;
    G.g = cur.g;
    G.tau = cur.tau;
    G.rid = cur.rid;
    G.err = (!(G.tau >= 0.f) || isnan(G.g)) ? DS_DEV_ERR_PARAM
                                            : ((G.g != 0.f && a.u == nullptr) ? DS_DEV_ERR_NO_UNCOND : 0u);
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

  uint4 rc[NCH], ru[NCH];
  uint32_t sc = 0u, su = 0u;
  CellGeo nxt = next_geo(cbeg);
  if (nxt.err == 0u) load_cell<NCH>(nxt, lane, rc, ru, sc, su);

  for (long long cell = cbeg; cell < cend; ++cell) {
    const CellGeo G = nxt;
    const bool has_next = cell + 1 < cend;
    auto prefetch_next = [&]() {
      if (has_next) {
        nxt = next_geo(cell + 1);
        if (nxt.err == 0u) load_cell<NCH>(nxt, lane, rc, ru, sc, su);
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
    const bool guided = g != 0.f;
    const int ns = G.ns, sid = G.sid;

    // ---- step 1: z, row max, moments of chunks 0..NCH-2 (always full)
    float2 z[NCH][4];
    const float2 g2 = make_float2(g, g);
    float m0 = -kInf, m1 = -kInf;
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const uint32_t wc[4] = {rc[j].x, rc[j].y, rc[j].z, rc[j].w};
      const uint32_t wu[4] = {ru[j].x, ru[j].y, ru[j].z, ru[j].w};
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
    float zs1;
    {
      const float cf = __uint_as_float(sc << 16);
      zs1 = (lane < ns) ? (guided ? cfg_combine(cf, __uint_as_float(su << 16), g) : cf) : -kInf;
    }
    const float m = warp_max(max3(m0, m1, zs1));
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
    if (NCH >= 2 && a.q_lo > -kInf) {
      const float n_s = (float)(32 * 8 * (NCH > 1 ? NCH - 1 : 1));
      const float S1 = warp_sum(s1.x + s1.y), S2 = warp_sum(s2.x + s2.y);
      const float mu = S1 / n_s;
      const float sd = sqrtf(fmaxf(S2 / n_s - mu * mu, 0.f));
      const float guess = fmaf(sd, a.q_lo, mu);
      if (isfinite(guess)) {
        tlo = fminf(guess, m);
        guessed = true;
      }
    }

    // ---- step 2: logsumexp and speculative compaction of z >= t_lo into this lane's column
    float2* colp = &sm.col[0][lane];
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
        *colp = make_float2(zz.x, __int_as_float(id0));
        colp += (zz.x >= tlo) ? 32 : 0;
        *colp = make_float2(zz.y, __int_as_float(id0 + 1));
        colp += (zz.y >= tlo) ? 32 : 0;
      }
    }
    float ssum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
    if (lane < ns) {
      ssum += ex2_approx((zs1 - m) * kLog2e);
      *colp = make_float2(zs1, __int_as_float(sid));
      colp += (zs1 >= tlo) ? 32 : 0;
    }
    int cnt = (int)(colp - &sm.col[0][lane]) >> 5;
    int ctot = warp_sum_i(cnt);

    // ---- step 3: the guess must cover the top k; otherwise keep every finite element
    if (guessed && ctot < k) {
      tlo = -FLT_MAX;
      colp = &sm.col[0][lane];
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int id0 = idb + 256 * j + 2 * i;
          *colp = make_float2(z[j][i].x, __int_as_float(id0));
          colp += (z[j][i].x >= tlo) ? 32 : 0;
          *colp = make_float2(z[j][i].y, __int_as_float(id0 + 1));
          colp += (z[j][i].y >= tlo) ? 32 : 0;
        }
      }
      if (lane < ns) {
        *colp = make_float2(zs1, __int_as_float(sid));
        colp += (zs1 >= tlo) ? 32 : 0;
      }
      cnt = (int)(colp - &sm.col[0][lane]) >> 5;
      ctot = warp_sum_i(cnt);
    }
    // z is dead from here on: start loading the next cell while this one races
    prefetch_next();
    const float lse = m + logf(warp_sum(ssum));
    __syncwarp();
    Items items;
    items.dense = ctot <= kDenseCap;
    if (items.dense) {
      const int base = warp_excl_scan(cnt, lane);
      for (int j = 0; j < cnt; ++j) sm.dense[base + j] = sm.col[j][lane];
      __syncwarp();
      items.n = ctot;
      items.n_it = (ctot + 31) >> 5;
    } else {
      items.n = cnt;
      items.n_it = -warp_min_i(-cnt);
    }

    // ---- step 4: Gumbel race, two candidates per iteration
    const uint32_t t32 = (uint32_t)G.t;
    const uint32_t ctr3 = a.iter_hi | (uint32_t)G.c;
    const uint32_t rid = G.rid;
    const float2 tau2 = make_float2(tau, tau);
    float loMax = -kInf;
    LaneTop2 tp;
    tp.init();
    for (int it = 0; it < items.n_it; it += 2) {
      float2 v0, v1;
      const bool ok0 = items.get(sm.col, sm.dense, it, lane, v0);
      const bool ok1 = items.get(sm.col, sm.dense, it + 1, lane, v1);
      if (!ok0) continue;
      const uint32_t x0 = noise_word((uint32_t)__float_as_int(v0.y), t32, rid, ctr3, a.rk0, a.rk1);
      uint32_t x1 = 0u;
      if (ok1) x1 = noise_word((uint32_t)__float_as_int(v1.y), t32, rid, ctr3, a.rk0, a.rk1);
      const float2 sc0 = __ffma2_rn(tau2, gumbel_bounds(x0), make_float2(v0.x, v0.x));  // (lo, hi)
      loMax = fmaxf(loMax, sc0.x);
      tp.insert(sc0.y, v0, x0);
      if (ok1) {
        const float2 sc1 = __ffma2_rn(tau2, gumbel_bounds(x1), make_float2(v1.x, v1.x));
        loMax = fmaxf(loMax, sc1.x);
        tp.insert(sc1.y, v1, x1);
      }
    }
    const float S = warp_max(loMax);
    float2 w = make_float2(0.f, __int_as_float(-1));
    bool exact = !(S > -kInf);
    if (!exact) {
      const float thr = S - (fabsf(S) + 1.f) * 0x1p-20f;
      const bool cA = (__float_as_int(tp.vA.y) >= 0) && (tp.hA >= thr);
      const bool cB = (__float_as_int(tp.vB.y) >= 0) && (tp.hB >= thr);
      const bool cplx = tp.h3 >= thr;
      const unsigned bA = __ballot_sync(0xffffffffu, cA);
      const unsigned bB = __ballot_sync(0xffffffffu, cB);
      const bool anyc = __any_sync(0xffffffffu, cplx);
      if (__popc(bA) + __popc(bB) == 1 && !anyc) {
        const int src = __ffs(bA) - 1;  // the single candidate is some lane's A
        w.x = __shfl_sync(0xffffffffu, tp.vA.x, src);
        w.y = __shfl_sync(0xffffffffu, tp.vA.y, src);
      } else {
        // exact G for the candidates the bounds cannot separate
        float bs = -kInf, bz = 0.f;
        int bid = INT_MAX;
        auto consider = [&](float2 v, uint32_t x) {
          const int id = __float_as_int(v.y);
          const float scr = __fmaf_rn(tau, gumbel_accurate(x), v.x);
          if (bid == INT_MAX || scr > bs || (scr == bs && id < bid)) {
            bs = scr;
            bid = id;
            bz = v.x;
          }
        };
        if (cplx) {
          for (int it = 0; it < items.n_it; ++it) {
            float2 v;
            if (!items.get(sm.col, sm.dense, it, lane, v)) continue;
            const uint32_t x = noise_word((uint32_t)__float_as_int(v.y), t32, rid, ctr3, a.rk0, a.rk1);
            if (__fmaf_rn(tau, gumbel_bounds(x).y, v.x) >= thr) consider(v, x);
          }
        } else {
          if (cA) consider(tp.vA, tp.xA);
          if (cB) consider(tp.vB, tp.xB);
        }
        const int wl = warp_argmax_lane(bs, bid);
        w.x = __shfl_sync(0xffffffffu, bz, wl);
        w.y = __int_as_float(__shfl_sync(0xffffffffu, bid, wl));
      }
      // membership of the winner in the exact top-k (rank by (z desc, id asc))
      if (ctot > k) {
        const int idw = __float_as_int(w.y);
        int rr = 0;
        for (int it = 0; it < items.n_it; ++it) {
          float2 v;
          if (!items.get(sm.col, sm.dense, it, lane, v)) continue;
          rr += (v.x > w.x || (v.x == w.x && __float_as_int(v.y) < idw)) ? 1 : 0;
        }
        if (warp_sum_i(rr) >= k) exact = true;
      }
    }
    if (exact) {
      // Exact kept set: the k-th largest composite key (z desc, id asc) among the
      // candidates, by an 8-bit radix select over shared-memory histograms; every
      // candidate is kept when ctot <= k.
      unsigned long long kth = 0ull;
      if (ctot > k) {
        int need = k;
        for (int shift = 56; shift >= 0; shift -= 8) {
          for (int b = lane; b < 256; b += 32) sm.hist[b] = 0;
          __syncwarp();
          for (int it = 0; it < items.n_it; ++it) {
            float2 v;
            if (!items.get(sm.col, sm.dense, it, lane, v)) continue;
            const unsigned long long key = rank_key(v.x, __float_as_int(v.y));
            const bool match = (shift == 56) || ((key >> (shift + 8)) == (kth >> (shift + 8)));
            if (match) atomicAdd(&sm.hist[(int)((key >> shift) & 255ull)], 1);
          }
          __syncwarp();
          // bins in descending digit order: lane l holds digits 255-8l .. 248-8l
          int cl[8], tot = 0;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            cl[e] = sm.hist[255 - 8 * lane - e];
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
      }
      float bs = -kInf, bz = 0.f;
      int bid = INT_MAX;
      for (int it = 0; it < items.n_it; ++it) {
        float2 v;
        if (!items.get(sm.col, sm.dense, it, lane, v)) continue;
        const int id = __float_as_int(v.y);
        if (rank_key(v.x, id) >= kth) {
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
      w.x = __shfl_sync(0xffffffffu, bz, wl);
      w.y = __int_as_float(__shfl_sync(0xffffffffu, bid, wl));
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
  k_sample_warp<NCH><<<(unsigned)blocks, kWarpKernelThreads, smem, st>>>(a);
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
