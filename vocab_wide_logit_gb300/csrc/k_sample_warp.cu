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
//   2. lse = m + log sum exp(z - m)
//   3. every element with z >= t_lo is written to a per-lane column of shared
//      memory (the store is unconditional, the column pointer advances only
//      for kept elements), t_lo being a threshold guessed from the moments; the
//      guess is verified exactly: count(z >= t_lo) >= k, so the kept set (the k
//      largest z, ties to the smallest id) lies inside the candidates
//   4. Gumbel race over the candidates: table bounds on G settle the winner
//      unless they overlap, in which case G is evaluated exactly for the few
//      that overlap; the winner's membership in the exact top-k is checked by
//      its rank, and a rare miss takes exact scores for every candidate and
//      the best one that ranks inside the top k
//   5. (token, logprob = z_tok - lse)
//
// Two instantiations share the body. The lean one runs every cell and carries
// only the paths above; a cell whose guess falls short twice, or whose
// candidates overflow the balanced list, is marked. The full one, launched
// right behind it in marker mode, finishes the marked cells (it can keep every
// element and race over the per-lane columns).
#include "ds_warp_common.cuh"

namespace ds {

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

// Occupancy: with the next cell's logits in shared memory rather than
// registers, 4 CTAs of 4 warps fit per SM.
#ifndef DS_WARP_MINB
#define DS_WARP_MINB 4
#endif
#ifndef DS_WARP_LEAN_MINB
#define DS_WARP_LEAN_MINB 4
#endif

template <int NCH, bool FULL>
constexpr int warp_min_blocks() {
  return (NCH <= 4) ? (FULL ? DS_WARP_MINB : DS_WARP_LEAN_MINB) : ((NCH <= 6) ? 3 : 2);
}


// Cell weights for the lean pass with per-request ratios: a request's cells cost
// about the same up to some 130 kept ids (the candidates fit the 5-slot
// straight-line race) and about 0.75% more per kept id above that (longer races
// and lists; measured at V = 1025: k = 205 costs 1.56 times k = 103).
__device__ __forceinline__ long long cell_weight(const SampleArgs& a, int r) {
  const float ratio = a.ratios[r];
  int kk = 1;
  if (ratio > 0.f && ratio <= 1.f) kk = min(max((int)ceilf(ratio * (float)a.V), 1), a.V);
  return 128 + max(0, kk - 130);
}

// Weight of one row of cells (every position once), by the whole warp.
__device__ __forceinline__ long long row_weight(const SampleArgs& a, int lane) {
  long long R = 0;
  for (int base = 0; base < a.B; base += 32) {
    const int r = base + lane;
    long long tw = 0;
    if (r < a.B) tw = (long long)max(a.seq_lens[r], 0) * cell_weight(a, r);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tw += __shfl_xor_sync(0xffffffffu, tw, o);
    R += tw;
  }
  return R;
}

// The first cell whose cumulative weight (cells in (c, p) order) reaches x,
// for 0 <= x <= C R; every lane returns the same cell.
__device__ long long cell_at_weight(const SampleArgs& a, long long x, long long R, int lane) {
  const long long c = x / R;
  if (c >= a.C) return (long long)a.C * a.P;
  const long long rem = x - c * R;
  long long acc = 0;
  int off = 0;
  for (int base = 0; base < a.B; base += 32) {
    const int r = base + lane;
    int T = 0;
    long long w = 1;
    if (r < a.B) {
      T = max(a.seq_lens[r], 0);
      w = cell_weight(a, r);
    }
    const long long tw = (long long)T * w;
    long long inc = tw;
    int incT = T;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, inc, o);
      const int tT = __shfl_up_sync(0xffffffffu, incT, o);
      if (lane >= o) {
        inc += t;
        incT += tT;
      }
    }
    const long long ex = inc - tw;
    const bool here = r < a.B && T > 0 && rem >= acc + ex && rem < acc + inc;
    const unsigned b = __ballot_sync(0xffffffffu, here);
    if (b) {
      // the first of this request's cells whose start weight reaches rem
      const long long t = (rem - acc - ex + w - 1) / w;
      const long long p = (long long)off + (incT - T) + t;
      return c * a.P + __shfl_sync(0xffffffffu, p, __ffs(b) - 1);
    }
    acc += __shfl_sync(0xffffffffu, inc, 31);
    off += __shfl_sync(0xffffffffu, incT, 31);
  }
  return (c + 1) * a.P;
}

// FULL = false: the lean pass (marks what it cannot settle with kStreamMark).
// FULL = true: every path; with only_marked set its warps scan their cell
// ranges for marks and finish just those cells.
// RAISE (lean pass of calls with per-request ratios, where k reaches the list's
// capacity): a first threshold that keeps more than kDenseCap candidates is
// raised once instead of leaving the cell to the exact pass. Calls with one ratio
// for every request run without it: the extra path costs them about 1%.
template <int NCH, bool FULL, bool RAISE>
__global__ void __launch_bounds__(kWarpKernelThreads, (warp_min_blocks<NCH, FULL>()))
    k_sample_warp(const SampleArgs a, int only_marked) {
  pdl_release();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  WarpSmem<NCH>& sm = reinterpret_cast<WarpSmem<NCH>*>(smem_raw)[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;

  const long long n_cells = (long long)a.C * a.P;
  const long long nw = (long long)gridDim.x * (kWarpKernelThreads / 32);
  const long long gw = (long long)blockIdx.x * (kWarpKernelThreads / 32) + (threadIdx.x >> 5);
  long long cbeg = gw * n_cells / nw;
  long long cend = (gw + 1) * n_cells / nw;
  if (!RAISE && cbeg >= cend) return;

  const bool marked_only = FULL && only_marked;
  // first cell at or after `from` in this warp's range that the lean pass marked
  auto next_marked = [&](long long from) -> long long {
    for (long long base = from; base < cend; base += 32) {
      const long long cj = base + lane;
      const unsigned b = __ballot_sync(0xffffffffu, cj < cend && a.out_tokens[cj] == kStreamMark);
      if (b) return base + (__ffs(b) - 1);
    }
    return cend;
  };
  long long cell0 = cbeg;
  if (marked_only) {
    cell0 = next_marked(cbeg);
    if (cell0 >= cend) return;
  }

  const int P = a.P;
  const BatchTotals bt = warp_batch_totals(a, lane);
  if (bt.bad || bt.tot != (long long)P) {
    if (marked_only) return;  // the lean pass has reported it and marked nothing
    for (long long cell = cbeg + lane; cell < cend; cell += 32) {
      a.out_tokens[cell] = -1;
      a.out_logprobs[cell] = __int_as_float(0x7fc00000);
    }
    if (lane == 0 && cbeg < cend) report(a.d_status, DS_DEV_ERR_LAYOUT);
    return;
  }
  if (RAISE) {
    // ranges of equal estimated cost instead of equal cell counts: with per-request
    // ratios the expensive requests would otherwise set the pass's time
    const long long R = row_weight(a, lane);
    const long long total = R * a.C;
    if (R > 0) {
      cbeg = cell_at_weight(a, gw * total / nw, R, lane);
      cend = (gw + 1 == nw) ? n_cells : cell_at_weight(a, (gw + 1) * total / nw, R, lane);
    }
    if (cbeg >= cend) return;
    cell0 = cbeg;
  }
  const long long P_u = bt.tot_u;
  const float2 l2e = make_float2(kLog2e, kLog2e);

  // position -> request walk over the warp's contiguous cell range (in marker
  // mode every visited cell gets a fresh lookup: marks are rare)
  CellWalker walk;
  walk.begin(a, cell0, P_u, lane);
  auto cdst = [&](int j) { return &sm.r.rawc[j][lane]; };
  auto udst = [&](int j) { return &sm.r.rawu[j][lane]; };

  uint32_t sc = 0u, su = 0u;
  CellGeo nxt = walk.geo(a, cell0, false, lane);
  if (nxt.err == 0u) prefetch_cell<NCH>(nxt, lane, cdst, udst, sc, su);

  long long ncell;
  for (long long cell = cell0; cell < cend; cell = ncell) {
    ncell = marked_only ? next_marked(cell + 1) : cell + 1;
    cp_async_wait_all();  // this lane's chunks of the cell have landed
    const CellGeo G = nxt;
    const float g = G.g, tau = G.tau;
    const int k = G.k;
    // Every path below ends at the one prefetch of the next cell (the copies land
    // in the candidate columns, so it comes once those are dead); `done` says the
    // cell's output is already written (or the cell marked for the exact pass).
    bool done = true;
    float lse = 0.f;
    int ctot = 0;
    if (G.err != 0u) {
      if (lane == 0) {
        a.out_tokens[cell] = -1;
        a.out_logprobs[cell] = __int_as_float(0x7fc00000);
        report(a.d_status, G.err);
      }
    } else {
      const bool guided = g != 0.f;
      const int ns = G.ns, sid = G.sid;
      // ---- step 1: z, row max, moments of chunks 0..NCH-2 (always full)
      float2 z[NCH][4];
      const float2 ng2 = make_float2(-g, -g);
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
            // fl(u - c), u widened to fp32 inside the subtraction; it is exactly
            // -fl(c - u) (round to nearest is symmetric), so (-g) fl(u - c) + c in
            // one fma is the combine fma(g, fl(c - u), c)
            float dx, dy;
            asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; sub.rn.f32.bf16 %0, lo, %3; sub.rn.f32.bf16 %1, hi, %4; }"
                : "=f"(dx), "=f"(dy) : "r"(wu[i]), "f"(cp.x), "f"(cp.y));
            z[j][i] = __ffma2_rn(ng2, make_float2(dx, dy), cp);
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
        if (lane == 0) {
          a.out_tokens[cell] = 0;
          a.out_logprobs[cell] = __int_as_float(0x7fc00000);
        }
      } else {
        // ---- step 2: logsumexp (every temperature)
        const float2 nml = make_float2(-m * kLog2e, -m * kLog2e);
        const int idb = G.h + 8 * lane;  // id of element (j, 0) is idb + 256 j
        {
          float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 tt = __ffma2_rn(z[j][i], l2e, nml);
              if (i & 1)
                acc1 = __fadd2_rn(acc1, make_float2(ex2_approx(tt.x), ex2_approx(tt.y)));
              else
                acc0 = __fadd2_rn(acc0, make_float2(ex2_approx(tt.x), ex2_approx(tt.y)));
            }
          }
          float ssum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
          ssum += (lane < ns) ? ex2_approx((zs1 - m) * kLog2e) : 0.f;
          lse = m + logf(warp_sum(ssum));
        }
        if (!(tau > 0.f)) {
          // ---- tau == 0: the smallest id attaining the max
          int am = INT_MAX;
#pragma unroll
          for (int j = NCH - 1; j >= 0; --j) {
#pragma unroll
            for (int i = 3; i >= 0; --i) {
              if (z[j][i].y == m) am = idb + 256 * j + 2 * i + 1;
              if (z[j][i].x == m) am = idb + 256 * j + 2 * i;
            }
          }
          if (lane < ns && zs1 == m) am = min(am, sid);
          am = warp_min_i(am);
          if (lane == 0) {
            a.out_tokens[cell] = am;
            a.out_logprobs[cell] = m - lse;
          }
        } else {
          // ---- threshold guess from the subsample moments
          float tlo = -FLT_MAX;  // -FLT_MAX: keep every finite element
          bool guessed = false;
          float sd = 0.f, mu = 0.f;
          if (NCH >= 2 && G.q_lo > -kInf) {
            const float inv_n = 1.0f / (float)(32 * 8 * (NCH > 1 ? NCH - 1 : 1));  // power of two: exact
            const float S1 = warp_sum(s1.x + s1.y), S2 = warp_sum(s2.x + s2.y);
            mu = S1 * inv_n;
            sd = sqrtf(fmaxf(fmaf(S2, inv_n, -mu * mu), 0.f));
            const float guess = fmaf(sd, G.q_lo, mu);
            if (isfinite(guess)) {
              tlo = fminf(guess, m);
              guessed = true;
            }
          }
          // ---- step 3: compaction of z >= t_lo into this lane's column (each
          // store is unconditional; the address advances by one row only past
          // kept elements, so the lane's last store lands in a row it owns).
          // The count must cover the top k. Otherwise the guess is lowered once
          // by 0.3 sd (a few dozen more candidates near the usual quantiles);
          // the full kernel then keeps every finite element, the lean one marks
          // the cell.
          const uint32_t col0 = (uint32_t)__cvta_generic_to_shared(&sm.col[0][lane]);
          int cnt = 0;
#pragma unroll 1
          for (int attempt = 0;; ++attempt) {
            uint32_t ca = col0;
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
            ca += (zs1 >= tlo) ? 256u : 0u;  // zs1 is -inf for lanes without a scalar element
            cnt = (int)((ca - col0) >> 8);
            ctot = warp_sum_i(cnt);
            // the lean kernel's list holds kDenseCap candidates: more than that
            // raises the threshold once, toward the middle of [k, kDenseCap]
            const bool over = RAISE && ctot > kDenseCap;
            if (!guessed || (ctot >= k && !over) || attempt == (FULL ? 2 : 1)) break;
            // lower the threshold by the shortfall (and a dozen more) over the
            // normal density at the first guess; the full kernel's third
            // attempt keeps every finite element
            float next = -FLT_MAX;
            if (attempt == 0 && sd > 0.f) {
              const float qe = (tlo - mu) / sd;
              const float dens = (float)a.V * 0.39894228f * __expf(-0.5f * qe * qe) / sd;
              next = over ? tlo + (float)(ctot - (k + kDenseCap) / 2) / dens : tlo - (float)(k + 12 - ctot) / dens;
            }
            if (over) {
              if (!(next > tlo)) break;  // no raise possible: the cell is left to the exact pass
              tlo = next;
            } else {
              tlo = (next < tlo && next > -FLT_MAX) ? next : -FLT_MAX;
            }
          }
          __syncwarp();
          if (!FULL && (ctot < k || ctot > kDenseCap)) {
            if (lane == 0) a.out_tokens[cell] = kStreamMark;  // left to the exact pass
          } else if (ctot <= kDenseCap) {
            // the balanced list, filled in rounds: round r copies each lane's
            // r-th candidate (a warp-uniform loop, so no divergent branches)
            const int base = warp_excl_scan(cnt, lane);
            const int rounds = __reduce_max_sync(0xffffffffu, cnt);
            for (int r = 0; r < rounds; ++r)
              if (r < cnt) sm.dense[base + r] = sm.col[r][lane];
            done = false;
          } else {
            // (full kernel only) too many candidates for the list: race over the columns
            Items items;
            items.dense = false;
            items.n = cnt;
            items.n_it = -warp_min_i(-cnt);
            const float2 w = race_generic<NCH>(a, sm, items, ctot, k, tau, (uint32_t)G.t, G.rid,
                                               G.iter_hi | (uint32_t)G.c, lane);
            if (lane == 0) {
              a.out_tokens[cell] = __float_as_int(w.y);
              a.out_logprobs[cell] = w.x - lse;
            }
          }
        }
      }
    }
    __syncwarp();
    // the next cell's logits load while this one races
    if (ncell < cend) {
      nxt = walk.geo(a, ncell, marked_only, lane);
      if (nxt.err == 0u) prefetch_cell<NCH>(nxt, lane, cdst, udst, sc, su);
    }
    if (done) continue;

    // ---- step 4: Gumbel race over the balanced list (a winner outside the top k
    // runs the exact select and race here, in both kernels: it is rare, and a
    // separate pass for it would cost more than its code)
    bool unsettled = false;
    const uint32_t t32 = (uint32_t)G.t, ctr3 = G.iter_hi | (uint32_t)G.c;
    float2 w;
    // 97..160 candidates (the usual count near k = ceil(0.1 V) at V = 1025): the
    // straight-line race over 4 or 5 candidates per lane; other counts: the
    // loop over pairs. Only two straight-line variants are kept: each adds about
    // 8 KB of code, and the kernel's hot code must stay within the SM's
    // instruction cache.
    switch ((ctot + 31) >> 5) {
      case 4: w = race_slots<4>(a, sm.dense, sm.r.hs, sm.r.hist, ctot, k, tau, t32, G.rid, ctr3, lane); break;
      case 5: w = race_slots<5>(a, sm.dense, sm.r.hs, sm.r.hist, ctot, k, tau, t32, G.rid, ctr3, lane); break;
      default:
        w = race_dense<true>(a, sm.dense, sm.r.hs, ctot, k, tau, t32, G.rid, ctr3, lane, sm.r.hist, unsettled);
    }
    // ---- step 5: output (or, in the lean kernel, a mark for the exact pass)
    if (lane == 0) {
      if (unsettled) {
        a.out_tokens[cell] = kStreamMark;
      } else {
        a.out_tokens[cell] = __float_as_int(w.y);
        a.out_logprobs[cell] = w.x - lse;
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- launcher
template <int NCH, bool FULL, bool RAISE = false>
static cudaError_t launch_nch(const SampleArgs& a, cudaStream_t st, int num_sms, int only_marked) {
  const size_t smem = (size_t)(kWarpKernelThreads / 32) * sizeof(WarpSmem<NCH>);
  auto kern = k_sample_warp<NCH, FULL, RAISE>;
  const int per_sm = cached(reinterpret_cast<const void*>(kern), (long long)smem, [&](int) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int n = 0;
    if (r == cudaSuccess) r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kWarpKernelThreads, smem);
    return r != cudaSuccess ? -(int)r : (n < 1 ? 1 : n);
  });
  if (per_sm <= 0) return per_sm < 0 ? (cudaError_t)(-per_sm) : cudaErrorUnknown;
  cudaError_t e;
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
  e = cudaLaunchKernelEx(&cfg, kern, a, only_marked);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

int warp_kernel_max_vocab() { return 8 * 256 + 7; }

template <bool FULL>
static cudaError_t launch_warp_variant(const SampleArgs& a, cudaStream_t st, int num_sms, int only_marked) {
  const int nch = ((a.V >> 3) + 31) / 32;
  if (!FULL && a.ratios) {  // k varies by request and can fill the list (V >= 520)
    switch (nch) {
      case 3: return launch_nch<3, false, true>(a, st, num_sms, only_marked);
      case 4: return launch_nch<4, false, true>(a, st, num_sms, only_marked);
      case 5: return launch_nch<5, false, true>(a, st, num_sms, only_marked);
      case 6: return launch_nch<6, false, true>(a, st, num_sms, only_marked);
      case 7: return launch_nch<7, false, true>(a, st, num_sms, only_marked);
      case 8: return launch_nch<8, false, true>(a, st, num_sms, only_marked);
      default: break;
    }
  }
  switch (nch < 1 ? 1 : nch) {
    case 1: return launch_nch<1, FULL>(a, st, num_sms, only_marked);
    case 2: return launch_nch<2, FULL>(a, st, num_sms, only_marked);
    case 3: return launch_nch<3, FULL>(a, st, num_sms, only_marked);
    case 4: return launch_nch<4, FULL>(a, st, num_sms, only_marked);
    case 5: return launch_nch<5, FULL>(a, st, num_sms, only_marked);
    case 6: return launch_nch<6, FULL>(a, st, num_sms, only_marked);
    case 7: return launch_nch<7, FULL>(a, st, num_sms, only_marked);
    case 8: return launch_nch<8, FULL>(a, st, num_sms, only_marked);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_sample_warp(const SampleArgs& a, cudaStream_t st, int num_sms, bool exact_pass) {
  // the lean pass over every cell, then (unless skipped) the full kernel over the cells it marked
  cudaError_t e = launch_warp_variant<false>(a, st, num_sms, 0);
  if (e == cudaSuccess && exact_pass) e = launch_warp_variant<true>(a, st, num_sms, 1);
  return e;
}

}  // namespace ds
