// k_sample_stream.cu -- sampling pass for large vocabularies, streaming form:
// one thread-block cluster per cell, the row split across its CTAs, each logit
// read once from HBM; only per-chunk maxima and a few candidates stay on chip.
//
// Per cell, in each CTA:
//   pass 1  stream the slice in 16-byte chunks: z = c + g (c - u), an online
//           (max, sum of exp(z - max), first argmax) per thread rescaled once
//           per batch, and an upper bound (bf16, rounded up) of every
//           8-element chunk's max into shared memory
//   R1      cluster merge of the triples ("perf: avoid full-vocab all-gather for
//           draft greedy sampling", LightLLM PR #1517, Design and invariants:
//           per-shard max, log-sum-exp and argmax, ties to the smallest id)
//   bound   the argmax element's lower-bound score SA = m + tau * G_lo(its
//           noise) is a score some element reaches, so nothing with
//           z + tau * G_max < SA can win the Gumbel race ("Sampler support for
//           discrete diffusion", Hert4's first comment): zmin = SA - tau * G_max
//   pass 2  re-read (from L2) only the chunks whose max reaches zmin and keep
//           their elements with z >= zmin as candidates
//   R3      race over the candidates with table bounds on G, cluster top-2 by
//           upper bound and C = count(z >= zmin); when C <= k every candidate
//           ranks inside the kept set (the k largest z, ties to the smallest
//           id) and every kept element below zmin cannot win, so the race is
//           exact without forming the kept set
//   R4      (only when the bounds leave several candidates) exact G for those
// A cell this cannot settle (C > k or a full candidate buffer) is marked in
// out_tokens and finished exactly by the staged kernel launched right after.
#include <cfloat>
#include <climits>
#include <cooperative_groups.h>
#include <type_traits>

#include "ds_launch.h"
#include "ds_sample_common.cuh"

namespace cg = cooperative_groups;

namespace ds {

namespace {

struct alignas(16) SRec {
  float f[8];
  int i[8];
};

struct SXchg {
  SRec slot[2];
  SRec comb;
};

__device__ __forceinline__ float max3s(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Smallest bf16 value >= f (f finite or -inf): an upper bound kept in 16 bits.
__device__ __forceinline__ uint16_t bf16_ceil(float f) {
  const uint32_t b = __float_as_uint(f);
  uint32_t hi = b >> 16;
  if ((b & 0xffffu) != 0u) hi += (b & 0x80000000u) ? 0u : 1u;  // positive: round up; negative: truncation rounds up
  return (uint16_t)hi;
}

// Online (max, sum of exp(x - max), first argmax) merge.
__device__ __forceinline__ void msa_merge(float& m, float& s, int& am, float m2, float s2, int am2) {
  const float mm = fmaxf(m, m2);
  if (mm == -kInf) {
    am = min(am, am2);
    s = 0.f;
    m = mm;
    return;
  }
  s = s * ex2_approx((m - mm) * kLog2e) + s2 * ex2_approx((m2 - mm) * kLog2e);
  am = (m > m2) ? am : ((m2 > m) ? am2 : min(am, am2));
  m = mm;
}

// Cluster-wide reduction of one record per CTA. Each warp passes a record already
// reduced over the warp (valid in every lane); warp 0 combines the CTA's NT/32
// warp records, then the cluster's CTAs (lane r reads CTA r's record over
// DSMEM). Only the first NF floats and NI ints are moved. Every CTA combines the
// same records in the same tree, so every CTA ends with the same result.
template <int NF, int NI, typename Comb>
__device__ __forceinline__ void warp_tree(SRec& r, int n, Comb comb) {
  const int lane = threadIdx.x & 31;
  for (int o = 1; o < n; o <<= 1) {
    SRec q;
#pragma unroll
    for (int j = 0; j < NF; ++j) q.f[j] = __shfl_down_sync(0xffffffffu, r.f[j], o);
#pragma unroll
    for (int j = 0; j < NI; ++j) q.i[j] = __shfl_down_sync(0xffffffffu, r.i[j], o);
    if ((lane & (2 * o - 1)) == 0 && lane + o < n) comb(r, q);
  }
}

template <int NT, int NF, int NI, typename Comb>
__device__ __forceinline__ SRec cluster_combine(cg::cluster_group& cl, SXchg& xs, SRec* wrec, const SRec& mine,
                                                int& parity, int cs, Comb comb) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) wrec[wid] = mine;
  __syncthreads();
  if (wid == 0) {
    SRec r = wrec[lane < NT / 32 ? lane : 0];
    warp_tree<NF, NI>(r, NT / 32, comb);
    if (lane == 0) xs.slot[parity] = r;
  }
  cl.sync();
  if (wid == 0) {
    SRec r = *cl.map_shared_rank(&xs.slot[parity], lane < cs ? lane : 0);
    warp_tree<NF, NI>(r, cs, comb);
    if (lane == 0) xs.comb = r;
  }
  __syncthreads();
  parity ^= 1;
  return xs.comb;
}

}  // namespace

constexpr int kStreamNT = 256;
constexpr int kStreamUnroll = 2;

template <int NT, int UNROLL>
__global__ void __launch_bounds__(NT, 4) k_sample_stream(const SampleArgs a, int chunk_cap, int cap) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float2* cand = reinterpret_cast<float2*>(smem_raw);           // [cap] (z, id bits)
  uint16_t* cmax = reinterpret_cast<uint16_t*>(cand + cap);     // [chunk_cap] chunk maxima, bf16 rounded up
  uint16_t* hot = cmax + chunk_cap;                             // [chunk_cap] chunks to revisit
  __shared__ SXchg xs;
  __shared__ SRec wrec[NT / 32];
  __shared__ int s_nhot, s_ncand;
  __shared__ ReqCursor s_cur;
  __shared__ long long s_Pu;
  __shared__ int s_bad;

  cg::cluster_group cl = cg::this_cluster();
  const int cs = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const long long n_cells = (long long)a.C * a.P;
  const long long n_clusters = (long long)gridDim.x / cs;
  const long long cluster_id = (long long)blockIdx.x / cs;
  const int P = a.P, V = a.V, k = a.k;
  const float2 neg1 = make_float2(-1.f, -1.f);
  const float2 l2e = make_float2(kLog2e, kLog2e);
  int parity = 0;

  if (wid == 0) {
    const BatchTotals bt = warp_batch_totals(a, lane);
    if (lane == 0) {
      s_bad = (bt.bad || bt.tot != (long long)P) ? 1 : 0;
      s_Pu = bt.tot_u;
    }
  }
  __syncthreads();
  if (s_bad) {
    if (rank == 0 && tid == 0) {
      for (long long cell = cluster_id; cell < n_cells; cell += n_clusters) {
        a.out_tokens[cell] = -1;
        a.out_logprobs[cell] = __int_as_float(0x7fc00000);
      }
      report(a.d_status, DS_DEV_ERR_LAYOUT);
    }
    return;  // uniform across the cluster; no shared memory was shared yet
  }
  const long long P_u = s_Pu;
  // every G lies below g_max, the upper bound of the last table bucket
  const float g_max = kGumbelBounds[(1u << (32 - DS_GUMBEL_BUCKET_SHIFT)) - 1].y;

  for (long long cell = cluster_id; cell < n_cells; cell += n_clusters) {
    const int c = (int)(cell / P);
    const int p = (int)(cell - (long long)c * P);
    if (wid == 0) {
      ReqCursor cur;
      warp_find_request(a, p, lane, cur);
      if (lane == 0) {
        s_cur = cur;
        s_nhot = 0;
        s_ncand = 0;
      }
    }
    __syncthreads();
    const ReqCursor cur = s_cur;
    const int t = p - cur.off;
    const float g = cur.g, tau = cur.tau;
    if (!(tau >= 0.f) || isnan(g) || (g != 0.f && a.u == nullptr)) {
      if (rank == 0 && tid == 0) {
        a.out_tokens[cell] = -1;
        a.out_logprobs[cell] = __int_as_float(0x7fc00000);
        report(a.d_status, (!(tau >= 0.f) || isnan(g)) ? DS_DEV_ERR_PARAM : DS_DEV_ERR_NO_UNCOND);
      }
      __syncthreads();
      continue;
    }
    const bool guided = g != 0.f;
    const bool sampled = tau > 0.f;
    const float2 g2 = make_float2(g, g);

    // ---- slice geometry
    const uint16_t* crow = a.c + cell * (long long)V;
    const uintptr_t ca = reinterpret_cast<uintptr_t>(crow);
    const uint4* cb = reinterpret_cast<const uint4*>(ca & ~(uintptr_t)15);
    const int dc = (int)((ca & 15) >> 1);
    const int nq = (dc + V + 7) >> 3;
    const int q_lo = (int)((long long)rank * nq / cs);
    const int q_hi = (int)((long long)(rank + 1) * nq / cs);
    const uint16_t* urow = nullptr;
    const uint4* ub = nullptr;
    bool u_aligned = true;
    if (guided) {
      urow = a.u + ((long long)c * P_u + cur.off_u + t) * (long long)V;
      const uintptr_t ua = reinterpret_cast<uintptr_t>(urow);
      ub = reinterpret_cast<const uint4*>(ua & ~(uintptr_t)15);
      u_aligned = (ua & 15) == (ca & 15);
    }
    // z of one 16-byte chunk (ids 8q - dc .. 8q - dc + 7), -inf outside the row
    auto chunk_z = [&](int q, uint4 vcw, uint4 vuw, float2 (&z)[4]) {
      const uint32_t wc[4] = {vcw.x, vcw.y, vcw.z, vcw.w};
      const uint32_t wu[4] = {vuw.x, vuw.y, vuw.z, vuw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 cp = make_float2(bf_lo(wc[i]), bf_hi(wc[i]));
        if (guided) {
          const float2 up = make_float2(bf_lo(wu[i]), bf_hi(wu[i]));
          z[i] = __ffma2_rn(g2, __ffma2_rn(up, neg1, cp), cp);  // fl(c - u), then one fma
        } else {
          z[i] = cp;
        }
      }
      if (q == 0 || q >= nq - 1) {  // row edges
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int id = 8 * q - dc + 2 * i;
          if (id < 0 || id >= V) z[i].x = -kInf;
          if (id + 1 < 0 || id + 1 >= V) z[i].y = -kInf;
        }
      }
    };
    auto load_u = [&](int q) -> uint4 {
      if (!guided) return make_uint4(0u, 0u, 0u, 0u);
      if (u_aligned) return ld_stream16(ub + q);
      const int id0 = 8 * q - dc;
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int i0 = id0 + 2 * h, i1 = i0 + 1;
        const uint32_t lo = (i0 >= 0 && i0 < V) ? (uint32_t)__ldg(urow + i0) : 0u;
        const uint32_t hi = (i1 >= 0 && i1 < V) ? (uint32_t)__ldg(urow + i1) : 0u;
        w[h] = lo | (hi << 16);
      }
      return make_uint4(w[0], w[1], w[2], w[3]);
    };

    // ---- pass 1: stream the slice once. Interior chunks go through full
    // batches with no per-chunk checks; the row's edge chunks and the last
    // partial batch go through a checked one-chunk path.
    float m = -kInf, s = 0.f;
    int am = INT_MAX;
    auto pass1 = [&](auto guided_tag) {
      constexpr bool GD = decltype(guided_tag)::value;
      // one batch of NCHK chunks at q0, q0 + NT, ...; CHECKED: mask edges and skip q >= q_hi
      auto load = [&](int q0, auto nchk_tag, auto checked_tag, uint4* vc, uint4* vu) {
        constexpr int NCHK = decltype(nchk_tag)::value;
        constexpr bool CHECKED = decltype(checked_tag)::value;
#pragma unroll
        for (int uu = 0; uu < NCHK; ++uu) {
          const int q = q0 + uu * NT;
          const bool ok = !CHECKED || q < q_hi;
          vc[uu] = ok ? ld_stream16(cb + q) : make_uint4(0u, 0u, 0u, 0u);
          if (GD) vu[uu] = ok ? load_u(q) : make_uint4(0u, 0u, 0u, 0u);
        }
      };
      auto compute = [&](int q0, auto nchk_tag, auto checked_tag, const uint4* vc, const uint4* vu) {
        constexpr int NCHK = decltype(nchk_tag)::value;
        constexpr bool CHECKED = decltype(checked_tag)::value;
        float2 z[NCHK][4];
        float bm = -kInf;
#pragma unroll
        for (int uu = 0; uu < NCHK; ++uu) {
          const int q = q0 + uu * NT;
          const uint32_t wc[4] = {vc[uu].x, vc[uu].y, vc[uu].z, vc[uu].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 cp = make_float2(bf_lo(wc[i]), bf_hi(wc[i]));
            if (GD) {
              const uint32_t wu = (i == 0) ? vu[uu].x : (i == 1) ? vu[uu].y : (i == 2) ? vu[uu].z : vu[uu].w;
              const float2 up = make_float2(bf_lo(wu), bf_hi(wu));
              z[uu][i] = __ffma2_rn(g2, __ffma2_rn(up, neg1, cp), cp);  // fl(c - u), then one fma
            } else {
              z[uu][i] = cp;
            }
          }
          if (CHECKED) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int id = 8 * q - dc + 2 * i;
              if (q >= q_hi || id < 0 || id >= V) z[uu][i].x = -kInf;
              if (q >= q_hi || id + 1 < 0 || id + 1 >= V) z[uu][i].y = -kInf;
            }
          }
          float cm = max3s(z[uu][0].x, z[uu][0].y, z[uu][1].x);
          cm = max3s(cm, z[uu][1].y, z[uu][2].x);
          cm = max3s(cm, z[uu][2].y, z[uu][3].x);
          cm = fmaxf(cm, z[uu][3].y);
          if (!CHECKED || q < q_hi) cmax[q - q_lo] = bf16_ceil(cm);
          bm = fmaxf(bm, cm);
        }
        if (bm >= m && bm > -kInf) {
          // a new (or equal) running max: rescale the sum; keep the smallest id
          // attaining it (chunks are not visited in id order, so take the min)
          if (bm > m) {
            s = (m == -kInf) ? 0.f : s * ex2_approx((m - bm) * kLog2e);
            m = bm;
            am = INT_MAX;
          }
          int aa = INT_MAX;
#pragma unroll
          for (int uu = NCHK - 1; uu >= 0; --uu) {
#pragma unroll
            for (int i = 3; i >= 0; --i) {
              const int id = 8 * (q0 + uu * NT) - dc + 2 * i;
              if (z[uu][i].y == bm) aa = id + 1;
              if (z[uu][i].x == bm) aa = id;
            }
          }
          am = min(am, aa);
        }
        if (m != -kInf) {
          const float2 nml = make_float2(-m * kLog2e, -m * kLog2e);
          float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int uu = 0; uu < NCHK; ++uu)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 tt = __ffma2_rn(z[uu][i], l2e, nml);
              const float2 ee = make_float2(ex2_approx(tt.x), ex2_approx(tt.y));
              if (i & 1) acc1 = __fadd2_rn(acc1, ee); else acc0 = __fadd2_rn(acc0, ee);
            }
          s += (acc0.x + acc0.y) + (acc1.x + acc1.y);
        }
      };
      // interior chunks [qa, qb): no row edges inside
      auto batch = [&](int q0, auto nchk_tag, auto checked_tag) {
        uint4 vc[decltype(nchk_tag)::value], vu[decltype(nchk_tag)::value];
        load(q0, nchk_tag, checked_tag, vc, vu);
        compute(q0, nchk_tag, checked_tag, vc, vu);
      };
      using UN = std::integral_constant<int, UNROLL>;
      using ONE = std::integral_constant<int, 1>;
      if (tid == 0 && q_lo == 0 && q_hi > 0) batch(0, ONE{}, std::true_type{});
      const int qa = max(q_lo, 1), qb = min(q_hi, nq - 1);
      const int n_full = (qb > qa) ? (qb - qa) / (NT * UNROLL) : 0;
      int q0 = qa + tid;
      if (n_full > 0) {
        // the next batch's loads are in flight while this one is reduced
        uint4 cc[UNROLL], cu[UNROLL], nc_[UNROLL], nu[UNROLL];
        load(q0, UN{}, std::false_type{}, cc, cu);
        for (int b = 0; b < n_full; ++b, q0 += NT * UNROLL) {
          if (b + 1 < n_full) load(q0 + NT * UNROLL, UN{}, std::false_type{}, nc_, nu);
          compute(q0, UN{}, std::false_type{}, cc, cu);
#pragma unroll
          for (int uu = 0; uu < UNROLL; ++uu) {
            cc[uu] = nc_[uu];
            cu[uu] = nu[uu];
          }
        }
      }
      // the rest of [qa, qb), then the row-edge chunk nq-1, one chunk at a time
      for (int q = qa + n_full * NT * UNROLL + tid; q < qb; q += NT) batch(q, ONE{}, std::true_type{});
      if (tid == 0 && nq - 1 >= max(q_lo, 1) && nq - 1 < q_hi) batch(nq - 1, ONE{}, std::true_type{});
    };
    if (guided)
      pass1(std::true_type{});
    else
      pass1(std::false_type{});

    // ---- R1: cluster max, sum and first argmax
    float lse;
    {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const int a2 = __shfl_xor_sync(0xffffffffu, am, o);
        msa_merge(m, s, am, m2, s2, a2);
      }
      SRec r{};
      r.f[0] = m; r.f[1] = s; r.i[0] = am;
      const SRec R = cluster_combine<NT, 2, 1>(cl, xs, wrec, r, parity, cs, [](SRec& x, const SRec& y) {
        msa_merge(x.f[0], x.f[1], x.i[0], y.f[0], y.f[1], y.i[0]);
      });
      m = R.f[0];
      am = R.i[0];
      lse = (m == -kInf) ? -kInf : m + logf(R.f[1]);
      if (m == -kInf || !sampled) {  // all -inf (token 0, logprob NaN) or temperature 0 (the argmax)
        if (rank == 0 && tid == 0) {
          a.out_tokens[cell] = (m == -kInf) ? 0 : am;
          a.out_logprobs[cell] = (m == -kInf) ? __int_as_float(0x7fc00000) : m - lse;
        }
        __syncthreads();
        continue;
      }
    }
    const uint32_t t32 = (uint32_t)t;
    const uint32_t ctr3 = a.iter_hi | (uint32_t)c;
    // the argmax element reaches at least SA, so nothing below zmin can win
    const float SA = __fmaf_rn(tau, gumbel_bounds(noise_word((uint32_t)am, t32, cur.rid, ctr3, a.rk0, a.rk1)).x, m);
    const float zmin = SA - (fabsf(SA) + 1.f) * 0x1p-20f - tau * g_max;

    // ---- chunks whose max reaches zmin (warp-aggregated list)
    const int n_loc = q_hi - q_lo;
    for (int j0 = 0; j0 < n_loc; j0 += NT) {
      const int j = j0 + tid;
      const bool h = (j < n_loc) && (__uint_as_float((uint32_t)cmax[j] << 16) >= zmin);
      const unsigned b = __ballot_sync(0xffffffffu, h);
      if (b) {
        int base = 0;
        if (lane == 0) base = atomicAdd(&s_nhot, __popc(b));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (h) hot[base + __popc(b & ((1u << lane) - 1u))] = (uint16_t)j;
      }
    }
    __syncthreads();
    // ---- pass 2: revisit those chunks (L2) and keep their elements >= zmin
    const int nhot = s_nhot;
    for (int h = tid; h < nhot; h += NT) {
      const int q = q_lo + hot[h];
      float2 z[4];
      chunk_z(q, ld_stream16(cb + q), load_u(q), z);
      const int id0 = 8 * q - dc;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (z[i].x >= zmin) {
          const int pos = atomicAdd(&s_ncand, 1);
          if (pos < cap) cand[pos] = make_float2(z[i].x, __int_as_float(id0 + 2 * i));
        }
        if (z[i].y >= zmin) {
          const int pos = atomicAdd(&s_ncand, 1);
          if (pos < cap) cand[pos] = make_float2(z[i].y, __int_as_float(id0 + 2 * i + 1));
        }
      }
    }
    __syncthreads();
    const int nc_all = s_ncand;
    const int nc = min(nc_all, cap);

    // ---- R3: the race over the candidates
    const float2 tau2 = make_float2(tau, tau);
    float zw;
    int idw;
    {
      float loMax = -kInf, hA = -kInf, hB = -kInf;
      int iA = -1;
      for (int i = tid; i < nc; i += NT) {
        const float2 v = cand[i];
        const uint32_t x = noise_word(__float_as_uint(v.y), t32, cur.rid, ctr3, a.rk0, a.rk1);
        const float2 sc = __ffma2_rn(tau2, gumbel_bounds(x), make_float2(v.x, v.x));
        loMax = fmaxf(loMax, sc.x);
        const bool gt = sc.y > hA;
        hB = gt ? hA : fmaxf(hB, sc.y);
        iA = gt ? i : iA;
        hA = fmaxf(hA, sc.y);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float lm2 = __shfl_xor_sync(0xffffffffu, loMax, o);
        const float hA2 = __shfl_xor_sync(0xffffffffu, hA, o);
        const float hB2 = __shfl_xor_sync(0xffffffffu, hB, o);
        const int iA2 = __shfl_xor_sync(0xffffffffu, iA, o);
        loMax = fmaxf(loMax, lm2);
        const bool take = hA2 > hA || (hA2 == hA && iA2 >= 0 && (iA < 0 || iA2 < iA));
        hB = fmaxf(fmaxf(hB, hB2), take ? hA : hA2);
        if (take) {
          hA = hA2;
          iA = iA2;
        }
      }
      SRec r{};
      r.f[0] = loMax;
      r.f[1] = hA;
      r.f[2] = hB;
      r.f[3] = (iA >= 0) ? cand[iA].x : 0.f;
      r.i[0] = (iA >= 0) ? __float_as_int(cand[iA].y) : -1;
      r.i[1] = (wid == 0) ? nc_all : 0;  // a CTA-wide value: count it once per CTA
      r.i[2] = (nc_all > cap) ? 1 : 0;
      const SRec R = cluster_combine<NT, 4, 3>(cl, xs, wrec, r, parity, cs, [](SRec& x, const SRec& y) {
        x.f[0] = fmaxf(x.f[0], y.f[0]);
        const bool take = y.f[1] > x.f[1] || (y.f[1] == x.f[1] && y.i[0] >= 0 && (x.i[0] < 0 || y.i[0] < x.i[0]));
        x.f[2] = fmaxf(fmaxf(x.f[2], y.f[2]), take ? x.f[1] : y.f[1]);
        if (take) {
          x.f[1] = y.f[1];
          x.f[3] = y.f[3];
          x.i[0] = y.i[0];
        }
        x.i[1] += y.i[1];
        x.i[2] |= y.i[2];
      });
      const float S = R.f[0];
      // a full buffer, or candidates that may not all rank inside the kept set
      if (R.i[2] != 0 || R.i[1] > k || !(S > -kInf)) {
        if (rank == 0 && tid == 0) a.out_tokens[cell] = kStreamMark;
        __syncthreads();
        continue;
      }
      const float thr = S - (fabsf(S) + 1.f) * 0x1p-20f;
      if (R.f[2] < thr) {
        zw = R.f[3];
        idw = R.i[0];
      } else {
        // R4: exact G for every candidate whose upper bound reaches thr
        float bs = -kInf, bz = 0.f;
        int bid = INT_MAX;
        for (int i = tid; i < nc; i += NT) {
          const float2 v = cand[i];
          const int id = __float_as_int(v.y);
          const uint32_t x = noise_word((uint32_t)id, t32, cur.rid, ctr3, a.rk0, a.rk1);
          if (__fmaf_rn(tau, gumbel_bounds(x).y, v.x) >= thr) {
            const float scr = __fmaf_rn(tau, gumbel_accurate(x), v.x);
            if (bid == INT_MAX || scr > bs || (scr == bs && id < bid)) {
              bs = scr; bz = v.x; bid = id;
            }
          }
        }
        const int wl = warp_argmax_lane(bs, bid);
        SRec r4{};
        r4.f[0] = __shfl_sync(0xffffffffu, bs, wl);
        r4.f[1] = __shfl_sync(0xffffffffu, bz, wl);
        r4.i[0] = __shfl_sync(0xffffffffu, bid, wl);
        const SRec R4 = cluster_combine<NT, 2, 1>(cl, xs, wrec, r4, parity, cs, [](SRec& x, const SRec& y) {
          if (y.f[0] > x.f[0] || (y.f[0] == x.f[0] && y.i[0] < x.i[0])) x = y;
        });
        zw = R4.f[1];
        idw = R4.i[0];
      }
    }
    if (rank == 0 && tid == 0) {
      a.out_tokens[cell] = idw;
      a.out_logprobs[cell] = zw - lse;
    }
    __syncthreads();
  }
  cl.sync();  // no CTA leaves while a peer may still read its exchange slots
}

// ---------------------------------------------------------------- launcher
cudaError_t launch_sample_stream(const SampleArgs& a, cudaStream_t st) {
  const int nq_max = (a.V + 7 + 7) >> 3;
  // up to 4 CTAs per row: enough logits per thread to amortise the per-cell rounds
  int cs = 1;
  while (cs < 4 && nq_max / cs > 2 * kStreamNT * kStreamUnroll) cs *= 2;
  const int chunk_cap = (nq_max + cs - 1) / cs + 1;
  if (chunk_cap > 65535) return cudaErrorInvalidValue;
  const int cap = 4096;
  auto kern = k_sample_stream<kStreamNT, kStreamUnroll>;
  const size_t smem = (size_t)cap * sizeof(float2) + (size_t)chunk_cap * 2 * sizeof(uint16_t) + 16;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kStreamNT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)cs, 1, 1);
  int max_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (max_clusters < 1) return cudaErrorLaunchOutOfResources;
  const long long n_cells = (long long)a.C * a.P;
  long long n_clusters = max_clusters;
  if (n_clusters > n_cells) n_clusters = n_cells;
  cfg.gridDim = dim3((unsigned)(n_clusters * cs), 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, a, chunk_cap, cap);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ds
