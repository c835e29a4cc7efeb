// k_sample_stream.cu -- sampling pass for large vocabularies, streaming form:
// one thread-block cluster per cell, the row split across its CTAs, each logit
// read once from HBM and never staged in full.
//
// Per cell, each CTA streams its slice in batches of 16-byte chunks and keeps:
//   * an online (max, sum of exp(z - max), first argmax) per thread, rescaled
//     once per batch ("perf: avoid full-vocab all-gather for draft greedy
//     sampling", LightLLM PR #1517, Design and invariants: per-shard max,
//     log-sum-exp and argmax, merged with ties to the smallest id);
//   * in shared memory, only the elements that could still win the Gumbel race
//     ("Sampler support for discrete diffusion", Hert4's first comment): with
//     G confined to [G_min, G_max] by the noise map, an element can only win
//     if z >= max z + tau * (G_min - G_max); the CTA's running max stands in
//     for max z, which keeps the cut conservative.
// Then, over distributed shared memory:
//   R1  max, sum, argmax, and SA = the best lower-bound score of the candidates
//       at each CTA's maximum
//   R3  the race over stored candidates with z >= zmin = SA - tau * G_max (no
//       other element can reach SA): table bounds on G, cluster top-2 by upper
//       bound, and C = count(z >= zmin). When C <= k every element above zmin
//       ranks inside the kept set (the k largest z, ties to the smallest id),
//       and every kept element below zmin cannot win, so the race is exact
//       without ever forming the kept set.
//   R4  (only if the bounds leave several candidates) exact G for those.
// A cell this cannot settle (C > k, a full candidate buffer) is marked in
// out_tokens and finished exactly by the staged kernel launched right after.
#include <cfloat>
#include <climits>
#include <cooperative_groups.h>

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

// Float from an order-preserving key (inverse of order_key).
__device__ __forceinline__ float from_order_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Cluster-wide reduction of one record per CTA: the caller passes a record that
// is already reduced over its warp (valid in every lane); warp 0 combines the
// CTA's warps, then the cluster's CTAs (lane r reads CTA r's record over DSMEM).
// Every CTA combines the same records in the same order.
template <int NT, typename Comb>
__device__ __forceinline__ SRec cluster_combine(cg::cluster_group& cl, SXchg& xs, SRec* wrec, const SRec& mine,
                                                int& parity, int cs, Comb comb) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) wrec[wid] = mine;
  __syncthreads();
  if (wid == 0) {
    SRec r = (lane < NT / 32) ? wrec[lane] : SRec{};
    bool has = lane < NT / 32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      SRec q;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        q.f[j] = __shfl_xor_sync(0xffffffffu, r.f[j], o);
        q.i[j] = __shfl_xor_sync(0xffffffffu, r.i[j], o);
      }
      const bool qhas = __shfl_xor_sync(0xffffffffu, has, o);
      if (qhas) {
        if (has) {
          // combine in a fixed orientation (lower lane first) for determinism
          if ((lane & o) == 0) comb(r, q); else { comb(q, r); r = q; }
        } else {
          r = q;
        }
        has = true;
      }
    }
    if (lane == 0) xs.slot[parity] = r;
  }
  cl.sync();
  if (wid == 0) {
    SRec r = *cl.map_shared_rank(&xs.slot[parity], lane < cs ? lane : 0);
    bool has = lane < cs;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      SRec q;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        q.f[j] = __shfl_xor_sync(0xffffffffu, r.f[j], o);
        q.i[j] = __shfl_xor_sync(0xffffffffu, r.i[j], o);
      }
      const bool qhas = __shfl_xor_sync(0xffffffffu, has, o);
      if (qhas) {
        if (has) {
          if ((lane & o) == 0) comb(r, q); else { comb(q, r); r = q; }
        } else {
          r = q;
        }
        has = true;
      }
    }
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
__global__ void __launch_bounds__(NT, 3) k_sample_stream(const SampleArgs a, int cap) {
  constexpr int EPB = 8 * UNROLL;  // elements per thread per batch
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float2* cand = reinterpret_cast<float2*>(smem_raw);                   // [cap] (z, id bits)
  float* stage = reinterpret_cast<float*>(cand + cap);                  // [NT][EPB] batch values
  __shared__ SXchg xs;
  __shared__ SRec wrec[NT / 32];
  __shared__ int s_ncand;
  __shared__ uint32_t s_maxkey;
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
  float* my_stage = stage + tid * EPB;
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
  // range of the noise map: every G lies in [g_min, g_max]
  const float g_max = kGumbelBounds[(1u << (32 - DS_GUMBEL_BUCKET_SHIFT)) - 1].y;
  const float g_min = kGumbelBounds[0].x;

  for (long long cell = cluster_id; cell < n_cells; cell += n_clusters) {
    const int c = (int)(cell / P);
    const int p = (int)(cell - (long long)c * P);
    if (wid == 0) {
      ReqCursor cur;
      warp_find_request(a, p, lane, cur);
      if (lane == 0) {
        s_cur = cur;
        s_ncand = 0;
        s_maxkey = 0u;  // order key below every float
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
    const float reach = tau * (g_max - g_min);  // the most noise can lift one element over another

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

    // ---- streaming pass
    float m = -kInf, s = 0.f;
    int am = INT_MAX;
    bool overflow = false;
    for (int q0 = q_lo + tid; q0 - tid < q_hi; q0 += NT * UNROLL) {
      uint4 vc[UNROLL], vu[UNROLL];
#pragma unroll
      for (int uu = 0; uu < UNROLL; ++uu) {
        const int q = q0 + uu * NT;
        vc[uu] = (q < q_hi) ? ld_stream16(cb + q) : make_uint4(0u, 0u, 0u, 0u);
      }
      if (guided) {
        if (u_aligned) {
#pragma unroll
          for (int uu = 0; uu < UNROLL; ++uu) {
            const int q = q0 + uu * NT;
            vu[uu] = (q < q_hi) ? ld_stream16(ub + q) : make_uint4(0u, 0u, 0u, 0u);
          }
        } else {
#pragma unroll
          for (int uu = 0; uu < UNROLL; ++uu) {
            const int id0 = 8 * (q0 + uu * NT) - dc;
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int i0 = id0 + 2 * h, i1 = i0 + 1;
              const uint32_t lo = (i0 >= 0 && i0 < V) ? (uint32_t)__ldg(urow + i0) : 0u;
              const uint32_t hi = (i1 >= 0 && i1 < V) ? (uint32_t)__ldg(urow + i1) : 0u;
              w[h] = lo | (hi << 16);
            }
            vu[uu] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      float2 z[UNROLL][4];
      float bm = -kInf;
#pragma unroll
      for (int uu = 0; uu < UNROLL; ++uu) {
        const int q = q0 + uu * NT;
        const uint32_t wc[4] = {vc[uu].x, vc[uu].y, vc[uu].z, vc[uu].w};
        const uint32_t wu[4] = {vu[uu].x, vu[uu].y, vu[uu].z, vu[uu].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 cp = make_float2(bf_lo(wc[i]), bf_hi(wc[i]));
          if (guided) {
            const float2 up = make_float2(bf_lo(wu[i]), bf_hi(wu[i]));
            z[uu][i] = __ffma2_rn(g2, __ffma2_rn(up, neg1, cp), cp);  // fl(c - u), then one fma
          } else {
            z[uu][i] = cp;
          }
        }
        if (q >= q_hi || q == 0 || q >= nq - 1) {  // outside the slice or at a row edge
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int id = 8 * q - dc + 2 * i;
            if (q >= q_hi || id < 0 || id >= V) z[uu][i].x = -kInf;
            if (q >= q_hi || id + 1 < 0 || id + 1 >= V) z[uu][i].y = -kInf;
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) bm = max3s(bm, z[uu][i].x, z[uu][i].y);
      }
      // online max / sum / first argmax (one rescale per batch)
      if (bm > m) {
        s = (m == -kInf) ? 0.f : s * ex2_approx((m - bm) * kLog2e);
        m = bm;
        if (!sampled) {
          int aa = INT_MAX;
#pragma unroll
          for (int uu = UNROLL - 1; uu >= 0; --uu)
#pragma unroll
            for (int i = 3; i >= 0; --i) {
              const int id = 8 * (q0 + uu * NT) - dc + 2 * i;
              if (z[uu][i].y == bm) aa = id + 1;
              if (z[uu][i].x == bm) aa = id;
            }
          am = aa;
        }
      }
      if (m != -kInf) {
        const float2 nml = make_float2(-m * kLog2e, -m * kLog2e);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int uu = 0; uu < UNROLL; ++uu)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 tt = __ffma2_rn(z[uu][i], l2e, nml);
            if (i & 1)
              acc1 = __fadd2_rn(acc1, make_float2(ex2_approx(tt.x), ex2_approx(tt.y)));
            else
              acc0 = __fadd2_rn(acc0, make_float2(ex2_approx(tt.x), ex2_approx(tt.y)));
          }
        s += (acc0.x + acc0.y) + (acc1.x + acc1.y);
      }
      if (sampled) {
        // keep the elements within `reach` of the CTA's running max
        const uint32_t old = atomicMax(&s_maxkey, order_key(bm));
        const float M = fmaxf(from_order_key(old), bm);
        const float cut = (M > -kInf) ? (M - reach) - (fabsf(M) + reach + 1.f) * 0x1p-16f : kInf;
        uint32_t mask = 0u;
#pragma unroll
        for (int uu = 0; uu < UNROLL; ++uu)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            mask |= (z[uu][i].x >= cut) ? (1u << (8 * uu + 2 * i)) : 0u;
            mask |= (z[uu][i].y >= cut) ? (1u << (8 * uu + 2 * i + 1)) : 0u;
          }
        if (__any_sync(0xffffffffu, mask != 0u)) {
          const int cnt = __popc(mask);
          const int ex = warp_excl_scan(cnt, lane);
          int base = 0;
          if (lane == 31) base = atomicAdd(&s_ncand, ex + cnt);
          base = __shfl_sync(0xffffffffu, base, 31);
          int pos = base + ex;
          if (pos + cnt > cap) {
            overflow = true;
          } else if (mask != 0u) {
            float4* st4 = reinterpret_cast<float4*>(my_stage);
#pragma unroll
            for (int uu = 0; uu < UNROLL; ++uu) {
              st4[2 * uu] = make_float4(z[uu][0].x, z[uu][0].y, z[uu][1].x, z[uu][1].y);
              st4[2 * uu + 1] = make_float4(z[uu][2].x, z[uu][2].y, z[uu][3].x, z[uu][3].y);
            }
            while (mask) {
              const int b = __ffs(mask) - 1;
              mask &= mask - 1u;
              const int id = 8 * (q0 + (b >> 3) * NT) - dc + (b & 7);
              cand[pos++] = make_float2(my_stage[b], __int_as_float(id));
            }
          }
        }
      }
    }

    // ---- R1: max, sum, first argmax, overflow, and SA from each CTA's top element(s)
    float lse, SA;
    {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const int a2 = __shfl_xor_sync(0xffffffffu, am, o);
        msa_merge(m, s, am, m2, s2, a2);
      }
      __syncthreads();  // s_ncand, s_maxkey and the candidates are final
      float lo = -kInf;
      if (sampled) {
        const float Mb = from_order_key(s_maxkey);
        const int ncl = min(s_ncand, cap);
        const uint32_t t32 = (uint32_t)t;
        const uint32_t ctr3 = a.iter_hi | (uint32_t)c;
        for (int i = tid; i < ncl; i += NT) {
          const float2 v = cand[i];
          if (v.x >= Mb) {  // this CTA's maximum
            const uint32_t x = noise_word(__float_as_uint(v.y), t32, cur.rid, ctr3, a.rk0, a.rk1);
            lo = fmaxf(lo, __fmaf_rn(tau, gumbel_bounds(x).x, v.x));
          }
        }
        lo = warp_max(lo);
      }
      SRec r{};
      r.f[0] = m; r.f[1] = s; r.i[0] = am;
      r.f[2] = lo;
      r.i[1] = __any_sync(0xffffffffu, overflow) ? 1 : 0;
      const SRec R = cluster_combine<NT>(cl, xs, wrec, r, parity, cs, [](SRec& x, const SRec& y) {
        msa_merge(x.f[0], x.f[1], x.i[0], y.f[0], y.f[1], y.i[0]);
        x.f[2] = fmaxf(x.f[2], y.f[2]);
        x.i[1] |= y.i[1];
      });
      m = R.f[0];
      lse = (m == -kInf) ? -kInf : m + logf(R.f[1]);
      SA = R.f[2];
      if (m == -kInf) {
        if (rank == 0 && tid == 0) {
          a.out_tokens[cell] = 0;
          a.out_logprobs[cell] = __int_as_float(0x7fc00000);
        }
        __syncthreads();
        continue;
      }
      if (!sampled) {
        if (rank == 0 && tid == 0) {
          a.out_tokens[cell] = R.i[0];
          a.out_logprobs[cell] = m - lse;
        }
        __syncthreads();
        continue;
      }
      if (R.i[1] != 0 || !(SA > -kInf)) {  // a full candidate buffer: finish in the staged kernel
        if (rank == 0 && tid == 0) a.out_tokens[cell] = kStreamMark;
        __syncthreads();
        continue;
      }
    }
    const int nc = min(s_ncand, cap);
    const uint32_t t32 = (uint32_t)t;
    const uint32_t ctr3 = a.iter_hi | (uint32_t)c;
    const float2 tau2 = make_float2(tau, tau);
    // nothing below zmin can reach SA, the lower bound of some candidate's score
    const float zmin = SA - (fabsf(SA) + 1.f) * 0x1p-20f - tau * g_max;

    // ---- R3: the race over the stored candidates >= zmin
    float zw;
    int idw;
    {
      float loMax = -kInf, hA = -kInf, hB = -kInf;
      int iA = -1, cnt = 0;
      for (int i = tid; i < nc; i += NT) {
        const float2 v = cand[i];
        if (v.x >= zmin) {
          ++cnt;
          const uint32_t x = noise_word(__float_as_uint(v.y), t32, cur.rid, ctr3, a.rk0, a.rk1);
          const float2 sc = __ffma2_rn(tau2, gumbel_bounds(x), make_float2(v.x, v.x));
          loMax = fmaxf(loMax, sc.x);
          const bool gt = sc.y > hA;
          hB = gt ? hA : fmaxf(hB, sc.y);
          iA = gt ? i : iA;
          hA = fmaxf(hA, sc.y);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float lm2 = __shfl_xor_sync(0xffffffffu, loMax, o);
        const float hA2 = __shfl_xor_sync(0xffffffffu, hA, o);
        const float hB2 = __shfl_xor_sync(0xffffffffu, hB, o);
        const int iA2 = __shfl_xor_sync(0xffffffffu, iA, o);
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
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
      r.i[1] = cnt;
      const SRec R = cluster_combine<NT>(cl, xs, wrec, r, parity, cs, [](SRec& x, const SRec& y) {
        x.f[0] = fmaxf(x.f[0], y.f[0]);
        const bool take = y.f[1] > x.f[1] || (y.f[1] == x.f[1] && y.i[0] >= 0 && (x.i[0] < 0 || y.i[0] < x.i[0]));
        x.f[2] = fmaxf(fmaxf(x.f[2], y.f[2]), take ? x.f[1] : y.f[1]);
        if (take) {
          x.f[1] = y.f[1];
          x.f[3] = y.f[3];
          x.i[0] = y.i[0];
        }
        x.i[1] += y.i[1];
      });
      const float S = R.f[0];
      // every candidate above zmin must rank inside the kept set: count <= k
      if (!(S > -kInf) || R.i[1] > k) {
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
          if (v.x >= zmin) {
            const int id = __float_as_int(v.y);
            const uint32_t x = noise_word((uint32_t)id, t32, cur.rid, ctr3, a.rk0, a.rk1);
            if (__fmaf_rn(tau, gumbel_bounds(x).y, v.x) >= thr) {
              const float scr = __fmaf_rn(tau, gumbel_accurate(x), v.x);
              if (bid == INT_MAX || scr > bs || (scr == bs && id < bid)) {
                bs = scr; bz = v.x; bid = id;
              }
            }
          }
        }
        const int wl = warp_argmax_lane(bs, bid);
        SRec r4{};
        r4.f[0] = __shfl_sync(0xffffffffu, bs, wl);
        r4.f[1] = __shfl_sync(0xffffffffu, bz, wl);
        r4.i[0] = __shfl_sync(0xffffffffu, bid, wl);
        const SRec R4 = cluster_combine<NT>(cl, xs, wrec, r4, parity, cs, [](SRec& x, const SRec& y) {
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
  // 8 CTAs per row for the large vocabularies, fewer for shorter rows
  int cs = 1;
  while (cs < 8 && nq_max / cs > 2 * kStreamNT * kStreamUnroll) cs *= 2;
  const int slice = 8 * ((nq_max + cs - 1) / cs);
  // candidate buffer: a quarter of the slice, at least 2048 entries
  int cap = slice / 4;
  if (cap < 2048) cap = 2048;
  if (cap > slice) cap = slice;
  if (cap > 8192) cap = 8192;
  auto kern = k_sample_stream<kStreamNT, kStreamUnroll>;
  const size_t smem = (size_t)cap * sizeof(float2) + (size_t)kStreamNT * 8 * kStreamUnroll * sizeof(float);
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
  e = cudaLaunchKernelEx(&cfg, kern, a, cap);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ds
