// k_sample_warp.cu -- sampling pass for small vocabularies: one warp per cell.
//
// A cell's whole row (V <= 8 * 256 - 7 elements) is loaded with 16-byte
// streaming loads and kept in registers as fp32 z; every later step (max,
// logsumexp, the top-ratio cut and the Gumbel race) runs on-chip, so the
// logits are read from HBM exactly once. Warps own contiguous cell ranges, so
// the position -> request walk advances in O(1) per cell.
//
// Steps per cell ("Sampler support for discrete diffusion", Hert4's first
// comment; "Add a sampler resource for discrete diffusion", Contract):
//   1. z = c + g (c - u)                 (u skipped for g == 0)
//   2. m = max z, lse = m + log sum exp(z - m), argmax (tau == 0)
//   3. kept set = k largest z, ties to the smallest id: a lower threshold
//      t_lo is guessed from the row's moments, verified by counting
//      (count(z >= t_lo) >= k) and the candidates compacted to shared memory
//   4. Gumbel race over the candidates: table bounds on G settle the winner
//      unless the bounds overlap, in which case G is evaluated exactly for the
//      overlapping few; the winner's membership in the exact top-k is
//      checked by its rank, and a rare miss falls back to an exact 64-bit
//      radix select of the k-th key
//   5. (token, logprob = z_tok - lse)
#include <climits>

#include "ds_launch.h"
#include "ds_sample_common.cuh"

namespace ds {

template <int NCH>
__global__ void __launch_bounds__(kWarpKernelThreads) k_sample_warp(const SampleArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  float2* Lb = reinterpret_cast<float2*>(smem_raw) + (size_t)wib * (NCH * 256);

  const long long n_cells = (long long)a.C * a.P;
  const long long nw = (long long)gridDim.x * (kWarpKernelThreads / 32);
  const long long gw = (long long)blockIdx.x * (kWarpKernelThreads / 32) + wib;
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

  ReqCursor cur;
  cur.r = -1;
  int cur_c = -1;

  for (long long cell = cbeg; cell < cend; ++cell) {
    const int c = (int)(cell / P);
    const int p = (int)(cell - (long long)c * P);
    if (c != cur_c || cur.r < 0 || p < cur.off) {
      warp_find_request(a, p, lane, cur);  // always found: the totals were checked
      cur_c = c;
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
    const int t = p - cur.off;
    const float g = cur.g, tau = cur.tau;
    {
      uint32_t err = 0;
      if (!(tau >= 0.f) || isnan(g)) err |= DS_DEV_ERR_PARAM;
      if (g != 0.f && a.u == nullptr) err |= DS_DEV_ERR_NO_UNCOND;
      if (err) {
        if (lane == 0) {
          a.out_tokens[cell] = -1;
          a.out_logprobs[cell] = __int_as_float(0x7fc00000);
          report(a.d_status, err);
        }
        continue;
      }
    }

    // ---- load the row (16-byte chunks of the aligned span covering it)
    const uint16_t* crow = a.c + cell * (long long)V;
    const uintptr_t ca = reinterpret_cast<uintptr_t>(crow);
    const uint4* cb = reinterpret_cast<const uint4*>(ca & ~(uintptr_t)15);
    const int dc = (int)((ca & 15) >> 1);  // elements of the first chunk before the row
    const int nq = (dc + V + 7) >> 3;      // chunks covering the row
    uint4 rc[NCH], ru[NCH];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int q = lane + 32 * j;
      rc[j] = (q < nq) ? ld_stream16(cb + q) : make_uint4(0u, 0u, 0u, 0u);
    }
    const bool guided = g != 0.f;
    if (guided) {
      const uint16_t* urow = a.u + ((long long)c * P_u + cur.off_u + t) * (long long)V;
      const uintptr_t ua = reinterpret_cast<uintptr_t>(urow);
      if (((ua & 15) >> 1) == (uintptr_t)dc) {
        const uint4* ub = reinterpret_cast<const uint4*>(ua & ~(uintptr_t)15);
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int q = lane + 32 * j;
          ru[j] = (q < nq) ? ld_stream16(ub + q) : make_uint4(0u, 0u, 0u, 0u);
        }
      } else {
        // u row aligned differently from the c row: gather element by element.
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int id0 = 8 * (lane + 32 * j) - dc;
          uint32_t w[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int i0 = id0 + 2 * h, i1 = i0 + 1;
            const uint32_t lo = (i0 >= 0 && i0 < V) ? (uint32_t)__ldg(urow + i0) : 0u;
            const uint32_t hi = (i1 >= 0 && i1 < V) ? (uint32_t)__ldg(urow + i1) : 0u;
            w[h] = lo | (hi << 16);
          }
          ru[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }

    // ---- step 1/2a: z, row max, moments of the interior chunks
    float z[NCH][8];
    float m = -kInf, s1 = 0.f, s2 = 0.f;
    int nsub = 0;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int q = lane + 32 * j;
      float cf[8];
      unpack8(rc[j], cf);
      if (guided) {
        float uf[8];
        unpack8(ru[j], uf);
#pragma unroll
        for (int e = 0; e < 8; ++e) z[j][e] = cfg_combine(cf[e], uf[e], g);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) z[j][e] = cf[e];
      }
      if (q == 0 || q >= nq - 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int id = 8 * q - dc + e;
          if (id < 0 || id >= V) z[j][e] = -kInf;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, z[j][e]);
      if (j >= 1 && j <= NCH - 2 && q < nq - 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          s1 += z[j][e];
          s2 = fmaf(z[j][e], z[j][e], s2);
        }
        nsub += 8;
      }
    }
    m = warp_max(m);
    if (m == -kInf) {  // every logit is -inf: token 0, logprob NaN
      if (lane == 0) {
        a.out_tokens[cell] = 0;
        a.out_logprobs[cell] = __int_as_float(0x7fc00000);
      }
      continue;
    }

    const bool sampled = tau > 0.f;
    float mu = 0.f, sd = 0.f, tlo = -kInf;
    bool all_mode = true;
    if (sampled) {
      const int n_s = warp_sum_i(nsub);
      const float S1 = warp_sum(s1), S2 = warp_sum(s2);
      if (n_s >= 64 && a.q_lo > -kInf) {
        mu = S1 / (float)n_s;
        sd = sqrtf(fmaxf(S2 / (float)n_s - mu * mu, 0.f));
        const float guess = fmaf(sd, a.q_lo, mu);
        if (isfinite(guess)) {
          tlo = fminf(guess, m);
          all_mode = false;
        }
      }
    }

    // ---- step 2b: logsumexp, count above t_lo (or argmax for tau == 0)
    float ssum = 0.f;
    int cnt = 0;
    int amin = INT_MAX;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        ssum += ex2_approx((z[j][e] - m) * kLog2e);
        cnt += (z[j][e] >= tlo) ? 1 : 0;
      }
    }
    const float lse = m + logf(warp_sum(ssum));
    if (!sampled) {
#pragma unroll
      for (int j = NCH - 1; j >= 0; --j) {
#pragma unroll
        for (int e = 7; e >= 0; --e) {
          if (z[j][e] == m) amin = 8 * (lane + 32 * j) - dc + e;
        }
      }
      const int am = warp_min_i(amin);
      if (lane == 0) {
        a.out_tokens[cell] = am;
        a.out_logprobs[cell] = m - lse;
      }
      continue;
    }

    // ---- step 3: verify the threshold guess and compact the candidates
    int ctot;
    if (!all_mode) {
      ctot = warp_sum_i(cnt);
      if (ctot < k) {
        const float guess = fmaf(sd, a.q_lo - 1.0f, mu);
        all_mode = true;
        if (isfinite(guess) && guess < tlo) {
          tlo = guess;
          cnt = 0;
#pragma unroll
          for (int j = 0; j < NCH; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) cnt += (z[j][e] >= tlo) ? 1 : 0;
          ctot = warp_sum_i(cnt);
          all_mode = ctot < k;
        }
      }
    }
    if (all_mode) {
      cnt = 0;
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int id0 = 8 * (lane + 32 * j) - dc;
#pragma unroll
        for (int e = 0; e < 8; ++e) cnt += (id0 + e >= 0 && id0 + e < V) ? 1 : 0;
      }
      ctot = V;
    }
    {
      int pos = warp_excl_scan(cnt, lane);
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int id0 = 8 * (lane + 32 * j) - dc;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int id = id0 + e;
          const bool keep = all_mode ? (id >= 0 && id < V) : (z[j][e] >= tlo);
          if (keep) {
            Lb[pos] = make_float2(z[j][e], __int_as_float(id));
            ++pos;
          }
        }
      }
    }
    __syncwarp();

    // ---- step 4: Gumbel race over the candidates
    const uint32_t t32 = (uint32_t)t;
    const uint32_t ctr3 = a.iter_hi | (uint32_t)c;
    float loMax = -kInf, hiA = -kInf, hi2 = -kInf;
    int iA = -1;
    uint32_t xA = 0;
    for (int i = lane; i < ctot; i += 32) {
      const float2 it = Lb[i];
      const uint32_t x = noise_word((uint32_t)__float_as_int(it.y), t32, cur.rid, ctr3, a.key0, a.key1);
      const float2 gb = gumbel_bounds(x);
      const float lo = __fmaf_rn(tau, gb.x, it.x);
      const float hi = __fmaf_rn(tau, gb.y, it.x);
      loMax = fmaxf(loMax, lo);
      if (iA < 0 || hi > hiA) {
        hi2 = hiA;
        hiA = hi;
        iA = i;
        xA = x;
      } else {
        hi2 = fmaxf(hi2, hi);
      }
    }
    const float S = warp_max(loMax);
    int w_item = -1;
    bool exact = !(S > -kInf);
    if (!exact) {
      const float thr = S - (fabsf(S) + 1.f) * 0x1p-20f;
      const bool cand = (iA >= 0) && (hiA >= thr);
      const bool cplx = hi2 >= thr;
      const unsigned bc = __ballot_sync(0xffffffffu, cand);
      const bool anyc = __any_sync(0xffffffffu, cplx);
      if (__popc(bc) == 1 && !anyc) {
        w_item = __shfl_sync(0xffffffffu, iA, __ffs(bc) - 1);
      } else {
        float bs = -kInf;
        int bid = INT_MAX, bit = -1;
        if (cplx) {
          for (int i = lane; i < ctot; i += 32) {
            const float2 it = Lb[i];
            const int id = __float_as_int(it.y);
            const uint32_t x = noise_word((uint32_t)id, t32, cur.rid, ctr3, a.key0, a.key1);
            const float hi = __fmaf_rn(tau, gumbel_bounds(x).y, it.x);
            if (hi >= thr) {
              const float sc = __fmaf_rn(tau, gumbel_accurate(x), it.x);
              if (bit < 0 || sc > bs || (sc == bs && id < bid)) {
                bs = sc;
                bid = id;
                bit = i;
              }
            }
          }
        } else if (cand) {
          const float2 it = Lb[iA];
          bs = __fmaf_rn(tau, gumbel_accurate(xA), it.x);
          bid = __float_as_int(it.y);
          bit = iA;
        }
        const int wl = warp_argmax_lane(bs, bid);
        w_item = __shfl_sync(0xffffffffu, bit, wl);
      }
      // membership of the winner in the exact top-k (rank by (z desc, id asc))
      if (ctot > k) {
        const float2 w = Lb[w_item];
        const int idw = __float_as_int(w.y);
        int rr = 0;
        for (int i = lane; i < ctot; i += 32) {
          const float2 it = Lb[i];
          rr += (it.x > w.x || (it.x == w.x && __float_as_int(it.y) < idw)) ? 1 : 0;
        }
        if (warp_sum_i(rr) >= k) exact = true;
      }
    }
    if (exact) {
      // k-th largest composite key among the candidates (all keys distinct),
      // one bit at a time from the top.
      unsigned long long kth = 0ull;
      for (int b = 63; b >= 0; --b) {
        const unsigned long long probe = kth | (1ull << b);
        int cb2 = 0;
        for (int i = lane; i < ctot; i += 32) {
          const float2 it = Lb[i];
          cb2 += (rank_key(it.x, __float_as_int(it.y)) >= probe) ? 1 : 0;
        }
        if (warp_sum_i(cb2) >= k) kth = probe;
      }
      float bs = -kInf;
      int bid = INT_MAX, bit = -1;
      for (int i = lane; i < ctot; i += 32) {
        const float2 it = Lb[i];
        const int id = __float_as_int(it.y);
        if (rank_key(it.x, id) >= kth) {
          const uint32_t x = noise_word((uint32_t)id, t32, cur.rid, ctr3, a.key0, a.key1);
          const float sc = __fmaf_rn(tau, gumbel_accurate(x), it.x);
          if (bit < 0 || sc > bs || (sc == bs && id < bid)) {
            bs = sc;
            bid = id;
            bit = i;
          }
        }
      }
      const int wl = warp_argmax_lane(bs, bid);
      w_item = __shfl_sync(0xffffffffu, bit, wl);
    }

    // ---- step 5: output
    if (lane == 0) {
      const float2 w = Lb[w_item];
      a.out_tokens[cell] = __float_as_int(w.y);
      a.out_logprobs[cell] = w.x - lse;
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- launcher
template <int NCH>
static cudaError_t launch_nch(const SampleArgs& a, cudaStream_t st, int num_sms) {
  const size_t smem = (size_t)(kWarpKernelThreads / 32) * NCH * 256 * sizeof(float2);
  static bool configured = false;  // per process; the attribute is per function
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_sample_warp<NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_sample_warp<NCH>,
                                                                kWarpKernelThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const long long n_cells = (long long)a.C * a.P;
  const long long warps_needed = n_cells;
  long long blocks = (long long)num_sms * per_sm;
  const long long max_useful = (warps_needed + (kWarpKernelThreads / 32) - 1) / (kWarpKernelThreads / 32);
  if (blocks > max_useful) blocks = max_useful;
  if (blocks < 1) blocks = 1;
  k_sample_warp<NCH><<<(unsigned)blocks, kWarpKernelThreads, smem, st>>>(a);
  return cudaGetLastError();
}

int warp_kernel_max_vocab() { return 8 * 256 - 7; }

cudaError_t launch_sample_warp(const SampleArgs& a, cudaStream_t st, int num_sms) {
  const int nq_max = (a.V + 7 + 7) >> 3;
  const int nch = (nq_max + 31) / 32;
  switch (nch) {
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
