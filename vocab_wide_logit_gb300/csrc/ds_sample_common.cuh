// ds_sample_common.cuh -- pieces of the sampling pass shared by the warp and cluster kernels.
#pragma once

#include "ds_device.cuh"
#include "gumbel_bounds.inc"

namespace ds {

// Position -> request mapping of the packed layout ("Add a sampler resource for
// discrete diffusion", Contract: [rows, positions, vocab] packed across
// requests; guidance 0 builds no unconditional document, so u packs only the
// guided requests).
struct ReqCursor {
  int32_t r;       // request index
  int32_t off;     // first position of request r
  int32_t T;       // seq_lens[r]
  int32_t off_u;   // first row of request r inside u's packed positions
  float g, tau;
  uint32_t rid;
  int32_t k;         // kept count of the request
  float q_lo, q_hi;  // N(0,1) quantiles seeding the request's threshold guesses
  float q_w;         // and the one-warp-per-cell kernel's first guess
  uint32_t iter_hi;  // the request's iteration << 8 (noise counter word 3)
  uint32_t perr;     // DS_DEV_ERR_PARAM when the request's ratio or iteration is invalid
};

// Upper-tail N(0,1) quantile of p (P(N > x) = p), for the threshold guesses
// only: -inf for p >= 1, +inf for p <= 0. Out of line: it runs once per
// request and cell walk, and its temporaries stay out of the kernels' loops.
static __device__ __noinline__ float upper_quantile(float p) {
  if (p >= 1.f) return -__builtin_huge_valf();
  if (p <= 0.f) return __builtin_huge_valf();
  return 1.41421356f * erfcinvf(2.f * p);
}

// The request's kept count, threshold quantiles and noise iteration: its own
// entries when the call passed per-request arrays, else the call's scalars.
// k = ceilf(ratio * V) in fp32, clamped to [1, V], as for the scalar; the
// quantiles aim the candidate count a little above and below k, as the host
// does for the scalar.
__device__ __forceinline__ void req_params(const SampleArgs& a, int r, ReqCursor& cur) {
  cur.perr = 0u;
  if (a.ratios) {
    const float ratio = a.ratios[r];
    if (!(ratio > 0.f && ratio <= 1.f)) {
      cur.perr = DS_DEV_ERR_PARAM;
      cur.k = 1;
      cur.q_lo = -__builtin_huge_valf();
      cur.q_hi = __builtin_huge_valf();
      cur.q_w = -__builtin_huge_valf();
    } else {
      int kk = (int)ceilf(ratio * (float)a.V);
      kk = kk < 1 ? 1 : (kk > a.V ? a.V : kk);
      cur.k = kk;
      const float kf = (float)kk, Vf = (float)a.V;
      const float spread = 1.5f * sqrtf(kf * (1.f - kf / Vf)) + 0.02f * kf + 4.f;
      cur.q_lo = (kf + spread >= Vf) ? -__builtin_huge_valf() : upper_quantile((kf + spread) / Vf);
      cur.q_hi = (kf - spread < 1.f) ? __builtin_huge_valf() : upper_quantile((kf - spread) / Vf);
      const float tw = kf + sqrtf(kf * (1.f - kf / Vf)) + 0.02f * kf + 2.f;
      cur.q_w = (tw >= Vf) ? -__builtin_huge_valf() : upper_quantile(tw / Vf);
    }
  } else {
    cur.k = a.k;
    cur.q_lo = a.q_lo;
    cur.q_hi = a.q_hi;
    cur.q_w = a.q_w;
  }
  if (a.iters) {
    const uint32_t it = a.iters[r];
    if (it > DS_MAX_ITERATION) cur.perr = DS_DEV_ERR_PARAM;
    cur.iter_hi = (it & 0xFFFFFFu) << 8;
  } else {
    cur.iter_hi = a.iter_hi;
  }
}

// Whole-batch totals, computed by each warp (O(B / 32)).
struct BatchTotals {
  long long tot;    // sum of seq_lens
  long long tot_u;  // sum over guided requests
  bool bad;         // a negative seq_len
};

__device__ __forceinline__ BatchTotals warp_batch_totals(const SampleArgs& a, int lane) {
  BatchTotals bt{0, 0, false};
  for (int base = 0; base < a.B; base += 32) {
    const int r = base + lane;
    int T = 0;
    float g = 0.f;
    if (r < a.B) {
      T = a.seq_lens[r];
      g = a.guidance[r];
    }
    const bool neg = T < 0;
    bt.bad |= __any_sync(0xffffffffu, neg);
    const int Tc = neg ? 0 : T;
    bt.tot += warp_sum_i(Tc);
    bt.tot_u += warp_sum_i(g != 0.f ? Tc : 0);
  }
  return bt;
}

// Find the request that owns position p by a warp-parallel scan from request 0.
// Returns false when no request owns p.
__device__ __forceinline__ bool warp_find_request(const SampleArgs& a, int p, int lane, ReqCursor& cur) {
  int off = 0, off_u = 0;
  for (int base = 0; base < a.B; base += 32) {
    const int r = base + lane;
    int T = 0;
    float g = 0.f;
    if (r < a.B) {
      T = max(a.seq_lens[r], 0);
      g = a.guidance[r];
    }
    const int Tu = (g != 0.f) ? T : 0;
    const int ex = warp_excl_scan(T, lane);
    const int exu = warp_excl_scan(Tu, lane);
    const bool own = (r < a.B) && (p >= off + ex) && (p < off + ex + T);
    const unsigned m = __ballot_sync(0xffffffffu, own);
    if (m) {
      const int src = __ffs(m) - 1;
      cur.r = base + src;
      cur.off = off + __shfl_sync(0xffffffffu, ex, src);
      cur.T = __shfl_sync(0xffffffffu, T, src);
      cur.off_u = off_u + __shfl_sync(0xffffffffu, exu, src);
      cur.g = a.guidance[cur.r];
      cur.tau = a.temperature[cur.r];
      cur.rid = (uint32_t)a.request_ids[cur.r];
      req_params(a, cur.r, cur);
      return true;
    }
    off += warp_sum_i(T);
    off_u += warp_sum_i(Tu);
  }
  return false;
}

// Gumbel bounds of one Philox word.
__device__ __forceinline__ float2 gumbel_bounds(uint32_t x) {
  return __ldg(&kGumbelBounds[x >> DS_GUMBEL_BUCKET_SHIFT]);
}

// 64-bit composite key of (z, id): larger key = earlier in the order (z desc, id asc).
// -0 is folded onto +0: the two are equal values, so they tie and the smaller id goes first.
__device__ __forceinline__ unsigned long long rank_key(float z, int id) {
  return ((unsigned long long)order_key(z == 0.f ? 0.f : z) << 32) | (unsigned long long)(0xffffffffu - (uint32_t)id);
}

}  // namespace ds
