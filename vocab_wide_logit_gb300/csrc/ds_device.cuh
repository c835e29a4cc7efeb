// ds_device.cuh -- device primitives shared by the libdsample kernels.
//
// bf16 unpacking, the order-preserving float key, Philox4x32-10, the Gumbel
// transform (table bounds and an accurate form), warp reductions and the
// streaming 16-byte loads. Written for sm_103a; nothing here is a dense
// contraction, so no tensor-core path appears.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ds {

constexpr float kInf = __builtin_huge_valf();
constexpr float kLog2e = 1.4426950408889634f;  // 1 / ln 2

// Launch-wide arguments of the sampling pass.
struct SampleArgs {
  const int32_t* request_ids;
  const uint16_t* c;
  const uint16_t* u;
  const int32_t* seq_lens;
  const float* guidance;
  const float* temperature;
  int32_t* out_tokens;
  float* out_logprobs;
  uint32_t* d_status;
  int32_t B, C, P, V;
  int32_t k;          // kept count
  float q_lo;         // N(0,1) quantile for the first lower threshold guess (-inf: keep all)
  float q_hi;         // N(0,1) quantile for the upper threshold (+inf: none)
  float q_w;          // N(0,1) quantile of the one-warp-per-cell kernel's first guess
  uint32_t key0, key1;
  uint32_t iter_hi;   // iteration << 8
  uint32_t rk0[10], rk1[10];  // Philox round keys (key + r * Weyl constants), computed on the host
  const float* ratios;        // per-request top ratio [B] (device) or null: k, q_lo, q_hi above
  const uint32_t* iters;      // per-request iteration [B] (device) or null: iter_hi above
  uint32_t keep_ties;         // 1: the kept set is every z reaching the k-th largest z
};

// Key used for kept-set membership: the full (z desc, id asc) composite key, or
// with keep_ties only its z part (every id tied with the k-th z is kept).
__device__ __forceinline__ unsigned long long member_key(unsigned long long key, uint32_t keep_ties) {
  return keep_ties ? (key | 0xffffffffull) : key;
}

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// bf16 pair in one 32-bit word: element 0 in the low half.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
  f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
  f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
  f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

// z = c + g (c - u): fp32 difference, then one fused multiply-add.
__device__ __forceinline__ float cfg_combine(float c, float u, float g) {
  return __fmaf_rn(g, __fsub_rn(c, u), c);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Monotone map of fp32 onto uint32 (larger float -> larger key), for finite and
// infinite values.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ---------------------------------------------------------------- Philox4x32-10
// Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): each
// round multiplies counter words 0 and 2 by two constants (32 x 32 -> 64 bits);
// the high halves are xored with the other words and the round key, the low
// halves move over. The round keys (the key bumped by two Weyl constants per
// round) come precomputed in rk0 / rk1.
__device__ __forceinline__ uint4 philox4x32_10(uint4 x, const uint32_t (&rk0)[10], const uint32_t (&rk1)[10]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const unsigned long long p0 = (unsigned long long)x.x * 0xD2511F53ull;
    const unsigned long long p1 = (unsigned long long)x.z * 0xCD9E8D57ull;
    x = make_uint4((uint32_t)(p1 >> 32) ^ x.y ^ rk0[r], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ x.w ^ rk1[r],
                   (uint32_t)p0);
  }
  return x;
}

// Word (id & 3) of the Philox block keyed for vocabulary id `id` of a cell.
__device__ __forceinline__ uint32_t noise_word(uint32_t id, uint32_t t, uint32_t rid, uint32_t ctr3,
                                               const uint32_t (&rk0)[10], const uint32_t (&rk1)[10]) {
  const uint4 o = philox4x32_10(make_uint4(id >> 2, t, rid, ctr3), rk0, rk1);
  const uint32_t s = id & 3u;
  const uint32_t a = (s & 1u) ? o.y : o.x;
  const uint32_t b = (s & 1u) ? o.w : o.z;
  return (s & 2u) ? b : a;
}

// Accurate G = -log(-log U), U = ((x >> 8) + 1/2) 2^-24, in fp32. U and 1 - U are
// formed exactly (each fits in 24 bits on its branch), so the inner logarithm
// keeps full relative accuracy as U approaches 1.
__device__ __forceinline__ float gumbel_accurate(uint32_t x) {
  const uint32_t j = x >> 8;
  float e;  // E = -log U > 0
  if (j < (1u << 23)) {
    const float u = (float)(2u * j + 1u) * 0x1p-25f;
    e = -logf(u);
  } else {
    const float w = (float)(2u * ((1u << 24) - j) - 1u) * 0x1p-25f;  // 1 - U
    e = -log1pf(-w);
  }
  return -logf(e);
}

// ---------------------------------------------------------------- warp reductions
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Max of a float across the warp in one reduce instruction over an
// order-preserving integer image; NaN is mapped below -inf, so it never wins
// (as with fmaxf).
__device__ __forceinline__ float warp_max_r(float v) {
  const int i = __float_as_int(v);
  const int key = (v != v) ? (int)0x807fffff : (i >= 0 ? i : (i ^ 0x7fffffff));
  const int mx = __reduce_max_sync(0xffffffffu, key);
  return __int_as_float(mx >= 0 ? mx : (mx ^ 0x7fffffff));
}

// Integer reductions use the warp-wide reduce instruction (one step instead of five shuffles).
__device__ __forceinline__ int warp_sum_i(int v) { return __reduce_add_sync(0xffffffffu, v); }
__device__ __forceinline__ int warp_min_i(int v) { return __reduce_min_sync(0xffffffffu, v); }
// Exclusive prefix sum over the warp.
__device__ __forceinline__ int warp_excl_scan(int v, int lane) {
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  return incl - v;
}

// (score desc, id asc) argmax across the warp; returns the winner's lane.
__device__ __forceinline__ int warp_argmax_lane(float s, int id) {
  float bs = s;
  int bi = id;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, bs, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (os > bs || (os == bs && oi < bi)) {
      bs = os;
      bi = oi;
    }
  }
  // lane holding (bs, bi)
  const unsigned m = __ballot_sync(0xffffffffu, s == bs && id == bi);
  return __ffs(m) - 1;
}

// Programmatic dependent launch. Every kernel of the library is launched so
// that it may be scheduled while the previous kernel on the stream drains;
// pdl_wait() blocks until that kernel has completed and its writes are
// visible, and comes before a kernel's first read of any input. pdl_release()
// lets the next kernel on the stream begin launching at once (it waits in its
// own pdl_wait() for this one to finish).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ void report(uint32_t* d_status, uint32_t bits) {
  if (d_status) atomicOr(d_status, bits);
}

}  // namespace ds
