// k_merge.cu -- the vocabulary-sharded side of the greedy path.
//
// "perf: avoid full-vocab all-gather for draft greedy sampling" (LightLLM PR
// #1517), Design and invariants: each tensor-parallel rank reduces its vocab
// shard to a triple of three FP32 words -- local max, local log-sum-exp, and
// the argmax's global token id with its bits kept in the third word -- the
// ranks exchange only those triples, and every rank merges them: the global
// max, the shard holding it giving the token (smallest global id on ties),
// and lse = m + log sum_s exp(lse_s - m). The same section keeps the dense
// fallback, which writes the full log-softmax; k_log_softmax_write is that
// fallback for callers that still need dense log-probabilities.
#include <climits>
#include <cuda_bf16.h>

#include "ds_device.cuh"
#include "ds_launch.h"

namespace ds {

// One thread per token: merge its `shards` triples.
__global__ void __launch_bounds__(256) k_merge_triples(const float* __restrict__ triples, int n, int shards,
                                                       float* __restrict__ out_max, float* __restrict__ out_lse,
                                                       int* __restrict__ out_argmax) {
  pdl_release();
  pdl_wait();
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < n; t += gridDim.x * blockDim.x) {
    const float* tr = triples + (long long)t * shards * 3;
    float m = -kInf;
    int a = INT_MAX;
    for (int s = 0; s < shards; ++s) {
      const float ms = tr[3 * s];
      const int as = __float_as_int(tr[3 * s + 2]);
      if (a == INT_MAX || ms > m || (ms == m && as < a)) {
        m = ms;
        a = as;
      }
    }
    float lse = -kInf;
    if (m != -kInf) {
      float acc = 0.f;
      for (int s = 0; s < shards; ++s) acc += expf(tr[3 * s + 1] - m);
      lse = m + logf(acc);
    }
    out_max[t] = m;
    out_lse[t] = lse;
    out_argmax[t] = (a == INT_MAX) ? 0 : a;
  }
}

// Dense log-softmax write-out: out[row][i] = x[row][i] - lse[row], fp32 or bf16
// (round to nearest even). One grid-stride pass over 16-byte chunks of the
// row-major [n][V] matrix; rows need not be 16-byte aligned, so chunk edges are
// handled element by element.
template <bool BF16_OUT>
__global__ void __launch_bounds__(256) k_log_softmax_write(const uint16_t* __restrict__ x, int n, int V,
                                                           const float* __restrict__ lse, void* __restrict__ out) {
  pdl_release();
  pdl_wait();
  const long long total = (long long)n * V;
  const long long n8 = total >> 3;
  const bool aligned = (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                       (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < (aligned ? n8 : 0); c += stride) {
    const uint4 v = ld_stream16(reinterpret_cast<const uint4*>(x) + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
    const long long e0 = c * 8;
    int row = (int)(e0 / V);
    int col = (int)(e0 - (long long)row * V);
    float l = lse[row];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = bf_lo(w[i]);
      f[2 * i + 1] = bf_hi(w[i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (col == V) {  // the chunk runs into the next row
        ++row;
        col = 0;
        l = lse[row];
      }
      f[i] -= l;
      ++col;
    }
    if (BF16_OUT) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
      reinterpret_cast<uint4*>(out)[c] = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      float4* o = reinterpret_cast<float4*>(out) + 2 * c;
      o[0] = make_float4(f[0], f[1], f[2], f[3]);
      o[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
  // element-wise: the tail after the last whole chunk, or everything when unaligned
  for (long long e = (aligned ? n8 * 8 : 0) + blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += stride) {
    const int row = (int)(e / V);
    const float v = __uint_as_float((uint32_t)x[e] << 16) - lse[row];
    if (BF16_OUT)
      reinterpret_cast<__nv_bfloat16*>(out)[e] = __float2bfloat16_rn(v);
    else
      reinterpret_cast<float*>(out)[e] = v;
  }
}

static cudaError_t launch_plain(const void* kern, void** args, long long work, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  long long blocks = (work + 255) / 256;
  const long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelExC(&cfg, kern, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_merge_triples(const float* triples, int n, int shards, float* out_max, float* out_lse,
                                 int* out_argmax, cudaStream_t st) {
  void* args[] = {&triples, &n, &shards, &out_max, &out_lse, &out_argmax};
  return launch_plain(reinterpret_cast<const void*>(&k_merge_triples), args, n, st);
}

cudaError_t launch_log_softmax_write(const uint16_t* x, int n, int V, const float* lse, void* out, bool bf16_out,
                                     cudaStream_t st) {
  void* args[] = {&x, &n, &V, &lse, &out};
  const long long work = ((long long)n * V + 7) / 8;
  return bf16_out ? launch_plain(reinterpret_cast<const void*>(&k_log_softmax_write<true>), args, work, st)
                  : launch_plain(reinterpret_cast<const void*>(&k_log_softmax_write<false>), args, work, st);
}

}  // namespace ds
