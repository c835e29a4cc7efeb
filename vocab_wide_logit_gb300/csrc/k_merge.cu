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
// (round to nearest even). Blocks stride over rows (blockIdx.y) and, within a
// row, over its 16-byte chunks of x (blockIdx.x), so a row's lse is read once
// and no flat index is divided. A row whose x and out both reach a 16-byte
// boundary after the same h head elements goes by chunks, four in flight per
// thread, with its head and tail element by element; any other row goes
// element by element.
template <bool BF16_OUT>
__global__ void __launch_bounds__(256) k_log_softmax_write(const uint16_t* __restrict__ x, int n, int V,
                                                           const float* __restrict__ lse, void* __restrict__ out) {
  pdl_release();
  pdl_wait();
  constexpr int OB = BF16_OUT ? 2 : 4;  // output bytes per element
  const int tpr = gridDim.x * blockDim.x;  // threads per row
  const int tr = blockIdx.x * blockDim.x + threadIdx.x;
  for (int row = blockIdx.y; row < n; row += gridDim.y) {
    const float l = lse[row];
    const uint16_t* xr = x + (long long)row * V;
    unsigned char* orow = reinterpret_cast<unsigned char*>(out) + (long long)row * V * OB;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(xr), oa = reinterpret_cast<uintptr_t>(orow);
    const int h = min((int)(((16u - (unsigned)(xa & 15)) & 15u) >> 1), V);
    const bool vec = ((oa + (uintptr_t)h * OB) & 15) == 0;
    const int nfc = vec ? (V - h) >> 3 : 0;
    const uint4* xc = reinterpret_cast<const uint4*>(xr + h);
    unsigned char* oc = orow + (long long)h * OB;
    for (int q0 = tr; q0 < nfc; q0 += 4 * tpr) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = q0 + u * tpr;
        v[u] = (q < nfc) ? ld_stream16(xc + q) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = q0 + u * tpr;
        if (q < nfc) {
          const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          float f[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            f[2 * i] = bf_lo(w[i]) - l;
            f[2 * i + 1] = bf_hi(w[i]) - l;
          }
          if (BF16_OUT) {
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __nv_bfloat162 hh = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
              o[i] = *reinterpret_cast<const uint32_t*>(&hh);
            }
            reinterpret_cast<uint4*>(oc)[q] = make_uint4(o[0], o[1], o[2], o[3]);
          } else {
            float4* o = reinterpret_cast<float4*>(oc) + 2 * q;
            o[0] = make_float4(f[0], f[1], f[2], f[3]);
            o[1] = make_float4(f[4], f[5], f[6], f[7]);
          }
        }
      }
    }
    // element by element: the head and the tail of a chunked row, or the whole row
    const int tail0 = h + 8 * nfc;
    const int ne = vec ? h + (V - tail0) : V;
    for (int j = tr; j < ne; j += tpr) {
      const int e = (vec && j >= h) ? tail0 + (j - h) : j;
      const float v = __uint_as_float((uint32_t)xr[e] << 16) - l;
      if (BF16_OUT)
        reinterpret_cast<__nv_bfloat16*>(orow)[e] = __float2bfloat16_rn(v);
      else
        reinterpret_cast<float*>(orow)[e] = v;
    }
  }
}

static cudaError_t launch_plain(const void* kern, void** args, long long work, cudaStream_t st) {
  const int sms = device_sms();
  if (sms <= 0) return cudaErrorUnknown;
  cudaError_t e;
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
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_merge_triples(const float* triples, int n, int shards, float* out_max, float* out_lse,
                                 int* out_argmax, cudaStream_t st) {
  void* args[] = {&triples, &n, &shards, &out_max, &out_lse, &out_argmax};
  return launch_plain(reinterpret_cast<const void*>(&k_merge_triples), args, n, st);
}

cudaError_t launch_log_softmax_write(const uint16_t* x, int n, int V, const float* lse, void* out, bool bf16_out,
                                     cudaStream_t st) {
  if (n <= 0 || V <= 0) return cudaSuccess;
  const int sms = device_sms();
  if (sms <= 0) return cudaErrorUnknown;
  cudaError_t e;
  // rows on y; per row enough blocks on x that the grid holds about 8 blocks per
  // SM, but no more than the row's chunks need at 4 per thread
  const int by = n < 65535 ? n : 65535;
  const long long want = ((long long)sms * 8 + by - 1) / by;
  const long long need = ((long long)V / 8 + 4 * 256 - 1) / (4 * 256);
  long long bx = want < need ? want : need;
  if (bx < 1) bx = 1;
  void* args[] = {&x, &n, &V, &lse, &out};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)bx, (unsigned)by, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const void* kern = bf16_out ? reinterpret_cast<const void*>(&k_log_softmax_write<true>)
                              : reinterpret_cast<const void*>(&k_log_softmax_write<false>);
  e = cudaLaunchKernelExC(&cfg, kern, args);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

}  // namespace ds
