// k_reveal.cu -- confidence ranking and reveal after the sampling pass.
//
// "Sampler support for discrete diffusion" (mstar issue #267), Hert4's first
// comment: each step scores the whole masked canvas, ranks the cells by
// confidence over the flattened [C, T] block of a request and commits only the
// top reveal_count. One CTA per request: an exact radix select finds the
// reveal_count-th key of the order (score desc, flattened index asc) -- keys
// are distinct 64-bit words, so exactly that many cells qualify -- and one
// more pass scatters their tokens into the canvas.
#include <climits>

#include "ds_device.cuh"
#include "ds_launch.h"

namespace ds {

namespace {

constexpr int kRevealNT = 256;

// Larger key = earlier in the reveal order: the score's order-preserving bits
// (-0 folded onto +0, so equal scores tie) above the inverted flattened index.
__device__ __forceinline__ unsigned long long reveal_key(float s, uint32_t f) {
  const float sc = (s == 0.f) ? 0.f : s;
  return ((unsigned long long)order_key(sc) << 32) | (unsigned long long)(0xffffffffu - f);
}

}  // namespace

__global__ void __launch_bounds__(kRevealNT) k_reveal(const float* __restrict__ scores,
                                                      const int32_t* __restrict__ tokens,
                                                      const int32_t* __restrict__ seq_lens,
                                                      const int32_t* __restrict__ reveal_counts, int B, int C, int P,
                                                      int32_t* __restrict__ canvas, uint8_t* __restrict__ revealed,
                                                      uint32_t* __restrict__ d_status) {
  __shared__ int hist[256];
  __shared__ long long s_tot, s_off;
  __shared__ int s_bad;
  __shared__ unsigned long long s_prefix;
  __shared__ int s_need;
  pdl_release();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

  for (int r = blockIdx.x; r < B; r += gridDim.x) {
    // the request's offset and the batch total, by a block-wide sum
    long long off = 0, tot = 0;
    int bad = 0;
    for (int j = tid; j < B; j += kRevealNT) {
      const int T = seq_lens[j];
      bad |= T < 0;
      const long long Tc = T < 0 ? 0 : T;
      tot += Tc;
      if (j < r) off += Tc;
    }
    if (tid == 0) {
      s_tot = 0;
      s_off = 0;
      s_bad = 0;
    }
    __syncthreads();
    atomicAdd(reinterpret_cast<unsigned long long*>(&s_tot), (unsigned long long)tot);
    atomicAdd(reinterpret_cast<unsigned long long*>(&s_off), (unsigned long long)off);
    if (bad) atomicOr(&s_bad, 1);
    __syncthreads();
    if (s_bad || s_tot != (long long)P) {
      if (tid == 0 && r == (int)blockIdx.x) report(d_status, DS_DEV_ERR_LAYOUT);
      return;  // uniform across the CTA; the layout is invalid for every request
    }
    const long long roff = s_off;
    const int T = seq_lens[r];
    const long long n = (long long)C * T;
    long long k = reveal_counts[r];
    k = k < 0 ? 0 : (k > n ? n : k);
    auto cell_of = [&](long long f) -> long long {
      const long long c = f / T;
      return c * (long long)P + roff + (f - c * T);
    };

    unsigned long long kth = 0ull;  // with k > 0, every key >= kth is revealed
    if (k > 0 && k < n) {
      if (tid == 0) {
        s_prefix = 0ull;
        s_need = (int)k;
      }
      for (int shift = 56; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += kRevealNT) hist[b] = 0;
        __syncthreads();
        const unsigned long long prefix = s_prefix;
        for (long long f = tid; f < n; f += kRevealNT) {
          const unsigned long long key = reveal_key(scores[cell_of(f)], (uint32_t)f);
          if (shift == 56 || (key >> (shift + 8)) == (prefix >> (shift + 8)))
            atomicAdd(&hist[(int)((key >> shift) & 255ull)], 1);
        }
        __syncthreads();
        if (wid == 0) {
          // bins in descending digit order: lane l holds digits 255-8l .. 248-8l
          int cl[8], sum = 0;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            cl[e] = hist[255 - 8 * lane - e];
            sum += cl[e];
          }
          const int need = s_need;
          const int above_lane = warp_excl_scan(sum, lane);
          const bool here = above_lane < need && need <= above_lane + sum;
          const int src = __ffs(__ballot_sync(0xffffffffu, here)) - 1;
          if (lane == src) {
            int run = above_lane;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (run + cl[e] >= need) {
                s_prefix = prefix | ((unsigned long long)(255 - 8 * lane - e) << shift);
                s_need = need - run;
                break;
              }
              run += cl[e];
            }
          }
        }
        __syncthreads();
      }
      kth = s_prefix;
    }
    // scatter (k == n: every cell, kth = 0)
    for (long long f = tid; f < n; f += kRevealNT) {
      const long long cell = cell_of(f);
      const bool on = k > 0 && reveal_key(scores[cell], (uint32_t)f) >= kth;
      if (on) canvas[cell] = tokens[cell];
      if (revealed) revealed[cell] = on ? 1 : 0;
    }
    __syncthreads();  // shared state is reused by the next request
  }
}

cudaError_t launch_reveal(const float* scores, const int32_t* tokens, const int32_t* seq_lens,
                          const int32_t* reveal_counts, int B, int C, int P, int32_t* canvas, uint8_t* revealed,
                          uint32_t* d_status, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  long long blocks = B;
  if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(kRevealNT, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_reveal, scores, tokens, seq_lens, reveal_counts, B, C, P, canvas, revealed,
                         d_status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ds
