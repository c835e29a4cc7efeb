// k_reveal.cu -- confidence ranking and reveal after the sampling pass.
//
// "Sampler support for discrete diffusion" (mstar issue #267), Hert4's first
// comment: each step scores the whole masked canvas, ranks the cells by
// confidence over the flattened [C, T] block of a request and commits only the
// top reveal_count. One CTA per request finds the reveal_count-th cell of the
// order (score desc, flattened index asc) and scatters the tokens of the cells
// up to it into the canvas. A request of at most kRevealStaged cells is staged
// once in shared memory as 32-bit score keys: four 8-bit radix rounds find the
// k-th key H, and the cells tied at H are taken in index order by a prefix
// count. A larger request runs an exact 64-bit radix select (score key above
// the inverted flattened index, so keys are distinct) over global memory.
#include <climits>

#include "ds_device.cuh"
#include "ds_launch.h"

namespace ds {

namespace {

constexpr int kRevealNT = 1024;  // short passes: a request holds about 2000 cells
constexpr int kRevealStaged = 16384;  // cells staged in shared memory (64 KB of keys)

// Larger key = earlier in the reveal order: the score's order-preserving bits
// (-0 folded onto +0, so equal scores tie) above the inverted flattened index.
__device__ __forceinline__ uint32_t score_key(float s) { return order_key((s == 0.f) ? 0.f : s); }
__device__ __forceinline__ unsigned long long reveal_key(float s, uint32_t f) {
  return ((unsigned long long)score_key(s) << 32) | (unsigned long long)(0xffffffffu - f);
}

// Warp 0 finds the digit of the need-th largest key from a 256-bin histogram:
// bins in descending digit order, lane l holding digits 255-8l .. 248-8l.
// Returns (digit, keys above it) in lane src; the caller broadcasts.
__device__ __forceinline__ void pick_digit(const int* hist, int need, int lane, int& digit, int& above) {
  int cl[8], sum = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    cl[e] = hist[255 - 8 * lane - e];
    sum += cl[e];
  }
  const int above_lane = warp_excl_scan(sum, lane);
  const bool here = above_lane < need && need <= above_lane + sum;
  const int src = __ffs(__ballot_sync(0xffffffffu, here)) - 1;
  digit = -1;
  above = 0;
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
  __shared__ int s_wcnt[kRevealNT / 32];
  extern __shared__ uint32_t skeys[];  // the staged request's score keys, in flattened order
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

    if (k > 0 && k < n && n <= kRevealStaged) {
      const int nn = (int)n, kk = (int)k;
      for (int f = tid; f < nn; f += kRevealNT) skeys[f] = score_key(scores[cell_of(f)]);
      if (tid == 0) {
        s_prefix = 0ull;
        s_need = kk;
      }
      __syncthreads();
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += kRevealNT) hist[b] = 0;
        __syncthreads();
        const uint32_t prefix = (uint32_t)s_prefix;
        for (int f = tid; f < nn; f += kRevealNT) {
          const uint32_t key = skeys[f];
          if (shift == 24 || (key >> (shift + 8)) == (prefix >> (shift + 8))) atomicAdd(&hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (wid == 0) {
          int digit, above;
          pick_digit(hist, s_need, lane, digit, above);
          if (digit >= 0) {
            s_prefix = (unsigned long long)(prefix | ((uint32_t)digit << shift));
            s_need -= above;
          }
        }
        __syncthreads();
      }
      // every key above H is revealed; of the keys equal to H, the first `need`
      // in flattened order (a running count over chunks of kRevealNT cells)
      const uint32_t H = (uint32_t)s_prefix;
      const int need = s_need;
      int run = 0;
      for (int base = 0; base < nn; base += kRevealNT) {
        const int f = base + tid;
        const uint32_t key = (f < nn) ? skeys[f] : 0u;
        const bool tied = f < nn && key == H;
        const unsigned bt = __ballot_sync(0xffffffffu, tied);
        if (lane == 0) s_wcnt[wid] = __popc(bt);
        __syncthreads();
        int before = run, total = 0;
#pragma unroll
        for (int w = 0; w < kRevealNT / 32; ++w) {
          const int cw = s_wcnt[w];
          before += (w < wid) ? cw : 0;
          total += cw;
        }
        before += __popc(bt & ((1u << lane) - 1u));
        if (f < nn) {
          const bool on = key > H || (tied && before < need);
          const long long cell = cell_of(f);
          if (on) canvas[cell] = tokens[cell];
          if (revealed) revealed[cell] = on ? 1 : 0;
        }
        run += total;
        __syncthreads();  // s_wcnt is rewritten by the next chunk
      }
      continue;  // uniform across the CTA
    }

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
          int digit, above;
          pick_digit(hist, s_need, lane, digit, above);
          if (digit >= 0) {
            s_prefix = prefix | ((unsigned long long)digit << shift);
            s_need -= above;
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
  e = cudaFuncSetAttribute(k_reveal, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(kRevealStaged * sizeof(uint32_t)));
  if (e != cudaSuccess) return e;
  long long blocks = B;
  if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(kRevealNT, 1, 1);
  cfg.dynamicSmemBytes = kRevealStaged * sizeof(uint32_t);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_reveal, scores, tokens, seq_lens, reveal_counts, B, C, P, canvas, revealed,
                         d_status);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

}  // namespace ds
