// k_reveal.cu -- confidence ranking and reveal after the sampling pass.
//
// "Sampler support for discrete diffusion" (mstar issue #267), Hert4's first
// comment: each step scores the whole masked canvas, ranks the cells by
// confidence over the flattened [C, T] block of a request and commits only the
// top reveal_count. One CTA per request finds the reveal_count-th cell of the
// order (score desc, flattened index asc) and scatters the tokens of the cells
// up to it into the canvas. A request of at most kRevealStaged cells is staged
// once in shared memory as 32-bit score keys. The top byte of the k-th key H
// comes from a 256-bin histogram built while staging, the next byte from a
// second histogram over the keys that share the first; 2-bit rounds (counting
// by warp reductions, one barrier each) go on only while more than 64 keys
// share the prefix, and one warp then ranks those keys against each other to
// settle H. When cells tied at H straddle the cut, a binary search over the
// flattened index finds the last one revealed. A larger request runs an exact
// 64-bit radix select (score key above the inverted flattened index, so keys
// are distinct) over global memory.
#include <climits>

#include "ds_device.cuh"
#include "ds_launch.h"

namespace ds {

namespace {

// A request holds about 800-3200 cells: 1024 threads stage them in one to four
// loads each (512 and 256 threads measured slower when the select ran 16 rounds).
constexpr int kRevealNT = 1024;
// Warps that run the 2-bit rounds: 16 behind a named barrier of their own (with
// all 16 rounds, 16 warps beat 8, 4 and 2 warps and all 32 behind block barriers).
constexpr int kSelWarps = 16;
constexpr int kRevealStaged = 16384;  // cells staged in shared memory (64 KB of keys, 64 KB of tokens)
// Once the keys that match the selected prefix number at most this many, one
// warp finishes the select by ranking them against each other.
constexpr int kCandMax = 64;

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

// Block-wide sums of three per-thread counts (one barrier: each warp writes
// its sums to its slot of this round's buffer, every thread adds them up).
__device__ __forceinline__ int3 block_sum3(int a, int b, int c, int (*slots)[kRevealNT / 32][4], int parity) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  a = __reduce_add_sync(0xffffffffu, a);
  b = __reduce_add_sync(0xffffffffu, b);
  c = __reduce_add_sync(0xffffffffu, c);
  if (lane == 0) {
    slots[parity][wid][0] = a;
    slots[parity][wid][1] = b;
    slots[parity][wid][2] = c;
  }
  __syncthreads();
  // lane w reads warp w's sums; three warp reductions give every lane the totals
  const int4 v = (lane < kRevealNT / 32) ? *reinterpret_cast<const int4*>(slots[parity][lane]) : make_int4(0, 0, 0, 0);
  return make_int3(__reduce_add_sync(0xffffffffu, v.x), __reduce_add_sync(0xffffffffu, v.y),
                   __reduce_add_sync(0xffffffffu, v.z));
}

__global__ void __launch_bounds__(kRevealNT) k_reveal(const float* __restrict__ scores,
                                                      const int32_t* __restrict__ tokens,
                                                      const int32_t* __restrict__ seq_lens,
                                                      const int32_t* __restrict__ reveal_counts, int B, int C, int P,
                                                      int32_t* __restrict__ canvas, uint8_t* __restrict__ revealed,
                                                      uint32_t* __restrict__ d_status) {
  __shared__ int hist[256];
  __shared__ __align__(16) int slots[2][kRevealNT / 32][4];
  __shared__ unsigned long long s_prefix;
  __shared__ int s_need, s_eq, s_cnt, s_bad;
  __shared__ int hist2[256];
  __shared__ long long s_off, s_tot;
  __shared__ uint32_t cand[kCandMax];
  extern __shared__ uint32_t skeys[];  // the staged request's score keys, in flattened order,
                                       // then its tokens (kRevealStaged entries each)
  int32_t* stok = reinterpret_cast<int32_t*>(skeys + kRevealStaged);
  pdl_release();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int parity = 0;

  for (int r = blockIdx.x; r < B; r += gridDim.x) {
    // the request's offset and the batch total (sums of non-negative int32, in
    // 64 bits), by warp 0; the previous request ended at a block barrier, so the
    // shared state is free
    const int T = seq_lens[r];
    long long k = reveal_counts[r];
    if (wid == 0) {
      long long off = 0, tot = 0;
      int bad = 0;
      for (int j = lane; j < B; j += 32) {
        const int Tj = seq_lens[j];
        bad |= Tj < 0;
        const long long Tc = Tj < 0 ? 0 : Tj;
        tot += Tc;
        if (j < r) off += Tc;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        off += __shfl_xor_sync(0xffffffffu, off, o);
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
      }
      bad = __any_sync(0xffffffffu, bad);
      if (lane == 0) {
        s_off = off;
        s_tot = tot;
        s_bad = bad;
        s_cnt = 0;
      }
    }
    if (tid < 256) {
      hist[tid] = 0;
      hist2[tid] = 0;
    }
    __syncthreads();
    const long long off = s_off, tot = s_tot;
    if (s_bad || tot != (long long)P) {
      if (tid == 0 && r == (int)blockIdx.x) report(d_status, DS_DEV_ERR_LAYOUT);
      return;  // uniform across the CTA; the layout is invalid for every request
    }
    const long long roff = off;
    const long long n = (long long)C * T;
    k = k < 0 ? 0 : (k > n ? n : k);
    auto cell_of = [&](long long f) -> long long {
      const long long c = f / T;
      return c * (long long)P + roff + (f - c * T);
    };

    if (k > 0 && k < n && n <= kRevealStaged) {
      // n < 2^15 here: 32-bit index arithmetic
      const int nn = (int)n, kk = (int)k;
      const unsigned Tu = (unsigned)T;
      auto cell32 = [&](int f) -> long long {
        const unsigned c = (unsigned)f / Tu;
        return (long long)c * P + roff + (long long)((unsigned)f - c * Tu);
      };
      for (int f = tid; f < nn; f += kRevealNT) {
        const long long cell = cell32(f);
        const uint32_t key = score_key(scores[cell]);
        stok[f] = tokens[cell];  // loaded now, with the score, so the scatter waits on no load
        skeys[f] = key;
        atomicAdd(&hist[key >> 24], 1);
      }
      __syncthreads();
      // the top two bytes of H from two 256-bin histograms: the first built while
      // staging, the second over the keys that match the first byte (skipped when
      // at most kCandMax keys share it)
      if (wid == 0) {
        int digit, above;
        pick_digit(hist, kk, lane, digit, above);
        if (digit >= 0) {
          s_prefix = (unsigned long long)digit << 24;
          s_need = kk - above;
          s_eq = hist[digit];
        }
      }
      __syncthreads();
      int shift = 24;
      if (s_eq > kCandMax) {
        const uint32_t top = (uint32_t)s_prefix >> 24;
        for (int f = tid; f < nn; f += kRevealNT) {
          const uint32_t key = skeys[f];
          if ((key >> 24) == top) atomicAdd(&hist2[(key >> 16) & 255u], 1);
        }
        __syncthreads();
        if (wid == 0) {
          int digit, above;
          const int need0 = s_need;
          pick_digit(hist2, need0, lane, digit, above);
          if (digit >= 0) {
            s_prefix |= (unsigned long long)digit << 16;
            s_need = need0 - above;
            s_eq = hist2[digit];
          }
        }
        __syncthreads();
        shift = 16;
      }
      // 2-bit radix select of the kk-th largest key H, MSB first, by the first
      // kSelWarps warps alone (a named barrier of their threads is much cheaper
      // than a block barrier): each round every selecting warp counts, among its
      // keys that match H above the current digit, those whose digit is >= 1, 2
      // and 3, publishes the sums in this round's slots, and after the barrier
      // adds all the warps' sums and picks the same digit (no atomics; the slots
      // alternate between rounds, so one barrier a round suffices). As soon as
      // at most kCandMax keys match the prefix chosen so far, those keys are
      // gathered and warp 0 ranks them against each other, which settles the
      // remaining digits at once.
      if (wid < kSelWarps) {
        uint32_t H = (uint32_t)s_prefix;
        int need = s_need, eq = s_eq, par = 0;
#pragma unroll 1
        while (eq > kCandMax && shift > 0) {
          shift -= 2;
          int c1 = 0, c2 = 0, c3 = 0;
          const uint32_t hi_mask = 0xffffffffu << (shift + 2);
          for (int f = tid; f < nn; f += kSelWarps * 32) {
            const uint32_t key = skeys[f];
            if ((key & hi_mask) == (H & hi_mask)) {
              const uint32_t d = (key >> shift) & 3u;
              c1 += d >= 1u;
              c2 += d >= 2u;
              c3 += d >= 3u;
            }
          }
          c1 = __reduce_add_sync(0xffffffffu, c1);
          c2 = __reduce_add_sync(0xffffffffu, c2);
          c3 = __reduce_add_sync(0xffffffffu, c3);
          if (lane == 0) {
            slots[par][wid][0] = c1;
            slots[par][wid][1] = c2;
            slots[par][wid][2] = c3;
          }
          asm volatile("bar.sync 1, %0;" ::"n"(kSelWarps * 32) : "memory");
          const int4 v = (lane < kSelWarps) ? *reinterpret_cast<const int4*>(slots[par][lane]) : make_int4(0, 0, 0, 0);
          const int C1 = __reduce_add_sync(0xffffffffu, v.x), C2 = __reduce_add_sync(0xffffffffu, v.y),
                    C3 = __reduce_add_sync(0xffffffffu, v.z);
          par ^= 1;
          uint32_t d;
          if (C3 >= need) {
            d = 3u;
            eq = C3;
          } else if (C2 >= need) {
            d = 2u;
            need -= C3;
            eq = C2 - C3;
          } else if (C1 >= need) {
            d = 1u;
            need -= C2;
            eq = C1 - C2;
          } else {
            d = 0u;
            need -= C1;
            eq = eq - C1;
          }
          H |= d << shift;
        }
        if (shift > 0) {
          // gather the eq keys that match H above `shift`
          const uint32_t mask = 0xffffffffu << shift;
          for (int fb = wid * 32; fb < nn; fb += kSelWarps * 32) {
            const int f = fb + lane;
            const uint32_t key = f < nn ? skeys[f] : 0u;
            const bool m = f < nn && (key & mask) == (H & mask);
            const unsigned b = __ballot_sync(0xffffffffu, m);
            if (b) {
              int base = 0;
              if (lane == 0) base = atomicAdd(&s_cnt, __popc(b));
              base = __shfl_sync(0xffffffffu, base, 0);
              const int pos = base + __popc(b & ((1u << lane) - 1u));
              if (m && pos < kCandMax) cand[pos] = key;  // pos < eq <= kCandMax
            }
          }
          asm volatile("bar.sync 1, %0;" ::"n"(kSelWarps * 32) : "memory");
          if (wid == 0) {
            // the need-th largest candidate is the one with fewer than need
            // candidates above it and at least need at or above it
            const bool on0 = lane < eq, on1 = lane + 32 < eq;
            const uint32_t k0 = on0 ? cand[lane] : 0u, k1 = on1 ? cand[lane + 32] : 0u;
            int gt0 = 0, ge0 = 0, gt1 = 0, ge1 = 0;
#pragma unroll 4
            for (int j = 0; j < eq; ++j) {
              const uint32_t v = cand[j];
              gt0 += v > k0;
              ge0 += v >= k0;
              gt1 += v > k1;
              ge1 += v >= k1;
            }
            const unsigned b0 = __ballot_sync(0xffffffffu, on0 && gt0 < need && need <= ge0);
            const unsigned b1 = __ballot_sync(0xffffffffu, on1 && gt1 < need && need <= ge1);
            const bool use1 = b0 == 0u;  // every such candidate has the same key
            const int src = __ffs(use1 ? b1 : b0) - 1;
            H = __shfl_sync(0xffffffffu, use1 ? k1 : k0, src);
            const int hgt = __shfl_sync(0xffffffffu, use1 ? gt1 : gt0, src);
            const int hge = __shfl_sync(0xffffffffu, use1 ? ge1 : ge0, src);
            need -= hgt;
            eq = hge - hgt;
          }
        }
        if (tid == 0) {
          s_prefix = (unsigned long long)H;
          s_need = need;
          s_eq = eq;
        }
      }
      __syncthreads();
      const uint32_t H = (uint32_t)s_prefix;
      const int need = s_need;
      const int eq_cnt = s_eq;
      // every key above H is revealed; of the eq_cnt keys equal to H, the first
      // `need` in flattened order: the need-th one's index by a binary search
      // (only when ties straddle the cut)
      int f_cut = nn;  // keys equal to H with f < f_cut are revealed
      if (eq_cnt > need) {
        int lo = 0, hi = nn - 1;
#pragma unroll 1
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          int c = 0;
          for (int f = tid; f <= mid; f += kRevealNT) c += skeys[f] == H;
          const int3 cs = block_sum3(c, 0, 0, slots, parity);
          parity ^= 1;
          if (cs.x >= need)
            hi = mid;
          else
            lo = mid + 1;
        }
        f_cut = lo + 1;
      }
      for (int f = tid; f < nn; f += kRevealNT) {
        const uint32_t key = skeys[f];
        const bool on = key > H || (key == H && f < f_cut);
        const long long cell = cell32(f);
        if (on) canvas[cell] = stok[f];
        if (revealed) revealed[cell] = on ? 1 : 0;
      }
      __syncthreads();  // skeys is restaged by the next request
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
  const int sms = device_sms();
  if (sms <= 0) return cudaErrorUnknown;
  const int ok = cached(reinterpret_cast<const void*>(k_reveal), 0, [](int) {
    const cudaError_t r = cudaFuncSetAttribute(k_reveal, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(2 * kRevealStaged * sizeof(uint32_t)));
    return r == cudaSuccess ? 1 : -(int)r;
  });
  if (ok <= 0) return ok < 0 ? (cudaError_t)(-ok) : cudaErrorUnknown;
  cudaError_t e;
  long long blocks = B;
  if (blocks > (long long)sms * 4) blocks = (long long)sms * 4;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(kRevealNT, 1, 1);
  cfg.dynamicSmemBytes = 2 * kRevealStaged * sizeof(uint32_t);
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
