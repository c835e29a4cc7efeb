// k_log_softmax.cu -- dense log-softmax with each row held on chip.
//
// "perf: avoid full-vocab all-gather for draft greedy sampling" (LightLLM PR
// #1517), Design and invariants: the dense fallback writes the full
// log-probabilities, out[row][i] = x[row][i] - lse[row], next to the per-row
// (max, log-sum-exp, argmax) triple. lse is known only after the whole row has
// been read, so a streaming write would read the row twice. Here a cluster of
// cs CTAs splits a row small enough to sit in their shared memory (at most
// kLsSliceMax 16-byte chunks per CTA):
//   load    each thread starts cp.async copies of all its chunks of the row
//           into shared memory at once, waits for them, then keeps an online
//           (max, sum of exp(x - max), first chunk holding the max) over them,
//           rescaled once per batch of chunks
//   merge   warp -> CTA -> cluster over DSMEM, in one fixed tree that every
//           CTA evaluates, so every CTA holds the same (max, sum, chunk); ties
//           go to the smaller chunk, hence to the smallest id
//   write   each thread writes its own chunks back as x - lse (fp32, or bf16
//           rounded to nearest even) from shared memory; the CTA that holds
//           the winning chunk names the argmax
// so every logit is read from HBM once. Clusters are persistent over rows.
#include <climits>
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "ds_device.cuh"
#include "ds_launch.h"

namespace cg = cooperative_groups;

namespace ds {

namespace {

constexpr int kLsNT = 256;
constexpr int kLsUnroll = 4;
constexpr int kLsSliceMax = 4096;  // 16-byte chunks of a row per CTA: 64 KB of shared memory

struct LsTrip {
  float m;  // max
  float s;  // sum of exp(x - m)
  int a;    // first 16-byte chunk attaining m
};

__device__ __forceinline__ LsTrip ls_merge(const LsTrip& p, const LsTrip& q) {
  LsTrip r;
  r.m = fmaxf(p.m, q.m);
  if (r.m == -kInf) {
    r.s = 0.f;
    r.a = min(p.a, q.a);
    return r;
  }
  r.s = p.s * ex2_approx((p.m - r.m) * kLog2e) + q.s * ex2_approx((q.m - r.m) * kLog2e);
  r.a = (p.m > q.m) ? p.a : (q.m > p.m) ? q.a : min(p.a, q.a);
  return r;
}

__device__ __forceinline__ LsTrip ls_warp_merge(LsTrip t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    LsTrip u;
    u.m = __shfl_xor_sync(0xffffffffu, t.m, o);
    u.s = __shfl_xor_sync(0xffffffffu, t.s, o);
    u.a = __shfl_xor_sync(0xffffffffu, t.a, o);
    t = ls_merge(t, u);
  }
  return t;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}

// The 8 logits of chunk q as fp32; ids outside [0, V) read as -inf.
__device__ __forceinline__ void chunk_values(const uint4& v, int q, int dc, int V, bool edge, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf_lo(w[i]);
    f[2 * i + 1] = bf_hi(w[i]);
  }
  if (edge) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = 8 * q - dc + i;
      if (e < 0 || e >= V) f[i] = -kInf;
    }
  }
}

}  // namespace

template <bool BF16_OUT>
__global__ void __launch_bounds__(kLsNT) k_log_softmax_fused(const uint16_t* __restrict__ x, int n, int V,
                                                             float* __restrict__ out_max, float* __restrict__ out_lse,
                                                             int* __restrict__ out_argmax, void* __restrict__ out) {
  pdl_wait();
  extern __shared__ uint4 slice[];  // this CTA's chunks of the current row
  __shared__ LsTrip warp_part[kLsNT / 32];
  __shared__ LsTrip cta_part[2];  // per row parity; read by the cluster's CTAs
  __shared__ LsTrip row_res;
  constexpr int OB = BF16_OUT ? 2 : 4;  // output bytes per element
  cg::cluster_group cl = cg::this_cluster();
  const int cs = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const long long n_clusters = (long long)gridDim.x / cs;
  const long long cid = (long long)blockIdx.x / cs;
  const float2 l2e = make_float2(kLog2e, kLog2e);

  // this CTA's slice of a row: 16-byte chunks [q_lo, q_hi) of the row's chunk
  // grid (chunk 0 starts at the row's first element rounded down to 16 bytes)
  struct Slice {
    const uint4* base;
    int dc, nq, q_lo, q_hi;
  };
  auto slice_of = [&](long long row) {
    Slice g;
    const uintptr_t ad = reinterpret_cast<uintptr_t>(x + row * (long long)V);
    g.base = reinterpret_cast<const uint4*>(ad & ~(uintptr_t)15);
    g.dc = (int)((ad & 15) >> 1);
    g.nq = (g.dc + V + 7) >> 3;
    g.q_lo = (int)((long long)rank * g.nq / cs);
    g.q_hi = (int)((long long)(rank + 1) * g.nq / cs);
    return g;
  };
  // The first row's copies; each later row's copies start during the previous
  // row's write pass, slot by slot as the slots are written out.
  if (cid < n) {
    const Slice g = slice_of(cid);
    for (int q = g.q_lo + tid; q < g.q_hi; q += kLsNT) cp_async16(&slice[q - g.q_lo], g.base + q);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");

  int it = 0;
  for (long long row = cid; row < n; row += n_clusters, ++it) {
    const Slice g = slice_of(row);
    const int dc = g.dc, nq = g.nq, q_lo = g.q_lo, q_hi = g.q_hi;

    // ---- load: this thread's chunks of the row (in flight since the previous
    // row's write pass), then an online (max, sum, first chunk) over them
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // a thread reads only the chunks it copied
    LsTrip t{-kInf, 0.f, INT_MAX};
    for (int q0 = q_lo + tid; q0 < q_hi; q0 += kLsNT * kLsUnroll) {
      float f[kLsUnroll][8];
      float bm = -kInf;
#pragma unroll
      for (int u = 0; u < kLsUnroll; ++u) {
        const int q = q0 + u * kLsNT;
        const uint4 v = (q < q_hi) ? slice[q - q_lo] : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
        chunk_values(v, q, dc, V, q == 0 || q == nq - 1, f[u]);
#pragma unroll
        for (int i = 0; i < 8; ++i) bm = fmaxf(bm, f[u][i]);
      }
      if (bm > t.m) {
        // a new running max: rescale the sum; the first chunk of this batch
        // holding it (an equal max later in the walk has larger ids)
        t.s = (t.m == -kInf) ? 0.f : t.s * ex2_approx((t.m - bm) * kLog2e);
        t.m = bm;
        int a = INT_MAX;
#pragma unroll
        for (int u = kLsUnroll - 1; u >= 0; --u) {
          float c = f[u][0];
#pragma unroll
          for (int i = 1; i < 8; ++i) c = fmaxf(c, f[u][i]);
          if (c == bm) a = q0 + u * kLsNT;
        }
        t.a = a;
      }
      if (t.m != -kInf) {
        const float2 nml = make_float2(-t.m * kLog2e, -t.m * kLog2e);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kLsUnroll; ++u)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 tt = __ffma2_rn(make_float2(f[u][2 * i], f[u][2 * i + 1]), l2e, nml);
            acc = __fadd2_rn(acc, make_float2(ex2_approx(tt.x), ex2_approx(tt.y)));
          }
        t.s += acc.x + acc.y;
      }
    }

    // ---- merge: warp, CTA, then the cluster's CTAs in one fixed tree
    t = ls_warp_merge(t);
    if (lane == 0) warp_part[wid] = t;
    __syncthreads();
    if (wid == 0) {
      LsTrip w = (lane < kLsNT / 32) ? warp_part[lane] : LsTrip{-kInf, 0.f, INT_MAX};
      w = ls_warp_merge(w);
      if (lane == 0) cta_part[it & 1] = w;
    }
    cl.sync();  // every CTA's partial of this row is written
    if (wid == 0) {
      LsTrip w = (lane < cs) ? *cl.map_shared_rank(&cta_part[it & 1], lane) : LsTrip{-kInf, 0.f, INT_MAX};
      w = ls_warp_merge(w);
      if (lane == 0) {
        row_res = w;
        // the row's triple; the argmax from the CTA that holds its chunk. Every
        // other thread of this CTA waits at the barrier below, so no slot of
        // the slice is rewritten while it is read here.
        if (rank == 0) {
          out_max[row] = w.m;
          out_lse[row] = (w.m == -kInf) ? -kInf : w.m + logf(w.s);
        }
        if (w.a == INT_MAX ? rank == 0 : (w.a >= q_lo && w.a < q_hi)) {
          int am = 0;
          if (w.a != INT_MAX) {
            float f[8];
            chunk_values(slice[w.a - q_lo], w.a, dc, V, true, f);
            am = INT_MAX;
#pragma unroll
            for (int i = 7; i >= 0; --i)
              if (f[i] == w.m) am = 8 * w.a - dc + i;
            if (am == INT_MAX) am = 0;  // not reached: the chunk holds the max
          }
          out_argmax[row] = am;
        }
      }
    }
    __syncthreads();
    const LsTrip R = row_res;
    const float lse = (R.m == -kInf) ? -kInf : R.m + logf(R.s);

    // ---- write: x - lse from shared memory, by 16-byte stores when the output
    // row lines up with the input chunks
    unsigned char* orow = reinterpret_cast<unsigned char*>(out) + row * (long long)V * OB;
    const bool vec = ((reinterpret_cast<uintptr_t>(orow) - (uintptr_t)dc * OB) & 15) == 0;
    const long long nrow = row + n_clusters;
    const Slice gn = slice_of(nrow < n ? nrow : row);
    const int n_next = (nrow < n) ? gn.q_hi - gn.q_lo : 0;  // slots the next row fills
    for (int q = q_lo + tid; q < q_hi; q += kLsNT) {
      const bool edge = q == 0 || q == nq - 1;
      float f[8];
      chunk_values(slice[q - q_lo], q, dc, V, false, f);
      // the slot is read: start the next row's copy into it
      if (q - q_lo < n_next) cp_async16(&slice[q - q_lo], gn.base + gn.q_lo + (q - q_lo));
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] -= lse;
      const long long e0 = 8LL * q - dc;  // id of the chunk's first element
      if (vec && !edge) {
        if (BF16_OUT) {
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            o[i] = *reinterpret_cast<const uint32_t*>(&h);
          }
          *reinterpret_cast<uint4*>(orow + e0 * OB) = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
          float4* o = reinterpret_cast<float4*>(orow + e0 * OB);
          o[0] = make_float4(f[0], f[1], f[2], f[3]);
          o[1] = make_float4(f[4], f[5], f[6], f[7]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const long long e = e0 + i;
          if (e < 0 || e >= V) continue;
          if (BF16_OUT)
            reinterpret_cast<__nv_bfloat16*>(orow)[e] = __float2bfloat16_rn(f[i]);
          else
            reinterpret_cast<float*>(orow)[e] = f[i];
        }
      }
    }
    // the next row's slots beyond this row's (its slice can be one chunk longer)
    for (int j = (q_hi - q_lo) + ((tid - (q_hi - q_lo)) % kLsNT + kLsNT) % kLsNT; j < n_next; j += kLsNT)
      cp_async16(&slice[j], gn.base + gn.q_lo + j);
    asm volatile("cp.async.commit_group;" ::: "memory");
    // A thread's chunks of the next row sit in the same slots of the slice (slot
    // j belongs to thread j % kLsNT in every row), so no barrier is needed
    // before it overwrites them; cta_part is the other parity's, and row_res
    // is rewritten only after the next row's cluster barrier, which every
    // thread reaches after reading it.
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  // The next kernel may start launching only now: this grid is persistent.
  pdl_release();
  cl.sync();  // no CTA leaves while a peer may still read its partials
}

// ---------------------------------------------------------------- launcher
bool log_softmax_fused_fits(int V) {
  const long long nq = ((long long)V + 14) >> 3;  // chunks of a row at any alignment
  return (nq + 7) / 8 <= kLsSliceMax;
}

cudaError_t launch_log_softmax_fused(const uint16_t* x, int n, int V, float* out_max, float* out_lse,
                                     int* out_argmax, void* out, bool bf16_out, cudaStream_t st, bool* refused) {
  *refused = false;
  if (n <= 0) return cudaSuccess;
  // the fewest CTAs per row whose slices fit (shared memory per CTA = one slice)
  const long long nq = ((long long)V + 14) >> 3;
  int cs = 1;
  while ((nq + cs - 1) / cs > kLsSliceMax) cs *= 2;
  if (cs > 8) return cudaErrorInvalidValue;
  const size_t smem = (size_t)((nq + cs - 1) / cs) * sizeof(uint4);
  auto kern = bf16_out ? k_log_softmax_fused<true> : k_log_softmax_fused<false>;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kLsNT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3((unsigned)cs, 1, 1);
  // No cluster of this shape fits the device (the query fails or finds none):
  // refuse before launching anything, so the caller can take the two-pass form.
  // Only the query's own error is cleared here.
  // (the shared-memory limit, one value per kernel, is set once per device for
  // the largest slice; the occupancy is kept per device and shape; a refusal is
  // asked again next time)
  const int attr_ok = cached(reinterpret_cast<const void*>(kern), -1, [&](int) {
    const cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)((size_t)kLsSliceMax * sizeof(uint4)));
    if (r != cudaSuccess) (void)cudaGetLastError();
    return r == cudaSuccess ? 1 : 0;
  });
  const int max_clusters = attr_ok <= 0 ? 0 : cached(reinterpret_cast<const void*>(kern), (long long)smem * 16 + cs, [&](int) {
    int v = 0;
    const cudaError_t r = cudaOccupancyMaxActiveClusters(&v, kern, &cfg);
    if (r != cudaSuccess) {
      (void)cudaGetLastError();
      return 0;
    }
    return v;
  });
  if (max_clusters < 1) {
    *refused = true;
    return cudaSuccess;
  }
  cudaError_t e;
  long long n_clusters = max_clusters;
  if (n_clusters > n) n_clusters = n;
  cfg.gridDim = dim3((unsigned)(n_clusters * cs), 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, x, n, V, out_max, out_lse, out_argmax, out);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

}  // namespace ds
