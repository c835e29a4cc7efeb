// k_greedy.cu -- per-row max, logsumexp and argmax over a large vocabulary.
//
// "perf: avoid full-vocab all-gather for draft greedy sampling" (LightLLM PR
// #1517), Design and invariants: every vocabulary shard reduces its slice to a
// (max, log-sum-exp, argmax) triple and the triples are merged with ties going
// to the smallest global id. Here the shards are the CTAs of one thread-block
// cluster that splits a row, and the merge runs over distributed shared
// memory instead of an all-gather between GPUs.
//
// One streaming pass: each thread walks 16-byte chunks in increasing id order
// keeping an online (max, sum of exp(x - max), first argmax); a chunk's eight
// values are folded with one rescale per chunk, so each logit costs one exp.
#include <climits>
#include <cooperative_groups.h>

#include "ds_device.cuh"
#include "ds_launch.h"

namespace cg = cooperative_groups;

namespace ds {

struct Triple {
  float m;  // max
  float s;  // sum of exp(x - m)
  int a;    // smallest id attaining m
};

__device__ __forceinline__ Triple merge(const Triple& p, const Triple& q) {
  Triple r;
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

__device__ __forceinline__ Triple warp_merge(Triple t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Triple u;
    u.m = __shfl_xor_sync(0xffffffffu, t.m, o);
    u.s = __shfl_xor_sync(0xffffffffu, t.s, o);
    u.a = __shfl_xor_sync(0xffffffffu, t.a, o);
    t = merge(t, u);
  }
  return t;
}

template <int NT, int UNROLL>
__global__ void __launch_bounds__(NT) k_greedy_lse(const uint16_t* __restrict__ x, int n, int V,
                                                  float* __restrict__ out_max, float* __restrict__ out_lse,
                                                  int* __restrict__ out_argmax) {
  __shared__ Triple warp_part[NT / 32];
  __shared__ Triple cta_part;
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

  for (int row = blockIdx.y; row < n; row += gridDim.y) {
    const uint16_t* xr = x + (long long)row * V;
    const uintptr_t ad = reinterpret_cast<uintptr_t>(xr);
    const uint4* base = reinterpret_cast<const uint4*>(ad & ~(uintptr_t)15);
    const int dc = (int)((ad & 15) >> 1);
    const int nq = (dc + V + 7) >> 3;
    const int q_lo = (int)((long long)rank * nq / cs);
    const int q_hi = (int)((long long)(rank + 1) * nq / cs);

    Triple t{-kInf, 0.f, INT_MAX};
    for (int q0 = q_lo + tid; q0 < q_hi; q0 += NT * UNROLL) {
      uint4 v[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int q = q0 + u * NT;
        v[u] = (q < q_hi) ? ld_stream16(base + q) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
      }
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int q = q0 + u * NT;
        float f[8];
        unpack8(v[u], f);
        if (q == 0 || q >= nq - 1) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int id = 8 * q - dc + e;
            if (id < 0 || id >= V) f[e] = -kInf;
          }
        }
        float cm = f[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) cm = fmaxf(cm, f[e]);
        if (cm > t.m) {
          t.s = (t.m == -kInf) ? 0.f : t.s * ex2_approx((t.m - cm) * kLog2e);
          t.m = cm;
          int a = INT_MAX;
#pragma unroll
          for (int e = 7; e >= 0; --e)
            if (f[e] == cm) a = 8 * q - dc + e;
          t.a = a;
        }
        if (t.m != -kInf) {
          const float mb = t.m * kLog2e;
#pragma unroll
          for (int e = 0; e < 8; ++e) t.s += ex2_approx(fmaf(f[e], kLog2e, -mb));
        }
      }
    }
    // block merge
    t = warp_merge(t);
    if (lane == 0) warp_part[wid] = t;
    __syncthreads();
    if (wid == 0) {
      Triple w = (lane < NT / 32) ? warp_part[lane] : Triple{-kInf, 0.f, INT_MAX};
      w = warp_merge(w);
      if (lane == 0) cta_part = w;
    }
    // cluster merge over distributed shared memory, in rank order
    cluster.sync();
    if (rank == 0 && tid == 0) {
      Triple r = cta_part;
      for (int j = 1; j < cs; ++j) {
        const Triple* peer = cluster.map_shared_rank(&cta_part, j);
        r = merge(r, *peer);
      }
      out_max[row] = r.m;
      out_lse[row] = (r.m == -kInf) ? -kInf : r.m + logf(r.s);
      out_argmax[row] = (r.a == INT_MAX) ? 0 : r.a;
    }
    cluster.sync();  // peers' partials stay alive until rank 0 has read them
  }
}

// ---------------------------------------------------------------- launcher
cudaError_t launch_greedy(const uint16_t* x, int n, int V, float* out_max, float* out_lse, int* out_argmax,
                          cudaStream_t st) {
  constexpr int NT = 512;
  constexpr int UNROLL = 4;
  // Slice of about 32K elements per CTA, cluster of up to 8 CTAs per row.
  int cs = 1;
  while (cs < 8 && (long long)V > 32768LL * cs) cs *= 2;
  const int rows_grid = n < 65535 ? n : 65535;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cs, (unsigned)rows_grid, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_greedy_lse<NT, UNROLL>, x, n, V, out_max, out_lse, out_argmax);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ds
