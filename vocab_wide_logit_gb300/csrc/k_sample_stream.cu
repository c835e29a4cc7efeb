// k_sample_stream.cu -- sampling pass for large vocabularies, streaming form:
// one thread-block cluster per cell, the row split across its CTAs, each logit
// read once from HBM, and the Gumbel race run inside that single pass.
//
// Per cell, in each CTA:
//   pass    stream the slice in 16-byte chunks: z = c + g (c - u) and an online
//           (max, sum of exp(z - max), first argmax) per thread, rescaled once
//           per batch of chunks
//   cut     S* (the best perturbed score z + tau G of the whole row) is at least
//           SA, the best lower-bound score z + tau G_lo found so far, and at
//           least m + tau G_min for any z = m already seen; G <= G_max for
//           every noise word, so nothing with z < SA - tau G_max can win
//           ("Sampler support for discrete diffusion", Hert4's first comment:
//           Gumbel-max over the kept set). SA is shared by the cluster's CTAs
//           through atomics on each other's shared memory.
//   stage   chunks whose max reaches the cut are copied (as 8 z values) to a
//           per-warp queue in shared memory; each full queue is expanded into
//           its elements that still reach the cut, and those get their noise
//           word and table bounds (lo, hi) on G, and raise SA
//   live    an element whose upper-bound score reaches SA stays on a short
//           per-warp list; every other element is out of the race
//   R1      one cluster merge: (max, sum, first argmax) ("perf: avoid
//           full-vocab all-gather for draft greedy sampling", LightLLM PR
//           #1517, Design and invariants: per-shard max, log-sum-exp and
//           argmax, ties to the smallest id), the live lists' best lower
//           bound S and two best upper bounds, and E, the number of elements
//           that got noise
//   R4      (only when the bounds leave two live elements in reach) exact G
//           for the live elements
// The race so decided is over the whole row. Its winner w ranks inside the
// kept set (the k largest z, ties to the smallest id) when E <= k: every
// element with z >= z_w got noise, so rank(w) <= E, and the whole-row winner
// is then also the kept-set winner. A cell that fails this (or fills a live
// list) is marked in out_tokens and finished exactly by the staged kernel
// launched right after.
#include <atomic>
#include <cfloat>
#include <climits>
#include <cooperative_groups.h>
#include <type_traits>

#include "ds_launch.h"
#include "ds_sample_common.cuh"

namespace cg = cooperative_groups;

namespace ds {

namespace {

struct alignas(16) SRec {
  float f[8];
  int i[8];
};

struct SXchg {
  SRec slot[2];
  SRec comb;
};

// Per-warp queues in shared memory.
constexpr int kStageCap = 96;   // staged chunks: up to 31 left + 2 chunks x 32 lanes per batch
constexpr int kElemCap = 288;   // elements awaiting noise: up to 31 left + 32 chunks x 8
constexpr int kLiveCap = 32;    // evaluated elements still in the race

struct alignas(16) WarpArea {
  float4 stz[kStageCap][2];  // a staged chunk's 8 z values
  int stq[kStageCap];        // its chunk index
  float2 eq[kElemCap];       // (z, id bits) awaiting noise
  float4 live[kLiveCap];     // (z, id bits, lower score, upper score)
};

__device__ __forceinline__ float max3s(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Order-preserving int image of a float (finite or -inf) for atomicMax.
__device__ __forceinline__ int ord_enc(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7fffffff);
}
__device__ __forceinline__ float ord_dec(int i) { return __int_as_float(i >= 0 ? i : (i ^ 0x7fffffff)); }

// Rounding allowance of a perturbed score near S.
__device__ __forceinline__ float score_eps(float S) { return (fabsf(S) + 1.f) * 0x1p-20f; }

// Online (max, sum of exp(x - max), first argmax) merge.
__device__ __forceinline__ void msa_merge(float& m, float& s, int& am, float m2, float s2, int am2) {
  const float mm = fmaxf(m, m2);
  if (mm == -kInf) {
    am = min(am, am2);
    s = 0.f;
    m = mm;
    return;
  }
  s = s * ex2_approx((m - mm) * kLog2e) + s2 * ex2_approx((m2 - mm) * kLog2e);
  am = (m > m2) ? am : ((m2 > m) ? am2 : min(am, am2));
  m = mm;
}

// Two best upper bounds (hA from element idA with z = zA; hB the runner-up),
// ties on hA to the smaller id.
__device__ __forceinline__ void top2_merge(float& hA, float& hB, float& zA, int& idA, float hA2, float hB2, float zA2,
                                           int idA2) {
  const bool take = hA2 > hA || (hA2 == hA && idA2 >= 0 && (idA < 0 || idA2 < idA));
  hB = fmaxf(fmaxf(hB, hB2), take ? hA : hA2);
  if (take) {
    hA = hA2;
    zA = zA2;
    idA = idA2;
  }
}

// Cluster-wide reduction of one record per CTA. Each warp passes a record already
// reduced over the warp (valid in every lane); warp 0 combines the CTA's NT/32
// warp records, then the cluster's CTAs (lane r reads CTA r's record over
// DSMEM). Only the first NF floats and NI ints are moved. Every CTA combines the
// same records in the same tree, so every CTA ends with the same result.
template <int NF, int NI, typename Comb>
__device__ __forceinline__ void warp_tree(SRec& r, int n, Comb comb) {
  const int lane = threadIdx.x & 31;
  for (int o = 1; o < n; o <<= 1) {
    SRec q;
#pragma unroll
    for (int j = 0; j < NF; ++j) q.f[j] = __shfl_down_sync(0xffffffffu, r.f[j], o);
#pragma unroll
    for (int j = 0; j < NI; ++j) q.i[j] = __shfl_down_sync(0xffffffffu, r.i[j], o);
    if ((lane & (2 * o - 1)) == 0 && lane + o < n) comb(r, q);
  }
}

template <int NT, int NF, int NI, typename Comb>
__device__ __forceinline__ SRec cluster_combine(cg::cluster_group& cl, SXchg& xs, SRec* wrec, const SRec& mine,
                                                int& parity, int cs, Comb comb) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) wrec[wid] = mine;
  __syncthreads();
  if (wid == 0) {
    SRec r = wrec[lane < NT / 32 ? lane : 0];
    warp_tree<NF, NI>(r, NT / 32, comb);
    if (lane == 0) xs.slot[parity] = r;
  }
  cl.sync();
  if (wid == 0) {
    SRec r = *cl.map_shared_rank(&xs.slot[parity], lane < cs ? lane : 0);
    warp_tree<NF, NI>(r, cs, comb);
    if (lane == 0) xs.comb = r;
  }
  __syncthreads();
  parity ^= 1;
  return xs.comb;
}

}  // namespace

constexpr int kStreamNT = 256;
constexpr int kStreamUnroll = 2;
// A noise word whose lower bound is at least this gets G evaluated exactly
// when it is drawn. The table's buckets are uniform in the word, so they widen
// without limit as U -> 1 (the top one spans G in [7.6, 17.3]); at large V
// the winner usually lies there, and exact values keep SA tight and the final
// bounds apart. About 0.25% of the draws take this branch.
constexpr float kExactGFrom = 6.0f;

// ALIGNED: every c and u row starts on a 16-byte boundary (V a multiple of 8,
// both buffers 16-byte aligned), so chunks never straddle rows and u never
// needs the element-wise gather.
// Programmatic-launch roles of a streaming launch (the call's kernels run in
// stream order; see launch_sample_stream):
//   kPdlAlone  wait for the previous kernel first, let the next one launch last
//   kPdlHead   the first of two launches: wait first, then let the tail launch
//              go at once (its CTAs take SM room only as this grid's CTAs exit)
//   kPdlTail   the second: its cells are its own and it reads only inputs, so
//              it starts without waiting; it waits for the head grid before it
//              exits, so that the pass behind it sees both launches complete
constexpr int kPdlAlone = 0, kPdlHead = 1, kPdlTail = 2;

template <int NT, int UNROLL, bool ALIGNED>
__global__ void __launch_bounds__(NT, 3)
    k_sample_stream(const SampleArgs a, long long cell_lo, long long cell_hi, int pdl_role) {
  if (pdl_role != kPdlTail) pdl_wait();
  if (pdl_role == kPdlHead) pdl_release();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ SXchg xs;
  __shared__ SRec wrec[NT / 32];
  __shared__ int s_sa[2];  // best lower-bound score of the cell, per cell parity (ord_enc)
  __shared__ ReqCursor s_cur;
  __shared__ long long s_Pu;
  __shared__ int s_bad;

  cg::cluster_group cl = cg::this_cluster();
  const int cs = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  WarpArea& W = reinterpret_cast<WarpArea*>(smem_raw)[wid];
  const long long n_clusters = (long long)gridDim.x / cs;
  const long long cluster_id = (long long)blockIdx.x / cs;
  const int P = a.P, V = a.V;
  const float2 l2e = make_float2(kLog2e, kLog2e);
  int parity = 0;

  if (wid == 0) {
    const BatchTotals bt = warp_batch_totals(a, lane);
    if (lane == 0) {
      s_bad = (bt.bad || bt.tot != (long long)P) ? 1 : 0;
      s_Pu = bt.tot_u;
    }
  }
  if (tid == 0) {
    s_sa[0] = ord_enc(-kInf);
    s_sa[1] = ord_enc(-kInf);
  }
  __syncthreads();
  if (s_bad) {
    if (rank == 0 && tid == 0) {
      for (long long cell = cell_lo + cluster_id; cell < cell_hi; cell += n_clusters) {
        a.out_tokens[cell] = -1;
        a.out_logprobs[cell] = __int_as_float(0x7fc00000);
      }
      report(a.d_status, DS_DEV_ERR_LAYOUT);
    }
    if (pdl_role == kPdlTail) pdl_wait();
    if (pdl_role != kPdlHead) pdl_release();
    return;  // uniform across the cluster; no shared memory was shared yet
  }
  cl.sync();  // peers may write s_sa from here on
  const long long P_u = s_Pu;
  // every G lies in [g_min, g_max], the outer bounds of the table
  const float g_max = kGumbelBounds[(1u << (32 - DS_GUMBEL_BUCKET_SHIFT)) - 1].y;
  const float g_min = kGumbelBounds[0].x;

  int it = 0;
  for (long long cell = cell_lo + cluster_id; cell < cell_hi; cell += n_clusters, ++it) {
    const int c = (int)(cell / P);
    const int p = (int)(cell - (long long)c * P);
    const int slot = it & 1;
    if (wid == 0) {
      ReqCursor cur;
      warp_find_request(a, p, lane, cur);
      if (lane == 0) s_cur = cur;
    }
    // The other parity's slot is next used by the next cell. Peers write it only
    // after they pass this cell's merge, which waits for this CTA.
    if (tid == 0) s_sa[slot ^ 1] = ord_enc(-kInf);
    __syncthreads();
    const ReqCursor cur = s_cur;
    const int t = p - cur.off;
    const float g = cur.g, tau = cur.tau;
    if (!(tau >= 0.f) || isnan(g) || cur.perr || (g != 0.f && a.u == nullptr)) {
      if (rank == 0 && tid == 0) {
        a.out_tokens[cell] = -1;
        a.out_logprobs[cell] = __int_as_float(0x7fc00000);
        report(a.d_status, (!(tau >= 0.f) || isnan(g) || cur.perr) ? DS_DEV_ERR_PARAM : DS_DEV_ERR_NO_UNCOND);
      }
      __syncthreads();
      continue;
    }
    const bool guided = g != 0.f;
    const bool sampled = tau > 0.f;
    const float2 ng2 = make_float2(-g, -g);
    const uint32_t t32 = (uint32_t)t;
    const uint32_t ctr3 = cur.iter_hi | (uint32_t)c;
    const int k = cur.k;
    const float tgmax = tau * g_max;

    // ---- slice geometry
    const uint16_t* crow = a.c + cell * (long long)V;
    const uintptr_t ca = reinterpret_cast<uintptr_t>(crow);
    const uint4* cb = reinterpret_cast<const uint4*>(ca & ~(uintptr_t)15);
    const int dc = ALIGNED ? 0 : (int)((ca & 15) >> 1);
    const int nq = (dc + V + 7) >> 3;
    const int q_lo = (int)((long long)rank * nq / cs);
    const int q_hi = (int)((long long)(rank + 1) * nq / cs);
    const uint16_t* urow = nullptr;
    const uint4* ub = nullptr;
    bool u_aligned = true;
    if (guided) {
      urow = a.u + ((long long)c * P_u + cur.off_u + t) * (long long)V;
      const uintptr_t ua = reinterpret_cast<uintptr_t>(urow);
      ub = reinterpret_cast<const uint4*>(ua & ~(uintptr_t)15);
      u_aligned = ALIGNED || (ua & 15) == (ca & 15);
    }
    auto load_u = [&](int q) -> uint4 {
      if (u_aligned) return ld_stream16(ub + q);
      const int id0 = 8 * q - dc;
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int i0 = id0 + 2 * h, i1 = i0 + 1;
        const uint32_t lo = (i0 >= 0 && i0 < V) ? (uint32_t)__ldg(urow + i0) : 0u;
        const uint32_t hi = (i1 >= 0 && i1 < V) ? (uint32_t)__ldg(urow + i1) : 0u;
        w[h] = lo | (hi << 16);
      }
      return make_uint4(w[0], w[1], w[2], w[3]);
    };

    // first id of chunk q whose z equals zt (INT_MAX if none): z formed from the
    // two logits exactly as in the pass, ids outside the row masked
    auto chunk_first_id = [&](int q, float zt) -> int {
      const uint4 vc = __ldg(cb + q);
      const uint4 vu = guided ? load_u(q) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t wc[4] = {vc.x, vc.y, vc.z, vc.w};
      const uint32_t wu[4] = {vu.x, vu.y, vu.z, vu.w};
      int id = INT_MAX;
#pragma unroll
      for (int i = 7; i >= 0; --i) {
        const float ci = (i & 1) ? bf_hi(wc[i >> 1]) : bf_lo(wc[i >> 1]);
        const float ui = (i & 1) ? bf_hi(wu[i >> 1]) : bf_lo(wu[i >> 1]);
        const float zi = guided ? __fmaf_rn(g, __fmaf_rn(ui, -1.f, ci), ci) : ci;
        const int e = 8 * q - dc + i;
        if (e >= 0 && e < V && zi == zt) id = e;
      }
      return id;
    };

    // ---- race state (queue lengths and flags are warp-uniform)
    float m = -kInf, s = 0.f;
    int am = INT_MAX;  // first chunk holding m
    int aid = INT_MAX;  // id of the first element equal to m (read by the anchor only)
    float SAl = -kInf;           // best lower-bound score this warp knows of
    int ns = 0, ne = 0, nl = 0;  // staged chunks, queued elements, live elements
    int E = 0;                   // elements this warp sent to the noise stage
    bool stop = false;           // cell left to the staged kernel: live list full or E > k

    auto slot_sa = [&]() -> float { return ord_dec(*reinterpret_cast<volatile int*>(&s_sa[slot])); };
    auto publish = [&](float v) {  // raise SA in every CTA of the cluster
      if (lane == 0) {
        const int e = ord_enc(v);
        for (int r = 0; r < cs; ++r) atomicMax(cl.map_shared_rank(&s_sa[slot], r), e);
      }
    };
    // lowest z that can still win, given the best known score bound and m
    // (+inf at temperature 0: no race, nothing is staged)
    // (never below -FLT_MAX, so a comparison with it also rejects -inf)
    auto cut_of = [&](float SA) -> float {
      const float sb = fmaxf(SA, __fmaf_rn(tau, g_min, m));
      return (sampled && !stop) ? fmaxf(sb - score_eps(sb) - tgmax, -FLT_MAX) : kInf;
    };
    // drop live entries whose upper score fell below thr (in place, in order)
    auto prune = [&](float thr) {
      int w = 0;
      for (int b0 = 0; b0 < nl; b0 += 32) {
        const int i = b0 + lane;
        const float4 v = (i < nl) ? W.live[i] : make_float4(0.f, 0.f, -kInf, -kInf);
        const bool keep = i < nl && v.w >= thr;
        const unsigned bk = __ballot_sync(0xffffffffu, keep);
        __syncwarp();
        if (keep) W.live[w + __popc(bk & lt_mask)] = v;
        w += __popc(bk);
        __syncwarp();
      }
      nl = w;
    };
    // noise for the last cnt queued elements; raise SA; keep the ones still in reach
    auto eval = [&](int cnt) {
      const int i = ne - cnt + lane;
      const bool on = lane < cnt;
      float2 v = make_float2(-kInf, 0.f);
      float lo = -kInf, hi = -kInf;
      if (on) {
        v = W.eq[i];
        const uint32_t x = noise_word(__float_as_uint(v.y), t32, cur.rid, ctr3, a.rk0, a.rk1);
        float2 gb = gumbel_bounds(x);
        if (gb.x >= kExactGFrom) {
          const float ge = gumbel_accurate(x);
          gb = make_float2(ge, ge);
        }
        lo = __fmaf_rn(tau, gb.x, v.x);
        hi = __fmaf_rn(tau, gb.y, v.x);
      }
      ne -= cnt;
      const float wlo = warp_max_r(lo);
      const float known = fmaxf(SAl, slot_sa());
      if (wlo > known) publish(wlo);
      SAl = fmaxf(known, wlo);
      const float thr = SAl - score_eps(SAl);
      const bool lv = on && hi >= thr && hi > -kInf;
      const unsigned b = __ballot_sync(0xffffffffu, lv);
      if (b) {
        if (nl + __popc(b) > kLiveCap) prune(thr);
        if (nl + __popc(b) > kLiveCap) {
          stop = true;
        } else {
          if (lv) W.live[nl + __popc(b & lt_mask)] = make_float4(v.x, v.y, lo, hi);
          nl += __popc(b);
        }
      }
      __syncwarp();
    };
    // expand the last cnt staged chunks into their elements that reach the cut
    auto drain = [&](int cnt) {
      const int e = ns - cnt + lane;
      const bool on = lane < cnt;
      float zz[8];
      int q = 0;
      if (on) {
        const float4 A = W.stz[e][0], Bv = W.stz[e][1];
        zz[0] = A.x; zz[1] = A.y; zz[2] = A.z; zz[3] = A.w;
        zz[4] = Bv.x; zz[5] = Bv.y; zz[6] = Bv.z; zz[7] = Bv.w;
        q = W.stq[e];
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) zz[j] = -kInf;
      }
      const float cut = cut_of(fmaxf(SAl, slot_sa()));
      uint32_t mk = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) mk |= (zz[j] >= cut) ? (1u << j) : 0u;
      const int n = __popc(mk);
      const int ex = warp_excl_scan(n, lane);
      const int tot = __shfl_sync(0xffffffffu, ex + n, 31);
      E += tot;
      if (E > k) stop = true;  // the cell goes to the staged kernel: stop staging
      __syncwarp();
      int pos = ne + ex;
      const int id0 = 8 * q - dc;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if ((mk >> j) & 1u) W.eq[pos++] = make_float2(zz[j], __int_as_float(id0 + j));
      ne += tot;
      ns -= cnt;
      __syncwarp();
    };
    auto work = [&]() {
      while (ns >= 32) {
        drain(32);
        while (ne >= 32) eval(32);
      }
    };

    // ---- the pass. Interior chunks go through full batches with no per-chunk
    // checks; the row's edge chunks and the last partial batch go through a
    // checked one-chunk path. MODE: 0 statistics, 1 statistics and staging,
    // 2 staging only. Guidance and temperature are per-cell flags here rather
    // than template parameters: one copy of the loop keeps register use low.
    auto pass = [&]() {
      auto load = [&](int q0, auto nchk_tag, auto checked_tag, bool act, uint4* vc, uint4* vu) {
        constexpr int NCHK = decltype(nchk_tag)::value;
        constexpr bool CHECKED = decltype(checked_tag)::value;
#pragma unroll
        for (int uu = 0; uu < NCHK; ++uu) {
          const int q = q0 + uu * NT;
          const bool ok = !CHECKED || (act && q < q_hi);
          vc[uu] = ok ? ld_stream16(cb + q) : make_uint4(0u, 0u, 0u, 0u);
          vu[uu] = (ok && guided) ? load_u(q) : make_uint4(0u, 0u, 0u, 0u);
        }
      };
      auto compute = [&](int q0, auto nchk_tag, auto checked_tag, auto mode_tag, bool act, const uint4* vc,
                         const uint4* vu) {
        constexpr int NCHK = decltype(nchk_tag)::value;
        constexpr bool CHECKED = decltype(checked_tag)::value;
        constexpr int MODE = decltype(mode_tag)::value;
        float2 z[NCHK][4];
        float cmx[NCHK];
        float bm = -kInf;
#pragma unroll
        for (int uu = 0; uu < NCHK; ++uu) {
          const int q = q0 + uu * NT;
          const uint32_t wc[4] = {vc[uu].x, vc[uu].y, vc[uu].z, vc[uu].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 cp = make_float2(bf_lo(wc[i]), bf_hi(wc[i]));
            const uint32_t wu = (i == 0) ? vu[uu].x : (i == 1) ? vu[uu].y : (i == 2) ? vu[uu].z : vu[uu].w;
            // fl(u - c), u widened to fp32 inside the subtraction; it is exactly
            // -fl(c - u) (round to nearest is symmetric), so (-g) fl(u - c) + c in
            // one fma is the combine fma(g, fl(c - u), c)
            float dx, dy;
            asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; sub.rn.f32.bf16 %0, lo, %3; sub.rn.f32.bf16 %1, hi, %4; }"
                : "=f"(dx), "=f"(dy) : "r"(wu), "f"(cp.x), "f"(cp.y));
            const float2 zg = __ffma2_rn(ng2, make_float2(dx, dy), cp);
            z[uu][i] = guided ? zg : cp;
          }
          if (CHECKED) {
            const bool ok = act && q < q_hi;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int id = 8 * q - dc + 2 * i;
              if (!ok || id < 0 || id >= V) z[uu][i].x = -kInf;
              if (!ok || id + 1 < 0 || id + 1 >= V) z[uu][i].y = -kInf;
            }
          }
          float cm = max3s(z[uu][0].x, z[uu][0].y, z[uu][1].x);
          cm = max3s(cm, z[uu][1].y, z[uu][2].x);
          cm = max3s(cm, z[uu][2].y, z[uu][3].x);
          cmx[uu] = fmaxf(cm, z[uu][3].y);
          bm = fmaxf(bm, cmx[uu]);
        }
        if (MODE != 2) {
          if (bm > m) {
            // a new running max: rescale the sum; remember the first chunk of the
            // batch holding it (a thread walks its chunks in increasing order, so
            // an equal max met later has larger ids)
            s = (m == -kInf) ? 0.f : s * ex2_approx((m - bm) * kLog2e);
            m = bm;
            int aa = INT_MAX, ai = INT_MAX;
#pragma unroll
            for (int uu = NCHK - 1; uu >= 0; --uu) {
              if (cmx[uu] == bm) {
                aa = q0 + uu * NT;
                int e = 0;
#pragma unroll
                for (int i = 3; i >= 0; --i) {
                  if (z[uu][i].y == bm) e = 2 * i + 1;
                  if (z[uu][i].x == bm) e = 2 * i;
                }
                ai = 8 * aa - dc + e;
              }
            }
            am = aa;
            aid = ai;
          }
          if (m != -kInf) {
            const float2 nml = make_float2(-m * kLog2e, -m * kLog2e);
            float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int uu = 0; uu < NCHK; ++uu)
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 tt = __ffma2_rn(z[uu][i], l2e, nml);
                const float2 ee = make_float2(ex2_approx(tt.x), ex2_approx(tt.y));
                if (i & 1) acc1 = __fadd2_rn(acc1, ee); else acc0 = __fadd2_rn(acc0, ee);
              }
            s += (acc0.x + acc0.y) + (acc1.x + acc1.y);
          }
        }
        if (MODE != 0) {
          const float cut = cut_of(fmaxf(SAl, slot_sa()));
#pragma unroll
          for (int uu = 0; uu < NCHK; ++uu) {
            const bool hot = cmx[uu] >= cut;
            const unsigned b = __ballot_sync(0xffffffffu, hot);
            if (hot) {
              const int pos = ns + __popc(b & lt_mask);
              W.stz[pos][0] = make_float4(z[uu][0].x, z[uu][0].y, z[uu][1].x, z[uu][1].y);
              W.stz[pos][1] = make_float4(z[uu][2].x, z[uu][2].y, z[uu][3].x, z[uu][3].y);
              W.stq[pos] = q0 + uu * NT;
            }
            ns += __popc(b);
          }
          __syncwarp();
          work();
        }
      };
      using UN = std::integral_constant<int, UNROLL>;
      using ONE = std::integral_constant<int, 1>;
      using STATS = std::integral_constant<int, 0>;
      using BOTH = std::integral_constant<int, 1>;
      using STAGE = std::integral_constant<int, 2>;
      auto batch1 = [&](int q, bool act) {  // one checked chunk
        uint4 vc[1], vu[1];
        load(q, ONE{}, std::true_type{}, act, vc, vu);
        compute(q, ONE{}, std::true_type{}, BOTH{}, act, vc, vu);
      };
      // row-edge chunk 0 (lane 0 of warp 0; the whole warp takes part in staging)
      if (wid == 0 && q_lo == 0 && q_hi > 0) batch1(0, lane == 0);
      const int qa = max(q_lo, 1), qb = min(q_hi, nq - 1);
      const int n_full = (qb > qa) ? (qb - qa) / (NT * UNROLL) : 0;
      int q0 = qa + tid;
      uint4 cc[UNROLL], cu[UNROLL], nc_[UNROLL], nu[UNROLL];
      if (n_full > 0) {
        load(q0, UN{}, std::false_type{}, true, cc, cu);
        if (n_full > 1) load(q0 + NT * UNROLL, UN{}, std::false_type{}, true, nc_, nu);
        compute(q0, UN{}, std::false_type{}, STATS{}, true, cc, cu);
      }
      if (sampled) {
        // Anchor: the warp's best z so far and its lower-bound score seed SA, so
        // that the first batch is staged against a useful cut. Each warp
        // publishes its own, with no CTA barrier: the cell's warps start
        // together, so the others' anchors land in SA within moments.
        float bz = m;
        int bi = aid;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float z2 = __shfl_xor_sync(0xffffffffu, bz, o);
          const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
          if (z2 > bz || (z2 == bz && i2 < bi)) {
            bz = z2;
            bi = i2;
          }
        }
        if (bz > -kInf && bi != INT_MAX) {  // the warp's first element holding its max
          const uint32_t x = noise_word((uint32_t)bi, t32, cur.rid, ctr3, a.rk0, a.rk1);
          const float lo = __fmaf_rn(tau, gumbel_bounds(x).x, bz);
          publish(lo);
          SAl = fmaxf(SAl, lo);
        }
        if (n_full > 0) compute(q0, UN{}, std::false_type{}, STAGE{}, true, cc, cu);
      }
      if (n_full > 0) {
#pragma unroll
        for (int uu = 0; uu < UNROLL; ++uu) {
          cc[uu] = nc_[uu];
          cu[uu] = nu[uu];
        }
        q0 += NT * UNROLL;
        for (int b = 1; b < n_full; ++b, q0 += NT * UNROLL) {
          // the next batch's loads are in flight while this one is reduced
          if (b + 1 < n_full) load(q0 + NT * UNROLL, UN{}, std::false_type{}, true, nc_, nu);
          compute(q0, UN{}, std::false_type{}, BOTH{}, true, cc, cu);
#pragma unroll
          for (int uu = 0; uu < UNROLL; ++uu) {
            cc[uu] = nc_[uu];
            cu[uu] = nu[uu];
          }
        }
      }
      // the rest of the slice (at most NT * UNROLL chunks, the row-edge chunk
      // nq-1 included), one checked chunk per thread and round; a warp whose
      // first chunk of the round lies past the slice has none and skips it
#pragma unroll 1
      for (int r = 0; r < UNROLL; ++r) {
        const int qw = qa + n_full * NT * UNROLL + r * NT + wid * 32;
        if (qw < q_hi) batch1(qw + lane, true);
      }
      if (sampled) {
        if (ns > 0) drain(ns);
        while (ne > 0) eval(min(ne, 32));
      }
    };
    pass();

    // ---- R1: one cluster merge of the statistics and of the race
    float lse, zw;
    int idw;
    {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const int a2 = __shfl_xor_sync(0xffffffffu, am, o);
        msa_merge(m, s, am, m2, s2, a2);
      }
      // this warp's live list: best lower score, two best upper scores
      float loMax = -kInf, hA = -kInf, hB = -kInf, zA = 0.f;
      int idA = -1;
      if (lane < nl) {
        const float4 v = W.live[lane];
        loMax = v.z;
        hA = v.w;
        zA = v.x;
        idA = __float_as_int(v.y);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        loMax = fmaxf(loMax, __shfl_xor_sync(0xffffffffu, loMax, o));
        const float hA2 = __shfl_xor_sync(0xffffffffu, hA, o);
        const float hB2 = __shfl_xor_sync(0xffffffffu, hB, o);
        const float zA2 = __shfl_xor_sync(0xffffffffu, zA, o);
        const int idA2 = __shfl_xor_sync(0xffffffffu, idA, o);
        top2_merge(hA, hB, zA, idA, hA2, hB2, zA2, idA2);
      }
      SRec r{};
      r.f[0] = m; r.f[1] = s; r.f[2] = loMax; r.f[3] = hA; r.f[4] = hB; r.f[5] = zA;
      r.i[0] = am; r.i[1] = idA; r.i[2] = E; r.i[3] = stop ? 1 : 0;
      const SRec R = cluster_combine<NT, 6, 4>(cl, xs, wrec, r, parity, cs, [](SRec& x, const SRec& y) {
        msa_merge(x.f[0], x.f[1], x.i[0], y.f[0], y.f[1], y.i[0]);
        x.f[2] = fmaxf(x.f[2], y.f[2]);
        top2_merge(x.f[3], x.f[4], x.f[5], x.i[1], y.f[3], y.f[4], y.f[5], y.i[1]);
        x.i[2] += y.i[2];
        x.i[3] |= y.i[3];
      });
      m = R.f[0];
      am = R.i[0];
      lse = (m == -kInf) ? -kInf : m + logf(R.f[1]);
      if (m == -kInf || !sampled) {  // all -inf (token 0, logprob NaN) or temperature 0 (the argmax)
        if (rank == 0 && tid == 0) {
          a.out_tokens[cell] = (m == -kInf) ? 0 : chunk_first_id(am, m);
          a.out_logprobs[cell] = (m == -kInf) ? __int_as_float(0x7fc00000) : m - lse;
        }
        __syncthreads();
        continue;
      }
      const float S = R.f[2];
      // a full live list, or a winner that may rank outside the kept set
      if (R.i[3] != 0 || R.i[2] > k || !(S > -kInf)) {
        if (rank == 0 && tid == 0) a.out_tokens[cell] = kStreamMark;
        __syncthreads();
        continue;
      }
      const float thr = S - score_eps(S);
      if (R.f[4] < thr) {
        zw = R.f[5];
        idw = R.i[1];
      } else {
        // R4: exact G for the live elements whose upper score reaches thr
        float bs = -kInf, bz = 0.f;
        int bid = INT_MAX;
        if (lane < nl) {
          const float4 v = W.live[lane];
          if (v.w >= thr) {
            const int id = __float_as_int(v.y);
            const uint32_t x = noise_word((uint32_t)id, t32, cur.rid, ctr3, a.rk0, a.rk1);
            bs = __fmaf_rn(tau, gumbel_accurate(x), v.x);
            bz = v.x;
            bid = id;
          }
        }
        const int wl = warp_argmax_lane(bs, bid);
        SRec r4{};
        r4.f[0] = __shfl_sync(0xffffffffu, bs, wl);
        r4.f[1] = __shfl_sync(0xffffffffu, bz, wl);
        r4.i[0] = __shfl_sync(0xffffffffu, bid, wl);
        const SRec R4 = cluster_combine<NT, 2, 1>(cl, xs, wrec, r4, parity, cs, [](SRec& x, const SRec& y) {
          if (y.f[0] > x.f[0] || (y.f[0] == x.f[0] && y.i[0] < x.i[0])) x = y;
        });
        zw = R4.f[1];
        idw = R4.i[0];
      }
    }
    if (rank == 0 && tid == 0) {
      a.out_tokens[cell] = idw;
      a.out_logprobs[cell] = zw - lse;
    }
    __syncthreads();
  }
  // The next kernel (the fix-up pass, or the tail launch already released by a
  // head launch) may start launching only now: this grid is persistent and sized
  // for an empty GPU, so the pass behind it should not take SM room before its
  // cells are done. A tail launch first waits for the head grid.
  if (pdl_role == kPdlTail) pdl_wait();
  if (pdl_role != kPdlHead) pdl_release();
  cl.sync();  // no CTA leaves while a peer may still read its exchange slots or write s_sa
}

// ---------------------------------------------------------------- launcher
namespace {

// Clusters of cs CTAs that fit on the device at once (cached per device, row
// alignment and cluster size; the answer depends on the kernel's resources only).
int stream_capacity(int dev, bool aligned, int cs, const void* kern, size_t smem) {
  static std::atomic<int> cache[16][2][3];
  const int ci = cs == 1 ? 0 : (cs == 2 ? 1 : 2);
  if (dev >= 0 && dev < 16) {
    const int v = cache[dev][aligned][ci].load(std::memory_order_relaxed);
    if (v != 0) return v;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kStreamNT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.gridDim = dim3((unsigned)cs, 1, 1);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) return -1;
  if (dev >= 0 && dev < 16) cache[dev][aligned][ci].store(n, std::memory_order_relaxed);
  return n;
}

// CTA time per cell relative to one CTA per cell, measured on GB300 at
// V = 248320 (1024 cells): 1.00, 1.10 and 1.19 for 1, 2 and 4 CTAs. A cell
// split over more CTAs finishes sooner but waits on more warps at its merge.
double stream_cell_cost(int cs) { return cs == 1 ? 1.0 : (cs == 2 ? 1.10 : 1.19); }

}  // namespace

// Up to two launches: the cheapest of one launch with 1, 2 or 4 CTAs per cell,
// or full rounds of one CTA per cell followed by the remaining cells on 2 or 4
// CTAs each (so that a partial last round still fills the GPU). Time in units
// of one CTA on one cell: rounds x cost(cs) / cs.
cudaError_t launch_sample_stream(const SampleArgs& a, cudaStream_t st) {
  const long long n_cells = (long long)a.C * a.P;
  if (n_cells <= 0) return cudaSuccess;
  const int nq_max = (a.V + 7 + 7) >> 3;
  // at most 4 CTAs per row, and no more than leave each CTA about two batches per thread
  int cs_max = 1;
  while (cs_max < 4 && nq_max / cs_max > 2 * kStreamNT * kStreamUnroll) cs_max *= 2;
  const bool aligned = (a.V % 8) == 0 && (reinterpret_cast<uintptr_t>(a.c) & 15) == 0 &&
                       (reinterpret_cast<uintptr_t>(a.u) & 15) == 0;
  auto kern = aligned ? k_sample_stream<kStreamNT, kStreamUnroll, true>
                      : k_sample_stream<kStreamNT, kStreamUnroll, false>;
  const size_t smem = sizeof(WarpArea) * (kStreamNT / 32);
  const int attr_ok = cached(reinterpret_cast<const void*>(kern), (long long)smem, [&](int) {
    const cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return r == cudaSuccess ? 1 : -(int)r;
  });
  if (attr_ok <= 0) return attr_ok < 0 ? (cudaError_t)(-attr_ok) : cudaErrorUnknown;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  long long cap[5] = {0, 0, 0, 0, 0};
  for (int cs = 1; cs <= cs_max; cs *= 2) {
    cap[cs] = stream_capacity(dev, aligned, cs, reinterpret_cast<const void*>(kern), smem);
    if (cap[cs] < 1) return cudaErrorLaunchOutOfResources;
  }
  auto t_of = [&](int cs, long long cells) {
    return (double)((cells + cap[cs] - 1) / cap[cs]) * stream_cell_cost(cs) / cs;
  };
  // the plan: cs1 for cells [0, split), cs2 for [split, n_cells)
  int cs1 = 1, cs2 = 1;
  long long split = n_cells;
  double best = t_of(1, n_cells);
  for (int cs = 2; cs <= cs_max; cs *= 2) {
    const double t = t_of(cs, n_cells);
    if (t < best) {
      best = t;
      cs1 = cs;
      split = n_cells;
    }
  }
  const long long full = (n_cells / cap[1]) * cap[1];
  if (full > 0 && full < n_cells) {
    for (int cs = 2; cs <= cs_max; cs *= 2) {
      const double t = (double)(full / cap[1]) + t_of(cs, n_cells - full);
      if (t < best) {
        best = t;
        cs1 = 1;
        cs2 = cs;
        split = full;
      }
    }
  }
  auto launch = [&](int cs, long long lo, long long hi, int role) -> cudaError_t {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kStreamNT, 1, 1);
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
    long long n_clusters = cap[cs];
    if (n_clusters > hi - lo) n_clusters = hi - lo;
    cfg.gridDim = dim3((unsigned)(n_clusters * cs), 1, 1);
    cudaError_t r = cudaLaunchKernelEx(&cfg, kern, a, lo, hi, role);
    if (r != cudaSuccess) return r;
    note_launch();
    return cudaGetLastError();
  };
  if (split < n_cells) {
    e = launch(cs1, 0, split, kPdlHead);
    if (e == cudaSuccess) e = launch(cs2, split, n_cells, kPdlTail);
  } else {
    e = launch(cs1, 0, split, kPdlAlone);
  }
  return e;
}

}  // namespace ds
