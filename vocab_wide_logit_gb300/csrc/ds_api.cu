// ds_api.cu -- the C ABI of libdsample: argument checks, launch parameters, dispatch.
//
// Host work per call is O(1): validate the scalars, derive the kept count k
// and the two normal quantiles that seed the kernels' threshold guesses, pick
// the kernel by vocabulary size, and launch asynchronously on the caller's
// stream. Nothing is allocated and nothing is synchronised.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>
#include <cuda_runtime.h>

#include "dsample.h"
#include "ds_launch.h"

namespace {

// Upper-tail standard normal quantile: x with P(N(0,1) > x) = p, by bisection on
// erfc (host-side, double). p <= 0 -> +inf, p >= 1 -> -inf.
double normal_upper_quantile(double p) {
  if (p <= 0.0) return INFINITY;
  if (p >= 1.0) return -INFINITY;
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 200; ++it) {
    const double mid = 0.5 * (lo + hi);
    const double tail = 0.5 * std::erfc(mid / std::sqrt(2.0));
    if (tail > p)
      lo = mid;
    else
      hi = mid;
  }
  return 0.5 * (lo + hi);
}

std::atomic<unsigned long long> g_launches{0};

std::mutex g_cache_mu;
std::map<std::tuple<const void*, int, long long>, int>& launch_cache() {
  static std::map<std::tuple<const void*, int, long long>, int> m;
  return m;
}

int device_sm_count() { return ds::device_sms(); }

}  // namespace

namespace ds {
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

bool cache_lookup(const void* site, int dev, long long param, int* value) {
  std::lock_guard<std::mutex> lk(g_cache_mu);
  const auto& m = launch_cache();
  const auto it = m.find(std::make_tuple(site, dev, param));
  if (it == m.end()) return false;
  *value = it->second;
  return true;
}

void cache_store(const void* site, int dev, long long param, int value) {
  std::lock_guard<std::mutex> lk(g_cache_mu);
  launch_cache()[std::make_tuple(site, dev, param)] = value;
}

int device_sms() {
  static const char site = 0;
  return cached(&site, 0, [](int dev) {
    int sms = 0;
    return cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? sms : -1;
  });
}
}  // namespace ds

extern "C" {

uint64_t ds_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* ds_status_string(ds_status s) {
  switch (s) {
    case DS_OK: return "ok";
    case DS_ERR_INVALID_ARG: return "invalid argument";
    case DS_ERR_UNSUPPORTED: return "unsupported size for this build";
    case DS_ERR_CUDA: return "CUDA launch or runtime error";
  }
  return "unknown status";
}

int32_t ds_top_k(float top_ratio, int32_t V) {
  if (V < 1 || !(top_ratio > 0.0f) || !(top_ratio <= 1.0f)) return 0;
  const float prod = top_ratio * (float)V;  // fp32 product, as the contract states
  long long k = (long long)ceilf(prod);
  if (k < 1) k = 1;
  if (k > V) k = V;
  return (int32_t)k;
}

ds_status ds_sample_ex(const int32_t* request_ids, const void* c_logits, const void* u_logits,
                       const int32_t* seq_lens, int32_t B, int32_t C, int32_t P, int32_t V,
                       const float* guidance, const float* temperature, const float* top_ratios,
                       float top_ratio, uint64_t seed, const uint32_t* iterations, uint32_t iteration,
                       uint32_t flags, int32_t* out_tokens, float* out_logprobs, uint32_t* d_status,
                       void* stream) {
  if (B < 0 || C < 0 || P < 0 || V < 1) return DS_ERR_INVALID_ARG;
  if ((flags & ~(uint32_t)(DS_FLAG_KEEP_TIES | DS_FLAG_SKIP_EXACT_PASS)) != 0u) return DS_ERR_INVALID_ARG;
  if (C > DS_MAX_ROWS) return DS_ERR_INVALID_ARG;
  if (!iterations && iteration > DS_MAX_ITERATION) return DS_ERR_INVALID_ARG;
  if (!top_ratios && !(top_ratio > 0.0f && top_ratio <= 1.0f)) return DS_ERR_INVALID_ARG;
  if (C == 0 || P == 0) return DS_OK;
  if (B == 0) return DS_ERR_INVALID_ARG;  // P > 0 positions need an owner
  if (!request_ids || !c_logits || !seq_lens || !guidance || !temperature || !out_tokens || !out_logprobs)
    return DS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(c_logits) & 1) || (reinterpret_cast<uintptr_t>(u_logits) & 1))
    return DS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(top_ratios) & 3) || (reinterpret_cast<uintptr_t>(iterations) & 3))
    return DS_ERR_INVALID_ARG;
  if (V > DS_MAX_VOCAB || V > ds::cluster_kernel_max_vocab()) return DS_ERR_UNSUPPORTED;
  if ((long long)C * (long long)P * (long long)V > (1LL << 46)) return DS_ERR_UNSUPPORTED;

  ds::SampleArgs a;
  a.request_ids = request_ids;
  a.c = static_cast<const uint16_t*>(c_logits);
  a.u = static_cast<const uint16_t*>(u_logits);
  a.seq_lens = seq_lens;
  a.guidance = guidance;
  a.temperature = temperature;
  a.out_tokens = out_tokens;
  a.out_logprobs = out_logprobs;
  a.d_status = d_status;
  a.B = B;
  a.C = C;
  a.P = P;
  a.V = V;
  a.ratios = top_ratios;
  a.iters = iterations;
  a.keep_ties = (flags & DS_FLAG_KEEP_TIES) ? 1u : 0u;
  // scalar kept count and threshold guesses (used when no per-request ratios are given)
  a.k = top_ratios ? 1 : ds_top_k(top_ratio, V);
  // Threshold guesses: aim the candidate count a little above k so that the
  // verified count rarely falls short, and the upper count a little below.
  const double kk = (double)a.k;
  const double spread = 1.5 * std::sqrt(kk * (1.0 - kk / (double)V)) + 0.02 * kk + 4.0;
  const double target_lo = kk + spread;
  const double target_hi = kk - spread;
  a.q_lo = (target_lo >= (double)V) ? -INFINITY : (float)normal_upper_quantile(target_lo / (double)V);
  a.q_hi = (target_hi < 1.0) ? INFINITY : (float)normal_upper_quantile(target_hi / (double)V);
  // The one-warp-per-cell kernel aims closer to k: its second guess is sized
  // to the shortfall, so a short first count costs one more compaction pass
  // while every candidate beyond 32 per lane costs a noise draw per lane.
  const double target_w = kk + (std::sqrt(kk * (1.0 - kk / (double)V)) + 0.02 * kk + 2.0);
  a.q_w = (target_w >= (double)V) ? -INFINITY : (float)normal_upper_quantile(target_w / (double)V);
  a.key0 = (uint32_t)(seed & 0xffffffffull);
  a.key1 = (uint32_t)(seed >> 32);
  a.iter_hi = iterations ? 0u : (iteration << 8);
  // Philox4x32-10 key schedule: round r uses key + r * (0x9E3779B9, 0xBB67AE85).
  for (int r = 0; r < 10; ++r) {
    a.rk0[r] = a.key0 + (uint32_t)r * 0x9E3779B9u;
    a.rk1[r] = a.key1 + (uint32_t)r * 0xBB67AE85u;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (V <= ds::warp_kernel_max_vocab()) {
    const int sms = device_sm_count();
    if (sms <= 0) return DS_ERR_CUDA;
    e = ds::launch_sample_warp(a, st, sms, !(flags & DS_FLAG_SKIP_EXACT_PASS));
  } else if (top_ratios || 4LL * a.k <= (long long)V) {
    // streaming pass; the cells it cannot finish exactly are marked and
    // finished by the staged kernel right behind it on the same stream (with
    // per-request ratios every k is possible, and this pair handles each)
    e = ds::launch_sample_stream(a, st);
    if (e == cudaSuccess && !(flags & DS_FLAG_SKIP_EXACT_PASS)) e = ds::launch_sample_cluster(a, st, 1);
  } else {
    e = ds::launch_sample_cluster(a, st, 0);
  }
  return e == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

ds_status ds_sample(const int32_t* request_ids, const void* c_logits, const void* u_logits,
                    const int32_t* seq_lens, int32_t B, int32_t C, int32_t P, int32_t V,
                    const float* guidance, const float* temperature, float top_ratio,
                    uint64_t seed, uint32_t iteration, int32_t* out_tokens, float* out_logprobs,
                    uint32_t* d_status, void* stream) {
  return ds_sample_ex(request_ids, c_logits, u_logits, seq_lens, B, C, P, V, guidance, temperature, nullptr,
                      top_ratio, seed, nullptr, iteration, 0u, out_tokens, out_logprobs, d_status, stream);
}

ds_status ds_greedy_lse(const void* logits, int32_t n, int32_t V, float* out_max, float* out_lse,
                        int32_t* out_argmax, void* stream) {
  if (n < 0 || V < 1) return DS_ERR_INVALID_ARG;
  if (n == 0) return DS_OK;
  if (!logits || !out_max || !out_lse || !out_argmax) return DS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) & 1) return DS_ERR_INVALID_ARG;
  const cudaError_t e = ds::launch_greedy(static_cast<const uint16_t*>(logits), n, V, out_max, out_lse,
                                          out_argmax, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

ds_status ds_merge_triples(const float* triples, int32_t n, int32_t shards, float* out_max, float* out_lse,
                           int32_t* out_argmax, void* stream) {
  if (n < 0 || shards < 1) return DS_ERR_INVALID_ARG;
  if (n == 0) return DS_OK;
  if (!triples || !out_max || !out_lse || !out_argmax) return DS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(triples) & 3) != 0) return DS_ERR_INVALID_ARG;
  if ((long long)n * shards * 3 > (1LL << 40)) return DS_ERR_UNSUPPORTED;
  const cudaError_t e =
      ds::launch_merge_triples(triples, n, shards, out_max, out_lse, out_argmax, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

ds_status ds_log_softmax(const void* logits, int32_t n, int32_t V, void* out, int32_t out_dtype, float* out_max,
                         float* out_lse, int32_t* out_argmax, void* stream) {
  if (n < 0 || V < 1) return DS_ERR_INVALID_ARG;
  if (out_dtype != DS_DTYPE_F32 && out_dtype != DS_DTYPE_BF16) return DS_ERR_INVALID_ARG;
  if (n == 0) return DS_OK;
  if (!logits || !out || !out_max || !out_lse || !out_argmax) return DS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 1) || (reinterpret_cast<uintptr_t>(out) & (out_dtype == DS_DTYPE_F32 ? 3 : 1)))
    return DS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint16_t* x = static_cast<const uint16_t*>(logits);
  const bool bf16_out = out_dtype == DS_DTYPE_BF16;
  cudaError_t e = cudaSuccess;
  bool two_pass = !ds::log_softmax_fused_fits(V);
  if (!two_pass) {
    // the row held on chip by a cluster: one read of the logits; refused (nothing
    // launched) when no cluster of that shape fits this device
    e = ds::launch_log_softmax_fused(x, n, V, out_max, out_lse, out_argmax, out, bf16_out, st, &two_pass);
  }
  if (e == cudaSuccess && two_pass) {
    // the triple pass, then the write pass (a second read of the logits)
    e = ds::launch_greedy(x, n, V, out_max, out_lse, out_argmax, st);
    if (e == cudaSuccess) e = ds::launch_log_softmax_write(x, n, V, out_lse, out, bf16_out, st);
  }
  return e == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

ds_status ds_reveal(const float* scores, const int32_t* tokens, const int32_t* seq_lens,
                    const int32_t* reveal_counts, int32_t B, int32_t C, int32_t P, int32_t* canvas,
                    uint8_t* revealed, uint32_t* d_status, void* stream) {
  if (B < 0 || C < 0 || P < 0) return DS_ERR_INVALID_ARG;
  if (C == 0 || (B == 0 && P == 0)) return DS_OK;
  if (B == 0) return DS_ERR_INVALID_ARG;  // P > 0 positions need an owner
  if (!scores || !tokens || !seq_lens || !reveal_counts || !canvas) return DS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scores) | reinterpret_cast<uintptr_t>(tokens) |
       reinterpret_cast<uintptr_t>(canvas)) & 3)
    return DS_ERR_INVALID_ARG;
  if ((long long)C * (long long)P >= (1LL << 32)) return DS_ERR_UNSUPPORTED;
  const cudaError_t e = ds::launch_reveal(scores, tokens, seq_lens, reveal_counts, B, C, P, canvas, revealed,
                                          d_status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

}  // extern "C"
