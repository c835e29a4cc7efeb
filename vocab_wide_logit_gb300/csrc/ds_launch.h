// ds_launch.h -- internal launch entry points of the libdsample kernels.
#pragma once

#include <cuda_runtime.h>

#include "dsample.h"
#include "ds_device.cuh"

namespace ds {

// Counts every kernel the library launches (read by ds_launch_count).
void note_launch();

// Launch-time queries (a kernel's occupancy, its shared-memory attribute, the
// SM count) cost microseconds of host time each; their answers depend only on
// the device, the kernel and its shared memory. cached(site, param, init) runs
// init(device) the first time a (site, current device, param) key is seen and
// returns its positive result from then on (a result <= 0 is an error and is
// not kept). Thread-safe.
bool cache_lookup(const void* site, int dev, long long param, int* value);
void cache_store(const void* site, int dev, long long param, int value);
template <typename F>
int cached(const void* site, long long param, F init) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  int v = 0;
  if (cache_lookup(site, dev, param, &v)) return v;
  v = init(dev);
  if (v > 0) cache_store(site, dev, param, v);
  return v;
}
// SM count of the current device (cached).
int device_sms();

constexpr int kWarpKernelThreads = 128;
constexpr int kStreamMark = DS_MARKED_TOKEN;  // out_tokens marker left by a fast pass for the exact one

// Largest V of the one-warp-per-cell kernel and of the cluster kernel.
int warp_kernel_max_vocab();
int cluster_kernel_max_vocab();

// One warp per cell: a lean pass that marks the cells it cannot settle on its
// common path (too few or too many candidates for its balanced list), then
// (exact_pass) the full kernel over the marked cells only.
cudaError_t launch_sample_warp(const SampleArgs& a, cudaStream_t st, int num_sms, bool exact_pass);

// Staged cluster kernel (z kept in shared memory); with only_marked it finishes
// just the cells the streaming kernel marked with kStreamMark.
cudaError_t launch_sample_cluster(const SampleArgs& a, cudaStream_t st, int only_marked);
// Streaming cluster kernel (candidates only in shared memory) for k well below V.
cudaError_t launch_sample_stream(const SampleArgs& a, cudaStream_t st);
cudaError_t launch_greedy(const uint16_t* x, int n, int V, float* out_max, float* out_lse, int* out_argmax,
                          cudaStream_t st);
cudaError_t launch_merge_triples(const float* triples, int n, int shards, float* out_max, float* out_lse,
                                 int* out_argmax, cudaStream_t st);
cudaError_t launch_reveal(const float* scores, const int32_t* tokens, const int32_t* seq_lens,
                          const int32_t* reveal_counts, int B, int C, int P, int32_t* canvas, uint8_t* revealed,
                          uint32_t* d_status, cudaStream_t st);
cudaError_t launch_log_softmax_write(const uint16_t* x, int n, int V, const float* lse, void* out, bool bf16_out,
                                     cudaStream_t st);

// Dense log-softmax with each row held in a cluster's shared memory (one read of
// the logits); fits when a row splits into at most 8 slices of 64 KB. When no
// cluster of the needed shape fits the device, *refused is set, nothing is
// launched and cudaSuccess is returned.
bool log_softmax_fused_fits(int V);
cudaError_t launch_log_softmax_fused(const uint16_t* x, int n, int V, float* out_max, float* out_lse,
                                     int* out_argmax, void* out, bool bf16_out, cudaStream_t st, bool* refused);

}  // namespace ds
