// ds_launch.h -- internal launch entry points of the libdsample kernels.
#pragma once

#include <cuda_runtime.h>

#include "dsample.h"
#include "ds_device.cuh"

namespace ds {

constexpr int kWarpKernelThreads = 128;  // 4 warps per CTA, one cell per warp at a time

// Largest V of the one-warp-per-cell kernel and of the cluster kernel.
int warp_kernel_max_vocab();
int cluster_kernel_max_vocab();

cudaError_t launch_sample_warp(const SampleArgs& a, cudaStream_t st, int num_sms);
cudaError_t launch_sample_cluster(const SampleArgs& a, cudaStream_t st);
cudaError_t launch_greedy(const uint16_t* x, int n, int V, float* out_max, float* out_lse, int* out_argmax,
                          cudaStream_t st);

}  // namespace ds
