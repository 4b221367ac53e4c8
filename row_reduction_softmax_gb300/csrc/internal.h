// Host-side interface between the C ABI (capi.cu) and the kernel translation
// units.  Not part of the public ABI: every symbol here has hidden visibility.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "rrs.h"

namespace rrs {

// Per-device facts the planner needs, queried once per device.
struct DeviceInfo {
  int sm_count = 0;
  int smem_optin = 0;       // max dynamic shared memory per CTA (opt-in), bytes
  int cluster_launch = 0;   // thread-block clusters supported
  int coop_launch = 0;      // cooperative launch supported
};

// Tuning limits shared by the planner and the launchers.
constexpr int kRowRegsMaxVec = 16;       // float4 registers per thread (warp-per-row)
constexpr int kSplitThreads = 256;       // CTA size of the cluster / two-phase kernels
constexpr int kClusterVec = 8;           // float4 per thread in a cluster CTA segment
constexpr int kClusterMax = 16;          // largest cluster (non-portable beyond 8)
constexpr int64_t kChunkAlign = 1024;    // two-phase chunk granularity (elements)

// ---- softmax launchers (return the launch's cudaError_t) ----
cudaError_t launch_softmax_row_regs(const rrs_plan& p, const float* x, float* y, int64_t M,
                                    int64_t N, int64_t ld, cudaStream_t s);
cudaError_t launch_softmax_cluster(const rrs_plan& p, const float* x, float* y, int64_t M,
                                   int64_t N, int64_t ld, cudaStream_t s);
cudaError_t launch_softmax_two_phase(const rrs_plan& p, const float* x, float* y, int64_t M,
                                     int64_t N, int64_t ld, void* workspace, cudaStream_t s);

// ---- row-sum launchers ----
cudaError_t launch_row_sum_rows(const rrs_plan& p, const float* x, float* out, int64_t M,
                                int64_t N, int64_t ld, cudaStream_t s);
cudaError_t launch_row_sum_split(const rrs_plan& p, const float* x, float* out, int64_t M,
                                 int64_t N, int64_t ld, void* workspace, cudaStream_t s);

// ---- device error word (set by kernels that wait on peers with a bound) ----
cudaError_t read_and_clear_device_error(cudaStream_t s, unsigned* value);

}  // namespace rrs
