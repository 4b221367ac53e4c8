// Elementwise GeLU, tanh approximation: y = 0.5 x (1 + tanh(a)),
// a = 0.79788456 (x + 0.044715 x^3) -- the pages' first kernel ("Kernels,
// Triton, XLA", section "GeLU three ways: the case for fusion" and the Triton
// GeLU walkthrough; "GPU High-Performance Programming", section 7.4.1), with
// the constants as printed there.
//
// Like the softmax it is HBM-bound (one 4-byte read and one 4-byte write per
// element, a few dozen flops), so the design is about bytes in flight: a
// grid of a few CTAs per SM strides over the vector in float4 units, each
// thread keeping kUnroll 128-bit loads in flight, streaming (evict-first)
// loads and stores, and a scalar tail for n % 4.
//
// Arithmetic: 0.5 (1 + tanh(a)) = 1 / (1 + e^(-2a)) exactly, so
// y = x / (1 + e^(-2a)).  This form has no cancellation where tanh(a) is near
// -1 (x well below 0), where 1 + tanh(a) computed in fp32 would lose most of
// its digits; e^(-2a) is 2^(-2a log2 e) on the SFU.  For a < -44 the
// exponential overflows to +inf and y = x / inf = -0, where the exact value
// is below 1e-37 in magnitude.
#include <algorithm>

#include "device_common.cuh"
#include "internal.h"
#include "launch_util.h"

namespace rrs {
namespace {

constexpr float kGeluC = 0.79788456f;
constexpr float kGeluK = 0.044715f;
constexpr int kGT = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ float gelu1(float x) {
  const float a = kGeluC * fmaf(kGeluK * x, x * x, x);   // c (x + k x^3)
  const float e = exp2_sfu(-2.0f * kLog2e * a);           // e^(-2a)
  return x / (1.0f + e);
}

__device__ __forceinline__ float4 gelu4(const float4& v) {
  return make_float4(gelu1(v.x), gelu1(v.y), gelu1(v.z), gelu1(v.w));
}

// V4: x and y 16-byte aligned.  Element i of x and y is read and written by
// the same thread, so x == y (in place) is safe.
template <bool V4>
__global__ void __launch_bounds__(kGT) gelu_kernel(const float* x, float* y, int64_t n) {
  pdl_entry();
  const int64_t stride = (int64_t)gridDim.x * kGT;
  const int64_t t = (int64_t)blockIdx.x * kGT + threadIdx.x;
  int64_t done = 0;
  if constexpr (V4) {
    const int64_t n4 = n >> 2;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float4* y4 = reinterpret_cast<float4*>(y);
    for (int64_t k = t; k < n4; k += stride * kUnroll) {
      float4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t idx = k + u * stride;
        if (idx < n4) v[u] = load_stream(x4 + idx);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t idx = k + u * stride;
        if (idx < n4) store_stream(y4 + idx, gelu4(v[u]));
      }
    }
    done = n4 << 2;
  }
  for (int64_t i = done + t; i < n; i += stride) store_stream(y + i, gelu1(load_stream(x + i)));
}

}  // namespace

int gelu_threads() { return kGT; }

cudaError_t launch_gelu(const float* x, float* y, int64_t n, int sm_count, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const bool v4 = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (reinterpret_cast<uintptr_t>(y) % 16 == 0);
  // enough CTAs to cover the vector once with kUnroll float4 per thread, at
  // most 8 resident CTAs per SM
  const int64_t per_cta = (int64_t)kGT * kUnroll * 4;
  const int64_t want = (n + per_cta - 1) / per_cta;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(want, 8 * (int64_t)sm_count));
  if (v4) return launch_pdl(gelu_kernel<true>, dim3((unsigned)grid), dim3(kGT), 0, s, 0, x, y, n);
  return launch_pdl(gelu_kernel<false>, dim3((unsigned)grid), dim3(kGT), 0, s, 0, x, y, n);
}

}  // namespace rrs
