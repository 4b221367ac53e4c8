// Row reductions: out[i] = sum_j x[i, j] (row_sum), max_j x[i, j] (row_max)
// and sum_j x[i, j] / N (row_mean).
//
// The pages' row sum ("Kernels, Triton, XLA", section "Reductions and
// tiling", paragraph "Row sum, when the row doesn't fit"; "GPU
// High-Performance Programming", section 7.5.1) gives one block a row, sweeps
// the row tile by tile into a vector of per-thread accumulators (masked lanes
// add the identity) and reduces that vector to a scalar at the end.  The row
// max is the first of the naive softmax's five steps (same section, the
// softmax paragraph); the mean is the sum divided by N.  All three share one
// skeleton, templated on the combining operation:
//  * ROW   -- a group of GW warps owns a row (GW = 1 for short rows, several
//    rows per CTA); each thread keeps 4 x kUnroll fp32 accumulators fed by
//    128-bit loads, kUnroll loads in flight per step; then a fixed-order
//    shuffle / shared-memory tree.  Bitwise reproducible.
//  * SPLIT -- for few long rows: CTAs reduce fixed chunks into a workspace and
//    a second kernel combines a row's chunk results in index order.
#include <algorithm>

#include "device_common.cuh"
#include "internal.h"
#include "launch_util.h"

namespace rrs {
namespace {

constexpr int kUnroll = 4;

// The combining operation: sum (row_sum, row_mean) or NaN-propagating max.
template <int OP>
struct Reduce {
  static __device__ __forceinline__ float identity() { return OP == kOpMax ? neg_inf() : 0.f; }
  static __device__ __forceinline__ float combine(float a, float b) {
    return OP == kOpMax ? max_nan(a, b) : a + b;
  }
  static __device__ __forceinline__ float warp(float v) {
    return OP == kOpMax ? warp_max(v) : warp_sum(v);
  }
  // The row's result from its reduced value: the mean divides by N (in
  // double, so N above 2^24 is exact; one division per row).
  static __device__ __forceinline__ float finish(float v, int64_t N) {
    return OP == kOpMean ? (float)((double)v / (double)N) : v;
  }
};

template <int GW>
__host__ __device__ constexpr int sum_threads() { return (32 * GW < 128) ? 128 : 32 * GW; }

// Reduction of columns [b, e) of row xr by `nthr` threads (thread index t),
// b a multiple of 4 when V4.  Per-thread accumulators, fixed order.
template <int OP, bool V4>
__device__ __forceinline__ float thread_range_reduce(const float* __restrict__ xr, int64_t b,
                                                     int64_t e, int64_t N, int t, int nthr) {
  using R = Reduce<OP>;
  const float id = R::identity();
  float4 acc[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) acc[u] = make_float4(id, id, id, id);
  int64_t scalar_from = b;
  if constexpr (V4) {
    const int64_t e4 = ((e == N) ? (N & ~int64_t(3)) : e) >> 2;
    const float4* x4 = reinterpret_cast<const float4*>(xr);
    for (int64_t k = (b >> 2) + t; k < e4; k += (int64_t)nthr * kUnroll) {
      float4 a[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t idx = k + (int64_t)u * nthr;
        a[u] = (idx < e4) ? load_stream(x4 + idx) : make_float4(id, id, id, id);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        acc[u].x = R::combine(acc[u].x, a[u].x);
        acc[u].y = R::combine(acc[u].y, a[u].y);
        acc[u].z = R::combine(acc[u].z, a[u].z);
        acc[u].w = R::combine(acc[u].w, a[u].w);
      }
    }
    scalar_from = e4 << 2;
  }
  for (int64_t j = scalar_from + t; j < e; j += (int64_t)nthr * kUnroll) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t idx = j + (int64_t)u * nthr;
      if (idx < e) acc[u].x = R::combine(acc[u].x, load_stream(xr + idx));
    }
  }
  float s = id;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u)
    s = R::combine(s, R::combine(R::combine(acc[u].x, acc[u].y), R::combine(acc[u].z, acc[u].w)));
  return s;
}

template <int OP, int GW, bool V4>
__global__ void __launch_bounds__(sum_threads<GW>())
row_reduce_rows_kernel(const float* __restrict__ x, float* __restrict__ out, int64_t M, int64_t N,
                       int64_t ld) {
  using R = Reduce<OP>;
  constexpr int kThreads = sum_threads<GW>();
  constexpr int kGroups = kThreads / (32 * GW);
  __shared__ float red[32];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int group = warp / GW;
  const int gw = warp % GW;
  const int gt = gw * 32 + lane;
  float* gred = red + group * GW;
  pdl_entry();

  for (int64_t row = (int64_t)blockIdx.x * kGroups + group; row < M;
       row += (int64_t)gridDim.x * kGroups) {
    float s = thread_range_reduce<OP, V4>(x + row * ld, 0, N, N, gt, 32 * GW);
    s = R::warp(s);
    if constexpr (GW > 1) {
      if (lane == 0) gred[gw] = s;
      named_barrier(1 + group, 32 * GW);
      s = R::warp((lane < GW) ? gred[lane] : R::identity());
      named_barrier(1 + group, 32 * GW);  // gred is rewritten by the next row
    }
    if (gt == 0) out[row] = R::finish(s, N);
  }
}

constexpr int kSplitT = 256;

template <int OP, bool V4>
__global__ void __launch_bounds__(kSplitT)
row_reduce_partials_kernel(const float* __restrict__ x, float* __restrict__ part, int64_t M,
                           int64_t N, int64_t ld, int64_t chunk, int64_t C) {
  using R = Reduce<OP>;
  __shared__ float red[kSplitT / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_entry();
  for (int64_t w = blockIdx.x; w < M * C; w += gridDim.x) {
    const int64_t row = w / C;
    const int64_t c = w - row * C;
    const int64_t b = c * chunk;
    const int64_t e = min(b + chunk, N);
    float s = R::warp(thread_range_reduce<OP, V4>(x + row * ld, b, e, N, threadIdx.x, kSplitT));
    if (lane == 0) red[warp] = s;
    __syncthreads();
    s = R::warp((lane < kSplitT / 32) ? red[lane] : R::identity());
    if (threadIdx.x == 0) part[w] = s;
    __syncthreads();
  }
}

// One warp per row combines the row's C chunk results: lane l takes chunks
// l, l + 32, ... in order, then a fixed shuffle tree.
template <int OP>
__global__ void __launch_bounds__(128)
row_reduce_finalize_kernel(const float* __restrict__ part, float* __restrict__ out, int64_t M,
                           int64_t C, int64_t N) {
  using R = Reduce<OP>;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * 4;
  pdl_entry();
  for (int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5); row < M; row += warps) {
    float s = R::identity();
    for (int64_t k = lane; k < C; k += 32) s = R::combine(s, part[row * C + k]);
    s = R::warp(s);
    if (lane == 0) out[row] = R::finish(s, N);
  }
}

// out[i] = v for i < M (the result of an empty row: 0, -inf or NaN).
__global__ void __launch_bounds__(256) fill_kernel(float* __restrict__ out, int64_t M, float v) {
  pdl_entry();
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < M; i += (int64_t)gridDim.x * 256)
    out[i] = v;
}

template <int OP, int GW>
cudaError_t launch_rows_gw(const rrs_plan& p, const float* x, float* out, int64_t M, int64_t N,
                           int64_t ld, cudaStream_t s) {
  constexpr int kThreads = sum_threads<GW>();
  if (p.threads != kThreads) return cudaErrorInvalidConfiguration;
  if (p.vector_io)
    return launch_pdl(row_reduce_rows_kernel<OP, GW, true>, dim3((unsigned)p.grid), dim3(kThreads), 0,
                      s, 0, x, out, M, N, ld);
  return launch_pdl(row_reduce_rows_kernel<OP, GW, false>, dim3((unsigned)p.grid), dim3(kThreads), 0,
                    s, 0, x, out, M, N, ld);
}

template <int OP>
cudaError_t launch_rows_op(const rrs_plan& p, const float* x, float* out, int64_t M, int64_t N,
                           int64_t ld, cudaStream_t s) {
  switch (p.warps_per_row) {
    case 1: return launch_rows_gw<OP, 1>(p, x, out, M, N, ld, s);
    case 2: return launch_rows_gw<OP, 2>(p, x, out, M, N, ld, s);
    case 4: return launch_rows_gw<OP, 4>(p, x, out, M, N, ld, s);
    case 8: return launch_rows_gw<OP, 8>(p, x, out, M, N, ld, s);
    case 16: return launch_rows_gw<OP, 16>(p, x, out, M, N, ld, s);
    case 32: return launch_rows_gw<OP, 32>(p, x, out, M, N, ld, s);
    default: return cudaErrorInvalidConfiguration;
  }
}

template <int OP>
cudaError_t launch_split_op(const rrs_plan& p, const float* x, float* out, int64_t M, int64_t N,
                            int64_t ld, void* workspace, cudaStream_t s) {
  if (p.threads != kSplitT) return cudaErrorInvalidConfiguration;
  float* part = static_cast<float*>(workspace);
  const dim3 grid((unsigned)p.grid), block(kSplitT);
  cudaError_t e = p.vector_io
                      ? launch_pdl(row_reduce_partials_kernel<OP, true>, grid, block, 0, s, 0, x,
                                   part, M, N, ld, p.chunk, p.ctas_per_row)
                      : launch_pdl(row_reduce_partials_kernel<OP, false>, grid, block, 0, s, 0, x,
                                   part, M, N, ld, p.chunk, p.ctas_per_row);
  if (e != cudaSuccess) return e;
  const int64_t fin_grid = (M + 3) / 4;
  return launch_pdl(row_reduce_finalize_kernel<OP>,
                    dim3((unsigned)(fin_grid < 65535 ? fin_grid : 65535)), dim3(128), 0, s, 0,
                    static_cast<const float*>(part), out, M, p.ctas_per_row, N);
}

}  // namespace

cudaError_t launch_row_reduce_rows(int op, const rrs_plan& p, const float* x, float* out,
                                   int64_t M, int64_t N, int64_t ld, cudaStream_t s) {
  switch (op) {
    case kOpSum: return launch_rows_op<kOpSum>(p, x, out, M, N, ld, s);
    case kOpMax: return launch_rows_op<kOpMax>(p, x, out, M, N, ld, s);
    case kOpMean: return launch_rows_op<kOpMean>(p, x, out, M, N, ld, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_row_reduce_split(int op, const rrs_plan& p, const float* x, float* out,
                                    int64_t M, int64_t N, int64_t ld, void* workspace,
                                    cudaStream_t s) {
  switch (op) {
    case kOpSum: return launch_split_op<kOpSum>(p, x, out, M, N, ld, workspace, s);
    case kOpMax: return launch_split_op<kOpMax>(p, x, out, M, N, ld, workspace, s);
    case kOpMean: return launch_split_op<kOpMean>(p, x, out, M, N, ld, workspace, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fill(float* out, int64_t M, float v, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((M + 255) / 256, 1024);
  return launch_pdl(fill_kernel, dim3((unsigned)blocks), dim3(256), 0, s, 0, out, M, v);
}

}  // namespace rrs
