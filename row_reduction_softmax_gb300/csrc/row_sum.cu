// Row sum: out[i] = sum_j x[i, j].
//
// The pages' version ("Kernels, Triton, XLA", section "Reductions and
// tiling", paragraph "Row sum, when the row doesn't fit"; "GPU
// High-Performance Programming", section 7.5.1) gives one block a row, sweeps
// the row tile by tile into a vector of per-thread accumulators (masked lanes
// add 0) and reduces that vector to a scalar at the end.  Here:
//  * ROW   -- a group of GW warps owns a row (GW = 1 for short rows, several
//    rows per CTA); each thread keeps 4 x kUnroll fp32 accumulators fed by
//    128-bit loads, kUnroll loads in flight per step; then a fixed-order
//    shuffle / shared-memory tree.  Bitwise reproducible.
//  * SPLIT -- for few long rows: CTAs sum fixed chunks into a workspace and a
//    second kernel adds a row's chunk sums in index order.
#include "device_common.cuh"
#include "internal.h"
#include "launch_util.h"

namespace rrs {
namespace {

constexpr int kUnroll = 4;

template <int GW>
__host__ __device__ constexpr int sum_threads() { return (32 * GW < 128) ? 128 : 32 * GW; }

// Sum of columns [b, e) of row xr by `nthr` threads (thread index t),
// b a multiple of 4 when V4.  Per-thread accumulators, fixed order.
template <bool V4>
__device__ __forceinline__ float thread_range_sum(const float* __restrict__ xr, int64_t b, int64_t e,
                                                  int64_t N, int t, int nthr) {
  float4 acc[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
  int64_t scalar_from = b;
  if constexpr (V4) {
    const int64_t e4 = ((e == N) ? (N & ~int64_t(3)) : e) >> 2;
    const float4* x4 = reinterpret_cast<const float4*>(xr);
    for (int64_t k = (b >> 2) + t; k < e4; k += (int64_t)nthr * kUnroll) {
      float4 a[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t idx = k + (int64_t)u * nthr;
        a[u] = (idx < e4) ? load_stream(x4 + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        acc[u].x += a[u].x;
        acc[u].y += a[u].y;
        acc[u].z += a[u].z;
        acc[u].w += a[u].w;
      }
    }
    scalar_from = e4 << 2;
  }
  for (int64_t j = scalar_from + t; j < e; j += (int64_t)nthr * kUnroll) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t idx = j + (int64_t)u * nthr;
      if (idx < e) acc[u].x += load_stream(xr + idx);
    }
  }
  float s = 0.f;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) s += (acc[u].x + acc[u].y) + (acc[u].z + acc[u].w);
  return s;
}

template <int GW, bool V4>
__global__ void __launch_bounds__(sum_threads<GW>())
row_sum_rows_kernel(const float* __restrict__ x, float* __restrict__ out, int64_t M, int64_t N,
                    int64_t ld) {
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
    float s = thread_range_sum<V4>(x + row * ld, 0, N, N, gt, 32 * GW);
    s = warp_sum(s);
    if constexpr (GW > 1) {
      if (lane == 0) gred[gw] = s;
      named_barrier(1 + group, 32 * GW);
      s = warp_sum((lane < GW) ? gred[lane] : 0.f);
      named_barrier(1 + group, 32 * GW);  // gred is rewritten by the next row
    }
    if (gt == 0) out[row] = s;
  }
}

constexpr int kSplitT = 256;

template <bool V4>
__global__ void __launch_bounds__(kSplitT)
row_sum_partials_kernel(const float* __restrict__ x, float* __restrict__ part, int64_t M,
                        int64_t N, int64_t ld, int64_t chunk, int64_t C) {
  __shared__ float red[kSplitT / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_entry();
  for (int64_t w = blockIdx.x; w < M * C; w += gridDim.x) {
    const int64_t row = w / C;
    const int64_t c = w - row * C;
    const int64_t b = c * chunk;
    const int64_t e = min(b + chunk, N);
    float s = warp_sum(thread_range_sum<V4>(x + row * ld, b, e, N, threadIdx.x, kSplitT));
    if (lane == 0) red[warp] = s;
    __syncthreads();
    s = warp_sum((lane < kSplitT / 32) ? red[lane] : 0.f);
    if (threadIdx.x == 0) part[w] = s;
    __syncthreads();
  }
}

// One warp per row adds the row's C chunk sums: lane l takes chunks
// l, l + 32, ... in order, then a fixed shuffle tree.
__global__ void __launch_bounds__(128)
row_sum_finalize_kernel(const float* __restrict__ part, float* __restrict__ out, int64_t M,
                        int64_t C) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * 4;
  pdl_entry();
  for (int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5); row < M; row += warps) {
    float s = 0.f;
    for (int64_t k = lane; k < C; k += 32) s += part[row * C + k];
    s = warp_sum(s);
    if (lane == 0) out[row] = s;
  }
}

template <int GW>
cudaError_t launch_rows_gw(const rrs_plan& p, const float* x, float* out, int64_t M, int64_t N,
                           int64_t ld, cudaStream_t s) {
  constexpr int kThreads = sum_threads<GW>();
  if (p.threads != kThreads) return cudaErrorInvalidConfiguration;
  if (p.vector_io)
    return launch_pdl(row_sum_rows_kernel<GW, true>, dim3((unsigned)p.grid), dim3(kThreads), 0, s, 0,
                      x, out, M, N, ld);
  return launch_pdl(row_sum_rows_kernel<GW, false>, dim3((unsigned)p.grid), dim3(kThreads), 0, s, 0,
                    x, out, M, N, ld);
}

}  // namespace

cudaError_t launch_row_sum_rows(const rrs_plan& p, const float* x, float* out, int64_t M,
                                int64_t N, int64_t ld, cudaStream_t s) {
  switch (p.warps_per_row) {
    case 1: return launch_rows_gw<1>(p, x, out, M, N, ld, s);
    case 2: return launch_rows_gw<2>(p, x, out, M, N, ld, s);
    case 4: return launch_rows_gw<4>(p, x, out, M, N, ld, s);
    case 8: return launch_rows_gw<8>(p, x, out, M, N, ld, s);
    case 16: return launch_rows_gw<16>(p, x, out, M, N, ld, s);
    case 32: return launch_rows_gw<32>(p, x, out, M, N, ld, s);
    default: return cudaErrorInvalidConfiguration;
  }
}

cudaError_t launch_row_sum_split(const rrs_plan& p, const float* x, float* out, int64_t M,
                                 int64_t N, int64_t ld, void* workspace, cudaStream_t s) {
  if (p.threads != kSplitT) return cudaErrorInvalidConfiguration;
  float* part = static_cast<float*>(workspace);
  const dim3 grid((unsigned)p.grid), block(kSplitT);
  cudaError_t e = p.vector_io
                      ? launch_pdl(row_sum_partials_kernel<true>, grid, block, 0, s, 0, x, part, M,
                                   N, ld, p.chunk, p.ctas_per_row)
                      : launch_pdl(row_sum_partials_kernel<false>, grid, block, 0, s, 0, x, part, M,
                                   N, ld, p.chunk, p.ctas_per_row);
  if (e != cudaSuccess) return e;
  const int64_t fin_grid = (M + 3) / 4;
  return launch_pdl(row_sum_finalize_kernel, dim3((unsigned)(fin_grid < 65535 ? fin_grid : 65535)),
                    dim3(128), 0, s, 0, static_cast<const float*>(part), out, M, p.ctas_per_row);
}

}  // namespace rrs
