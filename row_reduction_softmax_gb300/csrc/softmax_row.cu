// Single-pass row softmax with the whole row held in registers.
//
// The pages' fused kernel gives one block a whole row, loads it once with
// masked lanes set to -inf, and does max, subtract, exp, sum and divide on
// chip, so each element crosses HBM once each way ("Kernels, Triton, XLA",
// section "Reductions and tiling"; "GPU High-Performance Programming",
// section 7.5.1).  Here the unit that owns a row is a GROUP of GW warps
// (GW = 1 for rows up to 2048 floats, so short rows need no shared memory
// or barrier at all), each thread keeps VEC float4 of the row in registers
// (thread coarsening), and consecutive threads take consecutive float4 so
// every warp access is a full, coalesced 512-byte run.
#include "device_common.cuh"
#include "internal.h"
#include "launch_util.h"

namespace rrs {
namespace {

// Group-wide max / sum: warp shuffles, then one shared-memory step across the
// GW warps of the group, guarded by the group's own named barrier.
template <int GW>
__device__ __forceinline__ float group_max(float v, float* red, int gw, int lane, int bar_id) {
  v = warp_max(v);
  if constexpr (GW == 1) {
    return v;
  } else {
    if (lane == 0) red[gw] = v;
    named_barrier(bar_id, 32 * GW);
    float r = (lane < GW) ? red[lane] : neg_inf();
    return warp_max(r);
  }
}

template <int GW>
__device__ __forceinline__ float group_sum(float v, float* red, int gw, int lane, int bar_id) {
  v = warp_sum(v);
  if constexpr (GW == 1) {
    return v;
  } else {
    if (lane == 0) red[gw] = v;
    named_barrier(bar_id, 32 * GW);
    float r = (lane < GW) ? red[lane] : 0.f;
    return warp_sum(r);
  }
}

template <int GW>
__host__ __device__ constexpr int threads_for() { return (32 * GW < 128) ? 128 : 32 * GW; }

// Store of a thread's float4 slot i, in the slot layout of the kernel below.
template <bool V4, int kGT>
__device__ __forceinline__ void store_slot(float* yr, float4* yr4, int i, int gt, int n4, int N,
                                           const float4& o) {
  if constexpr (V4) {
    const int c = i * kGT + gt;
    if (c < n4) store_stream(yr4 + c, o);
  } else {
    const int j = 4 * i * kGT + gt;
    if (j < N) store_stream(yr + j, o.x);
    if (j + kGT < N) store_stream(yr + j + kGT, o.y);
    if (j + 2 * kGT < N) store_stream(yr + j + 2 * kGT, o.z);
    if (j + 3 * kGT < N) store_stream(yr + j + 3 * kGT, o.w);
  }
}

// V4: x, y 16-byte aligned, ldx % 4 == 0, ldy % 4 == 0; float4 slot i of a
// thread is columns 4 (i * groupsize + t) .. + 3, the N % 4 tail in `t`.
// !V4 (any alignment and stride): scalar loads, slot i component k is column
// (4 i + k) * groupsize + t, so every load instruction of a warp is one
// contiguous run.  Row r is owned by group (blockIdx.x * groups + group),
// striding by gridDim.x * groups.
// log_out != 0 writes log y = (x - m) - log(s) instead of y.  x == y (same
// stride) is safe: a group reads its whole row before writing it.
// The launch bound names one CTA per SM as the minimum, which leaves ptxas
// free to spend registers on the row (90 for a warp per row of 8 float4, 82
// for four warps per row): measured on GB300, 8192 x 1024 in 11.18 against
// 11.25 us with the default budget (62 registers, 8 CTAs per SM), 16384 x
// 4096 in 76.9 against 77.5 us; caps for 6 or 7 CTAs per SM were slower.
template <int VEC, int GW, bool V4>
__global__ void __launch_bounds__(threads_for<GW>(), 1)
softmax_row_regs_kernel(const float* x, float* y, int64_t M, int32_t N, int64_t ldx, int64_t ldy,
                        int32_t log_out) {
  constexpr int kThreads = threads_for<GW>();
  constexpr int kGroups = kThreads / (32 * GW);
  constexpr int kGT = 32 * GW;  // threads per group
  __shared__ float red_m[32];
  __shared__ float red_s[32];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int group = warp / GW;
  const int gw = warp % GW;
  const int gt = gw * 32 + lane;
  const int bar_id = 1 + group;
  float* gm = red_m + group * GW;
  float* gs = red_s + group * GW;

  const int n4 = N >> 2;
  const int rem = N & 3;
  const float kNeg = neg_inf();
  pdl_entry();

  for (int64_t row = (int64_t)blockIdx.x * kGroups + group; row < M;
       row += (int64_t)gridDim.x * kGroups) {
    const float* xr = x + row * ldx;
    float* yr = y + row * ldy;
    const float4* xr4 = reinterpret_cast<const float4*>(xr);
    float4* yr4 = reinterpret_cast<float4*>(yr);

    float4 v[VEC];
    float t = kNeg;
    if constexpr (V4) {
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const int c = i * kGT + gt;
        v[i] = (c < n4) ? load_last_use(xr4 + c) : make_float4(kNeg, kNeg, kNeg, kNeg);
      }
      t = (gt < rem) ? load_last_use(xr + 4 * n4 + gt) : kNeg;  // ragged tail, N % 4 != 0
    } else {
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const int j = 4 * i * kGT + gt;
        v[i].x = (j < N) ? load_last_use(xr + j) : kNeg;
        v[i].y = (j + kGT < N) ? load_last_use(xr + j + kGT) : kNeg;
        v[i].z = (j + 2 * kGT < N) ? load_last_use(xr + j + 2 * kGT) : kNeg;
        v[i].w = (j + 3 * kGT < N) ? load_last_use(xr + j + 3 * kGT) : kNeg;
      }
    }

    // (1) row max
    float m = t;
#pragma unroll
    for (int i = 0; i < VEC; ++i) m = max_nan(m, max4(v[i]));
    m = group_max<GW>(m, gm, gw, lane, bar_id);

    if (log_out) {
      // row sum of exp(x - m) with x kept, then log y = (x - m) - log(s)
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        s += (exp_shifted(v[i].x, m) + exp_shifted(v[i].y, m)) +
             (exp_shifted(v[i].z, m) + exp_shifted(v[i].w, m));
      }
      s += exp_shifted(t, m);
      s = group_sum<GW>(s, gs, gw, lane, bar_id);
      const float ls = logf(s);
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const float4 o = make_float4(log_softmax_of(v[i].x, m, ls), log_softmax_of(v[i].y, m, ls),
                                     log_softmax_of(v[i].z, m, ls), log_softmax_of(v[i].w, m, ls));
        store_slot<V4, kGT>(yr, yr4, i, gt, n4, N, o);
      }
      if (V4 && gt < rem) store_stream(yr + 4 * n4 + gt, log_softmax_of(t, m, ls));
      continue;
    }

    // (2)+(3) subtract and exponentiate in place, (4) row sum
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      v[i].x = exp_shifted(v[i].x, m);
      v[i].y = exp_shifted(v[i].y, m);
      v[i].z = exp_shifted(v[i].z, m);
      v[i].w = exp_shifted(v[i].w, m);
      s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    }
    t = exp_shifted(t, m);
    s += t;
    s = group_sum<GW>(s, gs, gw, lane, bar_id);

    // (5) divide: one reciprocal per row, then a multiply per element
    const float inv = 1.0f / s;
#pragma unroll
    for (int i = 0; i < VEC; ++i)
      store_slot<V4, kGT>(yr, yr4, i, gt, n4, N,
                          make_float4(v[i].x * inv, v[i].y * inv, v[i].z * inv, v[i].w * inv));
    if (V4 && gt < rem) store_stream(yr + 4 * n4 + gt, t * inv);
  }
}

template <int VEC, int GW>
cudaError_t launch_rr(const rrs_plan& p, const float* x, float* y, int64_t M, int64_t N,
                      const Layout& l, cudaStream_t s) {
  constexpr int kThreads = threads_for<GW>();
  if (p.threads != kThreads) return cudaErrorInvalidConfiguration;
  if (p.vector_io)
    return launch_pdl(softmax_row_regs_kernel<VEC, GW, true>, dim3((unsigned)p.grid), dim3(kThreads),
                      0, s, 0, x, y, M, (int32_t)N, l.ldx, l.ldy, (int32_t)l.log_out);
  return launch_pdl(softmax_row_regs_kernel<VEC, GW, false>, dim3((unsigned)p.grid), dim3(kThreads), 0,
                    s, 0, x, y, M, (int32_t)N, l.ldx, l.ldy, (int32_t)l.log_out);
}

}  // namespace

cudaError_t launch_softmax_row_regs(const rrs_plan& p, const float* x, float* y, int64_t M,
                                    int64_t N, const Layout& l, cudaStream_t s) {
  const int gw = p.warps_per_row;
  const int vec = p.vec;
#define RRS_RR(V, G) \
  if (vec == V && gw == G) return launch_rr<V, G>(p, x, y, M, N, l, s);
  RRS_RR(1, 1)
  RRS_RR(2, 1)
  RRS_RR(4, 1)
  RRS_RR(8, 1)
  RRS_RR(16, 1)
  RRS_RR(4, 2)
  RRS_RR(8, 2)
  RRS_RR(4, 4)
  RRS_RR(8, 4)
  RRS_RR(4, 8)
  RRS_RR(8, 8)
  RRS_RR(4, 16)
  RRS_RR(8, 16)
  RRS_RR(4, 32)
  RRS_RR(8, 32)
#undef RRS_RR
  return cudaErrorInvalidConfiguration;
}

}  // namespace rrs
