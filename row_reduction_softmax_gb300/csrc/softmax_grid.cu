// GRID path: a row too long for one CTA -- or for a cluster's registers --
// is split over C CTAs of a persistent, cooperative grid; each CTA keeps its
// segment in registers, and the segments' (max, sum) partials meet in global
// memory.
//
// The pages show the tile loop for rows that overflow a block only for the
// row sum ("Kernels, Triton, XLA", section "Reductions and tiling", "Row sum,
// when the row doesn't fit"); the softmax needs a max as well as a sum, so a
// segment's partial is (m_c, s_c = sum exp(x - m_c)) and partials merge by
//     m = max(m_a, m_b),   s = s_a exp(m_a - m) + s_b exp(m_b - m).
//
// Layout: G' = R * C CTAs; CTA g always holds segment c = g % C of rows
// g / C, g / C + R, g / C + 2R, ... so every round works on R whole rows and
// no row straddles two rounds.  For each of its rows a CTA
//   1. has the segment in registers (VEC float4 per thread, 128-bit loads),
//   2. forms (m_c, s_c), keeping e = exp(x - m_c) in registers, and
//      publishes the pair in the row's slot c under this launch's ticket
//      (release store),
//   3. issues the loads of its NEXT row's segment into the second register
//      buffer, so HBM stays busy through the wait,
//   4. waits (bounded) until all C slots of the row carry the ticket --
//      polling every slot at once with relaxed loads, then one acquire fence
//      -- merges them in slot order, identically in every CTA of the row, and
//      writes y = e * exp(m_c - m) / s with streaming stores.
// Every CTA publishes a round's partial before it waits in that round, all
// CTAs of a round's rows are in that round, and the cooperative launch makes
// them all resident: the waits always end.
#include "device_common.cuh"
#include "internal.h"
#include "sm100_async.cuh"

namespace rrs {

// Set when a CTA gave up waiting for its row's partials; read by rrs_device_error().
__device__ unsigned int g_grid_error = 0;

namespace {

constexpr int kT = kGridThreads;
constexpr int kW = kT / 32;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr unsigned kErrTimeout = 1u;

struct __align__(16) Slot {
  float m;
  float s;
  uint32_t ticket;
  uint32_t pad;
};

__device__ __forceinline__ float cta_max(float v, float* red, int warp, int lane) {
  v = warp_max(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const float r = warp_max((lane < kW) ? red[lane] : neg_inf());
  __syncthreads();  // `red` is rewritten by the next reduction
  return r;
}

__device__ __forceinline__ float cta_sum(float v, float* red, int warp, int lane) {
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const float r = warp_sum((lane < kW) ? red[lane] : 0.f);
  __syncthreads();
  return r;
}

template <int VEC>
__device__ __forceinline__ void load_segment(float4 (&v)[VEC], const float4* __restrict__ x4,
                                             int b4, int e4) {
  const float kNeg = neg_inf();
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const int c = b4 + i * kT + (int)threadIdx.x;
    v[i] = (c < e4) ? load_stream(x4 + c) : make_float4(kNeg, kNeg, kNeg, kNeg);
  }
}

template <int VEC>
__global__ void __launch_bounds__(kT, 2)
softmax_grid_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t M, int64_t N,
                    int64_t ld, int64_t seg, int32_t C, int32_t R, Slot* __restrict__ slots,
                    uint32_t ticket) {
  __shared__ float red[kW];
  __shared__ MaxSum whole;
  __shared__ int fail;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = (int)(blockIdx.x % C);
  const int64_t row0 = blockIdx.x / C;
  const int64_t b = (int64_t)c * seg;
  const int b4 = (int)(b >> 2);
  const int e4 = (int)(min(b + seg, N) >> 2);  // segment [b, e) relative to the row start
  if (threadIdx.x == 0) fail = 0;

  float4 cur[VEC], nxt[VEC];
  if (row0 < M) load_segment<VEC>(cur, reinterpret_cast<const float4*>(x + row0 * ld), b4, e4);

  for (int64_t row = row0; row < M; row += R) {
    // 2. the segment's partial; e = exp(x - m_c) stays in registers
    float mc = neg_inf();
#pragma unroll
    for (int i = 0; i < VEC; ++i) mc = max_nan(mc, max4(cur[i]));
    mc = cta_max(mc, red, warp, lane);
    const bool empty = (mc == neg_inf());  // only -inf in this segment (or nothing)
    float sc = 0.f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      cur[i].x = empty ? 0.f : exp_shifted(cur[i].x, mc);
      cur[i].y = empty ? 0.f : exp_shifted(cur[i].y, mc);
      cur[i].z = empty ? 0.f : exp_shifted(cur[i].z, mc);
      cur[i].w = empty ? 0.f : exp_shifted(cur[i].w, mc);
      sc += (cur[i].x + cur[i].y) + (cur[i].z + cur[i].w);
    }
    sc = cta_sum(sc, red, warp, lane);
    Slot* rs = slots + row * C;
    if (threadIdx.x == 0) {
      rs[c].m = mc;
      rs[c].s = sc;
      st_release_gpu(&rs[c].ticket, ticket);
    }

    // 3. the next row's segment is in flight while this row's partials meet
    const int64_t next = row + R;
    if (next < M) load_segment<VEC>(nxt, reinterpret_cast<const float4*>(x + next * ld), b4, e4);

    // 4. wait for the row's C partials, merge them in slot order.  Each lane
    //    polls all of its slots at once with relaxed loads; one acquire fence
    //    once every ticket is current orders the reads of (m, s) after them.
    if (warp == 0) {
      const uint64_t t0 = global_timer_ns();
      bool seen = false;
      uint32_t n = 0;
      while (true) {
        bool mine = true;
        for (int l = lane; l < C; l += 32) mine &= (ld_relaxed_gpu(&rs[l].ticket) == ticket);
        if (__all_sync(kFullMask, mine)) {
          seen = true;
          break;
        }
        if ((++n & 15u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) break;
      }
      fence_acquire_gpu();
      MaxSum acc{neg_inf(), 0.f};
      if (seen) {
        for (int l = lane; l < C; l += 32) acc = merge(acc, MaxSum{rs[l].m, rs[l].s});
      }
      acc = warp_merge(acc);  // same slots, same order in every CTA of the row
      if (lane == 0) {
        whole = acc;
        if (!seen) {
          atomicOr(&g_grid_error, kErrTimeout);
          fail = 1;
        }
      }
    }
    __syncthreads();
    if (fail) return;  // uniform: every thread reads the flag after the barrier
    const MaxSum w = whole;
    const bool bad = !(w.s == w.s) || w.m == neg_inf();  // NaN / inf / all -inf row
    const float scale = bad ? __int_as_float(0x7fc00000) : (empty ? 0.f : exp_shifted(mc, w.m) / w.s);
    float4* y4 = reinterpret_cast<float4*>(y + row * ld);
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const int cc = b4 + i * kT + (int)threadIdx.x;
      if (cc < e4) {
        store_stream(y4 + cc, make_float4(cur[i].x * scale, cur[i].y * scale, cur[i].z * scale,
                                          cur[i].w * scale));
      }
    }
#pragma unroll
    for (int i = 0; i < VEC; ++i) cur[i] = nxt[i];
    __syncthreads();  // `whole` is rewritten in the next round
  }
}

}  // namespace

cudaError_t launch_softmax_grid(const rrs_plan& p, const float* x, float* y, int64_t M, int64_t N,
                                int64_t ld, void* workspace, uint32_t ticket, cudaStream_t s) {
  if (p.threads != kT) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid, 1, 1);
  cfg.blockDim = dim3(kT, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  Slot* slots = static_cast<Slot*>(workspace);
  const int32_t C = (int32_t)p.ctas_per_row, R = p.rows_per_cta;
  switch (p.vec) {
    case 2:
      return cudaLaunchKernelEx(&cfg, softmax_grid_kernel<2>, x, y, M, N, ld, p.chunk, C, R, slots,
                                ticket);
    case 4:
      return cudaLaunchKernelEx(&cfg, softmax_grid_kernel<4>, x, y, M, N, ld, p.chunk, C, R, slots,
                                ticket);
    default:
      return cudaErrorInvalidConfiguration;
  }
}

int grid_blocks_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, softmax_grid_kernel<4>, kT, 0) != cudaSuccess)
    return 0;
  return n;
}

cudaError_t read_and_clear_grid_error(cudaStream_t s, unsigned* value) {
  unsigned host = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&host, g_grid_error, sizeof(host), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && host != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbolAsync(g_grid_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  *value = host;
  return e;
}

}  // namespace rrs
