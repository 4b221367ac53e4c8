// ROW_TWO_PASS: the row softmax's two passes as work items of one launch,
// for rows the register, cluster and staged grid kernels do not take
// (unaligned rows past 131072 floats, rows past the grid's segments).
//
// Item k = (row r, chunk c), k = r S + c, covers floats [c CH, min((c + 1)
// CH, N)) of row r, S = ceil(N / CH) chunks per row.
//   Pass 1 of item k: the chunk's max, then the sum of exponentials against
//   it (the pages' softmax steps on one tile: "Kernels, Triton, XLA",
//   section "Reductions and tiling"), over the CTA, published to item k's
//   slot as two ticket-tagged 64-bit words.
//   Pass 2 of item k: one warp merges the row's S pairs (m = max(m_a, m_b),
//   s = s_a e^(m_a - m) + s_b e^(m_b - m)) in a fixed order -- every lane
//   its chunks in increasing order, then the lanes in a fixed tree -- so
//   every CTA of the row gets the same pair bit for bit, while the other
//   warps' loads of the chunk are in flight; then the chunk, re-read from
//   the L2 where pass 1 left it moments before, is normalised and written.
// CTAs take their item by arrival order through the sequence of
// two_pass_item (lag D >= S), so a pass-2 CTA waits only for pass-1 items
// drawn before it, by CTAs that run: no co-residency is needed.  Every wait
// is bounded (1 s); on timeout the error words are set and the chunk is left
// unwritten.  Every element is read by pass 1 of its chunk before pass 2
// writes it, so x == y (in place) is safe.
//
// V4: x and y 16-byte aligned, strides and N multiples of 4: float4 loads
// and stores.  Otherwise each thread's 32 floats are scalars, consecutive
// lanes on consecutive floats.
#include <climits>

#include "device_common.cuh"
#include "internal.h"
#include "launch_util.h"
#include "sm100_async.cuh"
#include "two_pass_common.cuh"

namespace rrs {

// Set by ROW_TWO_PASS CTAs that gave up a bounded wait; read by rrs_device_error().
__device__ unsigned int g_rows_two_pass_error = 0;

namespace {

constexpr int kRT = 256;                   // threads per CTA
constexpr int kRW = kRT / 32;              // warps per CTA
constexpr int kRPer = 32;                  // floats per thread
constexpr int kChunk = kRT * kRPer;        // floats per item (32 KB)
constexpr int kPoll = 4;                   // pair slots a merging lane loads at once
constexpr unsigned kErrTimeout = 1u;

__device__ void report_timeout(unsigned* host_err) {
  atomicOr(&g_rows_two_pass_error, kErrTimeout);
  if (host_err) {
    *reinterpret_cast<volatile unsigned*>(host_err) = kErrTimeout;
    __threadfence_system();
  }
}

// Thread tid's floats of a chunk: float4 q (q < 8) at 4 (tid + kRT q) in the
// vector form, scalar q (q < 32) at tid + kRT q otherwise; v[q / 4] holds
// them four to a register slot either way.
template <bool V4>
__device__ __forceinline__ void load_chunk(const float* base, int n, int tid, float4 (&v)[kRPer / 4]) {
  const float kNeg = neg_inf();
  if constexpr (V4) {
#pragma unroll
    for (int q = 0; q < kRPer / 4; ++q) {
      const int j = 4 * (tid + kRT * q);
      v[q] = (j < n) ? load_stream(reinterpret_cast<const float4*>(base + j)) : make_float4(kNeg, kNeg, kNeg, kNeg);
    }
  } else {
#pragma unroll
    for (int q = 0; q < kRPer / 4; ++q) {
      const int j = tid + kRT * 4 * q;
      v[q].x = (j < n) ? load_stream(base + j) : kNeg;
      v[q].y = (j + kRT < n) ? load_stream(base + j + kRT) : kNeg;
      v[q].z = (j + 2 * kRT < n) ? load_stream(base + j + 2 * kRT) : kNeg;
      v[q].w = (j + 3 * kRT < n) ? load_stream(base + j + 3 * kRT) : kNeg;
    }
  }
}

template <bool V4>
__device__ __forceinline__ void store_chunk(float* base, int n, int tid, const float4 (&o)[kRPer / 4]) {
  if constexpr (V4) {
#pragma unroll
    for (int q = 0; q < kRPer / 4; ++q) {
      const int j = 4 * (tid + kRT * q);
      if (j < n) store_stream(reinterpret_cast<float4*>(base + j), o[q]);
    }
  } else {
#pragma unroll
    for (int q = 0; q < kRPer / 4; ++q) {
      const int j = tid + kRT * 4 * q;
      if (j < n) store_stream(base + j, o[q].x);
      if (j + kRT < n) store_stream(base + j + kRT, o[q].y);
      if (j + 2 * kRT < n) store_stream(base + j + 2 * kRT, o[q].z);
      if (j + 3 * kRT < n) store_stream(base + j + 3 * kRT, o[q].w);
    }
  }
}

// Five CTAs per SM (48 registers): measured on one GB300 against four (55-64
// registers) with the merging lane's poll 8 words wide, 46.7 against 48.8 us
// on 32 x 2^20, 52.0 against 55.0 with those rows off a 16-byte boundary,
// 286 against 310 on 1024 x 200001 unaligned; six (40 registers) spill and
// lose on the unaligned shapes.
template <bool V4, bool LOG>
__global__ void __launch_bounds__(kRT, 5)
softmax_rows_two_pass_kernel(const float* x, float* y, int64_t M, int64_t N, int64_t ldx, int64_t ldy,
                             int64_t S, int64_t D, unsigned long long* __restrict__ arrivals,
                             uint64_t* __restrict__ slots, int32_t fault, unsigned* host_err) {
  __shared__ float red[kRW];
  __shared__ MaxSum whole;
  __shared__ unsigned drawn[2];   // arrival index, ticket
  __shared__ int gave_up;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // every CTA draws before it lets the next kernel on the stream launch
  if (tid == 0) {
    drawn[0] = draw_arrival(arrivals, gridDim.x, &drawn[1]);
    gave_up = 0;
  }
  __syncthreads();
  pdl_entry();
  const uint32_t ticket = drawn[1];
  int pass;
  int64_t k;
  two_pass_item((int64_t)drawn[0], M * S, D, &pass, &k);
  const int64_t r = (int64_t)((uint32_t)k / (uint32_t)S);   // both below 2^31 (checked at launch)
  const int64_t c0 = (k - r * S) * kChunk;
  const int n = (int)min((int64_t)kChunk, N - c0);   // floats of this chunk
  const float* xb = x + r * ldx + c0;
  float* yb = y + r * ldy + c0;
  const float kNeg = neg_inf();
  const uint64_t log2e2 = f2_pack(kLog2e, kLog2e);
  float4 v[kRPer / 4];

  if (pass == 1) {
    load_chunk<V4>(xb, n, tid, v);
    float m = kNeg;
#pragma unroll
    for (int q = 0; q < kRPer / 4; ++q) m = max_nan(max_nan(m, max_nan(v[q].x, v[q].y)), max_nan(v[q].z, v[q].w));
    m = warp_max(m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < kRW; ++w) m = max_nan(m, red[w]);
    __syncthreads();   // red is rewritten below
    // exponentials against the chunk max (a chunk of -inf alone adds 0)
    const float sh = (m == kNeg) ? 0.f : -m;
    const uint64_t nm = f2_pack(sh, sh);
    uint64_t s2 = f2_pack(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kRPer / 4; ++q) {
      s2 = f2_add(s2, exp_shifted2(v[q].x, v[q].y, nm, log2e2));
      s2 = f2_add(s2, exp_shifted2(v[q].z, v[q].w, nm, log2e2));
    }
    float sa, sb;
    f2_unpack(s2, sa, sb);
    float s = warp_sum(sa + sb);
    if (lane == 0) red[warp] = s;
    __syncthreads();
    if (tid == 0 && !(fault != 0 && k == 0)) {   // fault: item 0's pair never appears
      s = 0.f;
#pragma unroll
      for (int w = 0; w < kRW; ++w) s += red[w];
      uint64_t* sl = slots + 2 * k;
      publish_gpu_u64(sl, tagged_word(ticket, m));
      publish_gpu_u64(sl + 1, tagged_word(ticket, s));
    }
    return;
  }

  // ---- pass 2: warps 1..7 load the chunk while warp 0 merges the row's
  // pairs (separate branches: the poll words and a chunk do not fit the
  // register budget together); warp 0 loads after the merge ----
  if (warp != 0) {
    load_chunk<V4>(xb, n, tid, v);
  } else {
    const uint64_t* rs = slots + 2 * (r * S);
    MaxSum acc{kNeg, 0.f};
    bool ok = true;
    const uint64_t t0 = global_timer_ns();
    for (int64_t b0 = 0; b0 < S && ok; b0 += 32 * kPoll) {
      uint64_t wm[kPoll], ws[kPoll];
      for (uint32_t polls = 1;; ++polls) {
        bool mine = true;
#pragma unroll
        for (int u = 0; u < kPoll; ++u) {
          const int64_t i = b0 + lane + 32 * u;
          wm[u] = (i < S) ? ld_relaxed_gpu_u64(rs + 2 * i) : tagged_word(ticket, kNeg);
          ws[u] = (i < S) ? ld_relaxed_gpu_u64(rs + 2 * i + 1) : tagged_word(ticket, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kPoll; ++u)
          mine &= ((uint32_t)(wm[u] >> 32) == ticket) && ((uint32_t)(ws[u] >> 32) == ticket);
        if (__all_sync(kFullMask, mine)) break;
        // one vote, so the warp leaves together
        if ((polls & 15u) == 0 && __any_sync(kFullMask, global_timer_ns() - t0 > kTwoPassWaitNs)) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
#pragma unroll
      for (int u = 0; u < kPoll; ++u)
        acc = merge(acc, MaxSum{__uint_as_float((uint32_t)wm[u]), __uint_as_float((uint32_t)ws[u])});
    }
    // the lanes in a fixed tree; lane 0 holds the row's pair
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      MaxSum q;
      q.m = __shfl_down_sync(kFullMask, acc.m, o);
      q.s = __shfl_down_sync(kFullMask, acc.s, o);
      if (lane < o) acc = merge(acc, q);
    }
    if (lane == 0) {
      whole = acc;
      if (!ok) {
        report_timeout(host_err);
        gave_up = 1;
      }
    }
  }
  __syncthreads();
  if (gave_up) return;
  if (warp == 0) load_chunk<V4>(xb, n, tid, v);
  const MaxSum w = whole;
  if constexpr (LOG) {   // (x - m) - log s
    const float ls = logf(w.s);
#pragma unroll
    for (int q = 0; q < kRPer / 4; ++q)
      v[q] = make_float4(log_softmax_of(v[q].x, w.m, ls), log_softmax_of(v[q].y, w.m, ls),
                         log_softmax_of(v[q].z, w.m, ls), log_softmax_of(v[q].w, w.m, ls));
  } else {
    const bool bad = !(w.s == w.s) || w.m == kNeg;   // NaN / inf / all -inf row
    const float inv = bad ? __int_as_float(0x7fc00000) : 1.0f / w.s;
    const uint64_t nwm = f2_pack(-w.m, -w.m), inv2 = f2_pack(inv, inv);
#pragma unroll
    for (int q = 0; q < kRPer / 4; ++q) {
      float4 o;
      f2_unpack(f2_mul(exp_shifted2(v[q].x, v[q].y, nwm, log2e2), inv2), o.x, o.y);
      f2_unpack(f2_mul(exp_shifted2(v[q].z, v[q].w, nwm, log2e2), inv2), o.z, o.w);
      v[q] = o;
    }
  }
  store_chunk<V4>(yb, n, tid, v);
}

}  // namespace

int rows_two_pass_threads() { return kRT; }
int rows_two_pass_chunk() { return kChunk; }

cudaError_t launch_softmax_rows_two_pass(const rrs_plan& p, const float* x, float* y, int64_t M, int64_t N,
                                         const Layout& l, void* workspace, int fault, unsigned* host_err,
                                         cudaStream_t s) {
  const int64_t S = p.ctas_per_row, D = p.stages;
  if (p.threads != kRT || p.chunk != kChunk || S != (N + kChunk - 1) / kChunk || D < S || D > M * S ||
      p.grid != 2 * M * S || p.grid > (int64_t)INT_MAX || (p.vector_io && (N % 4 != 0 || l.ldx % 4 != 0 || l.ldy % 4 != 0)))
    return cudaErrorInvalidConfiguration;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  auto* arrivals = reinterpret_cast<unsigned long long*>(ws);
  uint64_t* slots = reinterpret_cast<uint64_t*>(ws + kRowsTwoPassArrivalBytes);
  const dim3 grid((unsigned)p.grid), block(kRT);
  auto k = p.vector_io ? (l.log_out ? softmax_rows_two_pass_kernel<true, true> : softmax_rows_two_pass_kernel<true, false>)
                       : (l.log_out ? softmax_rows_two_pass_kernel<false, true> : softmax_rows_two_pass_kernel<false, false>);
  return launch_pdl(k, grid, block, 0, s, 0, x, y, M, N, l.ldx, l.ldy, S, D, arrivals, slots, (int32_t)fault,
                    host_err);
}

cudaError_t read_and_clear_rows_two_pass_error(cudaStream_t s, unsigned* value) {
  unsigned host = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&host, g_rows_two_pass_error, sizeof(host), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && host != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbolAsync(g_rows_two_pass_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  *value = host;
  return e;
}

}  // namespace rrs
