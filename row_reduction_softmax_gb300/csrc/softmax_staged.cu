// Persistent, TMA-staged softmax kernels.
//
// The pages' fused softmax reads each row into on-chip memory once, reduces
// it there and writes it once ("Kernels, Triton, XLA", section "Reductions
// and tiling"); their row sum shows the tile loop for rows that overflow one
// block (same section, "Row sum, when the row doesn't fit").  On GB300 the
// HBM stream is kept busy by decoupling the loads from the arithmetic:
//
//  * one CTA per SM (the grid never has a tail wave: every CTA gets the same
//    number of rows, +-1) runs a PRODUCER warp whose lanes issue 1-D bulk
//    async copies (the TMA engine) of row data into a ring of NS
//    shared-memory stages, each guarded by a "full" and an "empty" mbarrier
//    (small copies are issued from several lanes: one lane issues them at
//    only about one per 0.3 us);
//  * sixteen CONSUMER warps wait on "full", pull the stage into registers or
//    read it in place, reduce, and write y with 128-bit streaming stores,
//    then arrive on "empty" so the producer can refill the stage.
//
// Two kernels:
//  * staged_rows -- rows of at most 8192 floats.  A group of GW warps owns a
//    row; the stage is released as soon as the row sits in registers.
//    Stage s is always filled by producer lane s % G and drained by consumer
//    group s % G (G groups, NS a multiple of G), so each stage's uses are
//    ordered by one lane and one group -- which the parity waits need: a
//    wait for use u of a stage must never start before use u - 1 completed.
//  * staged_long -- rows up to about 32K floats: a whole row is staged as up
//    to four sub-tiles that stay resident while the next row's sub-tiles
//    stream in; pass 1 takes the row max, pass 2 the sum of exp(x - max),
//    pass 3 normalises from shared memory and releases the stages.
//  * staged_grid -- rows longer than a cluster's registers: each row is cut
//    into C segments held by C co-resident CTAs; a segment's (max, sum)
//    partial goes to a ticketed global slot, and each CTA publishes the next
//    row's partial before it waits for the current row's C partials, so the
//    exchange overlaps useful work while the ring keeps prefetching.
//
// Every wait is bounded (1 s, %globaltimer).  On timeout a kernel sets the
// device error word, makes the rest of its CTA stop, waits (bounded) for the
// copies it has in flight and returns; rrs_device_error() reports it.
#include <mutex>
#include <set>
#include <utility>

#include "device_common.cuh"
#include "internal.h"
#include "launch_util.h"
#include "sm100_async.cuh"

namespace rrs {

// Set by kernels that gave up a bounded wait; read by rrs_device_error().
__device__ unsigned int g_device_error = 0;

namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;  // + the producer warp
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kConsumerBar = 1;            // named barrier of the consumer threads
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrConfig = 2u;        // a launch whose stage count breaks the ring's rules

// Dynamic shared memory layout: a fixed header, then the NS stages.
constexpr int kMaxStages = 64;
constexpr int kFullOff = 0;                        // uint64_t[kMaxStages]
constexpr int kEmptyOff = kFullOff + 8 * kMaxStages;
constexpr int kAbortOff = kEmptyOff + 8 * kMaxStages;  // int
constexpr int kFailOff = kAbortOff + 16;               // int
constexpr int kRedMOff = kFailOff + 16;                // float[32]
constexpr int kRedSOff = kRedMOff + 128;               // float[32]
constexpr int kWholeOff = kRedSOff + 128;              // MaxSum
constexpr int kArrivalOff = kWholeOff + 16;            // int[2] (GRID: arrival index, ticket)
constexpr int kHeaderBytes = 2048;
static_assert(kArrivalOff + 16 <= kHeaderBytes, "header overflow");

// A wait ran out: set the device error word and, when the launch was given
// one, the host-visible word (pinned, mapped host memory the library checks
// at the start of later calls without synchronising).
__device__ void report_timeout(unsigned* host_err) {
  atomicOr(&g_device_error, kErrTimeout);
  if (host_err) {
    *reinterpret_cast<volatile unsigned*>(host_err) = kErrTimeout;
    __threadfence_system();
  }
}

// Bounded wait on an mbarrier phase.  False on timeout (error words and the
// CTA's abort flag set) or if another thread of the CTA already aborted.
__device__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                             unsigned* host_err = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        report_timeout(host_err);
        *abort_flag = 1;
        return false;
      }
    }
  }
  return true;
}

// After an abort: wait (bounded, one deadline) for the last copies the
// producer issued, so none lands in shared memory after the CTA exits.
__device__ void drain_copies(uint64_t* full, int64_t issued, int NS) {
  const uint64_t t0 = global_timer_ns();
  const int64_t first = issued > NS ? issued - NS : 0;
  for (int64_t q = first; q < issued; ++q) {
    const int s = (int)(q % NS);
    const uint32_t parity = (uint32_t)((q / NS) & 1);
    while (!mbar_try_wait(&full[s], parity)) {
      if (global_timer_ns() - t0 > kWaitLimitNs) return;
    }
  }
}

__device__ __forceinline__ void init_barriers(unsigned char* smem, int NS, uint32_t empty_count) {
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kFullOff);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + kEmptyOff);
  for (int s = 0; s < NS; ++s) {
    mbar_init(&full[s], 1);
    mbar_init(&empty[s], empty_count);
  }
  *reinterpret_cast<volatile int*>(smem + kAbortOff) = 0;
  *reinterpret_cast<volatile int*>(smem + kFailOff) = 0;
  fence_mbar_init();
}

template <int GW>
__device__ __forceinline__ float group_max(float v, float* red, int g, int gw, int lane) {
  v = warp_max(v);
  if constexpr (GW == 1) {
    return v;
  } else {
    if (lane == 0) red[g * GW + gw] = v;
    named_barrier(1 + g, 32 * GW);
    return warp_max((lane < GW) ? red[g * GW + lane] : neg_inf());
  }
}

template <int GW>
__device__ __forceinline__ float group_sum(float v, float* red, int g, int gw, int lane) {
  v = warp_sum(v);
  if constexpr (GW == 1) {
    return v;
  } else {
    if (lane == 0) red[g * GW + gw] = v;
    named_barrier(1 + g, 32 * GW);
    return warp_sum((lane < GW) ? red[g * GW + lane] : 0.f);
  }
}

// ------------------------------------------------------------ staged_rows ---
// Rows b, b + G, b + 2G, ... of CTA b (G = gridDim.x); local row j sits in
// stage j % NS, is issued by producer lane j % kGroups and consumed by warp
// group j % kGroups (NS % kGroups == 0).  Needs N % 4 == 0, 16-byte aligned
// x and y, ldx % 4 == 0, ldy % 4 == 0, N <= 32 * GW * VEC * 4.  x == y (in
// place) is safe: copies only ever read rows that are not yet written.
template <int VEC, int GW>
__global__ void __launch_bounds__(kThreads, 1)
softmax_staged_rows_kernel(const float* x, float* y, int64_t M, int32_t N, int64_t ldx,
                           int64_t ldy, int32_t NS, int32_t stage_stride) {
  constexpr int kGroups = kConsumerWarps / GW;
  constexpr int kGT = 32 * GW;
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kFullOff);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + kEmptyOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  float* red_m = reinterpret_cast<float*>(smem + kRedMOff);
  float* red_s = reinterpret_cast<float*>(smem + kRedSOff);
  unsigned char* stages = smem + kHeaderBytes;

  if (NS < kGroups || NS > kMaxStages || NS % kGroups != 0) {  // uniform: every thread returns
    if (threadIdx.x == 0) atomicOr(&g_device_error, kErrConfig);
    return;
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) init_barriers(smem, NS, GW);
  __syncthreads();
  pdl_entry();

  const int64_t G = gridDim.x;
  const int64_t b = blockIdx.x;
  const int64_t my_rows = (M > b) ? (M - b + G - 1) / G : 0;
  const uint32_t row_bytes = (uint32_t)N * 4u;

  if (warp == kProducerWarp) {
    if (lane < kGroups) {
      const uint64_t pol = l2_evict_first_policy();
      int64_t j = lane;
      bool ok = true;
      for (; j < my_rows; j += kGroups) {
        const int s = (int)(j % NS);
        if (j >= NS && !wait_bounded(&empty[s], (uint32_t)(((j / NS) - 1) & 1), abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], row_bytes);
        bulk_load(stages + (size_t)s * stage_stride, x + (b + j * G) * ldx, row_bytes, &full[s], pol);
      }
      if (!ok) drain_copies(full, j, NS);
    }
    return;
  }

  const int g = warp / GW;
  const int gw = warp % GW;
  const int gt = gw * 32 + lane;
  const int n4 = N >> 2;
  const float kNeg = neg_inf();

  for (int64_t j = g; j < my_rows; j += kGroups) {
    const int s = (int)(j % NS);
    bool ok = wait_bounded(&full[s], (uint32_t)((j / NS) & 1), abort_flag);
    if constexpr (GW > 1) ok = !barrier_or(1 + g, kGT, !ok);  // one decision per group
    if (!ok) break;

    const float4* sm = reinterpret_cast<const float4*>(stages + (size_t)s * stage_stride);
    float4 v[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const int c = i * kGT + gt;
      v[i] = (c < n4) ? sm[c] : make_float4(kNeg, kNeg, kNeg, kNeg);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // the row is in registers: stage free

    float m = kNeg;
#pragma unroll
    for (int i = 0; i < VEC; ++i) m = max_nan(m, max4(v[i]));
    m = group_max<GW>(m, red_m, g, gw, lane);

    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      v[i].x = exp_shifted(v[i].x, m);
      v[i].y = exp_shifted(v[i].y, m);
      v[i].z = exp_shifted(v[i].z, m);
      v[i].w = exp_shifted(v[i].w, m);
      sum += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    }
    sum = group_sum<GW>(sum, red_s, g, gw, lane);
    const float inv = 1.0f / sum;

    float4* yr4 = reinterpret_cast<float4*>(y + (b + j * G) * ldy);
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const int c = i * kGT + gt;
      if (c < n4) {
        store_stream(yr4 + c, make_float4(v[i].x * inv, v[i].y * inv, v[i].z * inv, v[i].w * inv));
      }
    }
  }
}

// ------------------------------------------------------------ staged_long ---
__device__ __forceinline__ float consumer_max(float v, float* red, int warp, int lane) {
  v = warp_max(v);
  if (lane == 0) red[warp] = v;
  named_barrier(kConsumerBar, kConsumers);
  const float r = warp_max((lane < kConsumerWarps) ? red[lane] : neg_inf());
  named_barrier(kConsumerBar, kConsumers);  // `red` is rewritten by the next reduction
  return r;
}

__device__ __forceinline__ float consumer_sum(float v, float* red, int warp, int lane) {
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  named_barrier(kConsumerBar, kConsumers);
  const float r = warp_sum((lane < kConsumerWarps) ? red[lane] : 0.f);
  named_barrier(kConsumerBar, kConsumers);
  return r;
}

constexpr int kLongUnroll = 4;

// CTA b takes rows b, b + G, b + 2G, ... (G = gridDim.x); each row is staged
// as n_sub <= 4 sub-tiles of tile_floats (the last may be shorter).  Every
// consumer thread goes through every row in order, so each stage's uses are
// ordered by the same threads.
__global__ void __launch_bounds__(kThreads, 1)
softmax_staged_long_kernel(const float* x, float* y, int64_t M, int64_t N, int64_t ldx,
                           int64_t ldy, int32_t tile_floats, int32_t NS) {
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kFullOff);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + kEmptyOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  float* red = reinterpret_cast<float*>(smem + kRedMOff);
  unsigned char* stages = smem + kHeaderBytes;
  const size_t stage_bytes = (size_t)tile_floats * 4;

  const int64_t G = gridDim.x;
  const int64_t b = blockIdx.x;
  const int n_sub = (int)((N + tile_floats - 1) / tile_floats);
  const int64_t items = (M > b) ? (M - b + G - 1) / G : 0;
  if (NS > kMaxStages || n_sub > NS || N <= 0) {  // uniform: every thread returns
    if (threadIdx.x == 0) atomicOr(&g_device_error, kErrConfig);
    return;
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) init_barriers(smem, NS, kConsumerWarps);
  __syncthreads();
  pdl_entry();

  if (warp == kProducerWarp) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int64_t q = 0;
      bool ok = true;
      for (int64_t k = 0; k < items && ok; ++k) {
        const float* src = x + (b + k * G) * ldx;
        for (int t = 0; t < n_sub; ++t, ++q) {
          const int s = (int)(q % NS);
          if (q >= NS && !wait_bounded(&empty[s], (uint32_t)(((q / NS) - 1) & 1), abort_flag)) {
            ok = false;
            break;
          }
          const int64_t t0 = (int64_t)t * tile_floats;
          const uint32_t bytes = (uint32_t)(min((int64_t)tile_floats, N - t0) * 4);
          mbar_arrive_expect_tx(&full[s], bytes);
          bulk_load(stages + (size_t)s * stage_bytes, src + t0, bytes, &full[s], pol);
        }
      }
      if (!ok) drain_copies(full, q, NS);
    }
    return;
  }

  const int tid = threadIdx.x;  // 0 .. kConsumers-1
  const float kNeg = neg_inf();
  int64_t q = 0;
  for (int64_t k = 0; k < items; ++k, q += n_sub) {
    const int64_t row = b + k * G;

    // pass 1: row max (each sub-tile as it lands)
    float m = kNeg;
    bool ok = true;
    for (int t = 0; t < n_sub; ++t) {
      const int s = (int)((q + t) % NS);
      ok = wait_bounded(&full[s], (uint32_t)(((q + t) / NS) & 1), abort_flag);
      ok = !barrier_or(kConsumerBar, kConsumers, !ok);
      if (!ok) break;
      const float4* sm = reinterpret_cast<const float4*>(stages + (size_t)s * stage_bytes);
      const int nf4 = (int)(min((int64_t)tile_floats, N - (int64_t)t * tile_floats) >> 2);
      for (int i = tid; i < nf4; i += kConsumers * kLongUnroll) {
#pragma unroll
        for (int u = 0; u < kLongUnroll; ++u) {
          const int idx = i + u * kConsumers;
          if (idx < nf4) m = max_nan(m, max4(sm[idx]));
        }
      }
    }
    if (!ok) break;
    m = consumer_max(m, red, warp, lane);

    // pass 2: sum of exp(x - m) (an all -inf row gives m = -inf, sum 0, y NaN)
    float sum = 0.f;
    if (m != kNeg) {
      for (int t = 0; t < n_sub; ++t) {
        const int s = (int)((q + t) % NS);
        const float4* sm = reinterpret_cast<const float4*>(stages + (size_t)s * stage_bytes);
        const int nf4 = (int)(min((int64_t)tile_floats, N - (int64_t)t * tile_floats) >> 2);
        for (int i = tid; i < nf4; i += kConsumers * kLongUnroll) {
#pragma unroll
          for (int u = 0; u < kLongUnroll; ++u) {
            const int idx = i + u * kConsumers;
            if (idx < nf4) {
              const float4 a = sm[idx];
              sum += (exp_shifted(a.x, m) + exp_shifted(a.y, m)) +
                     (exp_shifted(a.z, m) + exp_shifted(a.w, m));
            }
          }
        }
      }
    }
    sum = consumer_sum(sum, red, warp, lane);

    // pass 3: normalise from shared memory, store, release each sub-tile
    const float inv = 1.0f / sum;
    float* yr = y + row * ldy;
    for (int t = 0; t < n_sub; ++t) {
      const int s = (int)((q + t) % NS);
      const float4* sm = reinterpret_cast<const float4*>(stages + (size_t)s * stage_bytes);
      float4* y4 = reinterpret_cast<float4*>(yr + (int64_t)t * tile_floats);
      const int nf4 = (int)(min((int64_t)tile_floats, N - (int64_t)t * tile_floats) >> 2);
      for (int i = tid; i < nf4; i += kConsumers * kLongUnroll) {
#pragma unroll
        for (int u = 0; u < kLongUnroll; ++u) {
          const int idx = i + u * kConsumers;
          if (idx < nf4) {
            const float4 a = sm[idx];
            store_stream(y4 + idx, make_float4(exp_shifted(a.x, m) * inv,
                                               exp_shifted(a.y, m) * inv,
                                               exp_shifted(a.z, m) * inv,
                                               exp_shifted(a.w, m) * inv));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

// ------------------------------------------------------------ staged_grid ---
// Rows too long for a cluster: CTA g of a grid of R * C CTAs (one
// per SM) always holds segment c = g % C of rows g / C + k * R, k = 0, 1, ...
// Item k (one row segment of seg floats) is one ring stage, prefetched by the
// producer as far ahead as the ring allows.
//
// A segment's partial (m_c, s_c) goes to global slot [row, c] as two 64-bit
// words, (ticket << 32 | bits(m_c)) and (ticket << 32 | bits(s_c)), written
// and read with relaxed 64-bit accesses: each word is single-copy atomic, so
// a reader that sees this launch's ticket in a word has that word's value,
// and no fence is needed on either side.
//
// Warps 1..14 compute partials: P(k) = wait for stage k, copy this thread's
// float4 of it into registers and release the stage at once, reduce the
// segment max m_c over the 14 warps, form e = exp(x - m_c), reduce the sum
// s_c and publish (by atomic exchange, performed at L2, so peers see it
// promptly).  Warp 0 is the exchange warp:
// E(k) = poll the row's C slots (every load issued before any is used) and
// merge them in slot order, identically in every CTA of the row.  Partials
// run LEAD items ahead: iteration k runs P(k + LEAD) on warps 1..14 (into a
// spare register set) while warp 0 runs E(k); then the 15 consumer warps
// meet and warps 1..14 write y = e * exp(m_c - m) / s of item k.  E(k) needs
// P(k) of its row's CTAs, each published before that CTA's own E(k - LEAD);
// the CTAs of a row all start (see below), so the waits end.
//
// Which (row group, segment) a CTA takes is decided by its ARRIVAL order,
// not by blockIdx: the first CTA to start takes arrival index 0, and CTA a
// takes segment a % C of rows a / C + k R.  So the C CTAs a CTA waits on are
// the ones that arrived just before or just after it: at any time at most
// one row group is partly resident, every complete group runs to the end
// and frees its SMs, and the rest start.  No CTA waits on a CTA that can
// only start once it has finished, whatever else holds SMs (another
// stream's kernels, another process); only a group whose later members find
// no free SM for the whole bounded wait gives up, and that is reported.  The
// counter is one 64-bit word in the workspace, (epoch << 32 | count): a CTA's
// atomic add returns its arrival index (count) and its launch's ticket
// (epoch + 1) at once, and the CTA that draws the last index sets the word to
// (epoch + 1) << 32 before it lets the next kernel on the stream launch (and
// so before any CTA of that kernel draws).  Every launch thus gets a fresh
// ticket on the device -- also each replay of a captured CUDA graph, whose
// kernel arguments never change -- so a slot left by an earlier launch never
// looks current.
__device__ __forceinline__ uint64_t pack_tagged(uint32_t ticket, float v) {
  return ((uint64_t)ticket << 32) | (uint64_t)__float_as_uint(v);
}

// The grid kernel runs 16 warps (512 threads, so up to 128 registers):
// warp 0 exchanges, warps 1..14 compute partials, warp 15 produces.
constexpr int kGThreads = 512;
constexpr int kGProducerWarp = 15;
constexpr int kGConsumerWarps = 15;
constexpr int kGConsumers = 32 * kGConsumerWarps;
constexpr int kPartialBar = 2;                      // warps 1..14
constexpr int kPartialWarps = kGConsumerWarps - 1;
constexpr int kPartialThreads = 32 * kPartialWarps;
constexpr int kMaxSlotsPerLane = 5;                 // C <= 160: a row's slots over 32 lanes

template <int VEC, int LEAD>
__global__ void __launch_bounds__(kGThreads, 1)
softmax_staged_grid_kernel(const float* x, float* y, int64_t M, int64_t N, int64_t ldx,
                           int64_t ldy, int64_t seg, int32_t C, int32_t R, int32_t NS,
                           int32_t stage_stride, unsigned long long* __restrict__ arrivals,
                           uint64_t* __restrict__ slots, int32_t fault, int32_t log_out,
                           unsigned* host_err) {
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kFullOff);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + kEmptyOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  volatile int* fail_flag = reinterpret_cast<volatile int*>(smem + kFailOff);
  MaxSum* whole = reinterpret_cast<MaxSum*>(smem + kWholeOff);
  volatile int* arrival = reinterpret_cast<volatile int*>(smem + kArrivalOff);
  unsigned char* stages = smem + kHeaderBytes;

  // arrival index and ticket (every CTA draws, before anything can return)
  if (threadIdx.x == 0) {
    const unsigned long long old = atomicAdd(arrivals, 1ull);
    const unsigned a = (unsigned)(old & 0xffffffffull);
    const unsigned epoch = (unsigned)(old >> 32);
    if (a == gridDim.x - 1) {   // the last: the next launch's epoch and count 0, before it may start
      atomicExch(arrivals, (unsigned long long)(epoch == 0xfffffffeu ? 0u : epoch + 1u) << 32);
      __threadfence();
    }
    arrival[0] = (int)a;
    arrival[1] = (int)(epoch + 1u);   // never 0, the tag of a zero-filled slot
  }
  __syncthreads();
  const int me = arrival[0];
  const uint32_t ticket = (uint32_t)arrival[1];
  const int c = me % C;
  const int64_t row0 = me / C;
  const int64_t seg_begin = (int64_t)c * seg;
  const int64_t seg_n = min(seg, N - seg_begin);
  const int64_t items = (M > row0) ? (M - row0 + R - 1) / R : 0;
  const int nf4 = (int)(seg_n >> 2);
  if (NS < 2 || NS > kMaxStages || seg_n <= 0 || seg_n * 4 > stage_stride ||
      C > 32 * kMaxSlotsPerLane || nf4 > VEC * kPartialThreads || me >= (int)gridDim.x) {
    if (threadIdx.x == 0) atomicOr(&g_device_error, kErrConfig);
    return;
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) init_barriers(smem, NS, kPartialWarps);
  __syncthreads();
  pdl_launch_dependents();
  // the first two items' segments: into the L2 while the previous kernel
  // drains (on 32 x 2^20: one 46.1 -> 44.5 us, two 44.4, three 44.5, four 45.0)
  for (int64_t q = 0; q < 2 && q < items; ++q)
    prefetch_l2_range(x + (row0 + q * R) * ldx + seg_begin, seg_n * 4, threadIdx.x, kGThreads);
  pdl_wait();

  if (warp == kGProducerWarp) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const uint32_t bytes = (uint32_t)(seg_n * 4);
      int64_t k = 0;
      bool ok = true;
      for (; k < items; ++k) {
        const int st = (int)(k % NS);
        if (k >= NS && !wait_bounded(&empty[st], (uint32_t)(((k / NS) - 1) & 1), abort_flag, host_err)) {
          ok = false;
          break;
        }
        // every CTA's first segment gates the first exchange of its row: let
        // it land before the rest of the ring is queued behind it in HBM
        if (k == 2 && NS > 2 && !wait_bounded(&full[0], 0, abort_flag, host_err)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[st], bytes);
        bulk_load(stages + (size_t)st * stage_stride, x + (row0 + k * R) * ldx + seg_begin, bytes,
                  &full[st], pol);
      }
      if (!ok) drain_copies(full, k, NS);
    }
    return;
  }

  const float kNeg = neg_inf();
  const int ptid = threadIdx.x - 32;  // index among warps 1..14
  float* red_m = reinterpret_cast<float*>(smem + kRedMOff);
  float* red_s = reinterpret_cast<float*>(smem + kRedSOff);

  // P(k) on warps 1..14 into register set v: e = exp(x - m_c) against the
  // segment max m_c (a max reduction, then a sum reduction -- no exps in the
  // reduction trees).  False if a wait ran out (the same answer in all of them).
  auto partial = [&](int64_t k, float4 (&v)[VEC], float& mc_out) -> bool {
    const int st = (int)(k % NS);
    const bool got = wait_bounded(&full[st], (uint32_t)((k / NS) & 1), abort_flag, host_err);
    const float4* sm = reinterpret_cast<const float4*>(stages + (size_t)st * stage_stride);
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const int idx = ptid + i * kPartialThreads;
      v[i] = (got && idx < nf4) ? sm[idx] : make_float4(kNeg, kNeg, kNeg, kNeg);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // the segment is in registers: stage free
    float m = kNeg;
#pragma unroll
    for (int i = 0; i < VEC; ++i) m = max_nan(m, max4(v[i]));
    m = warp_max(m);
    if (lane == 0) red_m[warp] = m;
    if (barrier_or(kPartialBar, kPartialThreads, !got)) return false;
    m = warp_max((lane >= 1 && lane < kGConsumerWarps) ? red_m[lane] : kNeg);
    const bool none = (m == kNeg);  // only -inf (or nothing) in this segment
    float sum = 0.f;
    if (log_out) {  // keep x for the log form
      if (!none) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          sum += (exp_shifted(v[i].x, m) + exp_shifted(v[i].y, m)) +
                 (exp_shifted(v[i].z, m) + exp_shifted(v[i].w, m));
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        v[i].x = none ? 0.f : exp_shifted(v[i].x, m);
        v[i].y = none ? 0.f : exp_shifted(v[i].y, m);
        v[i].z = none ? 0.f : exp_shifted(v[i].z, m);
        v[i].w = none ? 0.f : exp_shifted(v[i].w, m);
        sum += (v[i].x + v[i].y) + (v[i].z + v[i].w);
      }
    }
    sum = warp_sum(sum);
    if (lane == 0) red_s[warp] = sum;
    named_barrier(kPartialBar, kPartialThreads);
    sum = warp_sum((lane >= 1 && lane < kGConsumerWarps) ? red_s[lane] : 0.f);
    mc_out = m;
    if (ptid == 0 && !(fault != 0 && me == 0 && k == 0)) {
      uint64_t* sl = slots + 2 * ((row0 + k * R) * C + c);
      publish_gpu_u64(sl, pack_tagged(ticket, m));
      publish_gpu_u64(sl + 1, pack_tagged(ticket, sum));
    }
    return true;
  };

  // E(k) on warp 0: merged (m, s) of the row into *whole; sets the fail flag
  // if the wait ran out.
  auto exchange = [&](int64_t k) {
    const uint64_t* rs = slots + 2 * (row0 + k * R) * C;
    const uint64_t t0 = global_timer_ns();
    bool seen = false;
    uint32_t n = 0;
    MaxSum acc{kNeg, 0.f};
    while (!*fail_flag) {
      uint64_t wm[kMaxSlotsPerLane], ws[kMaxSlotsPerLane];
#pragma unroll
      for (int j = 0; j < kMaxSlotsPerLane; ++j) {
        const int l = lane + 32 * j;
        wm[j] = (l < C) ? ld_relaxed_gpu_u64(rs + 2 * l) : pack_tagged(ticket, kNeg);
        ws[j] = (l < C) ? ld_relaxed_gpu_u64(rs + 2 * l + 1) : pack_tagged(ticket, 0.f);
      }
      bool mine = true;
#pragma unroll
      for (int j = 0; j < kMaxSlotsPerLane; ++j) {
        mine &= ((uint32_t)(wm[j] >> 32) == ticket) && ((uint32_t)(ws[j] >> 32) == ticket);
      }
      if (__all_sync(kFullMask, mine)) {
#pragma unroll
        for (int j = 0; j < kMaxSlotsPerLane; ++j) {
          acc = merge(acc, MaxSum{__uint_as_float((uint32_t)wm[j]), __uint_as_float((uint32_t)ws[j])});
        }
        seen = true;
        break;
      }
      if ((++n & 15u) == 0 && (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs)) break;
    }
    acc = warp_merge(acc);
    if (lane == 0) {
      *whole = acc;
      if (!seen) {
        report_timeout(host_err);
        *abort_flag = 1;
        *fail_flag = 1;
      }
    }
  };

  // The exchange warp and the partial warps run separate loops that meet at
  // the same two consumer barriers per item, so the partial warps' register
  // sets are never live in the exchange warp's code.
  if (warp == 0) {
    for (int64_t k = 0; k < items; ++k) {
      exchange(k);
      named_barrier(kConsumerBar, kGConsumers);
      const bool failed = *fail_flag != 0;
      named_barrier(kConsumerBar, kGConsumers);  // `whole` and the flag are rewritten next round
      if (failed) return;
    }
    return;
  }

  // Partial warps, one item: P(k + LEAD) into `ahead` (while warp 0 runs
  // E(k)), then y of item k from `cur`.  LEAD + 1 register sets rotate: the
  // item being written, those whose exchange is pending, the one being
  // formed.  False once the CTA must stop.
  auto step = [&](int64_t k, float4 (&cur)[VEC], float mtc, float4 (&ahead)[VEC], float& mta) {
    if (k + LEAD < items && !partial(k + LEAD, ahead, mta)) {
      if (ptid == 0) *fail_flag = 1;
    }
    named_barrier(kConsumerBar, kGConsumers);
    const bool failed = *fail_flag != 0;
    const MaxSum w = *whole;
    named_barrier(kConsumerBar, kGConsumers);
    if (failed) return false;
    float4* y4 = reinterpret_cast<float4*>(y + (row0 + k * R) * ldy + seg_begin);
    if (log_out) {
      const float ls = logf(w.s);
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const int idx = ptid + i * kPartialThreads;
        if (idx < nf4) {
          store_stream(y4 + idx, make_float4(log_softmax_of(cur[i].x, w.m, ls),
                                             log_softmax_of(cur[i].y, w.m, ls),
                                             log_softmax_of(cur[i].z, w.m, ls),
                                             log_softmax_of(cur[i].w, w.m, ls)));
        }
      }
      return true;
    }
    const bool bad = !(w.s == w.s) || w.m == kNeg;  // NaN / inf / all -inf row
    const float scale =
        bad ? __int_as_float(0x7fc00000) : (mtc == kNeg ? 0.f : exp_shifted(mtc, w.m) / w.s);
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const int idx = ptid + i * kPartialThreads;
      if (idx < nf4) {
        store_stream(y4 + idx, make_float4(cur[i].x * scale, cur[i].y * scale, cur[i].z * scale,
                                           cur[i].w * scale));
      }
    }
    return true;
  };

  float4 a[VEC], b[VEC];
  float ma = kNeg, mb = kNeg;
  bool ok = true;
  if constexpr (LEAD == 1) {
    if (items > 0) ok = partial(0, a, ma);
    if (!ok && ptid == 0) *fail_flag = 1;  // seen by every consumer warp at the first meeting
    for (int64_t k = 0; k < items; k += 2) {
      if (!step(k, a, ma, b, mb)) return;
      if (k + 1 >= items) break;
      if (!step(k + 1, b, mb, a, ma)) return;
    }
  } else {
    float4 cc[VEC];
    float mc = kNeg;
    if (items > 0) ok = partial(0, a, ma);
    if (ok && items > 1) ok = partial(1, b, mb);
    if (!ok && ptid == 0) *fail_flag = 1;
    for (int64_t k = 0; k < items; k += 3) {
      if (!step(k, a, ma, cc, mc)) return;
      if (k + 1 >= items) break;
      if (!step(k + 1, b, mb, a, ma)) return;
      if (k + 2 >= items) break;
      if (!step(k + 2, cc, mc, b, mb)) return;
    }
  }
}

// ---------------------------------------------------------------- launch ---
std::mutex g_attr_mu;
std::set<std::pair<const void*, int>> g_attr_done;

cudaError_t allow_dynamic_smem(const void* kernel) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (g_attr_done.count({kernel, dev})) return cudaSuccess;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess) g_attr_done.insert({kernel, dev});
  return e;
}

template <int VEC, int GW>
cudaError_t launch_rows_vg(const rrs_plan& p, const float* x, float* y, int64_t M, int64_t N,
                           const Layout& l, cudaStream_t s) {
  auto kern = softmax_staged_rows_kernel<VEC, GW>;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)p.grid), dim3(kThreads), (size_t)p.smem_bytes, s, 0, x, y,
                    M, (int32_t)N, l.ldx, l.ldy, p.stages, p.tile * 4);
}

}  // namespace

int staged_header_bytes() { return kHeaderBytes; }
int staged_max_stages() { return kMaxStages; }
int staged_threads() { return kThreads; }
int staged_consumer_warps() { return kConsumerWarps; }
int grid_threads() { return kGThreads; }
int grid_partial_threads() { return kPartialThreads; }

cudaError_t launch_softmax_staged_rows(const rrs_plan& p, const float* x, float* y, int64_t M,
                                       int64_t N, const Layout& l, cudaStream_t s) {
  if (p.threads != kThreads) return cudaErrorInvalidConfiguration;
  const int gw = p.warps_per_row, vec = p.vec;
#define RRS_SR(V, G) \
  if (vec == V && gw == G) return launch_rows_vg<V, G>(p, x, y, M, N, l, s);
  RRS_SR(1, 1)
  RRS_SR(2, 1)
  RRS_SR(4, 1)
  RRS_SR(8, 1)
  RRS_SR(16, 1)
  RRS_SR(8, 2)
  RRS_SR(8, 4)
  RRS_SR(8, 8)
#undef RRS_SR
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_softmax_staged_long(const rrs_plan& p, const float* x, float* y, int64_t M,
                                       int64_t N, const Layout& l, cudaStream_t s) {
  if (p.threads != kThreads) return cudaErrorInvalidConfiguration;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(softmax_staged_long_kernel));
  if (e != cudaSuccess) return e;
  return launch_pdl(softmax_staged_long_kernel, dim3((unsigned)p.grid), dim3(kThreads),
                    (size_t)p.smem_bytes, s, 0, x, y, M, N, l.ldx, l.ldy, p.tile, p.stages);
}

cudaError_t launch_softmax_staged_grid(const rrs_plan& p, const float* x, float* y, int64_t M,
                                       int64_t N, const Layout& l, void* workspace, int fault,
                                       unsigned* host_err, cudaStream_t s) {
  if (p.threads != kGThreads) return cudaErrorInvalidConfiguration;
  // segments of up to 4 float4 per thread run partials two items ahead (three
  // register sets); longer ones, up to 8 float4, one item ahead
  auto k2 = softmax_staged_grid_kernel<2, 2>;
  auto k4 = softmax_staged_grid_kernel<4, 2>;
  auto k8 = softmax_staged_grid_kernel<8, 1>;
  const void* kern = p.vec == 2 ? reinterpret_cast<const void*>(k2)
                   : p.vec == 4 ? reinterpret_cast<const void*>(k4)
                   : p.vec == 8 ? reinterpret_cast<const void*>(k8) : nullptr;
  if (!kern) return cudaErrorInvalidConfiguration;
  cudaError_t e = allow_dynamic_smem(kern);
  if (e != cudaSuccess) return e;
  // A plain launch with programmatic dependent launch, not a cooperative
  // one: a cooperative launch waits for every SM to be free, so it cannot
  // overlap the previous kernel's drain (measured on 32 x 2^20: 48.3 us
  // against 44.9 us).  The CTAs of a row are made co-resident by drawing
  // their work in arrival order instead (see the kernel).  Every wait is
  // still bounded: if one runs out, the kernel sets the device error word
  // and `host_err`, and later calls report RRS_ERR_TIMEOUT.
  auto* arrivals = static_cast<unsigned long long*>(workspace);
  uint64_t* slots = reinterpret_cast<uint64_t*>(static_cast<unsigned char*>(workspace) + kGridArrivalBytes);
  const int32_t C = (int32_t)p.ctas_per_row;
  const dim3 grid((unsigned)p.grid), block(kGThreads);
  const size_t smem = (size_t)p.smem_bytes;
  if (p.vec == 2)
    return launch_pdl(k2, grid, block, smem, s, 0, x, y, M, N, l.ldx, l.ldy, p.chunk, C,
                      p.rows_per_cta, p.stages, p.tile * 4, arrivals, slots, (int32_t)fault,
                      (int32_t)l.log_out, host_err);
  if (p.vec == 4)
    return launch_pdl(k4, grid, block, smem, s, 0, x, y, M, N, l.ldx, l.ldy, p.chunk, C,
                      p.rows_per_cta, p.stages, p.tile * 4, arrivals, slots, (int32_t)fault,
                      (int32_t)l.log_out, host_err);
  return launch_pdl(k8, grid, block, smem, s, 0, x, y, M, N, l.ldx, l.ldy, p.chunk, C,
                    p.rows_per_cta, p.stages, p.tile * 4, arrivals, slots, (int32_t)fault,
                    (int32_t)l.log_out, host_err);
}

// Testing only (rrs_test_occupy): holds an SM's shared memory for `ns`
// nanoseconds of the global timer, then returns; no memory is touched.
__global__ void occupy_kernel(int64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < (uint64_t)ns) __nanosleep(2000);
}

cudaError_t launch_occupy(int ctas, int smem_bytes, int64_t ns, cudaStream_t s) {
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(occupy_kernel));
  if (e != cudaSuccess) return e;
  occupy_kernel<<<ctas, 32, (size_t)smem_bytes, s>>>(ns);
  return cudaGetLastError();
}

cudaError_t read_and_clear_staged_error(cudaStream_t s, unsigned* value) {
  unsigned host = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&host, g_device_error, sizeof(host), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && host != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  *value = host;
  return e;
}

}  // namespace rrs
