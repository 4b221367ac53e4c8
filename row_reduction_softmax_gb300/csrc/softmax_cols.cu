// Column softmax: y[i, j] = exp(x[i, j] - m_j) / s_j with m_j = max_i x[i, j]
// and s_j = sum_i exp(x[i, j] - m_j) -- the pages' softmax ("Kernels, Triton,
// XLA", section "Reductions and tiling") with the reduction taken down each
// column.  The lecture transcript's question after the softmax kernel asks
// for it; the answer there is the same kernel with the strides swapped.  A
// thread per column reading down the rows would touch one float per 128-byte
// line per warp access -- the uncoalesced pattern of the pages' "memory
// coalescing" paragraph -- so here 8 lanes read 32 consecutive columns of a
// row (one float4 each: a full 128-byte line) and a warp access covers 4
// rows; the reduction runs across lanes groups, warps and CTAs.  A narrow
// band (32 columns) gives many CTAs, so that their load and store phases
// overlap instead of running in a few lockstep waves.
//
// COLS_CLUSTER -- a band of 32 columns per CTA group; the M rows are split
//   over a thread-block cluster of cs CTAs, each CTA's 32 row groups (8 warps
//   x 4 rows per access) hold VEC rows each in registers.  Per column: max and
//   sum over a thread's rows, then over the CTA's row groups (shared memory),
//   then over the cluster's CTAs (DSMEM), merged with m = max(m_a, m_b),
//   s = s_a e^(m_a - m) + s_b e^(m_b - m).  One read and one write per
//   element.  M <= 16 * 32 * 16 = 8192.
// COLS_BAND -- a band of 32 columns per cluster of cs <= 8 CTAs, each CTA
//   streaming its rows twice: pass 1 loads them at L2 evict-last priority
//   and forms per-column online (max, sum) partials, the cluster merges
//   them over DSMEM, pass 2 re-reads the rows -- from the L2, where pass 1
//   left them moments before -- and writes y.  HBM sees one read and one
//   write per element, with nothing but a few registers of state per
//   thread, so any M fits.  The planner sizes a CTA's rows (at most 1024 =
//   128 KB of x) so that the x of all resident CTAs (four per SM) fits the
//   L2 together.
// COLS_TWO_PHASE -- any M and alignment: kernel 1 writes each (row chunk,
//   column) online partial to a workspace, kernel 2 merges a column's
//   partials, re-reads its chunk and writes y (12 bytes per element unless
//   the re-read hits L2).
// COLS_TWO_PASS -- the band path's two passes as separate work items of one
//   launch, dealt out in arrival order so that every SM runs first passes
//   (HBM reads) beside second passes (L2 re-reads, HBM writes) and no CTA
//   waits at a cluster barrier; see the kernel.
#include <climits>

#include <cooperative_groups.h>

#include "device_common.cuh"
#include "internal.h"
#include "launch_util.h"
#include "sm100_async.cuh"
#include "two_pass_common.cuh"

namespace cg = cooperative_groups;

namespace rrs {

// Set by COLS_TWO_PASS CTAs that gave up a bounded wait; read by rrs_device_error().
__device__ unsigned int g_cols_error = 0;

namespace {

constexpr int kCT = 256;             // threads per CTA
constexpr int kCW = kCT / 32;        // warps per CTA
constexpr int kLPR = 8;              // lanes that share a row: 8 x float4 = 128 bytes
constexpr int kRPW = 32 / kLPR;      // rows per warp access
constexpr int kGroups = kCW * kRPW;  // row groups per CTA
constexpr int kBand = 4 * kLPR;      // columns per CTA

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Four consecutive columns j0..j0+3 of one row; lanes past N read `fill`.
// V4: the row is 16-byte aligned, so the float4 is aligned.
template <bool V4>
__device__ __forceinline__ float4 load_cols(const float* row, int64_t j0, int64_t N, float fill) {
  if (V4 && j0 + 3 < N) return load_stream(reinterpret_cast<const float4*>(row + j0));
  float4 v;
  v.x = (j0 + 0 < N) ? load_stream(row + j0 + 0) : fill;
  v.y = (j0 + 1 < N) ? load_stream(row + j0 + 1) : fill;
  v.z = (j0 + 2 < N) ? load_stream(row + j0 + 2) : fill;
  v.w = (j0 + 3 < N) ? load_stream(row + j0 + 3) : fill;
  return v;
}

template <bool V4>
__device__ __forceinline__ void store_cols(float* row, int64_t j0, int64_t N, const float4& v) {
  if (V4 && j0 + 3 < N) {
    store_stream(reinterpret_cast<float4*>(row + j0), v);
    return;
  }
  if (j0 + 0 < N) store_stream(row + j0 + 0, v.x);
  if (j0 + 1 < N) store_stream(row + j0 + 1, v.y);
  if (j0 + 2 < N) store_stream(row + j0 + 2, v.z);
  if (j0 + 3 < N) store_stream(row + j0 + 3, v.w);
}

__device__ __forceinline__ float comp(const float4& v, int c) {
  return c == 0 ? v.x : (c == 1 ? v.y : (c == 2 ? v.z : v.w));
}

// ------------------------------------------------------------ COLS_CLUSTER ---
// Grid: (bands * cs) CTAs in clusters of cs along x; cluster k owns columns
// [32k, 32k + 32).  Rank r owns rows [r * rseg, min((r + 1) * rseg, M)),
// rseg = ceil(M / cs) <= kGroups * VEC.  Thread (warp w, lane l) is in row
// group g = 4w + l / 8 and column slot l % 8; it holds rows
// r * rseg + g + kGroups * i, i < VEC, columns 4 (l % 8) .. + 3 of the band.
// x, y 16-byte aligned and ldx, ldy multiples of 4 (any N).  LOG writes
// (x - m) - log(s).
// Occupancy target per VEC: 4 CTAs per SM up to 4 rows per thread, then 3, 2.
template <int VEC>
__host__ __device__ constexpr int cols_min_blocks() { return VEC <= 4 ? 4 : (VEC == 8 ? 3 : 2); }

template <int VEC, bool LOG>
__global__ void __launch_bounds__(kCT, cols_min_blocks<VEC>())
softmax_cols_cluster_kernel(const float* x, float* y, int64_t M, int64_t N, int64_t ldx,
                            int64_t ldy) {
  __shared__ float red[kGroups][kBand];
  __shared__ MaxSum part[kBand];   // this CTA's per-column (m_c, s_c), read by its peers
  __shared__ MaxSum whole[kBand];  // the merged pair of each column

  cg::cluster_group cluster = cg::this_cluster();
  const int cs = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t band = blockIdx.x / cs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = lane % kLPR;
  const int g = warp * kRPW + lane / kLPR;
  const int64_t rseg = (M + cs - 1) / cs;
  const int64_t r0 = rank * rseg;
  const int64_t r1 = min(r0 + rseg, M);
  const int64_t j0 = band * kBand + 4 * slot;
  const float kNeg = neg_inf();
  pdl_entry();

  float4 v[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const int64_t r = r0 + g + (int64_t)kGroups * i;
    v[i] = (r < r1 && j0 < N) ? load_cols<true>(x + r * ldx, j0, N, kNeg)
                              : make_float4(kNeg, kNeg, kNeg, kNeg);
  }

  // per-column max over this thread's rows, then over the CTA's row groups
  float4 m = v[0];
#pragma unroll
  for (int i = 1; i < VEC; ++i) {
    m.x = max_nan(m.x, v[i].x);
    m.y = max_nan(m.y, v[i].y);
    m.z = max_nan(m.z, v[i].z);
    m.w = max_nan(m.w, v[i].w);
  }
  reinterpret_cast<float4*>(red[g])[slot] = m;
  __syncthreads();
  if (tid < kBand) {
    float cm = red[0][tid];
#pragma unroll 8
    for (int k = 1; k < kGroups; ++k) cm = max_nan(cm, red[k][tid]);
    part[tid].m = cm;
  }
  __syncthreads();
  float mc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) mc[c] = part[4 * slot + c].m;

  // per-column sum of exp(x - m_c); x stays in v for the log form
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    float4 e;
    e.x = (mc[0] == kNeg) ? 0.f : exp_shifted(v[i].x, mc[0]);
    e.y = (mc[1] == kNeg) ? 0.f : exp_shifted(v[i].y, mc[1]);
    e.z = (mc[2] == kNeg) ? 0.f : exp_shifted(v[i].z, mc[2]);
    e.w = (mc[3] == kNeg) ? 0.f : exp_shifted(v[i].w, mc[3]);
    s.x += e.x;
    s.y += e.y;
    s.z += e.z;
    s.w += e.w;
    if constexpr (!LOG) v[i] = e;
  }
  reinterpret_cast<float4*>(red[g])[slot] = s;  // red's max values were consumed before the barrier
  __syncthreads();
  if (tid < kBand) {
    float cs_sum = 0.f;
#pragma unroll 8
    for (int k = 0; k < kGroups; ++k) cs_sum += red[k][tid];
    part[tid].s = cs_sum;
  }
  cluster_arrive_release();  // publish part[] to the cluster
  cluster_wait_acquire();    // every peer's part[] is visible
  if (tid < kBand) {
    MaxSum q{kNeg, 0.f};
    for (int k = 0; k < cs; ++k) q = merge(q, *cluster.map_shared_rank(&part[tid], k));
    whole[tid] = q;  // the same ranks in the same order in every CTA
  }
  cluster_arrive_relaxed();  // done reading the peers' part[]
  __syncthreads();

  // per column: the merged max, and either log(s) or e^(m_c - m) / s
  float wm[4], k4[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const MaxSum w = whole[4 * slot + c];
    wm[c] = w.m;
    const bool bad = !(w.s == w.s) || w.m == kNeg;  // NaN / inf / all -inf column
    if constexpr (LOG) {
      k4[c] = logf(w.s);
    } else {
      k4[c] = bad ? __int_as_float(0x7fc00000)
                  : (mc[c] == kNeg ? 0.f : exp_shifted(mc[c], w.m) / w.s);
    }
  }
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const int64_t r = r0 + g + (int64_t)kGroups * i;
    if (r >= r1 || j0 >= N) continue;
    float4 o;
    if constexpr (LOG) {
      o = make_float4(log_softmax_of(v[i].x, wm[0], k4[0]), log_softmax_of(v[i].y, wm[1], k4[1]),
                      log_softmax_of(v[i].z, wm[2], k4[2]), log_softmax_of(v[i].w, wm[3], k4[3]));
    } else {
      o = make_float4(v[i].x * k4[0], v[i].y * k4[1], v[i].z * k4[2], v[i].w * k4[3]);
    }
    store_cols<true>(y + r * ldy, j0, N, o);
  }
  cluster_wait_acquire();  // peers finished reading part[] before this CTA exits
}

// --------------------------------------------------------------- COLS_BAND ---
// Grid: (bands * cs) CTAs in clusters of cs along x; cluster k owns columns
// [32k, 32k + 32).  Rank r owns rows [r * rseg, min((r + 1) * rseg, M)),
// rseg = ceil(M / cs).  Thread (warp w, lane l) is in row group
// g = 4w + l / 8 and column slot l % 8 (columns 4 (l % 8) .. + 3 of the
// band); it walks rows r0 + g, r0 + g + 32, ... with kBU rows in flight.
// x, y 16-byte aligned and ldx, ldy multiples of 4 (any M, N).  LOG writes
// (x - m) - log(s).  In place (x == y) is safe: every element is read by the
// thread that writes it, and pass 2 reads an element before writing it.
constexpr int kBU = 8;   // rows in flight per thread and batch

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ float4 load_evict_last(const float4* p, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p), "l"(pol));
  return v;
}


// A batch of kBU rows of a thread's four columns folded into its online
// (max, sum) pairs: the batch's column max rescales each pair once, then the
// exponentials against the pair's max are added in f32x2 pairs.  A column
// whose max is still -inf has seen only -inf: shifting by 0 gives 2^-inf = 0
// for all of them, which adds nothing.
__device__ __forceinline__ void fold_batch(MaxSum (&p)[4], const float4 (&a)[kBU], uint64_t log2e2) {
  const float kNeg = neg_inf();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float bm = comp(a[0], k);
#pragma unroll
    for (int u = 1; u < kBU; ++u) bm = max_nan(bm, comp(a[u], k));
    rescale_to(p[k], bm);
  }
  uint64_t nm[2], s2[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float ma = (p[2 * h].m == kNeg) ? 0.f : p[2 * h].m;
    const float mb = (p[2 * h + 1].m == kNeg) ? 0.f : p[2 * h + 1].m;
    nm[h] = f2_pack(-ma, -mb);
    s2[h] = f2_pack(p[2 * h].s, p[2 * h + 1].s);
  }
#pragma unroll
  for (int u = 0; u < kBU; ++u) {
    s2[0] = f2_add(s2[0], exp_shifted2(a[u].x, a[u].y, nm[0], log2e2));
    s2[1] = f2_add(s2[1], exp_shifted2(a[u].z, a[u].w, nm[1], log2e2));
  }
  f2_unpack(s2[0], p[0].s, p[1].s);
  f2_unpack(s2[1], p[2].s, p[3].s);
}

// Lanes l, l ^ 8, l ^ 16 and l ^ 24 of a warp hold the same four columns:
// their pairs merged by shuffles (merge is commutative, so each lane gets
// the same result).
__device__ __forceinline__ void merge_column_lanes(MaxSum (&p)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int o = kLPR; o < 32; o <<= 1) {
      MaxSum q;
      q.m = __shfl_xor_sync(kFullMask, p[k].m, o);
      q.s = __shfl_xor_sync(kFullMask, p[k].s, o);
      p[k] = merge(p[k], q);
    }
  }
}

// The second pass's arithmetic for a thread's four columns, from their
// merged pairs w[0..3]: y = 2^((x - m) log2 e) / s, or (x - m) - log s in
// the log form; a column that is all -inf or holds +inf or NaN gives NaN.
template <bool LOG>
struct ColumnScale {
  float wm[4], k4[4];
  uint64_t nwm[2], kk2[2];
  __device__ __forceinline__ explicit ColumnScale(const MaxSum* w) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      wm[c] = w[c].m;
      const bool bad = !(w[c].s == w[c].s) || w[c].m == neg_inf();
      if constexpr (LOG) {
        k4[c] = logf(w[c].s);
      } else {
        k4[c] = bad ? __int_as_float(0x7fc00000) : 1.0f / w[c].s;
      }
    }
    nwm[0] = f2_pack(-wm[0], -wm[1]);
    nwm[1] = f2_pack(-wm[2], -wm[3]);
    kk2[0] = f2_pack(k4[0], k4[1]);
    kk2[1] = f2_pack(k4[2], k4[3]);
  }
  __device__ __forceinline__ float4 operator()(const float4& v, uint64_t log2e2) const {
    float4 o;
    if constexpr (LOG) {
      o = make_float4(log_softmax_of(v.x, wm[0], k4[0]), log_softmax_of(v.y, wm[1], k4[1]),
                      log_softmax_of(v.z, wm[2], k4[2]), log_softmax_of(v.w, wm[3], k4[3]));
    } else {
      f2_unpack(f2_mul(exp_shifted2(v.x, v.y, nwm[0], log2e2), kk2[0]), o.x, o.y);
      f2_unpack(f2_mul(exp_shifted2(v.z, v.w, nwm[1], log2e2), kk2[1]), o.z, o.w);
    }
    return o;
  }
};

// Registers for four CTAs per SM (64, no spills in the softmax form).
// Measured on GB300 against three (80 registers), forced on the band path:
// 8192 x 16384 214.5 against 226.8 us, 8192 x 8192 109.8 against 119.7,
// 2048 x 65536 198.3 against 203.1, 4096 x 16384 109.1 against 107.7.
template <bool LOG>
__global__ void __launch_bounds__(kCT, 4)
softmax_cols_band_kernel(const float* x, float* y, int64_t M, int64_t N, int64_t ldx, int64_t ldy) {
  __shared__ MaxSum red[kCW][kBand];   // per warp, after the shuffle merge
  __shared__ MaxSum part[kBand];   // this CTA's per-column (m_c, s_c), read by its peers
  __shared__ MaxSum whole[kBand];  // the merged pair of each column

  cg::cluster_group cluster = cg::this_cluster();
  const int cs = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t band = blockIdx.x / cs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = lane % kLPR;
  const int g = warp * kRPW + lane / kLPR;
  const int64_t rseg = (M + cs - 1) / cs;
  const int64_t r0 = rank * rseg;
  const int64_t r1 = min(r0 + rseg, M);
  const int64_t j0 = band * kBand + 4 * slot;
  const bool live_col = j0 < N;   // N % 4 == 0 is not required: see the tail below
  const bool full4 = j0 + 3 < N;
  const float kNeg = neg_inf();
  const int64_t xstep = (int64_t)kGroups * ldx, ystep = (int64_t)kGroups * ldy;   // a thread's next row
  const uint64_t log2e2 = f2_pack(kLog2e, kLog2e);
  pdl_entry();
  const uint64_t pol = l2_evict_last_policy();

  auto load_row = [&](int64_t r, bool keep) -> float4 {
    const float* row = x + r * ldx;
    if (full4) return keep ? load_evict_last(reinterpret_cast<const float4*>(row + j0), pol)
                           : load_stream(reinterpret_cast<const float4*>(row + j0));
    float4 v;
    v.x = (j0 + 0 < N) ? row[j0 + 0] : kNeg;
    v.y = (j0 + 1 < N) ? row[j0 + 1] : kNeg;
    v.z = (j0 + 2 < N) ? row[j0 + 2] : kNeg;
    v.w = kNeg;
    return v;
  };
  // a batch is whole when its last row is inside the slice and the four
  // columns are: then it needs no per-row check
  auto whole_batch = [&](int64_t r) { return full4 && r + (int64_t)(kBU - 1) * kGroups < r1; };

  // ---- pass 1: online (max, sum) per column over this thread's rows ----
  MaxSum p[4] = {{kNeg, 0.f}, {kNeg, 0.f}, {kNeg, 0.f}, {kNeg, 0.f}};
  if (live_col) {
    const float* xr = x + (r0 + g) * ldx + j0;
    for (int64_t r = r0 + g; r < r1; r += (int64_t)kBU * kGroups, xr += kBU * xstep) {
      float4 a[kBU];
      if (whole_batch(r)) {
        const float* q = xr;
#pragma unroll
        for (int u = 0; u < kBU; ++u, q += xstep) a[u] = load_evict_last(reinterpret_cast<const float4*>(q), pol);
      } else {
#pragma unroll
        for (int u = 0; u < kBU; ++u) {
          const int64_t ru = r + (int64_t)u * kGroups;
          a[u] = (ru < r1) ? load_row(ru, true) : make_float4(kNeg, kNeg, kNeg, kNeg);
        }
      }
      fold_batch(p, a, log2e2);
    }
  }
  // ---- merge: a warp's 4 row groups by shuffles, the CTA's 8 warps in
  // order, then the cluster's ranks: a fixed order, and merge is
  // commutative, so the lanes of a column agree bit for bit ----
  merge_column_lanes(p);
  if (lane < kLPR) {
#pragma unroll
    for (int k = 0; k < 4; ++k) red[warp][4 * slot + k] = p[k];
  }
  __syncthreads();
  if (tid < kBand) {
    MaxSum q{kNeg, 0.f};
#pragma unroll
    for (int k = 0; k < kCW; ++k) q = merge(q, red[k][tid]);
    part[tid] = q;
  }
  cluster_arrive_release();  // publish part[] to the cluster
  // pass 2's first batch does not depend on the exchange: its loads are in
  // flight while the cluster barrier completes
  auto load_batch2 = [&](float4 (&a)[kBU], int64_t r, const float* xr) {
    if (whole_batch(r)) {
      const float* q = xr;
#pragma unroll
      for (int u = 0; u < kBU; ++u, q += xstep) a[u] = load_stream(reinterpret_cast<const float4*>(q));
    } else {
#pragma unroll
      for (int u = 0; u < kBU; ++u) {
        const int64_t ru = r + (int64_t)u * kGroups;
        if (ru < r1) a[u] = load_row(ru, false);
      }
    }
  };
  const int64_t rfirst = r0 + g;
  const bool any2 = live_col && rfirst < r1;
  float4 a2[kBU];
  if (any2) load_batch2(a2, rfirst, x + rfirst * ldx + j0);
  cluster_wait_acquire();    // every peer's part[] is visible
  if (tid < kBand) {
    MaxSum q{kNeg, 0.f};
    for (int k = 0; k < cs; ++k) q = merge(q, *cluster.map_shared_rank(&part[tid], k));
    whole[tid] = q;  // the same ranks in the same order in every CTA
  }
  cluster_arrive_relaxed();  // done reading the peers' part[]
  __syncthreads();

  // ---- pass 2: re-read (from the L2), normalise, write ----
  const ColumnScale<LOG> scale(&whole[4 * slot]);
  auto normalise = [&](const float4& v) -> float4 { return scale(v, log2e2); };
  if (any2) {
    int64_t r = rfirst;
    for (;;) {   // a2 holds the batch of rows r; the row pointers are formed
                 // from r each batch, so only r stays live across the loop
      if (whole_batch(r)) {
        float* o = y + r * ldy + j0;
#pragma unroll
        for (int u = 0; u < kBU; ++u, o += ystep) store_stream(reinterpret_cast<float4*>(o), normalise(a2[u]));
      } else {
#pragma unroll
        for (int u = 0; u < kBU; ++u) {
          const int64_t ru = r + (int64_t)u * kGroups;
          if (ru >= r1) continue;
          store_cols<true>(y + ru * ldy, j0, N, normalise(a2[u]));
        }
      }
      r += (int64_t)kBU * kGroups;
      if (r >= r1) break;
      load_batch2(a2, r, x + r * ldx + j0);
    }
  }
  cluster_wait_acquire();  // peers finished reading part[] before this CTA exits
}

// ----------------------------------------------------------- COLS_TWO_PASS ---
// Item k = (band b, slice r), k = b S + r, covers columns [32b, 32b + 32) of
// rows [r R, min((r + 1) R, M)), S = ceil(M / R) slices per band.
//   Pass 1 of item k: online (max, sum) per column over the slice, with the
//   loads at L2 evict-last priority, merged over the CTA (the band kernel's
//   shuffle and shared-memory steps) and published to item k's 32 column
//   slots as two tagged 64-bit words, (ticket << 32 | bits(m)) and
//   (ticket << 32 | bits(s)): each word is single-copy atomic, so a reader
//   that sees this launch's ticket in a word has its value.
//   Pass 2 of item k: one warp merges the band's S slice pairs of each
//   column in slice order (the same order in every CTA of the band, so they
//   agree bit for bit) while the other warps' first loads are in flight;
//   then the slice is re-read -- from the L2, where pass 1 left it -- and y
//   written.
// One CTA per (pass, item).  A CTA's (pass, item) follows from its arrival
// index t (an atomic counter in the workspace, as on the staged grid path:
// (epoch << 32 | count), the last CTA to draw opens the next epoch, and
// epoch + 1 is this launch's ticket) through a fixed sequence: pass 1 of items 0 .. D - 1, then pass 1
// of item D + i and pass 2 of item i alternately, then pass 2 of the last D
// items.  Pass 2 of an item thus trails its pass 1 by 2 D + 1 arrivals, and
// D >= S keeps pass 1 of every slice of a band ahead of the band's pass 2s.
// A pass-2 CTA waits only for pass-1 items drawn before it, by CTAs that are
// running or done, so the wait ends whatever else holds the GPU; it is still
// bounded (1 s), and on timeout the CTA sets the error words and leaves its
// slice of y unwritten.  Every element is read by pass 1 of its slice before
// pass 2 writes it, so x == y (in place) is safe.
constexpr uint64_t kColsWaitNs = kTwoPassWaitNs;
constexpr unsigned kColsErrTimeout = 1u;

// The item of a COLS_TWO_PASS CTA (t: its arrival index), by the whole
// CTA.  gave_up: set when the CTA's wait ran out; its slice of y is then
// left unwritten.
template <bool LOG, bool V4>
__device__ __forceinline__ void two_pass_run(const float* x, float* y, int64_t M, int64_t N, int64_t ldx,
                                             int64_t ldy, int64_t R, int64_t S, int64_t bands, int64_t D,
                                             uint64_t* __restrict__ slots, int32_t fault, unsigned* host_err,
                                             int64_t t, uint32_t ticket, MaxSum (*red)[kBand], MaxSum* whole,
                                             volatile int* gave_up) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = lane % kLPR;
  const int g = warp * kRPW + lane / kLPR;
  int pass;
  int64_t k;
  two_pass_item(t, bands * S, D, &pass, &k);
  const int64_t band = (int64_t)((uint32_t)k / (uint32_t)S);   // both below 2^31 (checked at launch)
  const int64_t r0 = (k - band * S) * R;
  const int nrows = (int)(min(r0 + R, M) - r0);   // rows of the slice, at most R
  const int64_t j0 = band * kBand + 4 * slot;
  const int ncol = (int)max((int64_t)0, min((int64_t)4, N - j0));   // this thread's columns inside the row
  const float kNeg = neg_inf();
  const int64_t xstep = (int64_t)kGroups * ldx;   // a thread's next row in pass 1
  const float* xs = x + r0 * ldx + j0;   // the slice's first row, this thread's columns
  const uint64_t log2e2 = f2_pack(kLog2e, kLog2e);

  // V4: a thread's four columns as one float4 (x, y 16-byte aligned, strides
  // multiples of 4); otherwise four scalars
  auto load4 = [&](const float* q, bool keep, uint64_t pol) -> float4 {
    if (V4 && ncol == 4) return keep ? load_evict_last(reinterpret_cast<const float4*>(q), pol)
                                     : load_stream(reinterpret_cast<const float4*>(q));
    float4 v;
    v.x = (ncol > 0) ? q[0] : kNeg;
    v.y = (ncol > 1) ? q[1] : kNeg;
    v.z = (ncol > 2) ? q[2] : kNeg;
    v.w = (ncol > 3) ? q[3] : kNeg;
    return v;
  };
  // a batch is whole when its last row is inside the slice and the four
  // columns are (float4 access): then it needs no per-row check (pass 1's
  // row groups)
  auto whole_batch = [&](int i) { return V4 && ncol == 4 && i + (kBU - 1) * kGroups < nrows; };

  if (pass == 1) {
    const uint64_t pol = l2_evict_last_policy();
    MaxSum p[4] = {{kNeg, 0.f}, {kNeg, 0.f}, {kNeg, 0.f}, {kNeg, 0.f}};
    if (ncol > 0) {
      const float* xr = xs + g * ldx;
      for (int i = g; i < nrows; i += kBU * kGroups, xr += kBU * xstep) {
        float4 a[kBU];
        if (whole_batch(i)) {
          const float* q = xr;
#pragma unroll
          for (int u = 0; u < kBU; ++u, q += xstep) a[u] = load_evict_last(reinterpret_cast<const float4*>(q), pol);
        } else {
          const float* q = xr;
#pragma unroll
          for (int u = 0; u < kBU; ++u, q += xstep)
            a[u] = (i + u * kGroups < nrows) ? load4(q, true, pol) : make_float4(kNeg, kNeg, kNeg, kNeg);
        }
        fold_batch(p, a, log2e2);
      }
    }
    merge_column_lanes(p);
    if (lane < kLPR) {
#pragma unroll
      for (int c = 0; c < 4; ++c) red[warp][4 * slot + c] = p[c];
    }
    __syncthreads();
    if (tid < kBand && !(fault != 0 && k == 0)) {   // fault: item 0's partials never appear
      MaxSum q{kNeg, 0.f};
#pragma unroll
      for (int w = 0; w < kCW; ++w) q = merge(q, red[w][tid]);
      uint64_t* sl = slots + 2 * (k * kBand + tid);
      publish_gpu_u64(sl, tagged_word(ticket, q.m));
      publish_gpu_u64(sl + 1, tagged_word(ticket, q.s));
    }
    return;
  }

  // ---- pass 2: warps 1..7 issue their first batch of loads while warp 0
  // merges (in separate branches: the poll words and a batch do not fit the
  // register budget together); warp 0 loads its batch after the merge.  (A
  // dedicated merge warp, with seven warps holding the rows, was slower:
  // 105.2 against 102.2 us on 4096 x 16384.) ----
  const int64_t ystep = (int64_t)kGroups * ldy;
  auto load_batch2 = [&](float4 (&a)[kBU], int i, const float* xr) {
    const float* q = xr;
    if (whole_batch(i)) {
#pragma unroll
      for (int u = 0; u < kBU; ++u, q += xstep) a[u] = load_stream(reinterpret_cast<const float4*>(q));
    } else {
#pragma unroll
      for (int u = 0; u < kBU; ++u, q += xstep)
        if (i + u * kGroups < nrows) a[u] = load4(q, false, 0);
    }
  };
  const bool any2 = ncol > 0 && g < nrows;
  float4 a2[kBU];
  if (warp != 0) {
    if (any2) load_batch2(a2, g, xs + g * ldx);
  } else {
    // lane c merges column c over the band's slices, 8 slices' words in flight
    const uint64_t* col = slots + 2 * (band * S * kBand + lane);
    MaxSum acc{kNeg, 0.f};
    bool ok = true;
    const uint64_t t0 = global_timer_ns();
    for (int64_t i0 = 0; i0 < S && ok; i0 += 8) {
      const int n = (S - i0 < 8) ? (int)(S - i0) : 8;
      uint64_t wm[8], ws[8];
      uint32_t polls = 0;
      for (;;) {
        bool mine = true;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (u < n) {
            const uint64_t* w = col + 2 * (i0 + u) * kBand;
            wm[u] = ld_relaxed_gpu_u64(w);
            ws[u] = ld_relaxed_gpu_u64(w + 1);
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (u < n) mine &= ((uint32_t)(wm[u] >> 32) == ticket) && ((uint32_t)(ws[u] >> 32) == ticket);
        }
        if (__all_sync(kFullMask, mine)) break;
        // one vote, so the warp leaves together
        if ((++polls & 15u) == 0 && __any_sync(kFullMask, global_timer_ns() - t0 > kColsWaitNs)) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (u < n) acc = merge(acc, MaxSum{__uint_as_float((uint32_t)wm[u]), __uint_as_float((uint32_t)ws[u])});
      }
    }
    whole[lane] = acc;
    if (!ok && lane == 0) {
      atomicOr(&g_cols_error, kColsErrTimeout);
      if (host_err) {
        *reinterpret_cast<volatile unsigned*>(host_err) = kColsErrTimeout;
        __threadfence_system();
      }
      *gave_up = 1;
    }
  }
  __syncthreads();
  if (*gave_up || !any2) return;
  if (warp == 0) load_batch2(a2, g, xs + g * ldx);

  const ColumnScale<LOG> scale(&whole[4 * slot]);
  auto normalise = [&](const float4& v) -> float4 { return scale(v, log2e2); };
  const float* xr = xs + g * ldx;
  float* yr = y + r0 * ldy + j0 + g * ldy;
  for (int i = g;;) {   // a2 holds the batch of rows i
    if (whole_batch(i)) {
      float* o = yr;
#pragma unroll
      for (int u = 0; u < kBU; ++u, o += ystep) store_stream(reinterpret_cast<float4*>(o), normalise(a2[u]));
    } else {
      float* o = yr;
#pragma unroll
      for (int u = 0; u < kBU; ++u, o += ystep) {
        if (i + u * kGroups >= nrows) continue;
        const float4 v = normalise(a2[u]);
        if (V4 && ncol == 4) {
          store_stream(reinterpret_cast<float4*>(o), v);
        } else {
          if (ncol > 0) store_stream(o + 0, v.x);
          if (ncol > 1) store_stream(o + 1, v.y);
          if (ncol > 2) store_stream(o + 2, v.z);
          if (ncol > 3) store_stream(o + 3, v.w);
        }
      }
    }
    i += kBU * kGroups;
    if (i >= nrows) break;
    xr += kBU * xstep;
    yr += kBU * ystep;
    load_batch2(a2, i, xr);
  }
}

template <bool LOG, bool V4>
__global__ void __launch_bounds__(kCT, 4)
softmax_cols_two_pass_kernel(const float* x, float* y, int64_t M, int64_t N, int64_t ldx, int64_t ldy,
                             int64_t R, int64_t S, int64_t bands, int64_t D,
                             unsigned long long* __restrict__ arrivals, uint64_t* __restrict__ slots,
                             int32_t fault, unsigned* host_err) {
  __shared__ MaxSum red[kCW][kBand];   // per warp, after the shuffle merge
  __shared__ MaxSum whole[kBand];      // the merged pair of each column
  __shared__ unsigned drawn[2];        // arrival index, ticket
  __shared__ int gave_up;
  // every CTA draws before it lets the next kernel on the stream launch
  if (threadIdx.x == 0) {
    drawn[0] = draw_arrival(arrivals, gridDim.x, &drawn[1]);
    gave_up = 0;
  }
  __syncthreads();
  pdl_entry();
  two_pass_run<LOG, V4>(x, y, M, N, ldx, ldy, R, S, bands, D, slots, fault, host_err, (int64_t)drawn[0], drawn[1], red,
                    whole, &gave_up);
}

// --------------------------------------------------------- COLS_TWO_PHASE ---
// Grid: bands x chunks CTAs, CTA (band b, chunk c) = blockIdx.x = c * bands + b.
// Chunk c holds rows [c * chunk, min((c + 1) * chunk, M)); row group g takes
// rows g, g + kGroups, ... of it, kTP rows in flight per thread.
// part[c * N + j] is chunk c's partial of column j.
constexpr int kTP = 4;

template <bool V4>
__global__ void __launch_bounds__(kCT, 4)
softmax_cols_partials_kernel(const float* x, MaxSum* __restrict__ part, int64_t M, int64_t N,
                             int64_t ldx, int64_t chunk, int64_t bands) {
  __shared__ MaxSum red[kGroups][kBand];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = lane % kLPR;
  const int g = warp * kRPW + lane / kLPR;
  const int64_t b = blockIdx.x % bands;
  const int64_t c = blockIdx.x / bands;
  const int64_t r0 = c * chunk;
  const int64_t r1 = min(r0 + chunk, M);
  const int64_t j0 = b * kBand + 4 * slot;
  const float kNeg = neg_inf();
  pdl_entry();

  MaxSum p[4] = {{kNeg, 0.f}, {kNeg, 0.f}, {kNeg, 0.f}, {kNeg, 0.f}};
  if (j0 < N) {
    for (int64_t r = r0 + g; r < r1; r += (int64_t)kTP * kGroups) {
      float4 a[kTP];
#pragma unroll
      for (int u = 0; u < kTP; ++u) {
        const int64_t ru = r + (int64_t)u * kGroups;
        a[u] = (ru < r1) ? load_cols<V4>(x + ru * ldx, j0, N, kNeg)
                         : make_float4(kNeg, kNeg, kNeg, kNeg);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float bm = comp(a[0], k);
#pragma unroll
        for (int u = 1; u < kTP; ++u) bm = max_nan(bm, comp(a[u], k));
        rescale_to(p[k], bm);
        if (p[k].m != kNeg) {
#pragma unroll
          for (int u = 0; u < kTP; ++u) p[k].s += exp_shifted(comp(a[u], k), p[k].m);
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) red[g][4 * slot + k] = p[k];
  __syncthreads();
  if (tid < kBand) {
    const int64_t j = b * kBand + tid;
    MaxSum q{kNeg, 0.f};
    for (int k = 0; k < kGroups; ++k) q = merge(q, red[k][tid]);
    if (j < N) part[c * N + j] = q;
  }
}

// Each CTA merges, for its 32 columns, the partials of all chunks in chunk
// order (so every CTA of a band gets the same pair), then re-reads its rows
// and writes y.  Every element is read and then written by one thread, so
// x == y (in place) is safe.
template <bool V4>
__global__ void __launch_bounds__(kCT, 4)
softmax_cols_finalize_kernel(const float* x, float* y, const MaxSum* __restrict__ part, int64_t M,
                             int64_t N, int64_t ldx, int64_t ldy, int64_t chunk, int64_t chunks,
                             int64_t bands, int32_t log_out) {
  __shared__ MaxSum whole[kBand];
  __shared__ MaxSum red[kCW][kBand];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = lane % kLPR;
  const int g = warp * kRPW + lane / kLPR;
  const int64_t b = blockIdx.x % bands;
  const int64_t c = blockIdx.x / bands;
  const int64_t r0 = c * chunk;
  const int64_t r1 = min(r0 + chunk, M);
  const int64_t j0 = b * kBand + 4 * slot;
  const float kNeg = neg_inf();
  pdl_entry();
  {
    // Merge the column's chunk partials: warp w takes chunks w, w + 8, ...
    // for column `lane` of the band, loading 4 partials before merging them;
    // then thread `lane` of warp 0 merges the 8 warps' results.  The order is
    // fixed, so every CTA of the band gets the same pair.
    static_assert(kBand == 32, "one lane per column of the band");
    const int64_t j = b * kBand + lane;
    MaxSum q{kNeg, 0.f};
    if (j < N) {
      for (int64_t k0 = warp; k0 < chunks; k0 += 4 * kCW) {
        MaxSum t[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t k = k0 + (int64_t)u * kCW;
          t[u] = (k < chunks) ? part[k * N + j] : MaxSum{kNeg, 0.f};
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) q = merge(q, t[u]);
      }
    }
    red[warp][lane] = q;
    __syncthreads();
    if (warp == 0) {
      MaxSum w = red[0][lane];
#pragma unroll
      for (int k = 1; k < kCW; ++k) w = merge(w, red[k][lane]);
      whole[lane] = w;
    }
  }
  __syncthreads();
  if (j0 >= N) return;
  float m[4], inv[4], ls[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const MaxSum w = whole[4 * slot + k];
    m[k] = w.m;
    inv[k] = 1.0f / w.s;
    ls[k] = logf(w.s);
  }
  for (int64_t r = r0 + g; r < r1; r += (int64_t)kTP * kGroups) {
    float4 a[kTP];
#pragma unroll
    for (int u = 0; u < kTP; ++u) {
      const int64_t ru = r + (int64_t)u * kGroups;
      if (ru < r1) a[u] = load_cols<V4>(x + ru * ldx, j0, N, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kTP; ++u) {
      const int64_t ru = r + (int64_t)u * kGroups;
      if (ru >= r1) continue;
      float4 o;
      if (log_out) {
        o = make_float4(log_softmax_of(a[u].x, m[0], ls[0]), log_softmax_of(a[u].y, m[1], ls[1]),
                        log_softmax_of(a[u].z, m[2], ls[2]), log_softmax_of(a[u].w, m[3], ls[3]));
      } else {
        o = make_float4(exp_shifted(a[u].x, m[0]) * inv[0], exp_shifted(a[u].y, m[1]) * inv[1],
                        exp_shifted(a[u].z, m[2]) * inv[2], exp_shifted(a[u].w, m[3]) * inv[3]);
      }
      store_cols<V4>(y + ru * ldy, j0, N, o);
    }
  }
}

template <int VEC, bool LOG>
cudaError_t launch_cols_cluster_vec(const rrs_plan& p, const float* x, float* y, int64_t M,
                                    int64_t N, const Layout& l, cudaStream_t s) {
  auto kern = softmax_cols_cluster_kernel<VEC, LOG>;
  if (p.cluster > 8) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(kern, dim3((unsigned)p.grid), dim3(kCT), 0, s, p.cluster, x, y, M, N, l.ldx,
                    l.ldy);
}

template <int VEC>
cudaError_t launch_cols_cluster_v(const rrs_plan& p, const float* x, float* y, int64_t M,
                                  int64_t N, const Layout& l, cudaStream_t s) {
  return l.log_out ? launch_cols_cluster_vec<VEC, true>(p, x, y, M, N, l, s)
                   : launch_cols_cluster_vec<VEC, false>(p, x, y, M, N, l, s);
}

}  // namespace

int cols_threads() { return kCT; }
int cols_row_groups() { return kGroups; }
int cols_band() { return kBand; }
int cols_rows_per_thread_max() { return 16; }

cudaError_t launch_softmax_cols_cluster(const rrs_plan& p, const float* x, float* y, int64_t M,
                                        int64_t N, const Layout& l, cudaStream_t s) {
  if (p.threads != kCT) return cudaErrorInvalidConfiguration;
  switch (p.vec) {
    case 1: return launch_cols_cluster_v<1>(p, x, y, M, N, l, s);
    case 2: return launch_cols_cluster_v<2>(p, x, y, M, N, l, s);
    case 4: return launch_cols_cluster_v<4>(p, x, y, M, N, l, s);
    case 8: return launch_cols_cluster_v<8>(p, x, y, M, N, l, s);
    case 16: return launch_cols_cluster_v<16>(p, x, y, M, N, l, s);
    default: return cudaErrorInvalidConfiguration;
  }
}

cudaError_t launch_softmax_cols_band(const rrs_plan& p, const float* x, float* y, int64_t M, int64_t N,
                                     const Layout& l, cudaStream_t s) {
  if (p.threads != kCT || p.cluster < 1 || p.cluster > 8 || p.vec != 4) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)p.grid), block(kCT);
  return l.log_out ? launch_pdl(softmax_cols_band_kernel<true>, grid, block, 0, s, p.cluster, x, y, M, N,
                                l.ldx, l.ldy)
                   : launch_pdl(softmax_cols_band_kernel<false>, grid, block, 0, s, p.cluster, x, y, M, N,
                                l.ldx, l.ldy);
}

cudaError_t launch_softmax_cols_two_pass(const rrs_plan& p, const float* x, float* y, int64_t M,
                                         int64_t N, const Layout& l, void* workspace, int fault,
                                         unsigned* host_err, cudaStream_t s) {
  const int64_t bands = (N + kBand - 1) / kBand;
  const int64_t R = p.chunk, S = p.ctas_per_row, D = p.stages;
  if (p.threads != kCT || R < 1 || S != (M + R - 1) / R || D < S || D > bands * S ||
      p.grid != 2 * bands * S || p.grid > (int64_t)INT_MAX)
    return cudaErrorInvalidConfiguration;
  auto* arrivals = static_cast<unsigned long long*>(workspace);
  uint64_t* slots = reinterpret_cast<uint64_t*>(static_cast<unsigned char*>(workspace) + kColsArrivalBytes);
  const dim3 grid((unsigned)p.grid), block(kCT);
  auto k = p.vector_io ? (l.log_out ? softmax_cols_two_pass_kernel<true, true> : softmax_cols_two_pass_kernel<false, true>)
                       : (l.log_out ? softmax_cols_two_pass_kernel<true, false> : softmax_cols_two_pass_kernel<false, false>);
  return launch_pdl(k, grid, block, 0, s, 0, x, y, M, N, l.ldx, l.ldy, R, S, bands, D, arrivals, slots,
                    (int32_t)fault, host_err);
}

void cols_two_pass_item(int64_t t, int64_t Q, int64_t D, int* pass, int64_t* k) { two_pass_item(t, Q, D, pass, k); }

cudaError_t read_and_clear_cols_error(cudaStream_t s, unsigned* value) {
  unsigned host = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&host, g_cols_error, sizeof(host), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && host != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbolAsync(g_cols_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  *value = host;
  return e;
}

cudaError_t launch_softmax_cols_two_phase(const rrs_plan& p, const float* x, float* y, int64_t M,
                                          int64_t N, const Layout& l, void* workspace,
                                          cudaStream_t s) {
  if (p.threads != kCT) return cudaErrorInvalidConfiguration;
  MaxSum* part = static_cast<MaxSum*>(workspace);
  const int64_t bands = (N + kBand - 1) / kBand;
  const int64_t chunks = p.ctas_per_row;  // row chunks
  const dim3 grid((unsigned)(bands * chunks)), block(kCT);
  const int32_t lo = (int32_t)l.log_out;
  cudaError_t e;
  if (p.vector_io) {
    e = launch_pdl(softmax_cols_partials_kernel<true>, grid, block, 0, s, 0, x, part, M, N, l.ldx,
                   p.chunk, bands);
    if (e == cudaSuccess)
      e = launch_pdl(softmax_cols_finalize_kernel<true>, grid, block, 0, s, 0, x, y,
                     static_cast<const MaxSum*>(part), M, N, l.ldx, l.ldy, p.chunk, chunks, bands, lo);
  } else {
    e = launch_pdl(softmax_cols_partials_kernel<false>, grid, block, 0, s, 0, x, part, M, N, l.ldx,
                   p.chunk, bands);
    if (e == cudaSuccess)
      e = launch_pdl(softmax_cols_finalize_kernel<false>, grid, block, 0, s, 0, x, y,
                     static_cast<const MaxSum*>(part), M, N, l.ldx, l.ldy, p.chunk, chunks, bands, lo);
  }
  return e;
}

}  // namespace rrs
