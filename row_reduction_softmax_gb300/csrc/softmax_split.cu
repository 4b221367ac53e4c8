// Split-row softmax: a row too long for one CTA's registers is cut into
// segments owned by different CTAs, each segment's partial (max, sum) is
// formed on chip, and the partials are merged with the rule
//     m = max(m_a, m_b),   s = s_a exp(m_a - m) + s_b exp(m_b - m),
// which follows from s = sum_j exp(x_j - m) (the pages stop at the row sum
// for rows that overflow a block -- "Kernels, Triton, XLA", section
// "Reductions and tiling", "Row sum, when the row doesn't fit" -- and the
// softmax needs a max as well as a sum, hence the pair).
//
// Two variants live here:
//  * CLUSTER  -- the CTAs of one row form a thread-block cluster; each keeps
//    its segment in registers, publishes (m_c, s_c) in its shared memory, and
//    every CTA reads all peers' pairs over DSMEM after one cluster barrier.
//    One HBM read and one write per element.
//  * TWO_PHASE -- any length and alignment: kernel 1 writes each chunk's
//    online (m, s) to a workspace, kernel 2 merges a row's partials, re-reads
//    its chunk and writes y.  12 bytes of traffic per element unless the
//    re-read hits L2; the fallback for shapes the other paths do not take.
#include <cooperative_groups.h>

#include "device_common.cuh"
#include "internal.h"
#include "launch_util.h"

namespace cg = cooperative_groups;

namespace rrs {

namespace {

constexpr int kT = kSplitThreads;
constexpr int kW = kT / 32;

__device__ __forceinline__ float cta_max(float v, float* red) {
  v = warp_max(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = (lane < kW) ? red[lane] : neg_inf();
  return warp_max(r);
}

__device__ __forceinline__ float cta_sum(float v, float* red) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = (lane < kW) ? red[lane] : 0.f;
  return warp_sum(r);
}

// CTA-wide merge of per-thread partials; every thread gets the result.
// `red` must not be in use by another reduction until the caller's next
// __syncthreads().
__device__ __forceinline__ MaxSum cta_merge(MaxSum p, MaxSum* red) {
  p = warp_merge(p);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = p;
  __syncthreads();
  MaxSum q = (lane < kW) ? red[lane] : MaxSum{neg_inf(), 0.f};
  return warp_merge(q);
}

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// Arrival that orders nothing: used once this CTA's reads of its peers'
// shared memory have been consumed (their values are already in registers).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ----------------------------------------------------------------- CLUSTER ---
// Grid: clusters of `cs` CTAs along x; cluster k owns rows k, k + nclusters, ...
// V4: rank r of a cluster owns float4 columns [r*seg4, min((r+1)*seg4, n4))
// of the row, seg4 = ceil(n4 / cs) <= VEC * kT; the last rank also owns the
// N % 4 scalar tail; x, y 16-byte aligned, ldx % 4 == 0, ldy % 4 == 0.
// Scalar (any alignment and stride): rank r owns columns [r*segs,
// min((r+1)*segs, N)), segs = ceil(N / cs) <= 4 * VEC * kT, each thread four
// scalars per register slot, so that every warp load is one contiguous run.
// Shifted (rows not 16-byte aligned, but x and y misaligned alike): each row
// is read through a window that starts o = (address of the row / 4) mod 4
// floats before it, so that float4 c of the window (columns 4c - o ..
// 4c - o + 3) is 16-byte aligned; rank r owns window float4s [r*seg4w,
// (r+1)*seg4w), seg4w = ceil(ceil((N + 3) / 4) / cs).  Lanes outside [0, N)
// read neighbouring bytes of the same 16-byte chunks (mapped memory) and are
// masked; stores of the two edge float4s go lane by lane.
// LOG writes log y = (x - m) - log(s) (a template parameter, so the softmax
// instantiation keeps the register count that lets 4 CTAs share an SM).  In
// place (x == y) is safe: a CTA reads its whole segment before writing it.
constexpr int kModeScalar = 0, kModeVec = 1, kModeShift = 2;

// Slot i of thread tid into the CTA's segment of the row: one float4 (V4),
// or four scalars kT apart (the scalar layout above).
template <bool V4>
__device__ __forceinline__ void store_segment(float* yr, float4* yr4, int i, int tid, int b4, int e4, int bs,
                                              int es, const float4& o) {
  if constexpr (V4) {
    const int c = b4 + i * kT + tid;
    if (c < e4) store_stream(yr4 + c, o);
  } else {
    const int j = bs + 4 * i * kT + tid;
    if (j < es) store_stream(yr + j, o.x);
    if (j + kT < es) store_stream(yr + j + kT, o.y);
    if (j + 2 * kT < es) store_stream(yr + j + 2 * kT, o.z);
    if (j + 3 * kT < es) store_stream(yr + j + 3 * kT, o.w);
  }
}

// Slot i into a shifted window (float4 c holds columns 4c - o .. 4c - o + 3).
__device__ __forceinline__ void store_window(float* yr, float4* yw, int c, int e4w, int o, int N, const float4& v) {
  if (c >= e4w) return;
  const int lo = 4 * c - o;
  if (lo >= 0 && lo + 3 < N) {
    store_stream(yw + c, v);
    return;
  }
  if (lo >= 0 && lo < N) store_stream(yr + lo, v.x);
  if (lo + 1 >= 0 && lo + 1 < N) store_stream(yr + lo + 1, v.y);
  if (lo + 2 >= 0 && lo + 2 < N) store_stream(yr + lo + 2, v.z);
  if (lo + 3 >= 0 && lo + 3 < N) store_stream(yr + lo + 3, v.w);
}

template <int VEC, bool LOG, int MODE>
__global__ void __launch_bounds__(kT, MODE == kModeShift ? 4 : 0)
softmax_cluster_kernel(const float* x, float* y, int64_t M, int32_t N, int64_t ldx, int64_t ldy) {
  constexpr bool V4 = MODE == kModeVec;
  __shared__ float red_m[kW];
  __shared__ float red_s[kW];
  __shared__ MaxSum part;   // this CTA's (m_c, s_c), read by its peers
  __shared__ MaxSum whole;  // the merged pair of the row

  cg::cluster_group cluster = cg::this_cluster();
  const int cs = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t nclusters = gridDim.x / cs;
  const int64_t cluster_id = blockIdx.x / cs;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  const int n4 = N >> 2;
  const int rem = N & 3;
  const int seg4 = (n4 + cs - 1) / cs;
  const int b4 = rank * seg4;
  const int e4 = min(b4 + seg4, n4);
  const bool has_tail = V4 && (rank == cs - 1) && (tid < rem);
  const int segs = (N + cs - 1) / cs;   // scalar layout
  const int bs = rank * segs;
  const int es = min(bs + segs, N);
  const int seg4w = (((N + 6) >> 2) + cs - 1) / cs;   // shifted layout
  const int b4w = rank * seg4w;
  const float kNeg = neg_inf();
  pdl_entry();

  for (int64_t row = cluster_id; row < M; row += nclusters) {
    const float* xr = x + row * ldx;
    float* yr = y + row * ldy;
    const float4* xr4 = reinterpret_cast<const float4*>(xr);
    float4* yr4 = reinterpret_cast<float4*>(yr);

    float4 v[VEC];
    float t = kNeg;
    int o = 0, e4w = 0;
    const float4* xw = nullptr;
    float4* yw = nullptr;
    if constexpr (MODE == kModeShift) {
      o = (int)((reinterpret_cast<uintptr_t>(xr) >> 2) & 3);
      xw = reinterpret_cast<const float4*>(xr - o);
      yw = reinterpret_cast<float4*>(yr - o);
      e4w = min(b4w + seg4w, (N + o + 3) >> 2);
      // every load first (all in flight), then the edge masks
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const int c = b4w + i * kT + tid;
        v[i] = (c < e4w) ? load_stream(xw + c) : make_float4(kNeg, kNeg, kNeg, kNeg);
      }
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const int lo = 4 * (b4w + i * kT + tid) - o;
        if (lo < 0 || lo + 3 >= N) {   // an edge of the row (or past it: already -inf)
          v[i].x = (lo >= 0 && lo < N) ? v[i].x : kNeg;
          v[i].y = (lo + 1 >= 0 && lo + 1 < N) ? v[i].y : kNeg;
          v[i].z = (lo + 2 >= 0 && lo + 2 < N) ? v[i].z : kNeg;
          v[i].w = (lo + 3 < N) ? v[i].w : kNeg;
        }
      }
    } else if constexpr (V4) {
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const int c = b4 + i * kT + tid;
        v[i] = (c < e4) ? load_stream(xr4 + c) : make_float4(kNeg, kNeg, kNeg, kNeg);
      }
      t = has_tail ? load_stream(xr + 4 * n4 + tid) : kNeg;
    } else {
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const int j = bs + 4 * i * kT + tid;
        v[i].x = (j < es) ? load_stream(xr + j) : kNeg;
        v[i].y = (j + kT < es) ? load_stream(xr + j + kT) : kNeg;
        v[i].z = (j + 2 * kT < es) ? load_stream(xr + j + 2 * kT) : kNeg;
        v[i].w = (j + 3 * kT < es) ? load_stream(xr + j + 3 * kT) : kNeg;
      }
    }

    float mc = t;
#pragma unroll
    for (int i = 0; i < VEC; ++i) mc = max_nan(mc, max4(v[i]));
    mc = cta_max(mc, red_m);
    const bool empty = (mc == kNeg);  // segment holds only -inf (or nothing)

    float sc = 0.f;
    if constexpr (LOG) {  // keep x for the log form
      if (!empty) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          sc += (exp_shifted(v[i].x, mc) + exp_shifted(v[i].y, mc)) +
                (exp_shifted(v[i].z, mc) + exp_shifted(v[i].w, mc));
        }
        sc += exp_shifted(t, mc);
      }
    } else {
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        v[i].x = empty ? 0.f : exp_shifted(v[i].x, mc);
        v[i].y = empty ? 0.f : exp_shifted(v[i].y, mc);
        v[i].z = empty ? 0.f : exp_shifted(v[i].z, mc);
        v[i].w = empty ? 0.f : exp_shifted(v[i].w, mc);
        sc += (v[i].x + v[i].y) + (v[i].z + v[i].w);
      }
      t = empty ? 0.f : exp_shifted(t, mc);
      sc += t;
    }
    sc = cta_sum(sc, red_s);

    if (tid == 0) part = MaxSum{mc, sc};
    // publish `part` to the cluster: its writer's warp arrives with release
    // semantics; the other warps wrote nothing the peers read, and a relaxed
    // arrival spares them the release's memory barrier (measured on
    // 4096 x 32768: 168.0 -> 163.2 us)
    if (warp == 0) cluster_arrive_release();
    else cluster_arrive_relaxed();
    cluster_wait_acquire();    // every peer's `part` is visible

    if (warp == 0) {
      MaxSum q{kNeg, 0.f};
      if (lane < cs) q = *cluster.map_shared_rank(&part, lane);
      q = warp_merge(q);  // same lanes, same order in every CTA: identical result
      if (lane == 0) whole = q;
    }
    cluster_arrive_relaxed();  // done reading the peers' `part`
    __syncthreads();
    const MaxSum w = whole;
    if constexpr (LOG) {
      const float ls = logf(w.s);
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const float4 r = make_float4(log_softmax_of(v[i].x, w.m, ls), log_softmax_of(v[i].y, w.m, ls),
                                     log_softmax_of(v[i].z, w.m, ls), log_softmax_of(v[i].w, w.m, ls));
        if constexpr (MODE == kModeShift) store_window(yr, yw, b4w + i * kT + tid, e4w, o, N, r);
        else store_segment<V4>(yr, yr4, i, tid, b4, e4, bs, es, r);
      }
      if (has_tail) store_stream(yr + 4 * n4 + tid, log_softmax_of(t, w.m, ls));
    } else {
      const bool bad = !(w.s == w.s) || w.m == kNeg;  // NaN / inf / all -inf row
      const float scale = bad ? __int_as_float(0x7fc00000)
                              : (empty ? 0.f : exp_shifted(mc, w.m) / w.s);
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const float4 r = make_float4(v[i].x * scale, v[i].y * scale, v[i].z * scale, v[i].w * scale);
        if constexpr (MODE == kModeShift) store_window(yr, yw, b4w + i * kT + tid, e4w, o, N, r);
        else store_segment<V4>(yr, yr4, i, tid, b4, e4, bs, es, r);
      }
      if (has_tail) store_stream(yr + 4 * n4 + tid, t * scale);
    }
    cluster_wait_acquire();  // peers finished reading `part` before it is reused / freed
  }
}

// --------------------------------------------------------------- TWO_PHASE ---
constexpr int kUnroll = 4;

// Per-thread online partial over columns [b, e) of row xr.
template <bool V4>
__device__ __forceinline__ MaxSum chunk_partial(const float* __restrict__ xr, int64_t b, int64_t e,
                                                int64_t N) {
  MaxSum p{neg_inf(), 0.f};
  const int tid = threadIdx.x;
  int64_t scalar_from = b;
  if constexpr (V4) {
    // b is a multiple of 4; the vector part stops at e, or at N & ~3 in the last chunk.
    const int64_t e4 = ((e == N) ? (N & ~int64_t(3)) : e) >> 2;
    const float4* x4 = reinterpret_cast<const float4*>(xr);
    for (int64_t k = (b >> 2) + tid; k < e4; k += (int64_t)kT * kUnroll) {
      float4 a[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t idx = k + (int64_t)u * kT;
        // plain (L2-allocating) load: the finalize kernel re-reads this chunk
        a[u] = (idx < e4) ? x4[idx] : make_float4(neg_inf(), neg_inf(), neg_inf(), neg_inf());
      }
      float bm = max4(a[0]);
#pragma unroll
      for (int u = 1; u < kUnroll; ++u) bm = max_nan(bm, max4(a[u]));
      rescale_to(p, bm);
      if (p.m != neg_inf()) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          p.s += (exp_shifted(a[u].x, p.m) + exp_shifted(a[u].y, p.m)) +
                 (exp_shifted(a[u].z, p.m) + exp_shifted(a[u].w, p.m));
        }
      }
    }
    scalar_from = e4 << 2;
  }
  for (int64_t j = scalar_from + tid; j < e; j += kT) {
    const float v = xr[j];
    rescale_to(p, v);
    if (p.m != neg_inf()) p.s += exp_shifted(v, p.m);
  }
  return p;
}

template <bool V4>
__global__ void __launch_bounds__(kT)
softmax_partials_kernel(const float* x, MaxSum* __restrict__ part, int64_t M, int64_t N,
                        int64_t ldx, int64_t chunk, int64_t C) {
  __shared__ MaxSum red[kW];
  const int64_t work = M * C;
  pdl_entry();
  for (int64_t w = blockIdx.x; w < work; w += gridDim.x) {
    const int64_t row = w / C;
    const int64_t c = w - row * C;
    const int64_t b = c * chunk;
    const int64_t e = min(b + chunk, N);
    MaxSum p = chunk_partial<V4>(x + row * ldx, b, e, N);
    p = cta_merge(p, red);
    if (threadIdx.x == 0) part[w] = p;
    __syncthreads();
  }
}

// Each thread reads an element and then writes the same element, so x == y
// (in place) is safe.  log_out != 0 writes log y = (x - m) - log(s).
template <bool V4>
__global__ void __launch_bounds__(kT)
softmax_finalize_kernel(const float* x, float* y, const MaxSum* __restrict__ part, int64_t M,
                        int64_t N, int64_t ldx, int64_t ldy, int64_t chunk, int64_t C,
                        int32_t log_out) {
  __shared__ MaxSum red[kW];
  const int64_t work = M * C;
  const int tid = threadIdx.x;
  pdl_entry();
  for (int64_t w = blockIdx.x; w < work; w += gridDim.x) {
    const int64_t row = w / C;
    const int64_t c = w - row * C;
    // Every CTA of the row merges the same partials in the same order.
    MaxSum q{neg_inf(), 0.f};
    for (int64_t k = tid; k < C; k += kT) q = merge(q, part[row * C + k]);
    q = cta_merge(q, red);
    const float m = q.m;
    const float inv = 1.0f / q.s;
    const float ls = logf(q.s);

    const int64_t b = c * chunk;
    const int64_t e = min(b + chunk, N);
    const float* xr = x + row * ldx;
    float* yr = y + row * ldy;
    int64_t scalar_from = b;
    if constexpr (V4) {
      const int64_t e4 = ((e == N) ? (N & ~int64_t(3)) : e) >> 2;
      const float4* x4 = reinterpret_cast<const float4*>(xr);
      float4* y4 = reinterpret_cast<float4*>(yr);
      for (int64_t k = (b >> 2) + tid; k < e4; k += (int64_t)kT * kUnroll) {
        float4 a[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t idx = k + (int64_t)u * kT;
          if (idx < e4) a[u] = load_stream(x4 + idx);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t idx = k + (int64_t)u * kT;
          if (idx < e4) {
            store_stream(y4 + idx, log_out ? make_float4(log_softmax_of(a[u].x, m, ls),
                                                         log_softmax_of(a[u].y, m, ls),
                                                         log_softmax_of(a[u].z, m, ls),
                                                         log_softmax_of(a[u].w, m, ls))
                                           : make_float4(exp_shifted(a[u].x, m) * inv,
                                                         exp_shifted(a[u].y, m) * inv,
                                                         exp_shifted(a[u].z, m) * inv,
                                                         exp_shifted(a[u].w, m) * inv));
          }
        }
      }
      scalar_from = e4 << 2;
    }
    for (int64_t j = scalar_from + tid; j < e; j += kT) {
      const float v = xr[j];
      yr[j] = log_out ? log_softmax_of(v, m, ls) : exp_shifted(v, m) * inv;
    }
    __syncthreads();
  }
}

template <int VEC, bool LOG, int MODE>
cudaError_t launch_cluster_vec(const rrs_plan& p, const float* x, float* y, int64_t M, int64_t N,
                               const Layout& l, cudaStream_t s) {
  auto kern = softmax_cluster_kernel<VEC, LOG, MODE>;
  if (p.cluster > 8) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(kern, dim3((unsigned)p.grid), dim3(kT), 0, s, p.cluster, x, y, M, (int32_t)N,
                    l.ldx, l.ldy);
}

}  // namespace

cudaError_t launch_softmax_cluster(const rrs_plan& p, const float* x, float* y, int64_t M,
                                   int64_t N, const Layout& l, cudaStream_t s) {
  if (p.threads != kT) return cudaErrorInvalidConfiguration;
  const bool lg = l.log_out != 0;
  switch (p.vector_io * 16 + p.vec) {   // (mode, VEC)
    case kModeScalar * 16 + 4: return lg ? launch_cluster_vec<4, true, kModeScalar>(p, x, y, M, N, l, s)
                                         : launch_cluster_vec<4, false, kModeScalar>(p, x, y, M, N, l, s);
    case kModeScalar * 16 + 8: return lg ? launch_cluster_vec<8, true, kModeScalar>(p, x, y, M, N, l, s)
                                         : launch_cluster_vec<8, false, kModeScalar>(p, x, y, M, N, l, s);
    case kModeVec * 16 + 4: return lg ? launch_cluster_vec<4, true, kModeVec>(p, x, y, M, N, l, s)
                                      : launch_cluster_vec<4, false, kModeVec>(p, x, y, M, N, l, s);
    case kModeVec * 16 + 8: return lg ? launch_cluster_vec<8, true, kModeVec>(p, x, y, M, N, l, s)
                                      : launch_cluster_vec<8, false, kModeVec>(p, x, y, M, N, l, s);
    case kModeShift * 16 + 4: return lg ? launch_cluster_vec<4, true, kModeShift>(p, x, y, M, N, l, s)
                                        : launch_cluster_vec<4, false, kModeShift>(p, x, y, M, N, l, s);
    case kModeShift * 16 + 8: return lg ? launch_cluster_vec<8, true, kModeShift>(p, x, y, M, N, l, s)
                                        : launch_cluster_vec<8, false, kModeShift>(p, x, y, M, N, l, s);
    default: return cudaErrorInvalidConfiguration;
  }
}

cudaError_t launch_softmax_two_phase(const rrs_plan& p, const float* x, float* y, int64_t M,
                                     int64_t N, const Layout& l, void* workspace, cudaStream_t s) {
  if (p.threads != kT) return cudaErrorInvalidConfiguration;
  MaxSum* part = static_cast<MaxSum*>(workspace);
  const dim3 grid((unsigned)p.grid), block(kT);
  const int32_t lo = (int32_t)l.log_out;
  cudaError_t e;
  if (p.vector_io) {
    e = launch_pdl(softmax_partials_kernel<true>, grid, block, 0, s, 0, x, part, M, N, l.ldx,
                   p.chunk, p.ctas_per_row);
    if (e == cudaSuccess)
      e = launch_pdl(softmax_finalize_kernel<true>, grid, block, 0, s, 0, x, y,
                     static_cast<const MaxSum*>(part), M, N, l.ldx, l.ldy, p.chunk, p.ctas_per_row, lo);
  } else {
    e = launch_pdl(softmax_partials_kernel<false>, grid, block, 0, s, 0, x, part, M, N, l.ldx,
                   p.chunk, p.ctas_per_row);
    if (e == cudaSuccess)
      e = launch_pdl(softmax_finalize_kernel<false>, grid, block, 0, s, 0, x, y,
                     static_cast<const MaxSum*>(part), M, N, l.ldx, l.ldy, p.chunk, p.ctas_per_row, lo);
  }
  return e;
}

}  // namespace rrs
