// Device-side helpers shared by the softmax and row-sum kernels (sm_103a).
//
// Reductions follow the pages' structure -- per-thread values, then a
// cross-thread reduction inside the block ("Kernels, Triton, XLA", section
// "Reductions and tiling") -- mapped onto warp shuffles (xor butterfly, fixed
// order, so results are bitwise reproducible) and a shared-memory step across
// the warps that share a row.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rrs {

// log2(e): exp(t) = 2^(t * log2 e).
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFullMask = 0xffffffffu;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// max that propagates NaN (PTX max.NaN): a row holding a NaN gets a NaN
// maximum, so every output of that row is NaN, as in the naive five steps.
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(kFullMask, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
  return v;
}

// 2^t on the SFU (PTX ex2.approx.ftz.f32: relative error about 2^-22 over
// the whole range; results below the smallest normal float flush to +0).
__device__ __forceinline__ float exp2_sfu(float t) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
  return r;
}

// Packed pairs of fp32 (PTX .f32x2 arithmetic: two lanes per instruction,
// each lane rounded as the scalar operation would round it).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// exp(v - m) as 2^((v - m) log2 e).  v - m is exact where v == m, so the
// row maximum always maps to exactly 1 and tied maxima stay tied; v = -inf
// gives exactly 0; m = -inf (a row with no finite entry) gives NaN.
__device__ __forceinline__ float exp_shifted(float v, float m) {
  return exp2_sfu((v - m) * kLog2e);
}

// One output of log-softmax: log y = (v - m) - log(s), with ls = log(s) of
// the row (CUDA's logf, once per row).  v = -inf gives -inf (log 0); a NaN
// row (m or ls NaN) gives NaN, as the softmax does.
__device__ __forceinline__ float log_softmax_of(float v, float m, float ls) { return (v - m) - ls; }

__device__ __forceinline__ float max4(const float4& v) {
  return max_nan(max_nan(v.x, v.y), max_nan(v.z, v.w));
}

// 128-bit streaming accesses: x is read once and y written once, so both are
// marked evict-first to keep them from displacing lines other work reuses.
__device__ __forceinline__ float4 load_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void store_stream(float4* p, const float4& v) { __stcs(p, v); }
__device__ __forceinline__ float load_stream(const float* p) { return __ldcs(p); }
__device__ __forceinline__ void store_stream(float* p, float v) { __stcs(p, v); }

// Loads marked last use (PTX ld.global.lu: on global memory a streaming
// load, like ld.cs).  Measured on GB300, the row-register softmax on
// 8192 x 1024 runs in 11.2 us with them against 11.7 us with ld.cs (and no
// other kernel here changed), so only that kernel uses them.
__device__ __forceinline__ float4 load_last_use(const float4* p) {
  float4 v;
  asm volatile("ld.global.lu.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ float load_last_use(const float* p) {
  float v;
  asm volatile("ld.global.lu.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

// Start of every kernel launched with launch_pdl(): allow the next kernel on
// the stream to be scheduled, then wait for the previous one to complete.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_entry() {
  pdl_launch_dependents();
  pdl_wait();
}

// L2 prefetch of the 128-byte line holding p (PTX prefetch.global.L2: a
// hint that returns no data).  Issued before pdl_wait() on a row the kernel
// is about to read, it overlaps the row's DRAM latency with the previous
// kernel's last stores.  That is safe even when the previous kernel writes
// the row: the L2 is the point of coherence for global memory, so the loads
// issued after pdl_wait() see that kernel's stores whatever the prefetch
// brought in; only the timing changes.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Threads t = 0 .. nt-1 prefetch the lines of bytes [0, n) from p (every
// address stays inside the range).
__device__ __forceinline__ void prefetch_l2_range(const void* p, int64_t n, int t, int nt) {
  const char* c = static_cast<const char*>(p);
  const int64_t first = -(int64_t)(reinterpret_cast<uintptr_t>(p) & 127);  // line start, relative
  for (int64_t o = first + 128 * (int64_t)t; o < n; o += 128 * (int64_t)nt)
    prefetch_l2(c + (o < 0 ? 0 : o));
}

// Named barrier over `threads` threads (a multiple of 32) of this CTA.
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// A partial of the split-row rule: m = max over a segment, s = sum of
// exp(x - m) over it; the empty / all -inf segment is (-inf, 0).
struct MaxSum {
  float m;
  float s;
};

// Merge of two partials of disjoint segments: m = max(m_a, m_b),
// s = s_a exp(m_a - m) + s_b exp(m_b - m); a side whose max is -inf adds 0
// (never exp(-inf - -inf)).  NaN in either s propagates.
__device__ __forceinline__ MaxSum merge(MaxSum a, MaxSum b) {
  const float m = max_nan(a.m, b.m);
  if (m == neg_inf()) return {m, 0.f};
  const float ta = (a.m == neg_inf()) ? 0.f : a.s * exp_shifted(a.m, m);
  const float tb = (b.m == neg_inf()) ? 0.f : b.s * exp_shifted(b.m, m);
  return {m, ta + tb};
}

__device__ __forceinline__ MaxSum warp_merge(MaxSum p) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MaxSum q;
    q.m = __shfl_xor_sync(kFullMask, p.m, o);
    q.s = __shfl_xor_sync(kFullMask, p.s, o);
    p = merge(p, q);
  }
  return p;
}

// Online update of a per-thread partial before it absorbs a batch of values
// whose max is bm: raise p.m to max(p.m, bm) and rescale p.s to the new max.
// Afterwards the batch's terms are exp_shifted(v, p.m), to be added only
// while p.m is not -inf (an all -inf prefix contributes nothing).
__device__ __forceinline__ void rescale_to(MaxSum& p, float bm) {
  const float nm = max_nan(p.m, bm);
  if (nm != p.m) {  // raised, or became NaN (NaN compares unequal)
    p.s = (p.m == neg_inf()) ? 0.f : p.s * exp_shifted(p.m, nm);
    p.m = nm;
  }
}

}  // namespace rrs
