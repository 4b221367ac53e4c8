// Fused attention forward on the tensor cores: O = softmax(Q K^T * scale) V
// per head, with the row-wise softmax taken online over key tiles.
//
// The pages build their kernels to this point and name FlashAttention as
// the fusion of them: elementwise work, the row-wise softmax reduction, and
// the tiled matmul ("Kernels, Triton, XLA", end of "Reductions and tiling";
// "CS336 2026 Lecture 6: Kernels, Triton", the assignment paragraph and the
// summary).  Over key tiles the softmax uses the split-row merge rule of the
// rest of this library: with m the running row max and l the running sum,
// a new tile with max m' rescales by e^(m - max(m, m')).
//
// One CTA owns 128 query rows of one head and walks the key tiles of 128:
//   warp 4, one thread: TMA loads of Q (once), K and V^T tiles (two-stage
//     rings with their own barriers, K two tiles ahead), and the tcgen05.mma
//     issue: S_{j+1} = Q K_{j+1}^T into the second of two TMEM S buffers
//     while the softmax warps read S_j, then O_j = P_j V_j into TMEM columns
//     [256, 256 + d) once P_j is written;
//   warps 0..7: query row r (TMEM lane r) belongs to warps r / 32 and
//     r / 32 + 4, each taking half of the row's columns: they read S from
//     TMEM (32 columns per tcgen05.ld), exchange their halves' maxima through
//     shared memory, take p = 2^(s log2e scale - m) on the SFU, write p as
//     bf16 into the 128-byte-swizzled P tile in shared memory (the A operand
//     of the second MMA), keep their halves' row sums in fp32, and, when the
//     row max rises, rescale their half of O, which accumulates in TMEM
//     across key tiles (O = alpha O + P_j V_j).
// Operands are bf16 (K-major, 128-byte swizzle, 1024-byte atoms, written by
// TMA for Q, K, V^T and by the softmax threads for P); accumulators fp32.
// V is transposed to V^T (d x S per head) by a small kernel first, so that
// both MMAs take K-major operands.  Every mbarrier wait is bounded (1 s): on
// timeout the CTA records an error, stops issuing, drains what it issued
// and frees its TMEM.
#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include <cudaTypedefs.h>

#include "device_common.cuh"
#include "internal.h"
#include "launch_util.h"
#include "sm100_async.cuh"
#include "sm100_tcgen05.cuh"

namespace rrs {

namespace {

__device__ unsigned int g_attn_error = 0;

constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrConfig = 2u;    // the dynamic shared memory was not 1024-byte aligned
constexpr int kBM = 128;               // query rows per CTA
constexpr int kBN = 128;               // keys per tile
// Warps sharing a group of 32 query rows (each takes a part of the key
// columns and of O's columns, at least 32 of the latter).  Two measured
// faster than four on d = 128 (0.81 against 0.85 ms on 64 heads of
// 4096^2): the group barrier and exchange grow with the split.  The softmax
// warps are 4 * split, then one warp issues loads and MMAs.
template <int D>
__host__ __device__ constexpr int attn_split() { return 2; }
template <int D>
__host__ __device__ constexpr int attn_threads() { return 32 * (4 * attn_split<D>() + 1); }

template <int D>
struct Layout2 {
  static constexpr int kQBytes = kBM * D * 2;   // D / 64 atom columns of 128 rows x 128 B
  static constexpr int kKBytes = kBN * D * 2;
  static constexpr int kVBytes = D * kBN * 2;   // V^T tile: 2 atom columns of D rows x 128 B
  static constexpr int kPBytes = kBM * kBN * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;               // 2 stages
  static constexpr int kV = kK + 2 * kKBytes;           // 2 stages
  static constexpr int kP = kV + 2 * kVBytes;           // 2 buffers
  static constexpr int kBar = kP + 2 * kPBytes;         // mbarriers and the TMEM address
  static constexpr int kX = kBar + 256;   // row-max exchange [2][split][128]; the row sums reuse it
  static constexpr int kBytes = kX + 2 * attn_split<D>() * kBM * 4;
  static constexpr int kAlloc = kBytes;                 // the dynamic base is 1024-aligned
  static constexpr uint32_t kTmemCols = 512;            // S: 2 x 128 columns, O_j: D columns
};

// Bounded parity wait; false (and the error word set) if it ran out or the
// CTA is aborting.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicOr(&g_attn_error, kErrTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
  return true;
}

// Address of the 16-byte chunk q (0..7) of row r in a K-major tile whose
// atom column holds `rows` rows (128-byte swizzle: chunk q of row r sits at
// chunk position q ^ (r % 8) of its 128-byte row).
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t base, int rows, int r, int col_atom, int q) {
  return base + (uint32_t)(col_atom * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((q ^ (r & 7)) << 4));
}

// Two floats rounded to bf16 (nearest even) and packed: a in the low half,
// b in the high half (PTX cvt.rn.bf16x2.f32 puts its first source high).
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// grid (ceil(L / 128), BH); block 32 * (4 kSplit + 1).  O, LSE: fp32, O row-major [BH, L, D].
template <int D>
__global__ void __launch_bounds__(attn_threads<D>(), 1)
attention_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, float* __restrict__ O,
                     float* __restrict__ LSE, int L, int S, int causal, float scale_log2e) {
  using Lay = Layout2<D>;
  constexpr int kSplit = attn_split<D>();
  constexpr int kSoftmaxWarps = 4 * kSplit;
  constexpr int kIssuerWarp = kSoftmaxWarps;
  extern __shared__ __align__(1024) unsigned char smem[];
  if (smem_addr(smem) & 1023u) {   // the swizzled tiles need 1024-byte alignment (uniform)
    if (threadIdx.x == 0) atomicOr(&g_attn_error, kErrConfig);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint64_t* bar_q = bars + 0;
  uint64_t* k_full = bars + 1;     // [2] K tile landed
  uint64_t* k_empty = bars + 3;    // [2] S MMA of that K tile done
  uint64_t* v_full = bars + 5;     // [2] V^T tile landed
  uint64_t* v_empty = bars + 7;    // [2] P V MMA of that tile done
  uint64_t* bar_s = bars + 9;      // [2] S_j in TMEM buffer j % 2
  // [2] S_j read and P_j written into P buffer j % 2 (one arrival per softmax
  // thread).  One barrier per buffer: the softmax warps may finish tile j + 1
  // before the issuer sees tile j, but tile j + 2 needs P_j V_j, issued only
  // after that, so no barrier runs two phases ahead of its waiter.
  uint64_t* bar_p = bars + 11;
  uint64_t* bar_o = bars + 13;     // [2] P_j V_j accumulated (P buffer j % 2 free again)
  uint64_t* bar_drain = bars + 15; // everything issued has completed (abort path)
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 17);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int q0 = blockIdx.x * kBM;
  // key tiles this query tile needs: all of them, or up to the causal bound
  // (query i sees keys j <= i + S - L)
  int n_tiles = (S + kBN - 1) / kBN;
  if (causal) {
    const int last_key = q0 + kBM - 1 + (S - L);
    n_tiles = min(n_tiles, last_key < 0 ? 0 : last_key / kBN + 1);
  }

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&bar_s[i], 1);
    }
    mbar_init(&bar_p[0], 32 * kSoftmaxWarps);
    mbar_init(&bar_p[1], 32 * kSoftmaxWarps);
    mbar_init(&bar_o[0], 1);
    mbar_init(&bar_o[1], 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kIssuerWarp) {
    tmem_alloc(tmem_base_slot, Lay::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_base_slot;
  const uint32_t tmem_s = tmem;              // two S buffers: columns [0, 128) and [128, 256)
  const uint32_t tmem_o = tmem + 2 * kBN;    // columns [256, 256 + D)
  const uint32_t sQ = smem_addr(smem + Lay::kQ);
  const uint32_t sK = smem_addr(smem + Lay::kK);
  const uint32_t sV = smem_addr(smem + Lay::kV);
  const uint32_t sP = smem_addr(smem + Lay::kP);
  pdl_entry();

  if (warp == kIssuerWarp) {
    // One thread: loads two tiles ahead, S_{j+1} (into the other S buffer)
    // while the softmax warps work on S_j, then P_j V_j once P_j is written.
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN);
      constexpr uint32_t kIdO = idesc_bf16_f32(kBM, D);
      int k_loads = 0, v_loads = 0, pv_done = 0;
      auto load_k = [&](int j) {
        const int st = j & 1;
        mbar_arrive_expect_tx(&k_full[st], Lay::kKBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + Lay::kK + st * Lay::kKBytes + c * kBN * 128, &tmk, c * 64, j * kBN, bh,
                      &k_full[st]);
        ++k_loads;
      };
      auto load_v = [&](int j) {
        const int st = j & 1;
        mbar_arrive_expect_tx(&v_full[st], Lay::kVBytes);
#pragma unroll
        for (int c = 0; c < kBN / 64; ++c)
          tma_load_3d(smem + Lay::kV + st * Lay::kVBytes + c * D * 128, &tmv, j * kBN + c * 64, 0, bh,
                      &v_full[st]);
        ++v_loads;
      };
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (!wait_bar(&k_full[st], (uint32_t)((j >> 1) & 1), abort_flag)) return false;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * 128 * 128 + (kk & 3) * 32);
          mma_bf16(tmem_s + st * kBN, smem_desc_sw128(sQ + off),
                   smem_desc_sw128(sK + st * Lay::kKBytes + off), kIdS, kk > 0);
        }
        mma_commit(&bar_s[st]);
        mma_commit(&k_empty[st]);
        return true;
      };
      mbar_arrive_expect_tx(bar_q, Lay::kQBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_3d(smem + Lay::kQ + c * kBM * 128, &tmq, c * 64, q0, bh, bar_q);
      load_k(0);
      load_v(0);
      if (n_tiles > 1) {
        load_k(1);
        load_v(1);
      }
      bool ok = wait_bar(bar_q, 0, abort_flag);
      ok = ok && issue_s(0);
      if (n_tiles > 1) ok = ok && issue_s(1);
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j & 1;
        const uint32_t use = (uint32_t)((j >> 1) & 1);
        if (j + 2 < n_tiles) {   // K stage st is free once S_j is done
          if (!(ok = wait_bar(&k_empty[st], use, abort_flag))) break;
          load_k(j + 2);
        }
        if (!(ok = wait_bar(&bar_p[st], use, abort_flag))) break;   // S_j read, P_j written
        if (!(ok = wait_bar(&v_full[st], use, abort_flag))) break;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t offp = (uint32_t)((kk >> 2) * kBM * 128 + (kk & 3) * 32);
          const uint32_t offv = (uint32_t)((kk >> 2) * D * 128 + (kk & 3) * 32);
          mma_bf16(tmem_o, smem_desc_sw128(sP + st * Lay::kPBytes + offp),
                   smem_desc_sw128(sV + st * Lay::kVBytes + offv), kIdO,
                   kk > 0 || j > 0);   // O accumulates in TMEM across key tiles
        }
        mma_commit(&bar_o[st]);
        mma_commit(&v_empty[st]);
        ++pv_done;
        if (j + 2 < n_tiles) {   // V stage st is free once P_j V_j is done
          if (!(ok = wait_bar(&v_empty[st], use, abort_flag))) break;
          load_v(j + 2);
          ok = issue_s(j + 2);   // S buffer st was read by the softmax warps (bar_p above)
        }
      }
      if (!ok) {
        // drain what was issued: the last load of each stage, then every MMA
        const uint64_t t0 = global_timer_ns();
        for (int st = 0; st < 2; ++st) {
          const int nk = (k_loads - st + 1) / 2, nv = (v_loads - st + 1) / 2;   // loads into stage st
          if (nk > 0)
            while (!mbar_try_wait(&k_full[st], (uint32_t)((nk - 1) & 1)) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
          if (nv > 0)
            while (!mbar_try_wait(&v_full[st], (uint32_t)((nv - 1) & 1)) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
        mma_commit(bar_drain);   // arrives once everything issued has completed
        (void)pv_done;
        while (!mbar_try_wait(bar_drain, 0u) && global_timer_ns() - t0 < 2 * kWaitLimitNs) {
        }
      }
    }
    __syncwarp();   // lanes 1..31 wait here for the issuing lane
  } else {
    // ---- softmax warps: warps w, w + 4, ... (kSplit of them) share query
    // rows 32 (w % 4) .. + 31 (TMEM lanes); warp w takes part w / 4 of every
    // key tile's columns and of O's columns ----
    constexpr int kHalf = kBN / kSplit;    // key columns per thread and tile
    constexpr int kDHalf = D / kSplit;     // O columns per thread
    const int h = warp >> 2;
    const int r = ((warp & 3) << 5) + lane;                 // query row within the tile
    const int qrow = q0 + r;
    const uint32_t lane_off = (uint32_t)(((warp & 3) * 32) << 16);
    const int pair_bar = 1 + (warp & 3);                     // named barrier of the row group's warps
    float* xmax = reinterpret_cast<float*>(smem + Lay::kX);          // [tile parity][part][row]
    const float kNeg = neg_inf();
    const int kmax = causal ? min(S - 1, qrow + (S - L)) : S - 1;   // last visible key
    float m = kNeg, l = 0.f;
    bool ok = true;
    // Waits are decided warp-uniformly, so the .sync.aligned TMEM accesses
    // below always run on a converged warp.  After a failed wait the loop
    // still runs to the end (the waits then return at once and the values
    // are discarded), so a row group's warps meet at every group barrier.
    for (int j = 0; j < n_tiles; ++j) {
      const uint32_t s_buf = tmem_s + (uint32_t)((j & 1) * kBN + h * kHalf) + lane_off;
      ok = __all_sync(kFullMask, ok && wait_bar(&bar_s[j & 1], (uint32_t)((j >> 1) & 1), abort_flag));
      tc_fence_after_sync();
      const int k0 = j * kBN + h * kHalf;
      // this part of the row's raw scores, masked, kept in registers (one
      // TMEM load of the 64 columns, one wait)
      static_assert(kHalf == 64, "one 64-column TMEM load per thread and tile");
      float sv[kHalf];
      tmem_ld64(s_buf, sv);
      tmem_wait_ld();
      if (k0 + kHalf - 1 > kmax) {   // the causal diagonal or the ragged end crosses this part
#pragma unroll
        for (int i = 0; i < kHalf; ++i) sv[i] = (k0 + i <= kmax) ? sv[i] : kNeg;
      }
      // max of the raw scores, then scaled (scale_log2e > 0 keeps the order)
      float tmax = kNeg;
#pragma unroll
      for (int i = 0; i < kHalf; ++i) tmax = max_nan(tmax, sv[i]);
      tmax *= scale_log2e;
      float* xm = xmax + (j & 1) * kSplit * kBM;
      xm[h * kBM + r] = tmax;
      named_barrier(pair_bar, 32 * kSplit);
#pragma unroll
      for (int k = 0; k < kSplit; ++k) tmax = max_nan(tmax, xm[k * kBM + r]);
      // The reference max moves only when the tile's max exceeds it by more
      // than 2^8 (or on the first visible key): p = 2^(s - m) then stays
      // below 256, exact in fp32 and in bf16's range, and O is rescaled far
      // less often.  The result is the same softmax: O and l share m.
      float m_new = m, alpha = 1.f;
      if (m == kNeg || !(tmax <= m + 8.f)) {
        m_new = max_nan(m, tmax);
        alpha = (m == kNeg) ? 0.f : exp2_sfu(m - m_new);
      }
      // O holds the tiles before j at scale m: if m moves, wait for P_{j-1} V_{j-1}
      // and rescale O to m_new
      bool waited_prev = false;
      if (j > 0 && __any_sync(kFullMask, alpha != 1.f)) {
        ok = __all_sync(kFullMask, ok && wait_bar(&bar_o[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1), abort_flag));
        waited_prev = true;
        tc_fence_after_sync();
        if (ok) {
          const uint32_t ta = tmem_o + lane_off + (uint32_t)(h * kDHalf);
          if constexpr (kDHalf == 64) {   // one load, one wait
            float v[64];
            tmem_ld64(ta, v);
            tmem_wait_ld();
            float lo[32], hi[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              lo[i] = v[i] * alpha;
              hi[i] = v[32 + i] * alpha;
            }
            tmem_st32(ta, lo);
            tmem_st32(ta + 32, hi);
          } else {
#pragma unroll
            for (int cb = 0; cb < kDHalf / 32; ++cb) {
              float v[32];
              tmem_ld32(ta + cb * 32, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] *= alpha;
              tmem_st32(ta + cb * 32, v);
            }
          }
          tmem_wait_st();
        }
      }
      // P buffer j % 2 was last read by P_{j-2} V_{j-2} (done if P_{j-1} V_{j-1} is)
      if (j >= 2 && !waited_prev) {
        ok = __all_sync(kFullMask, ok && wait_bar(&bar_o[j & 1], (uint32_t)(((j - 2) >> 1) & 1), abort_flag));
        tc_fence_after_sync();
      }
      const uint32_t sPj = sP + (uint32_t)((j & 1) * Lay::kPBytes);
      // p = 2^(s - m_new), this part's sum in fp32, P as bf16 into the swizzled tile
      float psum = 0.f;
#pragma unroll
      for (int cb = 0; cb < kHalf / 32; ++cb) {
        float v[32];
        if (m_new != kNeg) {   // p = 2^(s scale log2e - m): one FMA and one SFU op per key
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[i] = exp2_sfu(fmaf(sv[cb * 32 + i], scale_log2e, -m_new));
            psum += v[i];
          }
        } else {   // no visible key yet
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        // keys kc = h * kHalf + cb * 32 + 8 t .. + 7: atom column kc / 64, 16-byte chunk (kc % 64) / 8
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int kc = h * kHalf + cb * 32 + 8 * t;
          st_shared_v4(sw128_chunk(sPj, kBM, r, kc >> 6, (kc & 63) >> 3),
                       pack_bf16(v[8 * t + 0], v[8 * t + 1]), pack_bf16(v[8 * t + 2], v[8 * t + 3]),
                       pack_bf16(v[8 * t + 4], v[8 * t + 5]), pack_bf16(v[8 * t + 6], v[8 * t + 7]));
        }
      }
      l = l * alpha + psum;
      m = m_new;
      fence_proxy_async_smem();   // P (and the rescaled O) visible to the tensor cores
      tc_fence_before_sync();
      mbar_arrive(&bar_p[j & 1]);
    }
    // the row sum is the sum of the row group's parts (xsum: the exchange
    // buffer of the parity the last tile did not use, free since its barrier)
    float* xsum = xmax + ((n_tiles & 1) * kSplit * kBM);
    xsum[h * kBM + r] = l;
    named_barrier(pair_bar, 32 * kSplit);
    float l_row = 0.f;
#pragma unroll
    for (int k = 0; k < kSplit; ++k) l_row += xsum[k * kBM + r];
    const bool have_o = __all_sync(kFullMask, ok && n_tiles > 0 &&
                                                  wait_bar(&bar_o[(n_tiles - 1) & 1],
                                                           (uint32_t)(((n_tiles - 1) >> 1) & 1), abort_flag));
    if (have_o) tc_fence_after_sync();
    if (!*abort_flag && (have_o || n_tiles == 0)) {
      // O = O / l (a row that sees no key: 0 / 0 = NaN, its LSE -inf)
      const float inv = 1.0f / l_row;
      float* orow = O + ((size_t)bh * L + qrow) * D + h * kDHalf;
#pragma unroll
      for (int cb = 0; cb < kDHalf / 32; ++cb) {
        float v[32];
        if (have_o) {
          tmem_ld32(tmem_o + lane_off + (uint32_t)(h * kDHalf + cb * 32), v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        if (qrow < L) {
          float4* o4 = reinterpret_cast<float4*>(orow + cb * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o4[i] = make_float4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
        }
      }
      if (LSE && h == 0 && qrow < L)
        LSE[(size_t)bh * L + qrow] = (m == kNeg) ? kNeg : (m + log2f(l_row)) * 0.69314718055994531f;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kIssuerWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

// V [BH, S, D] -> V^T [BH, D, ldt] (bf16), 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) transpose_v_kernel(const uint16_t* __restrict__ v,
                                                          uint16_t* __restrict__ vt, int S, int D,
                                                          int ldt) {
  __shared__ uint16_t tile[32][33];
  pdl_entry();
  const int bh = blockIdx.z;
  const int s0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
  const uint16_t* src = v + (size_t)bh * S * D;
  uint16_t* dst = vt + (size_t)bh * D * ldt;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int s = s0 + i, d = d0 + threadIdx.x;
    if (s < S && d < D) tile[i][threadIdx.x] = src[(size_t)s * D + d];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int d = d0 + i, s = s0 + threadIdx.x;
    if (s < S && d < D) dst[(size_t)d * ldt + s] = tile[threadIdx.x][i];
  }
}

// ---- host: tensor maps ----
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D bf16 map over [dim2][dim1][dim0] (dim0 contiguous, row strides in
// elements), box {64, box1, 1}, 128-byte swizzle, out-of-range reads 0.
bool make_map(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
              uint64_t stride1_elems, uint64_t stride2_elems, uint32_t box1) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {dim0, dim1, dim2};
  const cuuint64_t strides[2] = {stride1_elems * 2, stride2_elems * 2};
  const cuuint32_t box[3] = {64, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

std::mutex g_attr_mu;
std::set<std::pair<const void*, int>> g_attr_done;

cudaError_t allow_smem(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (g_attr_done.count({kernel, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g_attr_done.insert({kernel, dev});
  return e;
}

template <int D>
cudaError_t launch_attn_d(const uint16_t* q, const uint16_t* k, const uint16_t* vt, int ldt, float* o,
                          float* lse, int BH, int L, int S, int causal, float scale, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, D, L, BH, D, (uint64_t)L * D, kBM) ||
      !make_map(&mk, k, D, S, BH, D, (uint64_t)S * D, kBN) ||
      !make_map(&mv, vt, S, D, BH, ldt, (uint64_t)D * ldt, D))
    return cudaErrorInvalidValue;
  auto kern = attention_fwd_kernel<D>;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), Layout2<D>::kAlloc);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((L + kBM - 1) / kBM), (unsigned)BH);
  return launch_pdl(kern, grid, dim3(attn_threads<D>()), (size_t)Layout2<D>::kAlloc, s, 0, mq, mk, mv, o, lse,
                    L, S, causal, scale * kLog2e);
}

}  // namespace

int attention_vt_stride(int S) { return (S + 7) / 8 * 8; }

cudaError_t launch_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* vt_ws,
                             float* o, float* lse, int BH, int L, int S, int D, int causal, float scale,
                             cudaStream_t s) {
  const int ldt = attention_vt_stride(S);
  const dim3 tgrid((unsigned)((S + 31) / 32), (unsigned)((D + 31) / 32), (unsigned)BH);
  cudaError_t e = launch_pdl(transpose_v_kernel, tgrid, dim3(32, 8), 0, s, 0, v, vt_ws, S, D, ldt);
  if (e != cudaSuccess) return e;
  if (D == 64) return launch_attn_d<64>(q, k, vt_ws, ldt, o, lse, BH, L, S, causal, scale, s);
  if (D == 128) return launch_attn_d<128>(q, k, vt_ws, ldt, o, lse, BH, L, S, causal, scale, s);
  return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_attn_error(cudaStream_t s, unsigned* value) {
  unsigned host = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&host, g_attn_error, sizeof(host), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && host != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbolAsync(g_attn_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  *value = host;
  return e;
}

}  // namespace rrs
