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
// One CTA owns 256 query rows of one head, as two tiles of 128 (TMEM lanes),
// and walks the key tiles of 128 keys:
//   warp 9, one thread: TMA loads of both query tiles (once), then K_j and
//     V_j into two-stage rings;
//   warp 8: the tcgen05.mma issue (one elected lane), per key tile in the
//     order P_0(j) V_j, S_0(j+1) = Q_0 K_{j+1}^T, P_1(j) V_j, S_1(j+1), so
//     the tensor cores work on one query tile while the other's softmax runs;
//   warps 0..3 and 4..7: the softmax warpgroup of query tile 0 and 1, one
//     thread per query row: it reads its 128 scores from TMEM, writes
//     p = 2^(s log2e scale - m) against the row's reference m as bf16 pairs
//     over the first half of the scores' TMEM columns (the A operand of P V,
//     read from TMEM), keeps the row sum in fp32, and rescales its row of O,
//     which accumulates in TMEM across key tiles (O = alpha O + P_j V_j),
//     when m moves (only when the tile sum shows that m can no longer hold).
// TMEM per query tile: S (128 fp32 columns, P over the first 64) and O (D
// columns): 512 columns for the two tiles.  Q and K are K-major operands,
// V [keys][d] is the MN-major B operand of P V (no transposed copy); all
// are bf16 in 128-byte-swizzled tiles written by TMA; accumulators fp32.
// Every mbarrier wait is bounded (1 s): on timeout the CTA records an
// error, stops issuing, drains what it issued and frees its TMEM.
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
constexpr int kBM = 128;                          // query rows per query tile (TMEM lanes)
constexpr int kBN = 128;                          // keys per key tile
constexpr int kQT = 2;                            // query tiles per CTA
constexpr int kSoftmaxWarps = 4 * kQT;            // a warpgroup per query tile, a thread per row
constexpr int kIssuerWarp = kSoftmaxWarps;        // one thread issues the MMAs
constexpr int kLoaderWarp = kSoftmaxWarps + 1;    // one thread issues the TMA loads
constexpr int kAttnThreads = 32 * (kSoftmaxWarps + 2);
constexpr int kStages = 2;                        // K and V ring depth
constexpr int kGroupHeads = 8;                    // causal launch order: heads per group

template <int D>
struct AttnLayout {
  static constexpr int kQBytes = kBM * D * 2;   // D / 64 atom columns of 128 rows x 128 B
  static constexpr int kKBytes = kBN * D * 2;
  static constexpr int kVBytes = kBN * D * 2;   // V tile: D / 64 blocks of 128 keys x 128 B
  static constexpr int kQ = 0;                          // kQT query tiles
  static constexpr int kK = kQ + kQT * kQBytes;         // kStages stages
  static constexpr int kV = kK + kStages * kKBytes;     // kStages stages
  static constexpr int kBar = kV + kStages * kVBytes;   // mbarriers, TMEM address, abort flag
  static constexpr int kBytes = kBar + 256;
  // The dynamic base is 1024-aligned.  At least 116 KB, so that one CTA
  // fits an SM: each CTA allocates all 512 TMEM columns.
  static constexpr int kAlloc = kBytes > 116 * 1024 ? kBytes : 116 * 1024;
  // TMEM: query tile t holds S (fp32, 128 columns, P as bf16 pairs over its
  // first 64 columns) at column 256 t and O (D columns) at 256 t + 128.
  static constexpr uint32_t kTmemCols = 512;
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

// Two floats rounded to bf16 (nearest even) and packed: a in the low half
// (the even key), b in the high half (PTX cvt.rn.bf16x2.f32 puts its first
// source high).
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// max of three that propagates NaN (PTX three-input max.NaN.f32)
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// grid (ceil(L / 256), BH); block kAttnThreads.  O, LSE: fp32, O row-major [BH, L, D].
template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
attention_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, float* __restrict__ O,
                     float* __restrict__ LSE, int L, int S, int causal, float scale_log2e) {
  using Lay = AttnLayout<D>;
  extern __shared__ __align__(1024) unsigned char smem[];
  if (smem_addr(smem) & 1023u) {   // the swizzled tiles need 1024-byte alignment (uniform)
    if (threadIdx.x == 0) atomicOr(&g_attn_error, kErrConfig);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint64_t* bar_q = bars + 0;      // both query tiles landed
  uint64_t* k_full = bars + 1;     // [kStages] K tile landed
  uint64_t* k_empty = bars + 3;    // [kStages] both S MMAs of that K tile done
  uint64_t* v_full = bars + 5;     // [kStages] V tile landed
  uint64_t* v_empty = bars + 7;    // [kStages] both P V MMAs of that tile done
  uint64_t* bar_s = bars + 9;      // [kQT] S_t(j) in TMEM (and everything issued before it done)
  uint64_t* bar_p = bars + 11;     // [kQT] P_t(j) written over S_t(j) (one arrival per row)
  uint64_t* bar_o = bars + 13;     // [kQT] the last P_t V MMA done
  uint64_t* bar_drain = bars + 15; // everything the issuer issued has completed (abort path)
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 17);
  static_assert(kStages == 2 && kQT == 2, "barrier slots above");
  static_assert(Lay::kQBytes >= 4 * 32 * 32 * 4, "a query tile's buffer stages its O blocks");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Which (head, query pair) this CTA takes.  Blocks start roughly in order
  // of their linear index.  Causal CTAs differ in work (query pair p sees
  // 2p + 2 key tiles), so heads go in groups of kGroupHeads and within a
  // group every head's heaviest pair starts first, then the next: the light
  // pairs fill the end of the grid, and a group's K and V (a few MB) stay in
  // the L2 while its CTAs run.  Unmasked CTAs are all alike: head-major.
  int bh, qp;
  if (causal) {
    const int npairs = (int)gridDim.x;
    const int i = (int)blockIdx.x + npairs * (int)blockIdx.y;
    const int per_group = kGroupHeads * npairs;
    const int g = i / per_group;
    const int r = i - g * per_group;
    const int gh = min(kGroupHeads, (int)gridDim.y - g * kGroupHeads);   // heads in this group
    qp = npairs - 1 - r / gh;
    bh = g * kGroupHeads + r % gh;
  } else {
    bh = (int)blockIdx.y;
    qp = (int)blockIdx.x;
  }
  const int q0 = qp * kQT * kBM;
  // key tiles each query tile needs: all of them, or up to the causal bound
  // (query i sees keys j <= i + S - L); the later tile never needs fewer
  const int n_all = (S + kBN - 1) / kBN;
  auto tiles_for = [&](int t) {
    if (!causal) return n_all;
    const int last_key = q0 + t * kBM + kBM - 1 + (S - L);
    return min(n_all, last_key < 0 ? 0 : last_key / kBN + 1);
  };
  const int n0 = tiles_for(0), n_max = tiles_for(1);

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int t = 0; t < kQT; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], kBM);
      mbar_init(&bar_o[t], 1);
    }
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
  const uint32_t sQ = smem_addr(smem + Lay::kQ);
  const uint32_t sK = smem_addr(smem + Lay::kK);
  const uint32_t sV = smem_addr(smem + Lay::kV);
  pdl_entry();

  if (warp == kLoaderWarp) {
    // ---- one thread: Q tiles once, then K_j and V_j into a two-stage ring ----
    if (lane == 0 && n_max > 0) {
      int k_loads = 0, v_loads = 0;
      bool ok = true;
      mbar_arrive_expect_tx(bar_q, kQT * Lay::kQBytes);
#pragma unroll
      for (int t = 0; t < kQT; ++t)
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + Lay::kQ + t * Lay::kQBytes + c * kBM * 128, &tmq, c * 64, q0 + t * kBM, bh, bar_q);
      for (int j = 0; ok && j < n_max; ++j) {
        const int st = j & 1;
        const uint32_t prev = (uint32_t)(((j >> 1) - 1) & 1);   // phase of the stage's previous use
        if (j >= kStages && !(ok = wait_bar(&k_empty[st], prev, abort_flag))) break;
        mbar_arrive_expect_tx(&k_full[st], Lay::kKBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + Lay::kK + st * Lay::kKBytes + c * kBN * 128, &tmk, c * 64, j * kBN, bh, &k_full[st]);
        ++k_loads;
        if (j >= kStages && !(ok = wait_bar(&v_empty[st], prev, abort_flag))) break;
        mbar_arrive_expect_tx(&v_full[st], Lay::kVBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + Lay::kV + st * Lay::kVBytes + c * kBN * 128, &tmv, c * 64, j * kBN, bh, &v_full[st]);
        ++v_loads;
      }
      if (!ok) {   // let the last load of each stage land before the CTA can exit
        const uint64_t t0 = global_timer_ns();
        for (int st = 0; st < kStages; ++st) {
          const int nk = (k_loads - st + 1) / 2, nv = (v_loads - st + 1) / 2;   // loads into stage st
          if (nk > 0)
            while (!mbar_try_wait(&k_full[st], (uint32_t)((nk - 1) & 1)) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
          if (nv > 0)
            while (!mbar_try_wait(&v_full[st], (uint32_t)((nv - 1) & 1)) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
      }
    }
    __syncwarp();
  } else if (warp == kIssuerWarp) {
    // ---- the MMAs, in this order per key tile j:
    //   P_0(j) V_j, S_0(j+1), P_1(j) V_j, S_1(j+1)
    // so the tensor cores work on one query tile while the other tile's
    // softmax runs.  S_t(j+1) overwrites the TMEM that P_t(j) V_j reads:
    // tcgen05 MMAs issued by one thread run in issue order.  The whole warp
    // runs the loop (so the descriptors stay warp-uniform) and one elected
    // lane issues each MMA and commit. ----
    if (n_max > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN);
      constexpr uint32_t kIdO = idesc_bf16_f32_bmn(kBM, D);   // B = V [keys][d]: MN-major
      const bool leader = elect_one();
      // descriptor bases; a K step adds its byte offset >> 4 to the start
      // address field (every address stays below 2^18, inside the field)
      const uint64_t dq0 = smem_desc_sw128(sQ), dk0 = smem_desc_sw128(sK);
      const uint64_t dv0 = smem_desc_sw128_mn(sV, kBN * 128);   // d blocks of 64 are 128 keys x 128 B apart
      auto issue_s = [&](int t, int j) {
        const uint64_t dq = dq0 + (uint64_t)((t * Lay::kQBytes) >> 4);
        const uint64_t dk = dk0 + (uint64_t)(((j & 1) * Lay::kKBytes) >> 4);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4);
            mma_bf16(tmem + (uint32_t)(t * 256), dq + off, dk + off, kIdS, kk > 0);
          }
          mma_commit(&bar_s[t]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int t, int j) {
        const uint64_t dv = dv0 + (uint64_t)(((j & 1) * Lay::kVBytes) >> 4);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {   // P: 8 TMEM columns (16 bf16 keys) per step
            const uint64_t offv = (uint64_t)((kk * 16 * 128) >> 4);   // V: 16 keys = two 1024-byte atoms
            mma_bf16_tmem_a(tmem + (uint32_t)(t * 256 + 128), tmem + (uint32_t)(t * 256 + 8 * kk), dv + offv,
                            kIdO, kk > 0 || j > 0);
          }
        }
        __syncwarp();
      };
      auto commit = [&](uint64_t* bar) {
        if (leader) mma_commit(bar);
        __syncwarp();
      };
      // every lane waits; the warp proceeds only if all of them saw the phase
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(kFullMask, wait_bar(bar, parity, abort_flag));
      };
      bool ok = wait_all(bar_q, 0) && wait_all(&k_full[0], 0);
      if (ok) {
        tc_fence_after_sync();
        if (n0 > 0) issue_s(0, 0);
        issue_s(1, 0);
        commit(&k_empty[0]);
      }
      for (int j = 0; ok && j < n_max; ++j) {
        const int st = j & 1;
        const uint32_t use = (uint32_t)((j >> 1) & 1);
        const int jn = j + 1;
        if (!(ok = wait_all(&v_full[st], use))) break;
        if (j < n0) {
          if (!(ok = wait_all(&bar_p[0], (uint32_t)(j & 1)))) break;
          tc_fence_after_sync();
          issue_pv(0, j);
          if (jn < n0) {
            if (!(ok = wait_all(&k_full[jn & 1], (uint32_t)((jn >> 1) & 1)))) break;
            tc_fence_after_sync();
            issue_s(0, jn);
          } else {
            commit(&bar_o[0]);
          }
        }
        if (!(ok = wait_all(&bar_p[1], (uint32_t)(j & 1)))) break;
        tc_fence_after_sync();
        issue_pv(1, j);
        commit(&v_empty[st]);
        if (jn < n_max) {
          if (!(ok = wait_all(&k_full[jn & 1], (uint32_t)((jn >> 1) & 1)))) break;
          tc_fence_after_sync();
          issue_s(1, jn);
          commit(&k_empty[jn & 1]);
        } else {
          commit(&bar_o[1]);
        }
      }
      if (!ok) {   // every MMA issued so far completes before TMEM is freed
        const uint64_t t0 = global_timer_ns();
        commit(bar_drain);
        while (!mbar_try_wait(bar_drain, 0u) && global_timer_ns() - t0 < 2 * kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ---- softmax warpgroup t: thread r owns query row r of tile t (TMEM
    // lane r): per key tile it reads its 128 scores, updates the row max,
    // writes p = 2^(s scale log2e - m) as bf16 over the scores, and rescales
    // its row of O when the reference max moves ----
    const int t = warp >> 2;
    const int r = ((warp & 3) << 5) + lane;
    const int qrow = q0 + t * kBM + r;
    const uint32_t lane_off = (uint32_t)(((warp & 3) * 32) << 16);
    const uint32_t ts = tmem + (uint32_t)(t * 256) + lane_off;        // S_t, then P_t
    const uint32_t to = tmem + (uint32_t)(t * 256 + 128) + lane_off;  // O_t
    const int nt = (t == 0) ? n0 : n_max;
    const float kNeg = neg_inf();
    const int kmax = causal ? min(S - 1, qrow + (S - L)) : S - 1;   // last visible key
    float m = kNeg, l = 0.f;
    bool ok = true;
    // Waits are decided warp-uniformly, so the .sync.aligned TMEM accesses
    // always run on a converged warp.
    for (int j = 0; j < nt; ++j) {
      ok = __all_sync(kFullMask, ok && wait_bar(&bar_s[t], (uint32_t)(j & 1), abort_flag));
      if (!ok) break;
      tc_fence_after_sync();
      float sa[64], sb[64];
      tmem_ld64(ts, sa);
      tmem_ld64(ts + 64, sb);
      tmem_wait_ld();
      const int k0 = j * kBN;
      if (k0 + kBN - 1 > kmax) {   // the causal diagonal or the ragged end crosses this tile
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          sa[i] = (k0 + i <= kmax) ? sa[i] : kNeg;
          sb[i] = (k0 + 64 + i <= kmax) ? sb[i] : kNeg;
        }
      }
      // p = 2^(s scale log2e - m_ref) for the tile's 128 keys: one FMA (in
      // pairs) and one SFU op per key; P as bf16 pairs over S, in four chunks
      // of 32 keys (16 columns each); returns the tile's part of l in fp32
      // (four chains of pairs).  A row with no visible key so far has only
      // -inf scores: shifting by 0 instead of -inf gives 2^-inf = 0 for all
      // of them (never -inf - -inf).
      const uint64_t c2 = f2_pack(scale_log2e, scale_log2e);
      auto write_p = [&](float m_ref) -> float {
        const float m_eff = (m_ref == kNeg) ? 0.f : m_ref;
        const uint64_t nm2 = f2_pack(-m_eff, -m_eff);
        uint64_t ps2[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) ps2[c] = 0ull;   // +0.0f in both halves
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          const float* sv = (cb < 2) ? sa + 32 * cb : sb + 32 * (cb - 2);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float xa, xb;
            f2_unpack(f2_fma(f2_pack(sv[2 * i], sv[2 * i + 1]), c2, nm2), xa, xb);
            const float a = exp2_sfu(xa);
            const float b = exp2_sfu(xb);
            ps2[i & 3] = f2_add(ps2[i & 3], f2_pack(a, b));
            pk[i] = pack_bf16(a, b);
          }
          tmem_st16u(ts + 16 * cb, pk);
        }
        float ps[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) f2_unpack(ps2[c], ps[2 * c], ps[2 * c + 1]);
        return ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      };
      // m is a reference value, not the running max: O and l share it, so
      // any m gives the same softmax as long as no p overflows.  Once m is
      // set, a tile takes p against it directly; its sum bounds every p, so
      // a sum below 2^64 shows that nothing overflowed (and P, l and O stay
      // far inside the fp32 / bf16 range).  Only the first visible tile, or
      // a tile whose sum is at or above 2^64 (or NaN: a NaN or +inf score),
      // takes the tile max -- and then the whole warp, whose TMEM accesses
      // are warp-wide.
      float psum = 0.f;
      bool done = false;
      if (__all_sync(kFullMask, m != kNeg)) {
        psum = write_p(m);
        done = !__any_sync(kFullMask, !(psum < 0x1p64f));
        if (done) l += psum;
        else tmem_wait_st();   // P is written again below
      }
      if (!done) {
        // row max of the raw scores (eight chains), then scaled (scale_log2e > 0 keeps the order)
        float mx[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) mx[c] = max_nan(sa[c], sb[c]);
#pragma unroll
        for (int i = 8; i < 64; ++i) mx[i & 7] = max3_nan(mx[i & 7], sa[i], sb[i]);
        float tmax = max3_nan(max3_nan(mx[0], mx[1], mx[2]), max3_nan(mx[3], mx[4], mx[5]),
                              max_nan(mx[6], mx[7]));
        tmax *= scale_log2e;
        // the reference moves to the tile max when that exceeds it by more
        // than 2^8 (or on the first visible key), so that p <= 256 here
        float m_new = m, alpha = 1.f;
        if (m == kNeg || !(tmax <= m + 8.f)) {
          m_new = max_nan(m, tmax);
          alpha = (m == kNeg) ? 0.f : exp2_sfu(m - m_new);
        }
        // O_t holds the tiles before j at scale m.  P_t(j-1) V_{j-1} is
        // complete: S_t(j) was issued after it and bar_s covers both.
        if (j > 0 && __any_sync(kFullMask, alpha != 1.f)) {
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb) {
            float v[32];
            tmem_ld32(to + cb * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha;
            tmem_st32(to + cb * 32, v);
          }
        }
        psum = write_p(m_new);
        l = l * alpha + psum;
        m = m_new;
      }
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(&bar_p[t]);
    }
    const bool have_o = __all_sync(kFullMask, ok && nt > 0 && wait_bar(&bar_o[t], 0u, abort_flag));
    if (have_o) tc_fence_after_sync();
    // A tile with no visible key still stages its NaN rows through its Q
    // buffer: wait until the Q load (issued whenever the other tile has work)
    // has landed there.
    const bool q_ready = nt > 0 || n_max == 0 || __all_sync(kFullMask, wait_bar(bar_q, 0u, abort_flag));
    if (!*abort_flag && q_ready && (have_o || nt == 0)) {
      // O = O / l (a row that sees no key: 0 / 0 = NaN, its LSE -inf).  Each
      // warp passes its 32 rows x 32 columns blocks through shared memory
      // (XOR-swizzled, conflict-free both ways) so that every global store
      // writes 128 contiguous bytes of one row.  The staging space is this
      // tile's Q buffer: the tile's last S MMA completed before bar_o.
      const float inv = 1.0f / l;
      float* stg = reinterpret_cast<float*>(smem + Lay::kQ + t * Lay::kQBytes) + (warp & 3) * 32 * 32;
      const int row0 = q0 + t * kBM + (warp & 3) * 32;   // the warp's first row
      float* obase = O + ((size_t)bh * L + row0) * D + lane;
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        float v[32];
        if (have_o) {
          tmem_ld32(to + cb * 32, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) stg[lane * 32 + (i ^ lane)] = v[i] * inv;
        __syncwarp();
#pragma unroll 8
        for (int k = 0; k < 32; ++k)
          if (row0 + k < L) obase[(size_t)k * D + cb * 32] = stg[k * 32 + (lane ^ k)];
        __syncwarp();
      }
      if (LSE && qrow < L)
        LSE[(size_t)bh * L + qrow] = (m == kNeg) ? kNeg : (m + log2f(l)) * 0.69314718055994531f;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kIssuerWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Lay::kTmemCols);
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
cudaError_t launch_attn_d(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* o,
                          float* lse, int BH, int L, int S, int causal, float scale, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, D, L, BH, D, (uint64_t)L * D, kBM) ||
      !make_map(&mk, k, D, S, BH, D, (uint64_t)S * D, kBN) ||
      !make_map(&mv, v, D, S, BH, D, (uint64_t)S * D, kBN))
    return cudaErrorInvalidValue;
  auto kern = attention_fwd_kernel<D>;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), AttnLayout<D>::kAlloc);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((L + kQT * kBM - 1) / (kQT * kBM)), (unsigned)BH);
  return launch_pdl(kern, grid, dim3(kAttnThreads), (size_t)AttnLayout<D>::kAlloc, s, 0, mq, mk, mv, o, lse,
                    L, S, causal, scale * kLog2e);
}

}  // namespace

cudaError_t launch_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* o, float* lse,
                             int BH, int L, int S, int D, int causal, float scale, cudaStream_t s) {
  if (D == 64) return launch_attn_d<64>(q, k, v, o, lse, BH, L, S, causal, scale, s);
  if (D == 128) return launch_attn_d<128>(q, k, v, o, lse, BH, L, S, causal, scale, s);
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
