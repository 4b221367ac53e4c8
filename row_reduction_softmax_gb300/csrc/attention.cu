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
//     ring), and the tcgen05.mma issue: S = Q K^T into TMEM columns
//     [0, 128), then O_j = P V into TMEM columns [128, 128 + d);
//   warps 0..3: thread r owns query row r (TMEM lane r): reads its S row
//     from TMEM (32 columns per tcgen05.ld), takes the row max and
//     p = 2^(s log2e scale - m) on the SFU, writes p as bf16 into the
//     128-byte-swizzled P tile in shared memory (the A operand of the second
//     MMA), keeps the row sum l in fp32, and accumulates O in registers:
//     O = alpha O + O_j.
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
constexpr int kBM = 128;               // query rows per CTA
constexpr int kBN = 128;               // keys per tile
constexpr int kAttnThreads = 160;      // warps 0..3 softmax, warp 4 loads + MMA issue
constexpr int kIssuerWarp = 4;

template <int D>
struct Layout2 {
  static constexpr int kQBytes = kBM * D * 2;   // D / 64 atom columns of 128 rows x 128 B
  static constexpr int kKBytes = kBN * D * 2;
  static constexpr int kVBytes = D * kBN * 2;   // V^T tile: 2 atom columns of D rows x 128 B
  static constexpr int kPBytes = kBM * kBN * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;               // 2 stages
  static constexpr int kV = kK + 2 * kKBytes;           // 2 stages
  static constexpr int kP = kV + 2 * kVBytes;
  static constexpr int kBar = kP + kPBytes;             // mbarriers and the TMEM address
  static constexpr int kBytes = kBar + 128;
  static constexpr int kAlloc = kBytes + 1024;          // slack to align the base to 1024
  static constexpr uint32_t kTmemCols = 256;            // S: 128 columns, O_j: D columns
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

// grid (ceil(L / 128), BH); block 160.  O, LSE: fp32, O row-major [BH, L, D].
template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
attention_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, float* __restrict__ O,
                     float* __restrict__ LSE, int L, int S, int causal, float scale_log2e) {
  using Lay = Layout2<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint64_t* bar_q = bars + 0;
  uint64_t* kv_full = bars + 1;    // [2]
  uint64_t* kv_empty = bars + 3;   // [2]
  uint64_t* bar_s = bars + 5;      // S_j in TMEM
  uint64_t* bar_p = bars + 6;      // S_j read and P_j written (128 arrivals)
  uint64_t* bar_o = bars + 7;      // O_j in TMEM
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(bars + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 9);

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
    mbar_init(&kv_full[0], 1);
    mbar_init(&kv_full[1], 1);
    mbar_init(&kv_empty[0], 1);
    mbar_init(&kv_empty[1], 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_p, kBM);
    mbar_init(bar_o, 1);
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
  const uint32_t tmem_s = tmem;            // columns [0, 128)
  const uint32_t tmem_o = tmem + kBN;      // columns [128, 128 + D)
  const uint32_t sQ = smem_addr(smem + Lay::kQ);
  const uint32_t sK = smem_addr(smem + Lay::kK);
  const uint32_t sV = smem_addr(smem + Lay::kV);
  const uint32_t sP = smem_addr(smem + Lay::kP);
  pdl_entry();

  if (warp == kIssuerWarp) {
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN);
      constexpr uint32_t kIdO = idesc_bf16_f32(kBM, D);
      constexpr uint32_t kKVBytes = Lay::kKBytes + Lay::kVBytes;
      int issued = 0;                       // KV tiles whose loads were issued
      auto load_kv = [&](int j) {
        const int st = j & 1;
        mbar_arrive_expect_tx(&kv_full[st], kKVBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + Lay::kK + st * Lay::kKBytes + c * kBN * 128, &tmk, c * 64, j * kBN, bh,
                      &kv_full[st]);
#pragma unroll
        for (int c = 0; c < kBN / 64; ++c)
          tma_load_3d(smem + Lay::kV + st * Lay::kVBytes + c * D * 128, &tmv, j * kBN + c * 64, 0, bh,
                      &kv_full[st]);
        ++issued;
      };
      mbar_arrive_expect_tx(bar_q, Lay::kQBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_3d(smem + Lay::kQ + c * kBM * 128, &tmq, c * 64, q0, bh, bar_q);
      load_kv(0);
      if (n_tiles > 1) load_kv(1);
      bool ok = wait_bar(bar_q, 0, abort_flag);
      auto issue_s = [&](int j) {
        const int st = j & 1;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * 128 * 128 + (kk & 3) * 32);
          mma_bf16(tmem_s, smem_desc_sw128(sQ + off), smem_desc_sw128(sK + st * Lay::kKBytes + off),
                   kIdS, kk > 0);
        }
        mma_commit(bar_s);
      };
      int mma_tiles = 0;                    // tiles whose S MMA was issued
      if (ok && (ok = wait_bar(&kv_full[0], 0, abort_flag))) {
        issue_s(0);
        mma_tiles = 1;
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j & 1;
        if (!(ok = wait_bar(bar_p, (uint32_t)(j & 1), abort_flag))) break;   // S_j read, P_j written
        tc_fence_after_sync();
        if (j + 1 < n_tiles) {
          if (!(ok = wait_bar(&kv_full[(j + 1) & 1], (uint32_t)(((j + 1) >> 1) & 1), abort_flag))) break;
          issue_s(j + 1);
          mma_tiles = j + 2;
        }
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t offp = (uint32_t)((kk >> 2) * kBM * 128 + (kk & 3) * 32);
          const uint32_t offv = (uint32_t)((kk >> 2) * D * 128 + (kk & 3) * 32);
          mma_bf16(tmem_o, smem_desc_sw128(sP + offp), smem_desc_sw128(sV + st * Lay::kVBytes + offv),
                   kIdO, kk > 0);
        }
        mma_commit(bar_o);
        mma_commit(&kv_empty[st]);
        if (j + 2 < n_tiles) {
          if (!(ok = wait_bar(&kv_empty[st], (uint32_t)((j >> 1) & 1), abort_flag))) break;
          load_kv(j + 2);
        }
      }
      if (!ok) {
        // drain: copies issued but not yet waited on, and the last MMAs
        for (int j = 0; j < issued; ++j) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(&kv_full[j & 1], (uint32_t)((j >> 1) & 1)) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
        (void)mma_tiles;
        mma_commit(bar_o);   // one more arrival once everything issued has completed
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar_o, (uint32_t)(n_tiles & 1)) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();   // lanes 1..31 wait here for the issuing lane
  } else {
    // ---- softmax warps: thread r owns query row r ----
    const int r = threadIdx.x;                              // 0..127
    const int qrow = q0 + r;
    const uint32_t lane_off = (uint32_t)((warp * 32) << 16);
    const float kNeg = neg_inf();
    float o[D];
#pragma unroll
    for (int c = 0; c < D; ++c) o[c] = 0.f;
    float m = kNeg, l = 0.f, alpha_prev = 0.f;
    bool ok = true;
    // waits are decided warp-uniformly, so the .sync.aligned TMEM loads below
    // always run on a converged warp
    for (int j = 0; j < n_tiles; ++j) {
      if (!(ok = __all_sync(kFullMask, wait_bar(bar_s, (uint32_t)(j & 1), abort_flag)))) break;
      tc_fence_after_sync();
      const int k0 = j * kBN;
      const int kmax = causal ? min(S - 1, qrow + (S - L)) : S - 1;   // last visible key
      // pass 1: row max of the scaled, masked scores (log2 units)
      float tmax = kNeg;
#pragma unroll
      for (int cb = 0; cb < kBN / 32; ++cb) {
        float v[32];
        tmem_ld32(tmem_s + lane_off + cb * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int key = k0 + cb * 32 + i;
          const float sv = (key <= kmax) ? v[i] * scale_log2e : kNeg;
          tmax = max_nan(tmax, sv);
        }
      }
      const float m_new = max_nan(m, tmax);
      const float alpha = (m == kNeg) ? 0.f : exp2_sfu(m - m_new);
      // O_{j-1} is complete: fold it in at the previous tile's scale
      if (j > 0) {
        if (!(ok = __all_sync(kFullMask, wait_bar(bar_o, (uint32_t)((j - 1) & 1), abort_flag)))) break;
        tc_fence_after_sync();
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          float v[32];
          tmem_ld32(tmem_o + lane_off + cb * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[cb * 32 + i] = o[cb * 32 + i] * alpha_prev + v[i];
        }
      }
      // pass 2: p = 2^(s - m_new), row sum in fp32, P row as bf16 into the swizzled tile
      float psum = 0.f;
#pragma unroll
      for (int cb = 0; cb < kBN / 32; ++cb) {
        float v[32];
        tmem_ld32(tmem_s + lane_off + cb * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int key = k0 + cb * 32 + i;
          v[i] = (key <= kmax && m_new != kNeg) ? exp2_sfu(v[i] * scale_log2e - m_new) : 0.f;
          psum += v[i];
        }
        // 32 bf16 = four 16-byte chunks, chunk index q = 4 (cb % 2) + t in atom column cb / 2
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          st_shared_v4(sw128_chunk(sP, kBM, r, cb >> 1, 4 * (cb & 1) + t),
                       pack_bf16(v[8 * t + 0], v[8 * t + 1]), pack_bf16(v[8 * t + 2], v[8 * t + 3]),
                       pack_bf16(v[8 * t + 4], v[8 * t + 5]), pack_bf16(v[8 * t + 6], v[8 * t + 7]));
        }
      }
      l = l * alpha + psum;
      m = m_new;
      alpha_prev = alpha;
      fence_proxy_async_smem();   // P visible to the tensor cores
      tc_fence_before_sync();
      mbar_arrive(bar_p);
    }
    if (ok && n_tiles > 0) {
      if (__all_sync(kFullMask, wait_bar(bar_o, (uint32_t)((n_tiles - 1) & 1), abort_flag))) {
        tc_fence_after_sync();
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          float v[32];
          tmem_ld32(tmem_o + lane_off + cb * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[cb * 32 + i] = o[cb * 32 + i] * alpha_prev + v[i];
        }
      }
    }
    // O = O / l (an all-masked row: 0 / 0 = NaN, its LSE -inf)
    if (qrow < L && !*abort_flag) {
      const float inv = 1.0f / l;
      float4* orow = reinterpret_cast<float4*>(O + ((size_t)bh * L + qrow) * D);
#pragma unroll
      for (int c = 0; c < D / 4; ++c)
        orow[c] = make_float4(o[4 * c] * inv, o[4 * c + 1] * inv, o[4 * c + 2] * inv, o[4 * c + 3] * inv);
      if (LSE) LSE[(size_t)bh * L + qrow] = (m == kNeg) ? kNeg : (m + log2f(l)) * 0.69314718055994531f;
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
  return launch_pdl(kern, grid, dim3(kAttnThreads), (size_t)Layout2<D>::kAlloc, s, 0, mq, mk, mv, o, lse,
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
