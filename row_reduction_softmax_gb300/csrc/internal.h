// Host-side interface between the C ABI (capi.cu) and the kernel translation
// units.  Not part of the public ABI: every symbol here has hidden visibility.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "rrs.h"

namespace rrs {

// ---- argument checks and error reporting shared by every entry point
// (capi.cu).  fail* record the calling thread's message for rrs_last_error
// and return the status; every entry point starts with clear_last_error().
void clear_last_error();
int fail(int status, const std::string& msg);
int fail_cuda(cudaError_t e, const char* what);
// RRS_OK if p is device memory of device `dev` or managed memory.
int check_device_pointer(const void* p, int dev, const char* name);
// M, N >= 0, ld >= max(N, 1), no overflow; *extent = elements spanned by a
// matrix of M rows of N entries at stride ld (0 when M or N is 0).
int check_shape(int64_t M, int64_t N, int64_t ld, int64_t* extent);
bool overlaps(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes);
// RRS_ERR_TIMEOUT (with its message) while a GRID kernel's timeout on `dev`
// has not been collected by rrs_device_error(); reads one host word and
// allocates nothing.
int check_no_pending_timeout(int dev);
// The plan softmax_rows would launch for these arguments (one stride for x
// and y) on device `dev`: true and *p set; false if the planner refuses the
// shape.  Leaves rrs_last_error clear.
bool plan_like_softmax_rows(const float* x, const float* y, int64_t M, int64_t N, int64_t ld, int dev,
                            rrs_plan* p);
// The device address of `dev`'s host error word if an earlier call made it,
// else null; allocates nothing.
unsigned* host_err_word_if_made(int dev);

// Per-device facts the planner needs, queried once per device.
struct DeviceInfo {
  int sm_count = 0;
  int smem_optin = 0;       // max dynamic shared memory per CTA (opt-in), bytes
  int cluster_launch = 0;   // thread-block clusters supported
};

// Row strides of x and y (elements) and the output form: 0 = softmax,
// 1 = log-softmax.  x == y with ldx == ldy is an in-place call.
struct Layout {
  int64_t ldx = 0;
  int64_t ldy = 0;
  int log_out = 0;
};

// Tuning limits shared by the planner and the launchers.
constexpr int kRowRegsMaxVec = 16;       // float4 registers per thread (warp-per-row)
constexpr int kSplitThreads = 256;       // CTA size of the cluster / two-phase kernels
constexpr int kClusterVec = 8;           // float4 per thread in a cluster CTA segment
constexpr int kClusterMax = 16;          // largest cluster (non-portable beyond 8)
constexpr int64_t kChunkAlign = 1024;    // two-phase chunk granularity (elements)
constexpr int64_t kGridArrivalBytes = 128;  // GRID workspace: the arrival counter, before the slots


// ---- softmax launchers (return the launch's cudaError_t) ----
// Every softmax launcher takes the strides and output form as a Layout;
// the staged launchers (ROW_STAGED, GRID) write the softmax only.
cudaError_t launch_softmax_row_regs(const rrs_plan& p, const float* x, float* y, int64_t M,
                                    int64_t N, const Layout& l, cudaStream_t s);
cudaError_t launch_softmax_cluster(const rrs_plan& p, const float* x, float* y, int64_t M,
                                   int64_t N, const Layout& l, cudaStream_t s);
cudaError_t launch_softmax_two_phase(const rrs_plan& p, const float* x, float* y, int64_t M,
                                     int64_t N, const Layout& l, void* workspace, cudaStream_t s);

// Persistent TMA-staged kernels (softmax_staged.cu): ROW_STAGED plans with
// vec > 0 run staged_rows (rows in registers), vec == 0 run staged_long
// (a row staged as <= 4 shared-memory sub-tiles).
int staged_header_bytes();
int staged_max_stages();
int staged_threads();
int staged_consumer_warps();
int grid_threads();
int grid_partial_threads();
cudaError_t launch_softmax_staged_rows(const rrs_plan& p, const float* x, float* y, int64_t M,
                                       int64_t N, const Layout& l, cudaStream_t s);
cudaError_t launch_softmax_staged_long(const rrs_plan& p, const float* x, float* y, int64_t M,
                                       int64_t N, const Layout& l, cudaStream_t s);
// GRID plans: rows split over a grid of R * C <= SMs CTAs (one per SM; a
// CTA takes its row group and segment in arrival order, so a row's CTAs
// are resident together; programmatic dependent launch).  `workspace`
// (zero-filled when allocated) holds the arrival counter, which also hands
// each launch its ticket, in its first kGridArrivalBytes, then 16 bytes per
// (row, segment) slot.
// `fault` != 0 (testing only, rrs_inject_fault): CTA 0 never publishes the
// partial of its first segment, so its row's waits run out.  `host_err`
// (device address of a mapped, pinned host word, or null) is set to
// RRS_ERR_TIMEOUT when a wait runs out.
cudaError_t launch_softmax_staged_grid(const rrs_plan& p, const float* x, float* y, int64_t M,
                                       int64_t N, const Layout& l, void* workspace, int fault,
                                       unsigned* host_err, cudaStream_t s);

// Testing only: `ctas` CTAs of one thread and `smem_bytes` of dynamic shared
// memory each, which hold their SMs for `ns` nanoseconds (global timer) and
// return on their own.
cudaError_t launch_occupy(int ctas, int smem_bytes, int64_t ns, cudaStream_t s);

// ---- ROW_TWO_PASS (softmax_rows_two_pass.cu): plans carry chunk (floats
// per item, rows_two_pass_chunk()), ctas_per_row (S, chunks per row),
// stages (the lag D, S <= D <= M S), grid = 2 M S and vector_io (float4
// when x, y, the strides and N allow); the workspace holds the arrival
// counter in its first kRowsTwoPassArrivalBytes, then 16 bytes per (row,
// chunk).  fault != 0: item 0's pair is never published (fault injection).
constexpr int64_t kRowsTwoPassArrivalBytes = 128;
int rows_two_pass_threads();
int rows_two_pass_chunk();
cudaError_t launch_softmax_rows_two_pass(const rrs_plan& p, const float* x, float* y, int64_t M, int64_t N,
                                         const Layout& l, void* workspace, int fault, unsigned* host_err,
                                         cudaStream_t s);
cudaError_t read_and_clear_rows_two_pass_error(cudaStream_t s, unsigned* value);

// ---- column softmax (softmax_cols.cu): COLS_CLUSTER plans carry cluster
// (CTAs per band of cols_band() columns) and vec (rows per thread; a CTA
// holds cols_row_groups() x vec rows); COLS_TWO_PHASE plans carry
// ctas_per_row (row chunks) and chunk (rows per chunk), workspace chunks x N
// (max, sum) pairs.
int cols_threads();
int cols_band();
int cols_row_groups();
int cols_rows_per_thread_max();
cudaError_t launch_softmax_cols_cluster(const rrs_plan& p, const float* x, float* y, int64_t M,
                                        int64_t N, const Layout& l, cudaStream_t s);
// COLS_BAND plans carry cluster (CTAs per band, <= 8) and rows_per_cta.
cudaError_t launch_softmax_cols_band(const rrs_plan& p, const float* x, float* y, int64_t M, int64_t N,
                                     const Layout& l, cudaStream_t s);
cudaError_t launch_softmax_cols_two_phase(const rrs_plan& p, const float* x, float* y, int64_t M,
                                          int64_t N, const Layout& l, void* workspace,
                                          cudaStream_t s);
// COLS_TWO_PASS plans carry chunk (rows per slice, R), ctas_per_row (slices
// per band, S = ceil(M / R)), stages (the lag D, S <= D <= bands x S) and
// grid = 2 x bands x S; the workspace holds the arrival counter in its first
// kColsArrivalBytes, then 16 bytes per (band, slice, column).  fault != 0:
// item 0's partials are never published (fault injection).  host_err: the
// mapped host error word (may be null).
constexpr int64_t kColsArrivalBytes = 128;
cudaError_t launch_softmax_cols_two_pass(const rrs_plan& p, const float* x, float* y, int64_t M,
                                         int64_t N, const Layout& l, void* workspace, int fault,
                                         unsigned* host_err, cudaStream_t s);
// The (pass, item) of arrival index t of a COLS_TWO_PASS launch with Q items
// per pass and lag D (host copy of the kernel's sequence, for tests).
void cols_two_pass_item(int64_t t, int64_t Q, int64_t D, int* pass, int64_t* k);

// ---- row-reduction launchers (row_sum.cu): op is one of kOp* ----
constexpr int kOpSum = 0;
constexpr int kOpMax = 1;
constexpr int kOpMean = 2;
cudaError_t launch_row_reduce_rows(int op, const rrs_plan& p, const float* x, float* out,
                                   int64_t M, int64_t N, int64_t ld, cudaStream_t s);
cudaError_t launch_row_reduce_split(int op, const rrs_plan& p, const float* x, float* out,
                                    int64_t M, int64_t N, int64_t ld, void* workspace,
                                    cudaStream_t s);
// out[0..M) = v (the result for rows with N == 0).
cudaError_t launch_fill(float* out, int64_t M, float v, cudaStream_t s);

// ---- elementwise GeLU (gelu.cu) ----
int gelu_threads();
cudaError_t launch_gelu(const float* x, float* y, int64_t n, int sm_count, cudaStream_t s);

// ---- fused attention forward (attention.cu) ----
// q, k, v: bf16 bit patterns, [BH, L | S, D] contiguous, 16-byte aligned;
// o: fp32 [BH, L, D]; lse: fp32 [BH, L] or null.  D is 64 or 128.
cudaError_t launch_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* o, float* lse,
                             int BH, int L, int S, int D, int causal, float scale, cudaStream_t s);

// ---- device error words (set by kernels whose bounded waits ran out) ----
cudaError_t read_and_clear_staged_error(cudaStream_t s, unsigned* value);
cudaError_t read_and_clear_attn_error(cudaStream_t s, unsigned* value);
cudaError_t read_and_clear_cols_error(cudaStream_t s, unsigned* value);

}  // namespace rrs
