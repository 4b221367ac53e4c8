/*
 * rrs.h -- C ABI of the GB300 row-wise softmax and row-sum library (librrs.so).
 *
 * The two operations are the ones the CS336 lecture 06 pages build their
 * reduction kernels around:
 *
 *   softmax_rows  "Kernels, Triton, XLA", section "Reductions and tiling:
 *                 softmax, row sum, matmul" (and "GPU High-Performance
 *                 Programming", section 7.5.1): for every row i,
 *                   m_i = max_j x[i,j],  s_i = sum_j exp(x[i,j] - m_i),
 *                   y[i,j] = exp(x[i,j] - m_i) / s_i.
 *   row_sum       same section, paragraph "Row sum, when the row doesn't
 *                 fit": out[i] = sum_j x[i,j].
 *
 * and variants on the same skeleton (declared further down, each with the
 * passage it rests on): softmax_rows_ex (separate strides for x and y, in
 * place, log-softmax), log_softmax_rows, softmax_cols, row_max, row_mean,
 * the elementwise gelu of the same pages, and the fused attention_fwd that
 * the pages build towards.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * - Data are fp32.  x, y and out are DEVICE pointers (cudaMalloc, a caching
 *   allocator or managed memory) owned by the caller; the library neither
 *   frees nor keeps them.  Host pointers are rejected (RRS_ERR_INVALID_ARG).
 * - Row i of x occupies x[i*ld .. i*ld + N).  y uses the same ld (except in
 *   softmax_rows_ex, which takes one stride for each).  The gap [N, ld) of
 *   every row of y is never written; the gap of x is never read.
 * - y may be x itself (the same pointer and stride): the softmax is then
 *   computed in place.  Any other overlap of x and y is RRS_ERR_ALIAS.
 * - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  All work is enqueued on it and the call returns without
 *   synchronising; results are ordered before later work on that stream.
 * - Any ld >= N and any 4-byte-aligned pointer is accepted.  The 128-bit
 *   vector paths run when x and y are 16-byte aligned and ld % 4 == 0;
 *   otherwise the scalar forms of the same single-pass kernels (rows up to
 *   131072 floats) or of the two-phase split give the same results.
 * - Arguments are checked before anything is enqueued.  A failed launch
 *   returns RRS_ERR_CUDA and rrs_last_error() holds the runtime's message.
 * - Rows that contain +inf or NaN, or are entirely -inf, come out as NaN
 *   (the naive five steps give (-inf) - (-inf) or inf - inf there).  -inf
 *   entries of other rows come out as exactly 0.
 * - Calls are thread-safe.  The split-row paths use a small per-(device,
 *   stream) workspace the library allocates on first use and keeps.
 * - Calls can be captured in a CUDA graph once each path has run eagerly on
 *   the capturing stream with at least the captured shape (the first call
 *   may allocate its workspace, which a capture may not): a captured call
 *   that would need to allocate returns RRS_ERR_UNSUPPORTED and enqueues
 *   nothing.  A captured call keeps using that stream's workspace, which
 *   the library then never frees before rrs_release_workspace(), even when
 *   a later eager call grows it: do not replay the graph concurrently with
 *   other calls on the capturing stream, with another replay of it, or
 *   after rrs_release_workspace().
 */
#ifndef RRS_H
#define RRS_H

#include <stdint.h>

#if defined(__GNUC__)
#define RRS_API __attribute__((visibility("default")))
#else
#define RRS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rrs_status {
  RRS_OK = 0,
  RRS_ERR_INVALID_ARG = 1, /* negative size, ld < N, null or host pointer, misaligned float */
  RRS_ERR_ALIAS = 2,       /* the byte ranges of x and y (or out) overlap */
  RRS_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed; see rrs_last_error() */
  RRS_ERR_TIMEOUT = 4,     /* a split-row kernel gave up waiting for its peers (rrs_device_error) */
  RRS_ERR_NOMEM = 5,       /* the workspace could not be allocated */
  RRS_ERR_UNSUPPORTED = 6  /* a forced path cannot run this shape on this device */
} rrs_status;

/* Execution paths of softmax_rows (the planner picks one; tests may force one). */
typedef enum rrs_path {
  RRS_PATH_AUTO = -1,
  RRS_PATH_TWO_PHASE = 0,   /* any shape/alignment: partial (max,sum) per chunk, then merge + re-read + write */
  RRS_PATH_ROW_REGS = 1,    /* a group of 1..32 warps keeps the whole row in registers; 1 read + 1 write */
  RRS_PATH_ROW_STAGED = 2,  /* persistent CTAs stage rows in shared memory with bulk async copies (TMA) */
  RRS_PATH_CLUSTER = 3,     /* row split over a thread-block cluster; (max,sum) merged through DSMEM */
  RRS_PATH_GRID = 4,        /* row split over co-resident CTAs; (max,sum) merged through global memory */
  RRS_PATH_TWO_PASS = 5,    /* any shape/alignment: the two passes as work items of one launch, dealt in arrival
                               order; the second pass re-reads its chunk from the L2 */
  RRS_PATH_COUNT = 6
} rrs_path;

/* Execution paths of row_sum. */
typedef enum rrs_sum_path {
  RRS_SUM_AUTO = -1,
  RRS_SUM_ROW = 0,          /* one CTA (or warp) per row, per-thread accumulators, fixed-order tree */
  RRS_SUM_SPLIT = 1,        /* rows split into chunks; partial sums merged in fixed order by a 2nd kernel */
  RRS_SUM_COUNT = 2
} rrs_sum_path;

/* A launch plan: what the host side decided for one call (pure host logic). */
/* Execution paths of softmax_cols. */
typedef enum rrs_cols_path {
  RRS_COLS_AUTO = -1,
  RRS_COLS_TWO_PHASE = 0,  /* any shape/alignment: per-(row chunk, column) partials, then merge + re-read + write */
  RRS_COLS_CLUSTER = 1,    /* a band of 32 columns over a cluster of CTAs, all rows in registers (M <= 8192) */
  RRS_COLS_BAND = 2,       /* a band of 32 columns over a cluster of CTAs, rows streamed twice (second read from L2) */
  RRS_COLS_TWO_PASS = 3,   /* the band path's two passes as work items of one launch, dealt out in arrival order */
  RRS_COLS_COUNT = 4
} rrs_cols_path;

typedef struct rrs_plan {
  int32_t path;          /* rrs_path or rrs_sum_path */
  int32_t threads;       /* threads per CTA */
  int64_t grid;          /* CTAs launched (first kernel for two-kernel paths) */
  int32_t cluster;       /* CTAs per cluster (1 = no cluster) */
  int32_t vec;           /* float4 registers per thread per row segment (0 for streaming paths; the
                            column band path: CTAs per SM its registers are budgeted for, 3 or 4) */
  int32_t warps_per_row; /* warps that share one row (ROW_REGS) */
  int32_t rows_per_cta;  /* rows one CTA holds at a time */
  int64_t ctas_per_row;  /* CTAs one row is split over (split paths) */
  int64_t chunk;         /* columns per CTA segment in split paths (last one shorter) */
  int64_t rounds;        /* persistent rounds (GRID / STAGED) */
  int32_t smem_bytes;    /* dynamic shared memory per CTA */
  int32_t vector_io;     /* 1: 128-bit loads/stores; 2: 128-bit through a window shifted per row to the
                            16-byte boundary (CLUSTER, rows not 16-byte aligned); 0: scalar */
  int64_t workspace_bytes;
  int32_t stages;        /* shared-memory ring depth (staged paths) */
  int32_t tile;          /* floats per shared-memory stage (staged paths) */
} rrs_plan;

/* y = softmax over each row of x (see the top of this file).
 * x, y: device fp32, M rows of N valid entries, row stride ld (elements).
 * M == 0 or N == 0: no work, RRS_OK.  Errors: RRS_ERR_INVALID_ARG (M < 0,
 * N < 0, ld < N, ld < 1, null/host pointer, pointer not 4-byte aligned,
 * extent overflow), RRS_ERR_ALIAS (x and y overlap, unless y == x: in
 * place), RRS_ERR_CUDA, RRS_ERR_NOMEM. */
RRS_API int softmax_rows(const float* x, float* y, int64_t M, int64_t N, int64_t ld, void* stream);

/* Flag bits of softmax_rows_ex. */
#define RRS_LOG_SOFTMAX 1 /* write log y[i,j] = (x[i,j] - m_i) - log(s_i) instead of y */

/* softmax_rows with a row stride for each matrix: row i of x at x + i*ldx,
 * row i of y at y + i*ldy (both >= max(N, 1)).  The pages' softmax kernel
 * takes the two row strides separately ("CS336 2026 Lecture 6: Kernels,
 * Triton", section 5.3, the row-wise softmax).  A softmax down the columns
 * is not a stride of this call (its reduction runs across rows): see
 * softmax_cols.  x == y with ldx == ldy computes in place; any other
 * overlap is RRS_ERR_ALIAS.
 *
 * flags = RRS_LOG_SOFTMAX writes the log-softmax, log y = (x - m) - log(s),
 * the logarithm of the softmax definition above (the pages do not show it;
 * it follows from y = exp(x - m) / s).  -inf entries give -inf; the rows
 * that give NaN in the softmax give NaN.  RRS_ERR_UNSUPPORTED if a forced
 * ROW_STAGED path is asked for the log form.  Unknown flag bits are
 * RRS_ERR_INVALID_ARG.  Other arguments and errors as softmax_rows. */
RRS_API int softmax_rows_ex(const float* x, int64_t ldx, float* y, int64_t ldy, int64_t M,
                            int64_t N, int flags, void* stream);

/* softmax_rows_ex(x, ld, y, ld, M, N, RRS_LOG_SOFTMAX, stream). */
RRS_API int log_softmax_rows(const float* x, float* y, int64_t M, int64_t N, int64_t ld,
                             void* stream);

/* Softmax down each column: for every j < N and i < M,
 *   m_j = max_i x[i,j],  s_j = sum_i exp(x[i,j] - m_j),
 *   y[i,j] = exp(x[i,j] - m_j) / s_j
 * (flags = RRS_LOG_SOFTMAX: (x[i,j] - m_j) - log(s_j)).  The pages' softmax
 * with the reduction over rows; the lecture transcript takes it up in the
 * questions after the softmax kernel, where only the strides change.  Element (i, j) of x is x[i*ldx + j], of y y[i*ldy + j];
 * columns are read along rows, full 128-byte lines.
 * Columns that are all -inf or hold +inf or NaN come out NaN.  x == y with
 * ldx == ldy computes in place.  Arguments, errors and the empty cases as
 * softmax_rows_ex.  On the two-pass path (large aligned inputs) CTAs wait
 * for other CTAs' column partials; every such wait is bounded (1 s), and one
 * that runs out leaves its slice of y unwritten and is reported like a grid
 * path timeout: rrs_device_error returns RRS_ERR_TIMEOUT, and later calls
 * on the device return it until then.  Its first call on a device, like the
 * grid path's, allocates (a workspace and the host error word), so make it
 * before capturing the call in a CUDA graph. */
RRS_API int softmax_cols(const float* x, int64_t ldx, float* y, int64_t ldy, int64_t M, int64_t N,
                         int flags, void* stream);

/* out[i] = sum_j x[i*ld + j] for i < M (fp32 accumulation, fixed order:
 * bitwise reproducible run to run).  N == 0 writes zeros (the sum's
 * identity).  out: device, M floats, must not overlap x.  Errors as for
 * softmax_rows. */
RRS_API int row_sum(const float* x, float* out, int64_t M, int64_t N, int64_t ld, void* stream);

/* out[i] = max_j x[i*ld + j]: the first of the naive softmax's five steps
 * ("Kernels, Triton, XLA", section "Reductions and tiling", the softmax
 * paragraph), on the row-sum skeleton.  Exact (a max does not round).  A row
 * holding a NaN gives NaN; N == 0 writes -inf (the max's identity).  Other
 * arguments and errors as row_sum. */
RRS_API int row_max(const float* x, float* out, int64_t M, int64_t N, int64_t ld, void* stream);

/* out[i] = (sum_j x[i*ld + j]) / N: row_sum's fp32 sum (same order), divided
 * by N once per row.  N == 0 writes NaN (0 / 0).  Other arguments and errors
 * as row_sum. */
RRS_API int row_mean(const float* x, float* out, int64_t M, int64_t N, int64_t ld, void* stream);

/* y[i] = GeLU(x[i]) for i < n, the tanh approximation with the pages'
 * constants: 0.5 x (1 + tanh(0.79788456 (x + 0.044715 x^3))) ("Kernels,
 * Triton, XLA", section "GeLU three ways: the case for fusion", and the
 * Triton GeLU walkthrough; "GPU High-Performance Programming", section
 * 7.4.1).  The lecture's first kernel: elementwise and HBM-bound like the
 * softmax.  Computed as x / (1 + exp(-2a)), the same value without the
 * cancellation of 1 + tanh(a) for negative x.  x, y: device fp32, n
 * contiguous elements; y == x computes in place, any other overlap is
 * RRS_ERR_ALIAS.  n == 0: no work.  +inf gives +inf, -inf and NaN give NaN.
 * Errors: RRS_ERR_INVALID_ARG (n < 0, null/host pointer, not 4-byte
 * aligned), RRS_ERR_ALIAS, RRS_ERR_CUDA. */
RRS_API int gelu(const float* x, float* y, int64_t n, void* stream);

/* Fused attention forward: for every head h < BH and query i < L,
 *   O[h,i,:] = sum_j softmax_j(Q[h,i,:] . K[h,j,:] * scale) V[h,j,:],
 *   LSE[h,i] = log sum_j exp(Q[h,i,:] . K[h,j,:] * scale).
 * The pages name FlashAttention as the fusion of their elementwise, row-wise
 * softmax and tiled matmul kernels ("Kernels, Triton, XLA", end of
 * "Reductions and tiling"; "CS336 2026 Lecture 6: Kernels, Triton", the
 * assignment paragraph); this is that fusion on the tcgen05 tensor cores,
 * with the row softmax taken online over key tiles by the merge rule of
 * softmax_rows' split paths.
 * q: [BH, L, d], k and v: [BH, S, d], bf16 (IEEE bfloat16 bit patterns),
 * contiguous, 16-byte aligned, device memory; o: [BH, L, d] fp32; lse: [BH, L]
 * fp32 or NULL.  d is 64 or 128.  scale = 0 selects 1/sqrt(d).  causal != 0
 * masks key j for query i when j > i + S - L (queries aligned to the last
 * keys); a query that sees no key gets NaN and LSE -inf.  The products and
 * sums accumulate in fp32; the softmax weights enter the second product
 * rounded to bf16.  BH == 0 or L == 0: no work.  Errors: RRS_ERR_INVALID_ARG
 * (sizes, d, scale, alignment, null/host pointers), RRS_ERR_ALIAS (an output
 * overlaps an input or the other output), RRS_ERR_CUDA; a bounded wait that
 * ran out shows in rrs_device_error.  No workspace is allocated. */
RRS_API int attention_fwd(const void* q, const void* k, const void* v, float* o, float* lse,
                          int64_t BH, int64_t L, int64_t S, int64_t d, int causal, float scale,
                          void* stream);

/* softmax_rows for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a deployment variant of the same operation.
 *
 * Some callers may not call cudaMalloc or anything that allocates: a
 * plugin's execute hook inside an inference engine that owns all device
 * memory, or a latency-critical loop where an allocation could synchronise
 * the device or fail mid-step.  softmax_rows may allocate a small workspace
 * the first time it meets a stream; this call never allocates.  Where
 * softmax_rows would run a kernel that needs no workspace (the register
 * kernel or the cluster split: aligned rows of up to 131072 floats, and
 * unaligned ones as the planner takes them), it runs that same kernel, with
 * the same result.  Where softmax_rows would run the grid split, it runs
 * that kernel too, with its workspace in a fixed 1 MiB array inside the
 * library (when the shape's (row, segment) slots fit it); a wait of that
 * kernel that runs out is reported by rrs_device_error, and makes later
 * calls refuse only if an earlier softmax_rows grid call made the host
 * error word.  Otherwise it runs the two-phase kernels with their
 * (max, sum) partials in another fixed 1 MiB array (131072 pairs).  Every
 * GPU that loads the library holds both arrays until the process exits.
 *
 * Same arguments, layout, results and error codes as softmax_rows (y == x
 * computes in place, any other overlap is RRS_ERR_ALIAS; rrs_last_error()
 * holds the message of a refused call), plus RRS_ERR_INVALID_ARG when the
 * two-phase kernels would run on M > 131072 rows (each row needs a slot).
 * Those kernels cut rows into at most 131072 / M chunks, so few-row calls
 * keep their parallelism.
 * The first grid or two-phase call on a device looks up the arrays' device
 * addresses with that device current; make that first call before any
 * stream capture.  All such calls on a device share the arrays, which keep
 * the last call's contents (nothing needs clearing: the two-phase kernels
 * write every slot they read, and the grid kernel's slots carry the ticket
 * of the launch that wrote them).  Grid or two-phase calls whose kernels
 * overlap on the GPU -- on different streams or host threads -- race on
 * them, so order them on one stream. */
RRS_API int softmax_rows_noalloc(const float* x, float* y, int64_t M, int64_t N, int64_t ld,
                                 void* stream);

/* Synchronises `stream`, then returns and clears the device-side error word
 * of the current device: RRS_ERR_TIMEOUT if a split-row kernel stopped
 * waiting for its peers since the last call (its output is then incomplete),
 * RRS_OK otherwise, RRS_ERR_CUDA if the synchronisation failed.
 *
 * A timeout is also visible without this call.  The CTAs of a GRID-path
 * row (RRS_PATH_GRID) wait for one another.  Each CTA takes its row and
 * segment in the order the CTAs start, so the CTAs a CTA waits on are the
 * ones that started around it: a complete row group always runs to the end
 * and frees its SMs, and no CTA waits on one that could only start after it
 * finished.  Every wait is also bounded (about a second), for a group whose
 * later CTAs find no free SM for that long (other work holding the SMs).
 * A GRID kernel whose wait runs out
 * also sets a word of pinned host memory, so that once that kernel has
 * finished, every later call of this library on the same device (any entry
 * point that enqueues work) returns RRS_ERR_TIMEOUT without enqueuing
 * anything, until rrs_device_error() reports and clears the timeout -- a
 * sticky error, in the manner of CUDA's own.  The word (pinned host
 * memory, cudaHostAlloc) is allocated with the first GRID-path call on a
 * device and kept until the process exits: make that first call before any
 * stream capture. */
RRS_API int rrs_device_error(void* stream);

/* Static string naming a status code. */
RRS_API const char* rrs_status_string(int status);

/* The calling thread's last error message ("" if none). */
RRS_API const char* rrs_last_error(void);

/* Frees every cached workspace (after a device synchronisation), including
 * those kept for CUDA graphs that captured calls (such graphs must not be
 * replayed afterwards).  Later calls allocate again on demand.  Returns
 * RRS_OK or RRS_ERR_CUDA. */
RRS_API int rrs_release_workspace(void);

/* Force a path for later calls from any thread (testing / measurement):
 * softmax_path is an rrs_path, sum_path an rrs_sum_path; AUTO restores the
 * planner.  A forced path that cannot run a shape makes the call return
 * RRS_ERR_UNSUPPORTED.  Returns RRS_OK or RRS_ERR_INVALID_ARG. */
RRS_API int rrs_force_path(int softmax_path, int sum_path);

/* The same for softmax_cols: an rrs_cols_path (AUTO restores the planner). */
RRS_API int rrs_force_cols_path(int cols_path);

/* Fault injection for failure-detection tests (no counterpart in the
 * pages).  kind 1: in later GRID launches, CTA 0 never publishes the
 * partial of its first row segment, so that row's bounded waits run out
 * (about 1 s); the kernel returns early, rrs_device_error() then reports
 * RRS_ERR_TIMEOUT, the output of that call is incomplete, and the CUDA
 * context stays usable.  kind 2: the same for COLS_TWO_PASS and the rows'
 * TWO_PASS launches, whose first pass-1 item never publishes its partials,
 * so the second passes of band 0 / row 0 time out.  kind 0 turns injection
 * off.  Nothing here faults
 * or hangs the GPU.  Returns RRS_OK or RRS_ERR_INVALID_ARG. */
RRS_API int rrs_inject_fault(int kind);

/* Testing only: the work item that arrival index t draws in a COLS_TWO_PASS
 * launch with Q items per pass and lag D (1 <= D <= Q): *pass = 1 (partials
 * of item *k) or 2 (normalise item *k), items k = band x S + slice.  Pure
 * host logic, the same function the kernel runs.  Returns RRS_OK or
 * RRS_ERR_INVALID_ARG (t outside [0, 2Q), D outside [1, Q], null outputs). */
RRS_API int rrs_cols_two_pass_item(int64_t t, int64_t Q, int64_t D, int* pass, int64_t* k);

/* Testing only (no counterpart in the pages): enqueue on `stream` `ctas`
 * CTAs that each hold `smem_bytes` of shared memory (at most the opt-in
 * limit) for `nanoseconds` (at most 2e8) of the GPU's global timer and then
 * return on their own, so that a test can run a call while other work holds
 * SMs.  Nothing is read or written.  Returns RRS_OK, RRS_ERR_INVALID_ARG or
 * RRS_ERR_CUDA. */
RRS_API int rrs_test_occupy(int ctas, int smem_bytes, int64_t nanoseconds, void* stream);

/* The planner, as pure host logic: the plan softmax_rows / row_sum would use
 * for this shape on a device with `sm_count` SMs and `smem_optin` bytes of
 * opt-in shared memory per CTA.  `vector_ok`: 1 if x and y are 16-byte
 * aligned with ld % 4 == 0; for rrs_plan_softmax also 2 if they are not but
 * are misaligned alike (the same address mod 16 bytes, strides equal mod 4);
 * 0 otherwise.  Honors rrs_force_path.  Returns RRS_OK, RRS_ERR_INVALID_ARG
 * or RRS_ERR_UNSUPPORTED; touches no GPU. */
RRS_API int rrs_plan_softmax(int64_t M, int64_t N, int64_t ld, int vector_ok, int sm_count,
                             int smem_optin, rrs_plan* plan);
RRS_API int rrs_plan_row_sum(int64_t M, int64_t N, int64_t ld, int vector_ok, int sm_count,
                             int smem_optin, rrs_plan* plan);
RRS_API int rrs_plan_softmax_cols(int64_t M, int64_t N, int64_t ld, int vector_ok, int sm_count,
                                  int smem_optin, rrs_plan* plan);

/* Occupancy arithmetic used by the planner ("Kernels, Triton, XLA", section
 * "Where the abstraction leaks", worked example on register pressure):
 * blocks of `threads` threads using `regs` registers each on an SM with
 * `sm_regs` registers and `max_warps` resident warps.  Writes the resident
 * blocks and warps; returns occupancy in basis points (1/100 %). */
RRS_API int rrs_occupancy(int threads, int regs, int sm_regs, int max_warps,
                          int* blocks, int* warps);

/* Wave arithmetic (same page, problem 6.2): `blocks` CTAs on `slots`
 * concurrent CTA slots.  Writes the size of the last wave and the idle slots
 * in it; returns the number of waves. */
RRS_API int64_t rrs_waves(int64_t blocks, int64_t slots, int64_t* last_wave, int64_t* idle);

/* Library version, major*10000 + minor*100 + patch. */
RRS_API int rrs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RRS_H */
