// C ABI of librrs: argument checks, the launch planner, the per-stream
// workspace cache and dispatch to the kernel translation units.
//
// The pages' wrapper conventions carry over ("GPU High-Performance
// Programming", section 7.4, the CUDA GeLU wrapper): check that inputs live on
// the device before launching, let the caller own the output, and check the
// launch afterwards -- here as status codes instead of exceptions.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <limits>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <utility>
#include <vector>

#include "internal.h"
#include "rrs.h"

namespace rrs {

// ------------------------------------------- checks shared by entry points ---
// (declared in internal.h: every entry point reports through the same
// per-thread message and applies the same shape, alias and pointer rules)
namespace {
thread_local std::string g_last_error;
}  // namespace

void clear_last_error() { g_last_error.clear(); }

int fail(int status, const std::string& msg) {
  g_last_error = msg;
  return status;
}

int fail_cuda(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return RRS_ERR_CUDA;
}

// A pointer the current device can use as global memory.
int check_device_pointer(const void* p, int dev, const char* name) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(RRS_ERR_INVALID_ARG, std::string(name) + " is not a CUDA pointer");
  }
  if (a.type == cudaMemoryTypeManaged) return RRS_OK;
  if (a.type == cudaMemoryTypeDevice && a.device == dev) return RRS_OK;
  if (a.type == cudaMemoryTypeDevice)
    return fail(RRS_ERR_INVALID_ARG, std::string(name) + " lives on another device");
  return fail(RRS_ERR_INVALID_ARG, std::string(name) + " is not device memory");
}

// Shape checks shared by the row operations; sets *extent (elements spanned
// by x) when M > 0.
int check_shape(int64_t M, int64_t N, int64_t ld, int64_t* extent) {
  if (M < 0 || N < 0) return fail(RRS_ERR_INVALID_ARG, "M and N must be >= 0");
  if (ld < 1 || ld < N) return fail(RRS_ERR_INVALID_ARG, "ld must be >= max(N, 1)");
  *extent = 0;
  if (M == 0 || N == 0) return RRS_OK;
  if (M - 1 > (INT64_MAX / 8 - N) / ld) return fail(RRS_ERR_INVALID_ARG, "extent overflows");
  *extent = (M - 1) * ld + N;
  return RRS_OK;
}

bool overlaps(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + (uintptr_t)b_bytes && b0 < a0 + (uintptr_t)a_bytes;
}

namespace {

std::atomic<int> g_force_softmax{RRS_PATH_AUTO};
std::atomic<int> g_force_sum{RRS_SUM_AUTO};
std::atomic<int> g_force_cols{RRS_COLS_AUTO};
std::atomic<int> g_fault{0};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
int pow2_ceil(int64_t v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// ------------------------------------------------------------- device info ---
std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;

int device_info(int dev, DeviceInfo* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_devices.find(dev);
  if (it != g_devices.end()) {
    *out = it->second;
    return RRS_OK;
  }
  DeviceInfo d;
  cudaError_t e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cluster_launch, cudaDevAttrClusterLaunch, dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
  g_devices[dev] = d;
  *out = d;
  return RRS_OK;
}

// ------------------------------------------------------ host error words ---
// One word of pinned, mapped host memory per device.  A GRID kernel whose
// bounded wait runs out writes RRS_ERR_TIMEOUT into it; every later call on
// that device reads it (a plain host load, no lock, no synchronisation) and
// refuses to enqueue with RRS_ERR_TIMEOUT until rrs_device_error() clears it.
constexpr int kMaxDevices = 64;
std::atomic<unsigned*> g_host_err[kMaxDevices];      // host address of each device's word
std::atomic<unsigned*> g_host_err_dev[kMaxDevices];  // the same word's device address

// The device address of `dev`'s word, allocated on first use (under g_mu;
// refused during a stream capture on `s`, which may not allocate).
bool capturing(cudaStream_t s);
int host_err_word(int dev, cudaStream_t s, unsigned** dptr) {
  if (dev < 0 || dev >= kMaxDevices) return fail(RRS_ERR_INVALID_ARG, "device ordinal out of range");
  if (unsigned* d = g_host_err_dev[dev].load(std::memory_order_acquire)) {
    *dptr = d;
    return RRS_OK;
  }
  if (capturing(s))
    return fail(RRS_ERR_UNSUPPORTED,
                "the first grid-path call on a device allocates pinned host memory, which a stream "
                "capture cannot: make an eager call first");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_host_err_dev[dev].load()) {
    void* p = nullptr;
    cudaError_t e = cudaHostAlloc(&p, 64, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return fail(RRS_ERR_NOMEM, std::string("cudaHostAlloc(error word): ") + cudaGetErrorString(e));
    }
    std::memset(p, 0, 64);
    void* d = nullptr;
    e = cudaHostGetDevicePointer(&d, p, 0);
    if (e != cudaSuccess) {
      (void)cudaFreeHost(p);
      return fail_cuda(e, "cudaHostGetDevicePointer(error word)");
    }
    g_host_err[dev].store(static_cast<unsigned*>(p), std::memory_order_release);
    g_host_err_dev[dev].store(static_cast<unsigned*>(d), std::memory_order_release);
  }
  *dptr = g_host_err_dev[dev].load();
  return RRS_OK;
}

// The word's value for `dev` (0 if it was never allocated); allocates nothing.
unsigned host_err_value(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return 0;
  const unsigned* h = g_host_err[dev].load(std::memory_order_acquire);
  return h ? *reinterpret_cast<const volatile unsigned*>(h) : 0;
}

void host_err_clear(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return;
  unsigned* h = g_host_err[dev].load(std::memory_order_acquire);
  if (h) *reinterpret_cast<volatile unsigned*>(h) = 0;
}

// --------------------------------------------------------------- workspace ---
// One buffer per (device, stream, kind): calls on one stream are ordered, so
// they can share it; calls on different streams never do.  Grown with the
// stream-ordered allocator (ordered after earlier work on the stream that
// still reads the old buffer) and zero-filled when (re)allocated (the GRID
// kind's kernels keep their own launch counter and tickets in it).
enum WorkspaceKind { kWsTwoPhase = 0, kWsGrid = 1, kWsRowSum = 2, kWsRowsTwoPass = 6 };

// Under stream capture: a call that needs more workspace than the stream has
// is refused (a capture may not allocate; make an eager call of the shape on
// that stream first), and a workspace handed to a captured call is never
// freed when it later grows -- a graph may still replay into it -- but kept
// until rrs_release_workspace().
struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  bool captured = false;   // handed to a call during a stream capture
};
std::map<std::tuple<int, uintptr_t, int>, Workspace> g_workspaces;
std::vector<std::pair<int, void*>> g_retired;   // (device, buffer) a captured graph may still use

bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return cs != cudaStreamCaptureStatusNone;
}

int get_workspace(int dev, cudaStream_t s, int kind, size_t bytes, void** ptr) {
  const bool cap = capturing(s);
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspaces[{dev, reinterpret_cast<uintptr_t>(s), kind}];
  if (w.bytes < bytes) {
    if (cap)
      return fail(RRS_ERR_UNSUPPORTED,
                  "this call needs a larger workspace, which a stream capture cannot allocate: make an "
                  "eager call of this shape on the capturing stream first");
    if (w.ptr) {
      if (w.captured) {
        g_retired.emplace_back(dev, w.ptr);
      } else {
        cudaError_t e = cudaFreeAsync(w.ptr, s);
        if (e != cudaSuccess) {
          w.ptr = nullptr;
          w.bytes = 0;
          return fail_cuda(e, "cudaFreeAsync(workspace)");
        }
      }
      w.ptr = nullptr;
      w.bytes = 0;
      w.captured = false;
    }
    const size_t want = std::max<size_t>(round_up((int64_t)bytes, 1 << 16), 1 << 16);
    cudaError_t e = cudaMallocAsync(&w.ptr, want, s);
    if (e != cudaSuccess) {
      w.ptr = nullptr;
      (void)cudaGetLastError();
      return fail(RRS_ERR_NOMEM, std::string("cudaMallocAsync(workspace): ") + cudaGetErrorString(e));
    }
    e = cudaMemsetAsync(w.ptr, 0, want, s);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(workspace)");
    w.bytes = want;
  }
  if (cap) w.captured = true;
  *ptr = w.ptr;
  return RRS_OK;
}

// ---------------------------------------------------------------- planner ---
// vector: float4 slots plus an N % 4 tail; scalar (unaligned x or y, or a
// stride not a multiple of 4): 4 scalars per slot, so the slots cover N.
void plan_row_regs(int64_t M, int64_t N, int sm_count, rrs_plan* p, bool vector = true) {
  const int64_t n4 = vector ? (N >> 2) : ceil_div(N, 4);
  int gw, vec;
  if (N <= 32 * 4 * kRowRegsMaxVec) {  // a warp per row
    gw = 1;
    vec = std::max(1, pow2_ceil(ceil_div(n4, 32)));
  } else {
    vec = 8;
    gw = pow2_ceil(ceil_div(n4, 32 * vec));
  }
  p->path = RRS_PATH_ROW_REGS;
  p->vec = vec;
  p->warps_per_row = gw;
  p->threads = std::max(32 * gw, 128);
  p->rows_per_cta = p->threads / (32 * gw);
  p->grid = std::min<int64_t>(ceil_div(M, p->rows_per_cta), INT_MAX);
  p->ctas_per_row = 1;
  p->chunk = N;
  p->rounds = 1;
  (void)sm_count;
}

bool row_regs_fits(int64_t N) { return N <= (int64_t)32 * 32 * 4 * 8; }

// mode 1 (vector): float4 slots plus an N % 4 tail in the last CTA; 0
// (scalar): 4 scalars per slot, so the slots cover N; 2 (shifted window):
// float4 slots over a window of up to N + 3 floats.
bool plan_cluster(int64_t M, int64_t N, rrs_plan* p, int mode = 1) {
  const int64_t n4 = mode == 1 ? (N >> 2) : (mode == 0 ? ceil_div(N, 4) : ceil_div(N + 3, 4));
  int vec = kClusterVec;
  int cs = pow2_ceil(std::max<int64_t>(1, ceil_div(n4, (int64_t)kSplitThreads * vec)));
  if (cs > kClusterMax) return false;
  // a cluster of one CTA per 4 KiB-aligned segment; shrink registers when the segment is short
  if (ceil_div(n4, cs) <= (int64_t)kSplitThreads * 4) vec = 4;
  p->path = RRS_PATH_CLUSTER;
  p->vector_io = mode;
  p->vec = vec;
  p->warps_per_row = kSplitThreads / 32;
  p->threads = kSplitThreads;
  p->cluster = cs;
  p->rows_per_cta = 1;
  p->ctas_per_row = cs;
  p->chunk = ceil_div(n4, cs) * 4;
  p->grid = std::min<int64_t>(M, INT_MAX / cs) * cs;
  p->rounds = 1;
  return true;
}

void plan_two_phase(int64_t M, int64_t N, int sm_count, rrs_plan* p) {
  const int64_t target = 4 * (int64_t)sm_count;
  int64_t C = std::max<int64_t>(1, std::min(ceil_div(target, M), ceil_div(N, 4096)));
  int64_t chunk = round_up(ceil_div(N, C), kChunkAlign);
  C = ceil_div(N, chunk);
  p->path = RRS_PATH_TWO_PHASE;
  p->threads = kSplitThreads;
  p->ctas_per_row = C;
  p->chunk = chunk;
  p->rows_per_cta = 1;
  p->grid = std::min<int64_t>(M * C, 32 * (int64_t)sm_count);
  p->workspace_bytes = M * C * 8;
  p->rounds = 1;
}

// Staged paths: one CTA per SM, shared-memory ring of `stages` stages.
int64_t staged_budget(int smem_optin) { return (int64_t)smem_optin - staged_header_bytes(); }

// Long rows keep a segment resident as 4 sub-tiles with at least 3 more
// stages to prefetch into: a sub-tile is at most budget / 7.
int64_t staged_tile_max(int smem_optin) { return (staged_budget(smem_optin) / 7) / 16 * 4; }

constexpr int64_t kStagedRowsMaxN = 8192;
constexpr int64_t kRowRegsFirstMaxN = 4096;   // the register kernel always, up to here
constexpr int64_t kRowRegsAutoMaxN = 16384;   // the register kernel or the cluster split, up to here
constexpr int64_t kClusterShortRowMaxN = 8192;      // rows this short ...
constexpr int64_t kClusterShortRowMinElems = 1 << 23;   // ... split only in matrices this large
constexpr double kPerSmBytesPerSec = 6.7e12 / 152.0;  // planning model only
constexpr double kItemSec = 0.4e-6;                    // per-segment fixed cost (planning model)
constexpr int64_t kGridMaxSegments = 160;              // slots one exchange warp polls

bool plan_staged_rows(int64_t M, int64_t N, int sm_count, int smem_optin, rrs_plan* p) {
  if (N % 4 != 0 || N > kStagedRowsMaxN) return false;
  const int64_t n4 = N / 4;
  int gw, vec;
  if (n4 <= 32 * 16) {
    gw = 1;
    vec = std::max(1, pow2_ceil(ceil_div(n4, 32)));
  } else {
    vec = 8;
    gw = pow2_ceil(ceil_div(n4, 32 * 8));
  }
  const int64_t G = std::min<int64_t>(M, sm_count);
  const int64_t rows_per_cta = ceil_div(M, G);
  const int64_t tile = round_up(N, 32);  // stage stride: a multiple of 128 bytes
  // Stage s is filled by producer lane s % groups and drained by consumer
  // group s % groups, so the ring depth is a multiple of the group count.
  const int64_t groups = staged_consumer_warps() / gw;
  int64_t ns = std::min<int64_t>(std::min<int64_t>(staged_max_stages(),
                                                   staged_budget(smem_optin) / (tile * 4)),
                                 round_up(rows_per_cta, groups));
  ns = ns / groups * groups;
  if (ns < groups) return false;
  p->path = RRS_PATH_ROW_STAGED;
  p->vec = vec;
  p->warps_per_row = gw;
  p->threads = staged_threads();
  p->grid = G;
  p->rows_per_cta = 1;
  p->ctas_per_row = 1;
  p->chunk = N;
  p->rounds = rows_per_cta;
  p->stages = (int32_t)ns;
  p->tile = (int32_t)tile;
  p->smem_bytes = (int32_t)(staged_header_bytes() + ns * tile * 4);
  return true;
}

bool plan_staged_long(int64_t M, int64_t N, int sm_count, int smem_optin, rrs_plan* p) {
  if (N % 4 != 0) return false;
  const int64_t tile = round_up(ceil_div(N, 4), 4);
  if (tile > staged_tile_max(smem_optin)) return false;
  const int64_t ns = std::min<int64_t>(staged_max_stages(), staged_budget(smem_optin) / (tile * 4));
  const int64_t G = std::min<int64_t>(M, sm_count);
  p->path = RRS_PATH_ROW_STAGED;
  p->vec = 0;
  p->warps_per_row = 8;
  p->threads = staged_threads();
  p->grid = G;
  p->rows_per_cta = 1;
  p->ctas_per_row = 1;
  p->chunk = N;
  p->rounds = ceil_div(M, G);
  p->stages = (int32_t)ns;
  p->tile = (int32_t)tile;
  p->smem_bytes = (int32_t)(staged_header_bytes() + ns * tile * 4);
  return true;
}

// GRID: C segments of a row on C CTAs (one per SM), R rows per round,
// R * C <= SMs; a segment is one shared-memory stage and, in registers, at
// most 8 float4 per thread of the grid kernel's partial warps.  The ring
// holds at least 2 stages.  C minimises rounds x (per-SM segment time + a
// fixed per-segment cost).

bool plan_grid(int64_t M, int64_t N, int sm_count, int smem_optin, rrs_plan* p) {
  if (N % 4 != 0) return false;
  const int64_t budget = staged_budget(smem_optin);
  const int64_t kGridMaxSegFloats = 8 * 4 * (int64_t)grid_partial_threads();
  double best = 1e300;
  int64_t b_seg = 0, b_c = 0, b_r = 0, b_ns = 0, b_stride = 0;
  for (int64_t c = std::max<int64_t>(1, ceil_div(N, kGridMaxSegFloats)); c <= sm_count; ++c) {
    const int64_t seg = round_up(ceil_div(N, c), 4);
    const int64_t C = ceil_div(N, seg);
    if (C > kGridMaxSegments || seg > kGridMaxSegFloats) continue;
    const int64_t stride = round_up(seg * 4, 128);
    const int64_t ns = std::min<int64_t>(staged_max_stages(), budget / stride);
    if (ns < 2) continue;
    const int64_t R = std::min<int64_t>(sm_count / C, M);
    if (R < 1) continue;
    const double rounds = (double)ceil_div(M, R);
    const double t = rounds * (8.0 * (double)seg / kPerSmBytesPerSec + kItemSec);
    if (t < best * (1.0 - 1e-9)) {
      best = t;
      b_seg = seg;
      b_c = C;
      b_r = R;
      b_ns = ns;
      b_stride = stride;
    }
  }
  if (b_seg == 0) return false;
  const int64_t per_thread = ceil_div(ceil_div(b_seg, 4), grid_partial_threads());
  p->path = RRS_PATH_GRID;
  p->vec = per_thread <= 2 ? 2 : (per_thread <= 4 ? 4 : 8);
  p->warps_per_row = grid_threads() / 32 - 1;
  p->threads = grid_threads();
  p->grid = b_r * b_c;
  p->rows_per_cta = (int32_t)b_r;
  p->ctas_per_row = b_c;
  p->chunk = b_seg;
  p->rounds = ceil_div(M, b_r);
  p->stages = (int32_t)b_ns;
  p->tile = (int32_t)(b_stride / 4);
  p->smem_bytes = (int32_t)(staged_header_bytes() + b_ns * b_stride);
  p->workspace_bytes = kGridArrivalBytes + M * b_c * 16;
  return true;
}

// ROW_TWO_PASS: items of rows_two_pass_chunk() floats, one CTA per (pass,
// item), and a lag of kRowTwoPassLagPerSm x SMs items (at least S, at most
// the item count); float4 access when x, y, the stride and N allow.
// A lag of 4 x SMs against 3: 46.1 against 46.7 us on 32 x 2^20, 51.3
// against 52.0 with those rows unaligned, 287 against 286 on 1024 x 200001.
constexpr int64_t kRowTwoPassLagPerSm = 4;
constexpr int64_t kRowTwoPassMaxChunks = 256;   // a row's pairs in two rounds of the merging warp's loads

bool plan_row_two_pass(int64_t M, int64_t N, int sm_count, bool vector_ok, rrs_plan* p) {
  const int64_t S = ceil_div(N, rows_two_pass_chunk());
  const int64_t Q = M * S;
  if (2 * Q > (int64_t)INT_MAX) return false;
  const int64_t D = std::min(Q, std::max(S, kRowTwoPassLagPerSm * (int64_t)sm_count));
  p->path = RRS_PATH_TWO_PASS;
  p->threads = rows_two_pass_threads();
  p->grid = 2 * Q;
  p->chunk = rows_two_pass_chunk();
  p->ctas_per_row = S;
  p->stages = (int32_t)D;
  p->rows_per_cta = 1;
  p->cluster = 1;
  p->vector_io = (vector_ok && N % 4 == 0) ? 1 : 0;
  p->workspace_bytes = kRowsTwoPassArrivalBytes + Q * 16;
  return true;
}

// vector_ok: 1 = x and y 16-byte aligned with strides multiples of 4; 2 =
// not, but misaligned alike (the same address mod 16 bytes, strides equal
// mod 4), so every row of both can be read and written through one shifted
// float4 window; 0 = neither.
int plan_softmax_impl(int64_t M, int64_t N, int64_t ld, int vector_ok_in, int sm_count,
                      int smem_optin, int cluster_ok, int forced, rrs_plan* p) {
  std::memset(p, 0, sizeof(*p));
  if (M < 0 || N < 0 || ld < 1 || ld < N || sm_count < 1 || vector_ok_in < 0 || vector_ok_in > 2)
    return fail(RRS_ERR_INVALID_ARG, "bad shape or device description");
  const int vector_ok = vector_ok_in == 1 ? 1 : 0;
  const int shift_mode = vector_ok_in == 2 ? 2 : 0;   // the cluster kernel's mode for unaligned rows
  p->cluster = 1;
  p->vector_io = vector_ok;
  if (M == 0 || N == 0) {
    p->path = (forced == RRS_PATH_AUTO) ? RRS_PATH_ROW_REGS : forced;
    return RRS_OK;
  }
  if (forced == RRS_PATH_AUTO) {
    // Measured on GB300 (N from 3584 to 16384; cluster split against register
    // kernel): the register kernel wins up
    // to 4096 floats (8192 rows of 4096: 39.6 against 47.9 us).  Past that
    // the cluster split wins where it fills its register slots at least as
    // well and the rows are more than one wave of CTAs (2^25 floats:
    // 16384-float rows 43.4 against 54.0 us, 12288 47.4 against 60.9, 10240
    // 51.8 against 67.1; 456 x 16384 13.2 against 14.4); with at most one
    // row per SM the register kernel's single pass has the shorter latency
    // (152 x 12288: 5.7 against 4.9 us), and rows of up to 8192 floats gain
    // only in matrices of 2^23 floats and more (8192: 1216 rows 15.4
    // against 15.9, 608 rows 9.2 both; 6144: 456 rows 7.1 against 7.0).  A
    // row that the register kernel fills and the cluster does not (an
    // unaligned 8191, whose shifted window spills into a second, half-empty
    // CTA: 63.0 against 50.2 us) stays on the register kernel.  Past 16384
    // the cluster split runs up to 16 CTAs' registers, then the staged grid
    // split, then the two-pass split for what the grid cannot hold or align
    // (one launch, its second pass re-reading from the L2: 32 x 1048577
    // unaligned 61.7 against 228 us on the two-phase pair, 1024 x 200001
    // unaligned 324 against 849, 32 x 1048575 58.3 against 69.8) up to 256
    // chunks a row, and the two-phase pair past that (4 x 2^24: 141 against
    // 157 us, where the two-pass merge takes eight rounds of loads).  Rows
    // whose start or stride is not 16-byte aligned take the shifted-window
    // or scalar forms; N % 4 != 0 the vector forms with a ragged tail (the
    // grid split needs whole float4 segments, the two-pass split scalars).
    rrs_plan c{}, r{}, t{};   // every field the planners leave alone stays 0
    r.cluster = c.cluster = t.cluster = 1;
    const int mode = vector_ok ? 1 : shift_mode;   // the cluster kernel's form for these rows
    auto cluster_plan = [&](rrs_plan* out) {
      return cluster_ok && (plan_cluster(M, N, out, mode) || (mode == 2 && plan_cluster(M, N, out, 0)));
    };
    auto slots = [](const rrs_plan& q, bool cluster) -> double {   // floats one row's register slots hold
      return cluster ? 4.0 * q.vec * q.threads * q.cluster : 4.0 * q.vec * 32 * q.warps_per_row;
    };
    if (N <= kRowRegsFirstMaxN) {
      plan_row_regs(M, N, sm_count, p, vector_ok != 0);
    } else if (N <= kRowRegsAutoMaxN) {
      plan_row_regs(M, N, sm_count, &r, vector_ok != 0);
      const bool many_rows = M > sm_count && (N > kClusterShortRowMaxN || M * N >= kClusterShortRowMinElems);
      if (many_rows && cluster_plan(&c) && slots(c, true) <= slots(r, false)) *p = c;
      else *p = r;
    } else if (cluster_plan(&c)) {
      *p = c;
    } else if (vector_ok && N % 4 == 0 && plan_grid(M, N, sm_count, smem_optin, p)) {
    } else if (plan_row_two_pass(M, N, sm_count, vector_ok != 0, &t) && t.ctas_per_row <= kRowTwoPassMaxChunks) {
      *p = t;
    } else {
      plan_two_phase(M, N, sm_count, p);
    }
    p->cluster = std::max(p->cluster, 1);
    if (p->path != RRS_PATH_CLUSTER && p->path != RRS_PATH_TWO_PASS) p->vector_io = vector_ok;
    return RRS_OK;
  }
  const int path = forced;
  switch (path) {
    case RRS_PATH_ROW_STAGED:
      if (vector_ok && (plan_staged_rows(M, N, sm_count, smem_optin, p) ||
                        plan_staged_long(M, N, sm_count, smem_optin, p))) {
        p->cluster = 1;
        p->vector_io = 1;
        return RRS_OK;
      }
      return fail(RRS_ERR_UNSUPPORTED, "ROW_STAGED needs 16-byte alignment, N % 4 == 0, N <= 32912");
    case RRS_PATH_GRID:
      if (vector_ok && plan_grid(M, N, sm_count, smem_optin, p)) {
        p->cluster = 1;
        p->vector_io = 1;
        return RRS_OK;
      }
      return fail(RRS_ERR_UNSUPPORTED, "GRID needs 16-byte alignment and N % 4 == 0");
    case RRS_PATH_ROW_REGS:
      if (!row_regs_fits(N)) return fail(RRS_ERR_UNSUPPORTED, "ROW_REGS needs N <= 32768");
      plan_row_regs(M, N, sm_count, p, vector_ok != 0);
      p->vector_io = vector_ok ? 1 : 0;
      return RRS_OK;
    case RRS_PATH_CLUSTER:
      if (!cluster_ok || !(plan_cluster(M, N, p, vector_ok ? 1 : shift_mode) ||
                           (!vector_ok && plan_cluster(M, N, p, 0))))
        return fail(RRS_ERR_UNSUPPORTED, "CLUSTER needs cluster launch and N <= 131072");
      return RRS_OK;
    case RRS_PATH_TWO_PHASE:
      plan_two_phase(M, N, sm_count, p);
      return RRS_OK;
    case RRS_PATH_TWO_PASS:
      if (plan_row_two_pass(M, N, sm_count, vector_ok != 0, p)) return RRS_OK;
      return fail(RRS_ERR_UNSUPPORTED, "TWO_PASS needs 2 x rows x chunks <= INT_MAX");
    default:
      return fail(RRS_ERR_UNSUPPORTED, "path not available");
  }
}

// Column softmax.  COLS_CLUSTER (forced only): a band of 32 columns per
// cluster; as many rows per thread as useful (vec a power of two, at most
// 16), so the fewest CTAs share a band: cs = ceil(M / (32 row groups x vec))
// <= 16 (M <= 8192).  COLS_TWO_PHASE: row chunks sized for about 4 CTAs per
// SM over all bands (unaligned inputs).  COLS_BAND: below.
enum WorkspaceKindCols { kWsCols = 3, kWsColsTwoPass = 4 };

bool plan_cols_cluster(int64_t M, int64_t N, int64_t max_cs, rrs_plan* p) {
  const int64_t groups = cols_row_groups();
  const int64_t vec = std::min<int64_t>(cols_rows_per_thread_max(),
                                        std::max<int64_t>(1, pow2_ceil(ceil_div(M, groups))));
  const int64_t cs = ceil_div(M, groups * vec);
  if (cs > std::min<int64_t>(max_cs, kClusterMax)) return false;
  p->path = RRS_COLS_CLUSTER;
  p->threads = cols_threads();
  p->vec = (int32_t)vec;
  p->cluster = (int32_t)cs;
  p->grid = ceil_div(N, cols_band()) * cs;
  p->rows_per_cta = (int32_t)(groups * vec);
  p->ctas_per_row = cs;
  p->chunk = ceil_div(M, cs);
  return true;
}

void plan_cols_two_phase(int64_t M, int64_t N, int sm_count, rrs_plan* p) {
  const int64_t bands = ceil_div(N, cols_band());
  const int64_t want = std::max<int64_t>(1, ceil_div(4 * (int64_t)sm_count, bands));
  const int64_t chunk = std::max<int64_t>(8, ceil_div(M, want));
  const int64_t chunks = ceil_div(M, chunk);
  p->path = RRS_COLS_TWO_PHASE;
  p->threads = cols_threads();
  p->grid = bands * chunks;
  p->ctas_per_row = chunks;
  p->chunk = chunk;
  p->rows_per_cta = (int32_t)std::min<int64_t>(chunk, INT_MAX);
  p->workspace_bytes = chunks * N * 8;
}

// COLS_BAND: the fewest CTAs per band (a power of two, at most 8) that keep
// a CTA's rows at most 512 (M < 2048) or 1024: measured on GB300,
// 1024 x 8192 ran fastest with 512 rows per CTA (18.3 us; 256 rows: 22.6,
// 1024: 25.5) and 4096 x 16384 with 1024 (119.8 us; 512: 128, 2048: 124.9).
// At most 1024 rows (128 KB of x) per CTA and four CTAs per SM keep the x
// that pass 2 re-reads within the L2.
bool bands_fit_grid(int64_t N) { return ceil_div(N, cols_band()) * 8 <= (int64_t)INT_MAX; }

void plan_cols_band(int64_t M, int64_t N, rrs_plan* p) {
  const int64_t bands = ceil_div(N, cols_band());
  const int64_t max_rows = (M < 2048) ? 512 : 1024;
  int64_t cs = 1;
  while (cs < 8 && ceil_div(M, cs) > max_rows) cs *= 2;
  p->path = RRS_COLS_BAND;
  p->threads = cols_threads();
  p->cluster = (int32_t)cs;
  p->grid = bands * cs;
  p->ctas_per_row = cs;
  p->chunk = ceil_div(M, cs);
  p->rows_per_cta = (int32_t)std::min<int64_t>(p->chunk, INT_MAX);
  // vec: the CTAs per SM the kernel's registers are budgeted for, four (a
  // budget of three, once faster on grids of three or more such waves, lost
  // everywhere once the four-CTA build stopped spilling)
  p->vec = 4;
}

// COLS_TWO_PASS: slices of kColsTwoPassRows rows, one CTA per (pass,
// item), and a lag of kColsTwoPassLagPerSm x SMs items between an item's
// first and second pass (at least the band's slice count, so every first
// pass of a band comes before its second passes; at most the item count).
constexpr int64_t kColsTwoPassRows = 512;
constexpr int64_t kColsTwoPassLagPerSm = 3;

bool plan_cols_two_pass(int64_t M, int64_t N, int sm_count, bool vector_ok, rrs_plan* p) {
  const int64_t bands = ceil_div(N, cols_band());
  const int64_t R = kColsTwoPassRows;
  const int64_t S = ceil_div(M, R);
  const int64_t Q = bands * S;
  if (2 * Q > (int64_t)INT_MAX) return false;
  const int64_t D = std::min(Q, std::max(S, kColsTwoPassLagPerSm * (int64_t)sm_count));
  p->path = RRS_COLS_TWO_PASS;
  p->threads = cols_threads();
  p->grid = 2 * Q;
  p->chunk = R;
  p->ctas_per_row = S;
  p->stages = (int32_t)D;
  p->rows_per_cta = (int32_t)R;
  p->workspace_bytes = kColsArrivalBytes + Q * cols_band() * 16;
  p->vector_io = vector_ok ? 1 : 0;
  return true;
}

int plan_cols_impl(int64_t M, int64_t N, int64_t ld, int vector_ok, int sm_count, int cluster_ok,
                   int forced, rrs_plan* p) {
  std::memset(p, 0, sizeof(*p));
  if (M < 0 || N < 0 || ld < 1 || ld < N || sm_count < 1)
    return fail(RRS_ERR_INVALID_ARG, "bad shape or device description");
  p->cluster = 1;
  p->vector_io = vector_ok ? 1 : 0;
  if (M == 0 || N == 0) {
    p->path = (forced == RRS_COLS_AUTO) ? RRS_COLS_TWO_PHASE : forced;
    return RRS_OK;
  }
  const bool cluster_fits = vector_ok && cluster_ok;
  if (forced == RRS_COLS_AUTO) {
    // Measured on GB300: the band path is the fastest of the cluster, band
    // and two-phase paths wherever it applies (1024 x 8192: 18.3 us against
    // 19.5 cluster and 28.6 two-phase; 4096 x 16384: 119.8 against 172.8 and
    // 140.9); the two-pass path beats it once there are items enough for
    // its passes to interleave, at least twice its lag, and at most 8
    // slices per band, so its merge takes one round of loads (4096 x 16384:
    // 102.1-102.6 against 106.8-108.5 us; 2048 x 65536: 192.9-196.5 against
    // 202.3-202.8; 4096 x 8192: 54.0 against 57.1, 55.1 on the band path
    // since its second pass stopped spilling); it loses where its passes
    // run one after the other (1024 x 8192: 16.2-16.5 against 15.3) and
    // ties or loses with 16-32 slices (8192 x 4096: 57.8 against 57.2,
    // 16384 x 2048: 63.3-65.8 against 63.0-63.7).
    rrs_plan t{};
    if (vector_ok && plan_cols_two_pass(M, N, sm_count, true, &t) && t.ctas_per_row <= 8 &&
        (int64_t)t.ctas_per_row * ceil_div(N, cols_band()) >= 2 * kColsTwoPassLagPerSm * (int64_t)sm_count) {
      *p = t;
    } else if (cluster_fits && bands_fit_grid(N)) {
      plan_cols_band(M, N, p);
      p->vector_io = 1;
    } else if (!vector_ok && plan_cols_two_pass(M, N, sm_count, false, &t) && t.ctas_per_row <= 8) {
      // unaligned: the two-pass path's scalar form beats the two-phase pair
      // at every size measured (4096 x 16384, ld 16385: 166.8 against 207.9
      // us; 1024 x 8192, ld 8193: 28.3 against 34.1; 2048 x 65536, ld 65537,
      // offset 3 floats: 317.9 against 402.3)
      *p = t;
    } else {
      plan_cols_two_phase(M, N, sm_count, p);
      p->vector_io = vector_ok ? 1 : 0;
    }
    return RRS_OK;
  }
  if (forced == RRS_COLS_CLUSTER) {
    if (cluster_fits && plan_cols_cluster(M, N, kClusterMax, p)) {
      p->vector_io = 1;
      return RRS_OK;
    }
    return fail(RRS_ERR_UNSUPPORTED, "COLS_CLUSTER needs 16-byte alignment, cluster launch and M <= 8192");
  }
  if (forced == RRS_COLS_TWO_PHASE) {
    plan_cols_two_phase(M, N, sm_count, p);
    p->vector_io = vector_ok ? 1 : 0;
    return RRS_OK;
  }
  if (forced == RRS_COLS_BAND) {
    if (cluster_fits && bands_fit_grid(N)) {
      plan_cols_band(M, N, p);
      p->vector_io = 1;
      return RRS_OK;
    }
    return fail(RRS_ERR_UNSUPPORTED, "COLS_BAND needs 16-byte alignment and cluster launch");
  }
  if (forced == RRS_COLS_TWO_PASS) {
    if (plan_cols_two_pass(M, N, sm_count, vector_ok != 0, p)) return RRS_OK;
    return fail(RRS_ERR_UNSUPPORTED, "COLS_TWO_PASS needs 2 x items <= INT_MAX");
  }
  return fail(RRS_ERR_UNSUPPORTED, "column path not available");
}

int plan_row_sum_impl(int64_t M, int64_t N, int64_t ld, int vector_ok, int sm_count,
                      int smem_optin, int forced, rrs_plan* p) {
  std::memset(p, 0, sizeof(*p));
  if (M < 0 || N < 0 || ld < 1 || ld < N || sm_count < 1)
    return fail(RRS_ERR_INVALID_ARG, "bad shape or device description");
  (void)smem_optin;
  p->cluster = 1;
  p->vector_io = vector_ok ? 1 : 0;
  int path = forced;
  if (path == RRS_SUM_AUTO) {
    path = (M < 2 * (int64_t)sm_count && N >= 65536) ? RRS_SUM_SPLIT : RRS_SUM_ROW;
  }
  if (path == RRS_SUM_ROW) {
    // about 32 floats per thread before a CTA holds more than 8 warps (a
    // 256-thread CTA per long row measured faster than 512 on 4096 x 32768)
    const int gw = (int)std::min<int64_t>(8, std::max<int64_t>(1, pow2_ceil(ceil_div(N, 32 * 32 * 2))));
    p->path = RRS_SUM_ROW;
    p->warps_per_row = gw;
    p->threads = std::max(32 * gw, 128);
    p->rows_per_cta = p->threads / (32 * gw);
    p->grid = std::max<int64_t>(1, std::min<int64_t>(ceil_div(M, p->rows_per_cta), INT_MAX));
    p->ctas_per_row = 1;
    p->chunk = N;
    return RRS_OK;
  }
  if (path == RRS_SUM_SPLIT) {
    const int64_t target = 4 * (int64_t)sm_count;
    int64_t C = std::max<int64_t>(1, std::min(ceil_div(target, std::max<int64_t>(M, 1)),
                                              ceil_div(std::max<int64_t>(N, 1), 8192)));
    int64_t chunk = round_up(ceil_div(std::max<int64_t>(N, 1), C), kChunkAlign);
    C = ceil_div(std::max<int64_t>(N, 1), chunk);
    p->path = RRS_SUM_SPLIT;
    p->threads = 256;
    p->ctas_per_row = C;
    p->chunk = chunk;
    p->rows_per_cta = 1;
    p->grid = std::max<int64_t>(1, std::min<int64_t>(M * C, 32 * (int64_t)sm_count));
    p->workspace_bytes = M * C * 4;
    return RRS_OK;
  }
  return fail(RRS_ERR_UNSUPPORTED, "row_sum path not available");
}

bool vector_ok(const void* x, const void* y, int64_t ld) {
  return (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (reinterpret_cast<uintptr_t>(y) % 16 == 0) &&
         (ld % 4 == 0);
}

}  // namespace

int check_no_pending_timeout(int dev) {
  if (host_err_value(dev) != 0)
    return fail(RRS_ERR_TIMEOUT,
                "an earlier split-row kernel on this device stopped waiting for its peers (its output "
                "is incomplete); rrs_device_error() reports and clears this");
  return RRS_OK;
}

}  // namespace rrs

using namespace rrs;

namespace rrs {

// For softmax_rows_noalloc: the plan softmax_rows would launch for these
// arguments on `dev` (true, *p set), or false when the planner refuses the
// shape (a forced path that cannot run it); rrs_last_error is left clear
// either way.
bool plan_like_softmax_rows(const float* x, const float* y, int64_t M, int64_t N, int64_t ld, int dev,
                            rrs_plan* p) {
  DeviceInfo info;
  if (device_info(dev, &info) != RRS_OK) {
    clear_last_error();
    return false;
  }
  const bool vec = vector_ok(x, y, ld);
  const bool alike = (reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) % 16 == 0;
  const int st = plan_softmax_impl(M, N, ld, vec ? 1 : (alike ? 2 : 0), info.sm_count, info.smem_optin,
                                   info.cluster_launch, g_force_softmax.load(), p);
  clear_last_error();
  return st == RRS_OK;
}

// The device address of `dev`'s host error word if an earlier call made it,
// else null (allocates nothing).
unsigned* host_err_word_if_made(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  return g_host_err_dev[dev].load(std::memory_order_acquire);
}

}  // namespace rrs

extern "C" {

RRS_API int rrs_version(void) { return 100; }

RRS_API const char* rrs_status_string(int status) {
  switch (status) {
    case RRS_OK: return "RRS_OK";
    case RRS_ERR_INVALID_ARG: return "RRS_ERR_INVALID_ARG";
    case RRS_ERR_ALIAS: return "RRS_ERR_ALIAS";
    case RRS_ERR_CUDA: return "RRS_ERR_CUDA";
    case RRS_ERR_TIMEOUT: return "RRS_ERR_TIMEOUT";
    case RRS_ERR_NOMEM: return "RRS_ERR_NOMEM";
    case RRS_ERR_UNSUPPORTED: return "RRS_ERR_UNSUPPORTED";
    default: return "RRS_ERR_UNKNOWN";
  }
}

RRS_API const char* rrs_last_error(void) { return rrs::g_last_error.c_str(); }

RRS_API int rrs_force_path(int softmax_path, int sum_path) {
  if (softmax_path < RRS_PATH_AUTO || softmax_path >= RRS_PATH_COUNT) return RRS_ERR_INVALID_ARG;
  if (sum_path < RRS_SUM_AUTO || sum_path >= RRS_SUM_COUNT) return RRS_ERR_INVALID_ARG;
  g_force_softmax.store(softmax_path);
  g_force_sum.store(sum_path);
  return RRS_OK;
}

RRS_API int rrs_force_cols_path(int cols_path) {
  if (cols_path < RRS_COLS_AUTO || cols_path >= RRS_COLS_COUNT) return RRS_ERR_INVALID_ARG;
  g_force_cols.store(cols_path);
  return RRS_OK;
}

RRS_API int rrs_inject_fault(int kind) {
  if (kind < 0 || kind > 2) return RRS_ERR_INVALID_ARG;
  g_fault.store(kind);
  return RRS_OK;
}

RRS_API int rrs_cols_two_pass_item(int64_t t, int64_t Q, int64_t D, int* pass, int64_t* k) {
  if (!pass || !k || Q < 1 || D < 1 || D > Q || t < 0 || t >= 2 * Q) return RRS_ERR_INVALID_ARG;
  cols_two_pass_item(t, Q, D, pass, k);
  return RRS_OK;
}

RRS_API int rrs_plan_softmax(int64_t M, int64_t N, int64_t ld, int vector_ok_flag, int sm_count,
                             int smem_optin, rrs_plan* plan) {
  if (!plan) return RRS_ERR_INVALID_ARG;
  return plan_softmax_impl(M, N, ld, vector_ok_flag, sm_count, smem_optin, 1, g_force_softmax.load(),
                           plan);
}

RRS_API int rrs_plan_row_sum(int64_t M, int64_t N, int64_t ld, int vector_ok_flag, int sm_count,
                             int smem_optin, rrs_plan* plan) {
  if (!plan) return RRS_ERR_INVALID_ARG;
  return plan_row_sum_impl(M, N, ld, vector_ok_flag, sm_count, smem_optin, g_force_sum.load(),
                           plan);
}

RRS_API int rrs_plan_softmax_cols(int64_t M, int64_t N, int64_t ld, int vector_ok_flag,
                                  int sm_count, int smem_optin, rrs_plan* plan) {
  if (!plan) return RRS_ERR_INVALID_ARG;
  (void)smem_optin;
  return plan_cols_impl(M, N, ld, vector_ok_flag, sm_count, 1, g_force_cols.load(), plan);
}

RRS_API int rrs_occupancy(int threads, int regs, int sm_regs, int max_warps, int* blocks,
                          int* warps) {
  if (threads <= 0 || regs <= 0 || sm_regs <= 0 || max_warps <= 0) return 0;
  const int warps_per_block = (threads + 31) / 32;
  int b = std::min(sm_regs / (threads * regs), max_warps / warps_per_block);
  if (b < 0) b = 0;
  if (blocks) *blocks = b;
  if (warps) *warps = b * warps_per_block;
  return (int)((int64_t)b * warps_per_block * 10000 / max_warps);
}

RRS_API int64_t rrs_waves(int64_t blocks, int64_t slots, int64_t* last_wave, int64_t* idle) {
  if (blocks <= 0 || slots <= 0) {
    if (last_wave) *last_wave = 0;
    if (idle) *idle = slots > 0 ? slots : 0;
    return 0;
  }
  const int64_t waves = ceil_div(blocks, slots);
  const int64_t last = blocks - (waves - 1) * slots;
  if (last_wave) *last_wave = last;
  if (idle) *idle = slots - last;
  return waves;
}

RRS_API int softmax_rows_ex(const float* x, int64_t ldx, float* y, int64_t ldy, int64_t M,
                            int64_t N, int flags, void* stream) {
  clear_last_error();
  if (flags & ~RRS_LOG_SOFTMAX) return fail(RRS_ERR_INVALID_ARG, "unknown flag bits");
  int64_t xext = 0, yext = 0;
  int st = check_shape(M, N, ldx, &xext);
  if (st != RRS_OK) return st;
  if ((st = check_shape(M, N, ldy, &yext)) != RRS_OK) return st;
  if (M == 0 || N == 0) return RRS_OK;
  if (!x || !y) return fail(RRS_ERR_INVALID_ARG, "null pointer");
  if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(y) % 4)
    return fail(RRS_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
  // in place (the same matrix, the same stride) is allowed; any other overlap is not
  const bool in_place = (static_cast<const void*>(x) == static_cast<const void*>(y)) && ldx == ldy;
  if (!in_place && overlaps(x, xext * 4, y, yext * 4)) return fail(RRS_ERR_ALIAS, "x and y overlap");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if ((st = check_no_pending_timeout(dev)) != RRS_OK) return st;
  if ((st = check_device_pointer(x, dev, "x")) != RRS_OK) return st;
  if ((st = check_device_pointer(y, dev, "y")) != RRS_OK) return st;
  DeviceInfo info;
  if ((st = device_info(dev, &info)) != RRS_OK) return st;

  const bool vec = vector_ok(x, y, ldx) && ldy % 4 == 0;
  const bool alike = (reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) % 16 == 0 &&
                     (ldx - ldy) % 4 == 0;   // every row of x and of y misaligned the same way
  rrs_plan plan;
  st = plan_softmax_impl(M, N, std::max(ldx, ldy), vec ? 1 : (alike ? 2 : 0), info.sm_count, info.smem_optin,
                         info.cluster_launch, g_force_softmax.load(), &plan);
  if (st != RRS_OK) return st;
  Layout l;
  l.ldx = ldx;
  l.ldy = ldy;
  l.log_out = (flags & RRS_LOG_SOFTMAX) ? 1 : 0;
  if (l.log_out && plan.path == RRS_PATH_ROW_STAGED)
    return fail(RRS_ERR_UNSUPPORTED, "ROW_STAGED writes the softmax only");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (plan.path) {
    case RRS_PATH_ROW_REGS:
      e = launch_softmax_row_regs(plan, x, y, M, N, l, s);
      break;
    case RRS_PATH_CLUSTER:
      e = launch_softmax_cluster(plan, x, y, M, N, l, s);
      break;
    case RRS_PATH_ROW_STAGED:
      e = (plan.vec > 0) ? launch_softmax_staged_rows(plan, x, y, M, N, l, s)
                         : launch_softmax_staged_long(plan, x, y, M, N, l, s);
      break;
    case RRS_PATH_GRID: {
      void* ws = nullptr;
      unsigned* herr = nullptr;
      if ((st = host_err_word(dev, s, &herr)) != RRS_OK) return st;
      if ((st = get_workspace(dev, s, kWsGrid, (size_t)plan.workspace_bytes, &ws)) != RRS_OK) return st;
      e = launch_softmax_staged_grid(plan, x, y, M, N, l, ws, g_fault.load() == 1 ? 1 : 0, herr, s);
      break;
    }
    case RRS_PATH_TWO_PHASE: {
      void* ws = nullptr;
      if ((st = get_workspace(dev, s, kWsTwoPhase, (size_t)plan.workspace_bytes, &ws)) != RRS_OK)
        return st;
      e = launch_softmax_two_phase(plan, x, y, M, N, l, ws, s);
      break;
    }
    case RRS_PATH_TWO_PASS: {
      void* ws = nullptr;
      unsigned* herr = nullptr;
      if ((st = host_err_word(dev, s, &herr)) != RRS_OK) return st;
      if ((st = get_workspace(dev, s, kWsRowsTwoPass, (size_t)plan.workspace_bytes, &ws)) != RRS_OK) return st;
      e = launch_softmax_rows_two_pass(plan, x, y, M, N, l, ws, g_fault.load() == 2 ? 1 : 0, herr, s);
      break;
    }
    default:
      return fail(RRS_ERR_UNSUPPORTED, "planned path has no launcher");
  }
  if (e != cudaSuccess) return fail_cuda(e, "softmax launch");
  return RRS_OK;
}

RRS_API int softmax_cols(const float* x, int64_t ldx, float* y, int64_t ldy, int64_t M, int64_t N,
                         int flags, void* stream) {
  clear_last_error();
  if (flags & ~RRS_LOG_SOFTMAX) return fail(RRS_ERR_INVALID_ARG, "unknown flag bits");
  int64_t xext = 0, yext = 0;
  int st = check_shape(M, N, ldx, &xext);
  if (st != RRS_OK) return st;
  if ((st = check_shape(M, N, ldy, &yext)) != RRS_OK) return st;
  if (M == 0 || N == 0) return RRS_OK;
  if (!x || !y) return fail(RRS_ERR_INVALID_ARG, "null pointer");
  if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(y) % 4)
    return fail(RRS_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
  const bool in_place = (static_cast<const void*>(x) == static_cast<const void*>(y)) && ldx == ldy;
  if (!in_place && overlaps(x, xext * 4, y, yext * 4)) return fail(RRS_ERR_ALIAS, "x and y overlap");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if ((st = check_no_pending_timeout(dev)) != RRS_OK) return st;
  if ((st = check_device_pointer(x, dev, "x")) != RRS_OK) return st;
  if ((st = check_device_pointer(y, dev, "y")) != RRS_OK) return st;
  DeviceInfo info;
  if ((st = device_info(dev, &info)) != RRS_OK) return st;

  const bool vec = vector_ok(x, y, ldx) && ldy % 4 == 0;
  rrs_plan plan;
  st = plan_cols_impl(M, N, std::max(ldx, ldy), vec ? 1 : 0, info.sm_count, info.cluster_launch,
                      g_force_cols.load(), &plan);
  if (st != RRS_OK) return st;
  Layout l;
  l.ldx = ldx;
  l.ldy = ldy;
  l.log_out = (flags & RRS_LOG_SOFTMAX) ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (plan.path == RRS_COLS_CLUSTER) {
    e = launch_softmax_cols_cluster(plan, x, y, M, N, l, s);
  } else if (plan.path == RRS_COLS_BAND) {
    e = launch_softmax_cols_band(plan, x, y, M, N, l, s);
  } else if (plan.path == RRS_COLS_TWO_PASS) {
    void* ws = nullptr;
    unsigned* herr = nullptr;
    if ((st = host_err_word(dev, s, &herr)) != RRS_OK) return st;
    if ((st = get_workspace(dev, s, kWsColsTwoPass, (size_t)plan.workspace_bytes, &ws)) != RRS_OK) return st;
    e = launch_softmax_cols_two_pass(plan, x, y, M, N, l, ws, g_fault.load() == 2 ? 1 : 0, herr, s);
  } else {
    void* ws = nullptr;
    if ((st = get_workspace(dev, s, kWsCols, (size_t)plan.workspace_bytes, &ws)) != RRS_OK) return st;
    e = launch_softmax_cols_two_phase(plan, x, y, M, N, l, ws, s);
  }
  if (e != cudaSuccess) return fail_cuda(e, "softmax_cols launch");
  return RRS_OK;
}

RRS_API int softmax_rows(const float* x, float* y, int64_t M, int64_t N, int64_t ld,
                         void* stream) {
  return softmax_rows_ex(x, ld, y, ld, M, N, 0, stream);
}

RRS_API int log_softmax_rows(const float* x, float* y, int64_t M, int64_t N, int64_t ld,
                             void* stream) {
  return softmax_rows_ex(x, ld, y, ld, M, N, RRS_LOG_SOFTMAX, stream);
}

}  // extern "C"

namespace rrs {
namespace {

// row_sum / row_max / row_mean: one planner and one kernel family (op).
int row_reduce_impl(int op, const char* name, const float* x, float* out, int64_t M, int64_t N,
                    int64_t ld, void* stream) {
  clear_last_error();
  int64_t extent = 0;
  int st = check_shape(M, N, ld, &extent);
  if (st != RRS_OK) return st;
  if (M == 0) return RRS_OK;
  if (!out || (N > 0 && !x)) return fail(RRS_ERR_INVALID_ARG, "null pointer");
  if (reinterpret_cast<uintptr_t>(out) % 4 || reinterpret_cast<uintptr_t>(x) % 4)
    return fail(RRS_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
  if (N > 0 && overlaps(x, extent * 4, out, M * 4)) return fail(RRS_ERR_ALIAS, "x and out overlap");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if ((st = check_no_pending_timeout(dev)) != RRS_OK) return st;
  if ((st = check_device_pointer(out, dev, "out")) != RRS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {  // the empty row's value: the sum's identity 0, the max's -inf, the mean 0/0
    const float v = op == kOpSum ? 0.f
                  : op == kOpMax ? -std::numeric_limits<float>::infinity()
                                 : std::numeric_limits<float>::quiet_NaN();
    e = launch_fill(out, M, v, s);
    return e == cudaSuccess ? RRS_OK : fail_cuda(e, (std::string(name) + " fill").c_str());
  }
  if ((st = check_device_pointer(x, dev, "x")) != RRS_OK) return st;
  DeviceInfo info;
  if ((st = device_info(dev, &info)) != RRS_OK) return st;

  rrs_plan plan;
  const bool vok = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (ld % 4 == 0);
  st = plan_row_sum_impl(M, N, ld, vok ? 1 : 0, info.sm_count, info.smem_optin,
                         g_force_sum.load(), &plan);
  if (st != RRS_OK) return st;
  switch (plan.path) {
    case RRS_SUM_ROW:
      e = launch_row_reduce_rows(op, plan, x, out, M, N, ld, s);
      break;
    case RRS_SUM_SPLIT: {
      void* ws = nullptr;
      if ((st = get_workspace(dev, s, kWsRowSum, (size_t)plan.workspace_bytes, &ws)) != RRS_OK)
        return st;
      e = launch_row_reduce_split(op, plan, x, out, M, N, ld, ws, s);
      break;
    }
    default:
      return fail(RRS_ERR_UNSUPPORTED, "planned path has no launcher");
  }
  if (e != cudaSuccess) return fail_cuda(e, (std::string(name) + " launch").c_str());
  return RRS_OK;
}

}  // namespace
}  // namespace rrs

extern "C" {

RRS_API int row_sum(const float* x, float* out, int64_t M, int64_t N, int64_t ld, void* stream) {
  return row_reduce_impl(kOpSum, "row_sum", x, out, M, N, ld, stream);
}

RRS_API int row_max(const float* x, float* out, int64_t M, int64_t N, int64_t ld, void* stream) {
  return row_reduce_impl(kOpMax, "row_max", x, out, M, N, ld, stream);
}

RRS_API int row_mean(const float* x, float* out, int64_t M, int64_t N, int64_t ld, void* stream) {
  return row_reduce_impl(kOpMean, "row_mean", x, out, M, N, ld, stream);
}

RRS_API int gelu(const float* x, float* y, int64_t n, void* stream) {
  clear_last_error();
  if (n < 0) return fail(RRS_ERR_INVALID_ARG, "n must be >= 0");
  if (n == 0) return RRS_OK;
  if (n > INT64_MAX / 8) return fail(RRS_ERR_INVALID_ARG, "extent overflows");
  if (!x || !y) return fail(RRS_ERR_INVALID_ARG, "null pointer");
  if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(y) % 4)
    return fail(RRS_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
  if (static_cast<const void*>(x) != static_cast<const void*>(y) && overlaps(x, n * 4, y, n * 4))
    return fail(RRS_ERR_ALIAS, "x and y overlap");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  int st;
  if ((st = check_no_pending_timeout(dev)) != RRS_OK) return st;
  if ((st = check_device_pointer(x, dev, "x")) != RRS_OK) return st;
  if ((st = check_device_pointer(y, dev, "y")) != RRS_OK) return st;
  DeviceInfo info;
  if ((st = device_info(dev, &info)) != RRS_OK) return st;
  e = launch_gelu(x, y, n, info.sm_count, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "gelu launch");
  return RRS_OK;
}

RRS_API int attention_fwd(const void* q, const void* k, const void* v, float* o, float* lse,
                          int64_t BH, int64_t L, int64_t S, int64_t d, int causal, float scale,
                          void* stream) {
  clear_last_error();
  if (BH < 0 || L < 0 || S < 0) return fail(RRS_ERR_INVALID_ARG, "BH, L and S must be >= 0");
  if (d != 64 && d != 128) return fail(RRS_ERR_INVALID_ARG, "head dimension must be 64 or 128");
  if (BH == 0 || L == 0) return RRS_OK;
  if (S == 0) return fail(RRS_ERR_INVALID_ARG, "S must be >= 1 when L >= 1");
  if (BH > 65535 || L > INT_MAX - 256 || S > INT_MAX - 256)
    return fail(RRS_ERR_INVALID_ARG, "BH <= 65535, L and S < 2^31 - 256");
  if (!(scale >= 0.f) || std::isinf(scale)) return fail(RRS_ERR_INVALID_ARG, "scale must be finite and >= 0");
  if (!q || !k || !v || !o) return fail(RRS_ERR_INVALID_ARG, "null pointer");
  const void* ptrs[4] = {q, k, v, o};
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) % 16)
      return fail(RRS_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (lse && reinterpret_cast<uintptr_t>(lse) % 4) return fail(RRS_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  const int64_t qb = BH * L * d * 2, kb = BH * S * d * 2, ob = BH * L * d * 4, lb = BH * L * 4;
  if (overlaps(o, ob, q, qb) || overlaps(o, ob, k, kb) || overlaps(o, ob, v, kb) ||
      (lse && (overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kb) || overlaps(lse, lb, v, kb) ||
               overlaps(lse, lb, o, ob))))
    return fail(RRS_ERR_ALIAS, "outputs overlap inputs or each other");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  int st;
  if ((st = check_no_pending_timeout(dev)) != RRS_OK) return st;
  if ((st = check_device_pointer(q, dev, "q")) != RRS_OK) return st;
  if ((st = check_device_pointer(k, dev, "k")) != RRS_OK) return st;
  if ((st = check_device_pointer(v, dev, "v")) != RRS_OK) return st;
  if ((st = check_device_pointer(o, dev, "o")) != RRS_OK) return st;
  if (lse && (st = check_device_pointer(lse, dev, "lse")) != RRS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt((float)d);
  e = launch_attention(static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
                       static_cast<const uint16_t*>(v), o, lse, (int)BH, (int)L, (int)S, (int)d,
                       causal ? 1 : 0, sc, s);
  if (e != cudaSuccess) return fail_cuda(e, "attention_fwd launch");
  return RRS_OK;
}

RRS_API int rrs_device_error(void* stream) {
  clear_last_error();
  unsigned v = 0, w = 0;
  cudaError_t e = read_and_clear_staged_error(static_cast<cudaStream_t>(stream), &v);
  if (e == cudaSuccess) e = read_and_clear_attn_error(static_cast<cudaStream_t>(stream), &w);
  unsigned c = 0, r2 = 0;
  if (e == cudaSuccess) e = read_and_clear_cols_error(static_cast<cudaStream_t>(stream), &c);
  if (e == cudaSuccess) e = read_and_clear_rows_two_pass_error(static_cast<cudaStream_t>(stream), &r2);
  if (e != cudaSuccess) return fail_cuda(e, "rrs_device_error");
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    if (host_err_value(dev) != 0) v |= 1u;
    host_err_clear(dev);
  }
  v |= w | c | r2;
  return v ? fail(RRS_ERR_TIMEOUT, "a split-row kernel stopped waiting for its peers") : RRS_OK;
}

RRS_API int rrs_test_occupy(int ctas, int smem_bytes, int64_t nanoseconds, void* stream) {
  clear_last_error();
  if (ctas < 1 || ctas > 65535 || smem_bytes < 0 || nanoseconds < 0 || nanoseconds > 200000000)
    return fail(RRS_ERR_INVALID_ARG, "1 <= ctas <= 65535, smem_bytes >= 0, 0 <= ns <= 2e8");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  DeviceInfo info;
  int st;
  if ((st = device_info(dev, &info)) != RRS_OK) return st;
  if (smem_bytes > info.smem_optin) return fail(RRS_ERR_INVALID_ARG, "smem_bytes above the opt-in limit");
  e = launch_occupy(ctas, smem_bytes, nanoseconds, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "rrs_test_occupy launch");
  return RRS_OK;
}

RRS_API int rrs_release_workspace(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  (void)cudaGetDevice(&cur);
  int status = RRS_OK;
  for (auto& kv : g_workspaces) {
    if (!kv.second.ptr) continue;
    if (cudaSetDevice(std::get<0>(kv.first)) == cudaSuccess) {
      cudaError_t e = cudaDeviceSynchronize();
      if (e == cudaSuccess) e = cudaFree(kv.second.ptr);
      if (e != cudaSuccess) status = fail_cuda(e, "rrs_release_workspace");
    }
  }
  g_workspaces.clear();
  for (auto& r : g_retired) {
    if (cudaSetDevice(r.first) == cudaSuccess) {
      cudaError_t e = cudaDeviceSynchronize();
      if (e == cudaSuccess) e = cudaFree(r.second);
      if (e != cudaSuccess) status = fail_cuda(e, "rrs_release_workspace");
    }
  }
  g_retired.clear();
  (void)cudaSetDevice(cur);
  return status;
}

}  // extern "C"
