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
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "internal.h"
#include "rrs.h"

namespace rrs {
namespace {

thread_local std::string g_last_error;
std::atomic<int> g_force_softmax{RRS_PATH_AUTO};
std::atomic<int> g_force_sum{RRS_SUM_AUTO};

int fail(int status, const std::string& msg) {
  g_last_error = msg;
  return status;
}

int fail_cuda(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return RRS_ERR_CUDA;
}

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
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&d.coop_launch, cudaDevAttrCooperativeLaunch, dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
  g_devices[dev] = d;
  *out = d;
  return RRS_OK;
}

// --------------------------------------------------------------- workspace ---
// One buffer per (device, stream): calls on one stream are ordered, so they
// can share it; calls on different streams never do.  Grown with the
// stream-ordered allocator, so growth is ordered after earlier work on the
// stream that still reads the old buffer.
struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, uintptr_t>, Workspace> g_workspaces;

int get_workspace(int dev, cudaStream_t s, size_t bytes, void** ptr) {
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspaces[{dev, reinterpret_cast<uintptr_t>(s)}];
  if (w.bytes < bytes) {
    if (w.ptr) {
      cudaError_t e = cudaFreeAsync(w.ptr, s);
      w.ptr = nullptr;
      w.bytes = 0;
      if (e != cudaSuccess) return fail_cuda(e, "cudaFreeAsync(workspace)");
    }
    const size_t want = std::max<size_t>(round_up((int64_t)bytes, 1 << 16), 1 << 16);
    cudaError_t e = cudaMallocAsync(&w.ptr, want, s);
    if (e != cudaSuccess) {
      w.ptr = nullptr;
      (void)cudaGetLastError();
      return fail(RRS_ERR_NOMEM, std::string("cudaMallocAsync(workspace): ") + cudaGetErrorString(e));
    }
    w.bytes = want;
  }
  *ptr = w.ptr;
  return RRS_OK;
}

// ----------------------------------------------------------------- checks ---
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

// Shape checks shared by both operations; sets *extent (elements spanned by
// x) when M > 0.
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

// ---------------------------------------------------------------- planner ---
void plan_row_regs(int64_t M, int64_t N, int sm_count, rrs_plan* p) {
  const int64_t n4 = N >> 2;
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

bool plan_cluster(int64_t M, int64_t N, rrs_plan* p) {
  const int64_t n4 = N >> 2;
  int vec = kClusterVec;
  int cs = pow2_ceil(std::max<int64_t>(1, ceil_div(n4, (int64_t)kSplitThreads * vec)));
  if (cs > kClusterMax) return false;
  // a cluster of one CTA per 4 KiB-aligned segment; shrink registers when the segment is short
  if (ceil_div(n4, cs) <= (int64_t)kSplitThreads * 4) vec = 4;
  p->path = RRS_PATH_CLUSTER;
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

int plan_softmax_impl(int64_t M, int64_t N, int64_t ld, int vector_ok, int sm_count,
                      int smem_optin, int cluster_ok, int forced, rrs_plan* p) {
  std::memset(p, 0, sizeof(*p));
  if (M < 0 || N < 0 || ld < 1 || ld < N || sm_count < 1)
    return fail(RRS_ERR_INVALID_ARG, "bad shape or device description");
  (void)smem_optin;
  p->cluster = 1;
  p->vector_io = vector_ok ? 1 : 0;
  if (M == 0 || N == 0) {
    p->path = (forced == RRS_PATH_AUTO) ? RRS_PATH_ROW_REGS : forced;
    return RRS_OK;
  }
  int path = forced;
  if (path == RRS_PATH_AUTO) {
    if (!vector_ok) {
      path = RRS_PATH_TWO_PHASE;
    } else if (N <= 16384) {
      path = RRS_PATH_ROW_REGS;
    } else if (cluster_ok && N <= (int64_t)kClusterMax * kSplitThreads * kClusterVec * 4) {
      path = RRS_PATH_CLUSTER;
    } else {
      path = RRS_PATH_TWO_PHASE;
    }
  }
  switch (path) {
    case RRS_PATH_ROW_REGS:
      if (!vector_ok || !row_regs_fits(N))
        return fail(RRS_ERR_UNSUPPORTED, "ROW_REGS needs 16-byte alignment and N <= 32768");
      plan_row_regs(M, N, sm_count, p);
      return RRS_OK;
    case RRS_PATH_CLUSTER:
      if (!vector_ok || !cluster_ok || !plan_cluster(M, N, p))
        return fail(RRS_ERR_UNSUPPORTED, "CLUSTER needs 16-byte alignment, cluster launch and N <= 131072");
      return RRS_OK;
    case RRS_PATH_TWO_PHASE:
      plan_two_phase(M, N, sm_count, p);
      return RRS_OK;
    default:
      return fail(RRS_ERR_UNSUPPORTED, "path not available");
  }
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
    // about 32 floats per thread before a CTA holds more than 16 warps
    const int gw = (int)std::min<int64_t>(16, std::max<int64_t>(1, pow2_ceil(ceil_div(N, 32 * 32 * 2))));
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
}  // namespace rrs

using namespace rrs;

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

RRS_API const char* rrs_last_error(void) { return g_last_error.c_str(); }

RRS_API int rrs_force_path(int softmax_path, int sum_path) {
  if (softmax_path < RRS_PATH_AUTO || softmax_path >= RRS_PATH_COUNT) return RRS_ERR_INVALID_ARG;
  if (sum_path < RRS_SUM_AUTO || sum_path >= RRS_SUM_COUNT) return RRS_ERR_INVALID_ARG;
  g_force_softmax.store(softmax_path);
  g_force_sum.store(sum_path);
  return RRS_OK;
}

RRS_API int rrs_plan_softmax(int64_t M, int64_t N, int64_t ld, int vector_ok_flag, int sm_count,
                             int smem_optin, rrs_plan* plan) {
  if (!plan) return RRS_ERR_INVALID_ARG;
  return plan_softmax_impl(M, N, ld, vector_ok_flag, sm_count, smem_optin, 1,
                           g_force_softmax.load(), plan);
}

RRS_API int rrs_plan_row_sum(int64_t M, int64_t N, int64_t ld, int vector_ok_flag, int sm_count,
                             int smem_optin, rrs_plan* plan) {
  if (!plan) return RRS_ERR_INVALID_ARG;
  return plan_row_sum_impl(M, N, ld, vector_ok_flag, sm_count, smem_optin, g_force_sum.load(),
                           plan);
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

RRS_API int softmax_rows(const float* x, float* y, int64_t M, int64_t N, int64_t ld,
                         void* stream) {
  g_last_error.clear();
  int64_t extent = 0;
  int st = check_shape(M, N, ld, &extent);
  if (st != RRS_OK) return st;
  if (M == 0 || N == 0) return RRS_OK;
  if (!x || !y) return fail(RRS_ERR_INVALID_ARG, "null pointer");
  if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(y) % 4)
    return fail(RRS_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
  if (overlaps(x, extent * 4, y, extent * 4)) return fail(RRS_ERR_ALIAS, "x and y overlap");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if ((st = check_device_pointer(x, dev, "x")) != RRS_OK) return st;
  if ((st = check_device_pointer(y, dev, "y")) != RRS_OK) return st;
  DeviceInfo info;
  if ((st = device_info(dev, &info)) != RRS_OK) return st;

  rrs_plan plan;
  st = plan_softmax_impl(M, N, ld, vector_ok(x, y, ld) ? 1 : 0, info.sm_count, info.smem_optin,
                         info.cluster_launch, g_force_softmax.load(), &plan);
  if (st != RRS_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (plan.path) {
    case RRS_PATH_ROW_REGS:
      e = launch_softmax_row_regs(plan, x, y, M, N, ld, s);
      break;
    case RRS_PATH_CLUSTER:
      e = launch_softmax_cluster(plan, x, y, M, N, ld, s);
      break;
    case RRS_PATH_TWO_PHASE: {
      void* ws = nullptr;
      if ((st = get_workspace(dev, s, (size_t)plan.workspace_bytes, &ws)) != RRS_OK) return st;
      e = launch_softmax_two_phase(plan, x, y, M, N, ld, ws, s);
      break;
    }
    default:
      return fail(RRS_ERR_UNSUPPORTED, "planned path has no launcher");
  }
  if (e != cudaSuccess) return fail_cuda(e, "softmax_rows launch");
  return RRS_OK;
}

RRS_API int row_sum(const float* x, float* out, int64_t M, int64_t N, int64_t ld, void* stream) {
  g_last_error.clear();
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
  if ((st = check_device_pointer(out, dev, "out")) != RRS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    e = cudaMemsetAsync(out, 0, (size_t)M * sizeof(float), s);
    return e == cudaSuccess ? RRS_OK : fail_cuda(e, "cudaMemsetAsync");
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
      e = launch_row_sum_rows(plan, x, out, M, N, ld, s);
      break;
    case RRS_SUM_SPLIT: {
      void* ws = nullptr;
      if ((st = get_workspace(dev, s, (size_t)plan.workspace_bytes, &ws)) != RRS_OK) return st;
      e = launch_row_sum_split(plan, x, out, M, N, ld, ws, s);
      break;
    }
    default:
      return fail(RRS_ERR_UNSUPPORTED, "planned path has no launcher");
  }
  if (e != cudaSuccess) return fail_cuda(e, "row_sum launch");
  return RRS_OK;
}

RRS_API int rrs_device_error(void* stream) {
  unsigned v = 0;
  cudaError_t e = read_and_clear_device_error(static_cast<cudaStream_t>(stream), &v);
  if (e != cudaSuccess) return fail_cuda(e, "rrs_device_error");
  return v ? fail(RRS_ERR_TIMEOUT, "a split-row kernel stopped waiting for its peers") : RRS_OK;
}

RRS_API int rrs_release_workspace(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  (void)cudaGetDevice(&cur);
  int status = RRS_OK;
  for (auto& kv : g_workspaces) {
    if (!kv.second.ptr) continue;
    if (cudaSetDevice(kv.first.first) == cudaSuccess) {
      cudaError_t e = cudaDeviceSynchronize();
      if (e == cudaSuccess) e = cudaFree(kv.second.ptr);
      if (e != cudaSuccess) status = fail_cuda(e, "rrs_release_workspace");
    }
  }
  g_workspaces.clear();
  (void)cudaSetDevice(cur);
  return status;
}

}  // extern "C"
