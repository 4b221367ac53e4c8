// softmax_rows_noalloc: the row softmax for callers that may not allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) on the
// path that calls this library: a plugin's execute/enqueue hook inside an
// inference engine, where the host framework owns every byte of device
// memory and allocation there is forbidden; or a latency-critical loop where
// an allocation could synchronise the device or fail under memory pressure
// halfway through a step.  softmax_rows may allocate a small workspace on
// first use of a stream; this entry point never does.  Where softmax_rows
// would run a kernel that needs no workspace (the register kernel or the
// cluster split), it runs that same kernel; where it would run the grid
// split or the two-pass split, it runs that kernel with its workspace in a
// fixed array of device memory that is part of the library image (when the
// shape's slots fit);
// otherwise it runs the two-phase kernels (per-chunk (max, sum) partials,
// then merge, re-read and write) with the partials in another such array.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it until the process exits.  In host code its name is only a
// host-side stand-in, never a device address: the device address is taken
// once per device with cudaGetSymbolAddress, with that device current, and
// passed to the kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstring>
#include <map>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"
#include "rrs.h"

namespace rrs {
namespace {

// Capacity: (max, sum) pairs, one per (row, chunk) of a call.  8 bytes each,
// so 1 MiB of device memory per GPU.
constexpr int64_t kNoAllocPairs = 131072;
// Smallest chunk a row is cut into before the SM count asks for more.
constexpr int64_t kNoAllocMinChunk = 4096;

static __device__ __align__(256) MaxSum g_noalloc_partials[kNoAllocPairs];

// The grid and two-pass splits' workspace (an arrival counter, then 16
// bytes per (row, segment) or (row, chunk) slot).  Zero at load, and each
// launch leaves it ready for the next: the last CTA to draw opens the next
// epoch, and a slot only counts when it carries the current launch's ticket.
constexpr int64_t kNoAllocGridBytes = 1 << 20;
static __device__ __align__(256) unsigned char g_noalloc_grid_ws[kNoAllocGridBytes];

struct NoAllocDevice {
  void* scratch = nullptr;   // device address of g_noalloc_partials on this device
  void* grid_ws = nullptr;   // device address of g_noalloc_grid_ws on this device
  int sm_count = 0;
};

std::mutex g_noalloc_mu;
std::map<int, NoAllocDevice> g_noalloc_devices;

// Set-up, once per device, with that device current (the caller's current
// device at its first call): look up the scratch array's device address.
int noalloc_device(int dev, NoAllocDevice* out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  auto it = g_noalloc_devices.find(dev);
  if (it != g_noalloc_devices.end()) {
    *out = it->second;
    return RRS_OK;
  }
  NoAllocDevice d;
  cudaError_t e = cudaGetSymbolAddress(&d.scratch, g_noalloc_partials);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(noalloc scratch)");
  e = cudaGetSymbolAddress(&d.grid_ws, g_noalloc_grid_ws);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(noalloc grid workspace)");
  if (d.scratch == nullptr || d.grid_ws == nullptr) return fail(RRS_ERR_CUDA, "noalloc scratch has no device address");
  e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
  g_noalloc_devices[dev] = d;
  *out = d;
  return RRS_OK;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace
}  // namespace rrs

using namespace rrs;

extern "C" RRS_API int softmax_rows_noalloc(const float* x, float* y, int64_t M, int64_t N,
                                            int64_t ld, void* stream) {
  // The same checks and messages as softmax_rows (shared with capi.cu).
  clear_last_error();
  int64_t extent = 0;
  int st = check_shape(M, N, ld, &extent);
  if (st != RRS_OK) return st;
  if (M == 0 || N == 0) return RRS_OK;
  if (!x || !y) return fail(RRS_ERR_INVALID_ARG, "null pointer");
  if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(y) % 4)
    return fail(RRS_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
  // In place (y == x, one shared stride) is allowed, as in softmax_rows:
  // every kernel reads each element before the same thread writes it.  Any
  // other overlap is refused.
  const bool in_place = static_cast<const void*>(x) == static_cast<const void*>(y);
  if (!in_place && overlaps(x, extent * 4, y, extent * 4)) return fail(RRS_ERR_ALIAS, "x and y overlap");
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x), ya = reinterpret_cast<uintptr_t>(y);

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if ((st = check_no_pending_timeout(dev)) != RRS_OK) return st;
  if ((st = check_device_pointer(x, dev, "x")) != RRS_OK) return st;
  if ((st = check_device_pointer(y, dev, "y")) != RRS_OK) return st;
  Layout l;
  l.ldx = ld;
  l.ldy = ld;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  rrs_plan plan;
  const bool planned = plan_like_softmax_rows(x, y, M, N, ld, dev, &plan);
  if (planned && (plan.path == RRS_PATH_ROW_REGS || plan.path == RRS_PATH_CLUSTER)) {
    e = plan.path == RRS_PATH_ROW_REGS ? launch_softmax_row_regs(plan, x, y, M, N, l, s)
                                       : launch_softmax_cluster(plan, x, y, M, N, l, s);
    if (e != cudaSuccess) return fail_cuda(e, "softmax_rows_noalloc launch");
    return RRS_OK;
  }
  NoAllocDevice d;
  if ((st = noalloc_device(dev, &d)) != RRS_OK) return st;
  if (planned && (plan.path == RRS_PATH_GRID || plan.path == RRS_PATH_TWO_PASS) &&
      plan.workspace_bytes <= kNoAllocGridBytes) {
    // Both kernels keep an arrival counter (epoch << 32 | count) and
    // ticket-tagged slots in the same layout, so they share the array: each
    // launch opens the next epoch for whichever comes next.  A wait that
    // runs out sets the device error word (rrs_device_error); the host word
    // that makes later calls refuse is used only if an earlier call made it,
    // since making it allocates.
    unsigned* herr = host_err_word_if_made(dev);
    e = plan.path == RRS_PATH_GRID ? launch_softmax_staged_grid(plan, x, y, M, N, l, d.grid_ws, 0, herr, s)
                                   : launch_softmax_rows_two_pass(plan, x, y, M, N, l, d.grid_ws, 0, herr, s);
    if (e != cudaSuccess) return fail_cuda(e, "softmax_rows_noalloc launch");
    return RRS_OK;
  }
  // Every row needs at least one (max, sum) slot of the fixed scratch.
  if (M > kNoAllocPairs)
    return fail(RRS_ERR_INVALID_ARG,
                "softmax_rows_noalloc takes at most 131072 rows where its two-phase kernels run");

  // Chunks per row: enough CTAs to fill the GPU (about 4 per SM), chunks of
  // about kNoAllocMinChunk columns or more (rounded up to kChunkAlign), and
  // never more (row, chunk) pairs than the scratch holds.
  int64_t C = std::max<int64_t>(1, std::min(cdiv(4 * (int64_t)d.sm_count, M), cdiv(N, kNoAllocMinChunk)));
  C = std::min<int64_t>(C, kNoAllocPairs / M);
  const int64_t chunk = cdiv(cdiv(N, C), kChunkAlign) * kChunkAlign;
  C = cdiv(N, chunk);

  std::memset(&plan, 0, sizeof(plan));
  plan.path = RRS_PATH_TWO_PHASE;
  plan.threads = kSplitThreads;
  plan.cluster = 1;
  plan.ctas_per_row = C;
  plan.chunk = chunk;
  plan.rows_per_cta = 1;
  plan.rounds = 1;
  plan.grid = std::min<int64_t>(M * C, 32 * (int64_t)d.sm_count);
  plan.vector_io = (xa % 16 == 0 && ya % 16 == 0 && ld % 4 == 0) ? 1 : 0;
  plan.workspace_bytes = 0;

  // All calls on this device share the one scratch array and it keeps the
  // last call's partials.  Nothing in it needs to start at zero: the first
  // kernel writes every slot the second kernel reads.  Two calls whose
  // kernels overlap on the GPU (other streams, other host threads) race on it.
  e = launch_softmax_two_phase(plan, x, y, M, N, l, d.scratch, s);
  if (e != cudaSuccess) return fail_cuda(e, "softmax_rows_noalloc launch");
  return RRS_OK;
}
