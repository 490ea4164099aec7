// Allocation-free variant of the route sort (moe_route_sort_noalloc).
//
// Some callers cannot allocate device memory at the moment they need the
// sort: a plugin's enqueue callback inside an inference engine that has
// already handed all device memory to its own pool, a server that reserved
// the whole device up front for its caches, or a latency-critical loop in which
// a cudaMalloc (which can synchronise the device) is not allowed.  For them,
// the sort's scratch (the per-block histograms of the multi-block path) lives in
// a fixed array in this library's device memory
// instead of a caller-provided workspace.  The caller still passes the inputs
// and outputs.
//
// The array is a file-scope __device__ symbol: every GPU that loads the
// library holds it until the process exits (or the context is reset).  Host code
// cannot use the symbol's name as a device address, so the first call in each
// context of a device looks the address up with cudaGetSymbolAddress (with that
// device current) and caches it together with the context's ID; a call in a new
// context (after a cudaDeviceReset, or once the primary context was released and
// created again, which loads the module at a new address) looks it up again.
// That look-up should therefore not fall inside a stream capture.
#include <mutex>

#include "abi_checks.h"
#include "common.cuh"
#include "kernels.h"
#include "tensor_map.h"

namespace {

// Multi-block path: at most kMaxBlocks blocks (8192 routes each at the largest R),
// E + 1 <= 1024 buckets, one histogram per block.
constexpr int kMaxBlocks = 64;
static_assert(MOE_ROUTE_SORT_NOALLOC_MAX_ROUTES <= kMaxBlocks * 8192, "blocks of the largest sort");
constexpr size_t kScratchInts = kMaxBlocks * 1024u;  // 64 Ki int32 = 256 KiB

static __device__ __align__(256) int32_t g_route_sort_scratch[kScratchInts];

std::mutex g_scratch_mutex;
int32_t* g_scratch_addr[moe::kMaxDevices] = {};
unsigned long long g_scratch_ctx[moe::kMaxDevices] = {};

// Device address of the scratch array in the current device's current context.
cudaError_t scratch_address(int32_t** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= moe::kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  const unsigned long long ctx = moe::context_id();
  if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_sort_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<int32_t*>(p);
    g_scratch_ctx[dev] = moe::context_id();  // the look-up made the context current if it was not
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int32_t moe_route_sort_noalloc(const moe_dims_t* d, const int32_t* expert_idx, int32_t* sorted_src_route,
                                          int32_t* expanded_row_idx, int32_t* tokens_per_expert, int32_t* cumsum,
                                          void* stream) {
  // the checks moe_route_sort makes, in the same order, plus the size limit of the fixed scratch
  int32_t rc = moe::check_dims(d);
  if (rc != MOE_OK) return rc;
  const int64_t R = (int64_t)d->M * d->topK;
  if (R > MOE_ROUTE_SORT_NOALLOC_MAX_ROUTES) return MOE_ERR_SHAPE;  // beyond the fixed scratch
  if (!expert_idx || !sorted_src_route || !expanded_row_idx || !tokens_per_expert || !cumsum) return MOE_ERR_NULL;
  if (!moe::all_aligned16({expert_idx, sorted_src_route, expanded_row_idx, tokens_per_expert, cumsum}))
    return MOE_ERR_ALIGN;
  if ((rc = moe::check_device()) != MOE_OK) return rc;
  int32_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_LAUNCH;
  // The kernels write every scratch entry they later read (the histograms), so
  // the previous call's contents need no clearing.
  return moe::launch_status(moe::launch_route_sort(expert_idx, (int)R, d->E, sorted_src_route, expanded_row_idx,
                                                   tokens_per_expert, cumsum, scratch,
                                                   static_cast<cudaStream_t>(stream), kMaxBlocks));
}
