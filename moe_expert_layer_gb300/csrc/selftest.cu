// Self-tests of the bounded device-side waits the pipeline kernels use.
//
// One warp initialises an mbarrier that nothing will ever arrive on and waits for
// its first phase with the same bounded wait the GEMM pipelines use.  The wait must
// give up after `limit_us`, record MOE_ERR_TIMEOUT in the status word and let the
// kernel return normally, leaving the CUDA context usable.
#include "common.cuh"

namespace {

__global__ void wait_timeout_probe_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t never;
  if (threadIdx.x == 0) {
    moe::mbar_init(&never, 1);
    moe::fence_barrier_init();
  }
  __syncwarp();
  if (!moe::mbar_wait_bounded(&never, 0, limit_ns)) moe::record_status(status, MOE_ERR_TIMEOUT);
}

// The bounded wait on a count other CTAs raise (the fused SwiGLU's), on a count
// nothing raises.
__global__ void count_timeout_probe_kernel(int32_t* status, const int32_t* count, uint64_t limit_ns) {
  if (threadIdx.x == 0 && !moe::count_wait_bounded(count, 1, limit_ns)) moe::record_status(status, MOE_ERR_TIMEOUT);
}

}  // namespace

extern "C" int32_t moe_selftest_count_timeout(int32_t* status, int32_t* count, uint32_t limit_us, void* stream) {
  if (!status || !count) return MOE_ERR_NULL;
  if (limit_us == 0 || limit_us > 2000000u) return MOE_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess ||
      cudaMemsetAsync(count, 0, sizeof(int32_t), st) != cudaSuccess)
    return MOE_ERR_LAUNCH;
  count_timeout_probe_kernel<<<1, 32, 0, st>>>(status, count, (uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

extern "C" int32_t moe_selftest_wait_timeout(int32_t* status, uint32_t limit_us, void* stream) {
  if (!status) return MOE_ERR_NULL;
  if (limit_us == 0 || limit_us > 2000000u) return MOE_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_LAUNCH;
  wait_timeout_probe_kernel<<<1, 32, 0, st>>>(status, (uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}
