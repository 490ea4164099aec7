// Host-side argument checks shared by the C entry points (include/moe_layer.h,
// "Conventions shared by every entry point"): shapes, pointer alignment and the
// device architecture, all decided before anything is launched.
#pragma once
#include <cstdint>
#include <initializer_list>

#include <cuda_runtime.h>

#include "../../include/moe_layer.h"

namespace moe {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every given (non-null) device pointer 16-byte aligned; optional arguments may be null.
inline bool all_aligned16(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p && !aligned16(p)) return false;
  return true;
}

// The shape preconditions (d->weight_layout not read).
inline int32_t check_shape(const moe_dims_t* d) {
  if (!d) return MOE_ERR_NULL;
  if (d->M < 1 || d->topK < 1 || d->E < d->topK || d->E > 1023) return MOE_ERR_SHAPE;
  if (d->K < 128 || d->K > 16384 || d->K % 128) return MOE_ERR_SHAPE;
  if (d->I < 64 || d->I > 8192 || d->I % 64) return MOE_ERR_SHAPE;
  const int64_t R = (int64_t)d->M * d->topK;
  if (R >= (int64_t)1 << 24) return MOE_ERR_SHAPE;
  return MOE_OK;
}

// The shape preconditions and a valid weight layout.
inline int32_t check_dims(const moe_dims_t* d) {
  const int32_t rc = check_shape(d);
  if (rc != MOE_OK) return rc;
  if (d->weight_layout != MOE_WEIGHTS_ROWS && d->weight_layout != MOE_WEIGHTS_TILES) return MOE_ERR_SHAPE;
  return MOE_OK;
}

// The current device is an sm_103 GPU (its compute capability cached per device).
inline int32_t check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_ARCH;
  static int cached_dev = -2, cached_ok = 0;
  if (dev != cached_dev) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_ARCH;
    cached_ok = (major == 10 && minor == 3);
    cached_dev = dev;
  }
  return cached_ok ? MOE_OK : MOE_ERR_ARCH;
}

inline int32_t launch_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH; }

}  // namespace moe
