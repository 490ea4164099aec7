// Host-side helpers shared by the GEMM engines: TMA descriptors and the SM count.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
inline PFN_encodeTiled tensor_map_encoder() {
  static PFN_encodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  }
  return fn;
}

// 2-D row-major tensor [outer][inner] of `elem`-byte elements, box {box_inner, box_outer},
// 128-byte swizzle, 256-byte L2 promotion, zero fill out of bounds.
inline bool encode_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, size_t elem, const void* base,
                                 uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  PFN_encodeTiled fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * elem};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device, once-only host state (kernel attributes, SM counts): devices 0..63.
constexpr int kMaxDevices = 64;
inline int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  return dev;
}

// Unique ID (cuCtxGetId) of the CUDA context current on this thread; 0 while the
// runtime has not yet made one current, or if the driver lacks the query.  Host
// state cached per device that belongs to a context -- kernel attributes, the
// address of a __device__ array -- is valid only in the context it was made in: a
// cudaDeviceReset, or a primary context released and created again, loads the
// module anew.  Such caches keep this ID beside what they hold and redo the set-up
// when it changes.
inline unsigned long long context_id() {
  typedef CUresult (*PFN_ctxGetCurrent)(CUcontext*);
  typedef CUresult (*PFN_ctxGetId)(CUcontext, unsigned long long*);
  static PFN_ctxGetCurrent get_current = nullptr;
  static PFN_ctxGetId get_id = nullptr;
  if (!get_current || !get_id) {
    void* p = nullptr;
    void* q = nullptr;
    cudaDriverEntryPointQueryResult r1, r2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r1) != cudaSuccess ||
        r1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) != cudaSuccess ||
        r2 != cudaDriverEntryPointSuccess)
      return 0;
    get_id = reinterpret_cast<PFN_ctxGetId>(q);
    get_current = reinterpret_cast<PFN_ctxGetCurrent>(p);
  }
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// A one-time set-up per device and context: needed(dev) is true until done(dev) has
// been called in the context current now (and again after that context is replaced).
struct PerContextOnce {
  unsigned long long ctx[kMaxDevices] = {};
  bool needed(int dev) const { return ctx[dev] == 0 || ctx[dev] != context_id(); }
  void done(int dev) { ctx[dev] = context_id(); }
};

inline int sm_count() {
  static int sms[kMaxDevices] = {};
  const int dev = current_device();
  if (!sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    sms[dev] = n;
  }
  return sms[dev];
}

}  // namespace moe
