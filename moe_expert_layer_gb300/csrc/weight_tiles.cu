// Weight tiles (MOE_WEIGHTS_TILES in include/moe_layer.h): a row-layout weight
// W[E][N][D] rewritten once as 16 KiB tiles of 128 channels x 128 reduction bytes,
// each tile contiguous and already in the 128-byte-swizzled order that a tensor copy
// of the same box leaves in shared memory, so the GEMMs move it with one untiled bulk
// copy; each weight v is stored as the byte v + 128.  The tiles stand in for the
// pre-packed weight of the PTO-ISA MegaMoE operator page (section "3. GMM1"), laid
// out offline for GB300's copy engine.
#include <cuda_runtime.h>

#include "kernels.h"

namespace moe {
namespace {

// One thread per 16-byte chunk of the tile buffer: chunk (tile, r, s) is tile row r's
// swizzled chunk s, which holds source chunk c = s ^ (r % 8) of that row.
__global__ void pack_weight_tiles_kernel(const int4* __restrict__ w, int N, int D, int KB, size_t n_chunks,
                                         int4* __restrict__ tiles) {
  const int NB = N / kWTileRows;
  const int d16 = D / 16;  // source row length in chunks
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_chunks; i += (size_t)gridDim.x * blockDim.x) {
    const size_t tile = i >> 10;
    const int within = (int)(i & 1023);
    const int r = within >> 3, s = within & 7;
    const int c = s ^ (r & 7);
    const int kb = (int)(tile % KB);
    const size_t eb = tile / KB;  // e * NB + nb
    const int nb = (int)(eb % NB);
    const size_t e = eb / NB;
    const int kc = kb * (kWTileDepth / 16) + c;  // source chunk along D
    int4 v = make_int4(0, 0, 0, 0);  // depth padding: the code of 0
    if (kc < d16) v = __ldg(w + ((e * N + (size_t)nb * kWTileRows + r) * (size_t)d16 + kc));
    // each byte v stored as v + 128 (the sign bit flipped), the form the GEMMs widen
    // to binary16 with one instruction less per four weights
    constexpr int kExcess = (int)0x80808080u;
    tiles[i] = make_int4(v.x ^ kExcess, v.y ^ kExcess, v.z ^ kExcess, v.w ^ kExcess);
  }
}

}  // namespace

cudaError_t launch_pack_weight_tiles(const int8_t* w, int E, int N, int D, int8_t* tiles, cudaStream_t stream) {
  const int KB = weight_tile_kb(D);
  const size_t n_chunks = weight_tiles_bytes(E, N, D) / 16;
  const int threads = 256;
  const size_t want = (n_chunks + threads - 1) / threads;
  const int blocks = (int)(want < (size_t)1 << 20 ? want : (size_t)1 << 20);
  pack_weight_tiles_kernel<<<blocks, threads, 0, stream>>>(reinterpret_cast<const int4*>(w), N, D, KB, n_chunks,
                                                           reinterpret_cast<int4*>(tiles));
  return cudaGetLastError();
}

}  // namespace moe
