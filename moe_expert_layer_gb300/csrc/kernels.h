// Internal launch interface of the layer's kernels (host side).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// route_sort.cu
// The multi-block path (more than 8192 routes) uses max_blocks blocks of up to 8192
// routes each, more blocks only beyond max_blocks * 8192 routes; its scratch (two
// [blocks][E+1] int32 tables) grows with them.  Few blocks of several passes beat
// many one-pass blocks: the scan walks every block's table (R = 524288: 103 us with
// 512 blocks, 44 us with 64).
constexpr int kMaxSortBlocks = 64;
size_t route_sort_workspace_bytes(int R, int E, int max_blocks = kMaxSortBlocks);
cudaError_t launch_route_sort(const int32_t* expert_idx, int R, int E, int32_t* sorted_src_route,
                              int32_t* expanded_row_idx, int32_t* tokens_per_expert, int32_t* cumsum,
                              void* workspace, cudaStream_t stream, int max_blocks = kMaxSortBlocks);

// elementwise.cu
// Activation bounds (include/moe_layer.h): per expert, per 1024-deep segment
constexpr int kBoundSegment = 1024;
constexpr int kBoundSegments = 16;
cudaError_t launch_quant_tokens(const uint16_t* x, int M, int K, int8_t* xq_i8, uint16_t* xq_f16,
                                float* pts1, const int32_t* expanded_row_idx, int topK, uint16_t* a1,
                                const int32_t* expert_idx, int E, int32_t* bounds, cudaStream_t stream);
// FrontReorder in one call: the route sort and the quant-scatter.  Up to 4096 routes
// the sort runs inside the quant kernel (each token's CTA counts all routes itself);
// above, the route-sort kernels run first (sort_workspace: route_sort_workspace_bytes).
cudaError_t launch_front_reorder(const uint16_t* x, int M, int K, const int32_t* expert_idx, int topK, int E,
                                 int32_t* sorted_src_route, int32_t* expanded_row_idx, int32_t* tokens_per_expert,
                                 int32_t* cumsum, uint16_t* a1, float* pts1, int32_t* bounds, void* sort_workspace,
                                 cudaStream_t stream);
cudaError_t launch_swiglu_quant(const uint16_t* c1, int R, int I, int E, int topK, const float* pts1,
                                const int32_t* sorted_src_route, const int32_t* cumsum, int8_t* q2_i8,
                                uint16_t* q2_f16, float* pts2, const int32_t* expert_idx, int32_t* bounds,
                                cudaStream_t stream);
cudaError_t launch_combine_unpermute(const uint16_t* c2, const float* pts2, const int32_t* expanded_row_idx,
                                     const float* probs, int M, int K, int topK, uint16_t* out,
                                     cudaStream_t stream);

// Grouped W8A8 GEMM over expert-major rows (GMM1 and GMM2):
//   C[row][n] = sat_f16(float(sum_k act[row][k] * W[e][n][k]) * scale[e][n]),  n < N
struct GroupedGemmProblem {
  const uint16_t* act;              // [act_rows][Kd] binary16-coded int8 activations: expert-major
                                    // rows, or (gather_route set) token rows
  const int32_t* gather_route;      // null, or [R] route of each expert-major row: row d's
                                    // activations are act[gather_route[d] / topK] (TMA gather)
  int topK, act_rows;
  const int32_t* cumsum;            // [E] inclusive prefix of rows per expert
  const int8_t* w;                  // [E][N][Kd] rows, or (w_kb > 0) the tile layout
  int w_kb;                         // 0: rows; else 128-deep tiles per 128-channel block
  const float* scale;               // [E][N]
  uint16_t* C;                      // [R][N]
  int R, E, N, Kd;
  int32_t* status;                  // device status word
  int split_rows;                   // experts with <= split_rows rows run on the warp-MMA engine,
                                    // the others on the tcgen05 pairs (set by launch_grouped_gemm)
  int min_rows;                     // the warp-MMA engine skips experts of <= min_rows rows (0: none)
  const int32_t* bounds;            // [E][kBoundSegments] activation bounds, or null
  // GMM1 only, set by launch_gemm1_swiglu: SwiGLU + requant fused into the tcgen05 pairs
  const float* sw_pts1;             // [M] token scales (null: a plain GEMM)
  const int32_t* sw_sorted;         // [R] route of each expanded row
  uint16_t* sw_q2;                  // [R][N/2] binary16-coded codes
  float* sw_pts2;                   // [R]
  int32_t* sw_bounds;               // [E][kBoundSegments] or null
  int32_t* sw_done;                 // [E] int32, zero at launch
};
cudaError_t launch_grouped_gemm(const GroupedGemmProblem& p, cudaStream_t stream);     // picks an engine
bool grouped_gemm_reads_bounds(int R, int E);  // whether the engine it picks uses activation bounds
cudaError_t launch_grouped_gemm_hmma(const GroupedGemmProblem& p, int T, cudaStream_t stream);  // gemm_hmma.cu
cudaError_t launch_grouped_gemm_tc(const GroupedGemmProblem& p, cudaStream_t stream);  // gemm_tc.cu
// Whether every CTA pair of the tcgen05 kernel's grid can be resident at once on the
// current device (the fused SwiGLU's waits rely on it).
bool pair_grid_coresident();
// The largest I the tcgen05 pairs fuse SwiGLU for (the ABI's largest I).
constexpr int kFusedSwigluMaxI = 8192;
// GMM1 (g1: c1 written as usual) followed by SwiGLU + requant of its rows (q2 as
// binary16 codes, pts2, q2_bounds if not null), as launch_grouped_gemm then
// launch_swiglu_quant would compute them.  When the tcgen05 pairs run (more than 24
// rows per expert on average; the warp-MMA engine's share, if any, first), the
// operand is tiled and the pairs can all be resident, the SwiGLU runs inside the
// pairs' GMM1 kernel (sw_done: [E] int32 the caller has zeroed); otherwise GMM1 and
// the SwiGLU kernel run one after the other.  Returns in *fused which happened.
cudaError_t launch_gemm1_swiglu(const GroupedGemmProblem& g1, int I, int topK, const float* pts1,
                                const int32_t* sorted_src_route, const int32_t* expert_idx, uint16_t* q2,
                                float* pts2, int32_t* q2_bounds, int32_t* sw_done, cudaStream_t stream,
                                bool* fused = nullptr);

// weight_tiles.cu: the MOE_WEIGHTS_TILES layout (include/moe_layer.h) of a weight
// [E][N][D]: 16 KiB tiles of 128 channels x 128 reduction bytes, 128-byte swizzled,
// weight_tile_kb(D) tiles per 128-channel block (the depth zero-padded to 256).
constexpr int kWTileRows = 128, kWTileDepth = 128, kWTileBytes = kWTileRows * kWTileDepth;
inline int weight_tile_kb(int D) { return 2 * ((D + 255) / 256); }
inline size_t weight_tiles_bytes(int E, int N, int D) {
  return (size_t)E * (size_t)(N / kWTileRows) * (size_t)weight_tile_kb(D) * kWTileBytes;
}
cudaError_t launch_pack_weight_tiles(const int8_t* w, int E, int N, int D, int8_t* tiles, cudaStream_t stream);

}  // namespace moe
