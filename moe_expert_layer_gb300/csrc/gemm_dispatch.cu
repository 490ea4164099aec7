// Engine choice of the grouped W8A8 GEMM (PTO-ISA MegaMoE operator page, "3. GMM1"
// and "5. GMM2"): the warp-MMA engine (gemm_hmma.cu) for few rows per expert, the
// tcgen05 CTA pairs (gemm_tc.cu) for many, or both, split by expert on the device.
#include "kernels.h"

namespace moe {

// Engine choice.  A tcgen05.mma costs ~90 cycles for any N up to 128 (measured on
// GB300) and consumes 2 KB of int8 weights per SM in that time: with few rows per
// expert that caps weight streaming at about the HBM rate before any overhead.
// Warp-level HMMA (m16n8k16) consumes weights several times faster at N=8.  So
// batches with at most 24 rows per expert on average run entirely on the warp-MMA
// engine (GMM1 at K=7168, I=2048, E=256, 16 rows per expert: 1.64 ms with 16-row
// tiles against 2.92 ms on single-CTA tcgen05).  Larger batches split by expert
// on the device: experts with at most kSplitRows rows go to the warp-MMA engine
// (32-row tiles: one work item per expert and channel block), the others to the
// tcgen05 pairs; both kernels derive their share from cumsum, so the host never
// reads device counts (a kernel with no share exits at once).  Skewed routing
// (K=7168, I=2048, E=256, Zipf): GMM1 1.90 ms at 32 rows, 1.97 at 16.
constexpr int kSplitRows = 32;

// Above kPairsOnlyRows rows per expert on average (prefill-sized batches) the pairs
// take every expert, small ones as single short tiles (small MMA N): an expert of at most
// kSplitRows rows is then rare, while the warp-MMA kernel's launch, work-list set-up
// and exit (~4 us per GEMM at M = 8192, E = 64, measured) would be paid on every call.
constexpr double kPairsOnlyRows = 256.0;

// The warp-MMA engine alone (up to 24 rows per expert on average) keeps 512-deep
// chunks and reads no activation bounds.
bool grouped_gemm_reads_bounds(int R, int E) { return (double)R / (double)E > 24.0; }

// The warp-MMA engine's share of experts with more than lo and at most hi rows: 16-row
// tiles for the experts of up to 16 rows, 32-row tiles for the larger ones (one launch
// each).  An expert of 9-16 rows streams its weights once either way, and the 16-row
// tiles' kernel (a 16-row token box, four partial accumulators per fragment) runs its
// stages faster; an expert of 17-32 rows would stream them twice on 16-row tiles.
// Skewed routing (181 experts of <= 32 rows, 125 of them <= 16): GMM1 1609 -> 1591 us,
// GMM2 889 -> 880 us against 32-row tiles for all.
constexpr int kWarpTile16Rows = 16;
cudaError_t launch_warp_share(const GroupedGemmProblem& p, int lo, int hi, cudaStream_t stream) {
  GroupedGemmProblem q = p;
  if (lo < kWarpTile16Rows) {
    q.min_rows = lo;
    q.split_rows = min(hi, kWarpTile16Rows);
    cudaError_t e = launch_grouped_gemm_hmma(q, 16, stream);
    if (e != cudaSuccess || hi <= kWarpTile16Rows) return e;
  }
  q.min_rows = max(lo, kWarpTile16Rows);
  q.split_rows = hi;
  return launch_grouped_gemm_hmma(q, 32, stream);
}

cudaError_t launch_grouped_gemm(const GroupedGemmProblem& p, cudaStream_t stream) {
  GroupedGemmProblem q = p;
  const double mean_rows = (double)p.R / (double)p.E;
  if (!grouped_gemm_reads_bounds(p.R, p.E)) {
    // 16-row tiles up to 8 rows per expert on average (decode); 32-row tiles above,
    // so that an expert of up to 32 rows streams its weights through one work item
    // (splitting off the experts of up to 16 rows onto 16-row tiles, as below, measured
    // no gain at 16 rows per expert: GMM1 1297 -> 1296 us, GMM2 726 -> 733 us)
    q.split_rows = 0x7fffffff;
    return launch_grouped_gemm_hmma(q, mean_rows <= 8.0 ? 16 : 32, stream);
  }
  if (mean_rows >= kPairsOnlyRows) {
    q.split_rows = 0;
    return launch_grouped_gemm_tc(q, stream);
  }
  cudaError_t err = launch_warp_share(q, 0, kSplitRows, stream);
  if (err != cudaSuccess) return err;
  q.split_rows = kSplitRows;
  return launch_grouped_gemm_tc(q, stream);
}

cudaError_t launch_gemm1_swiglu(const GroupedGemmProblem& g1, int I, int topK, const float* pts1,
                                const int32_t* sorted_src_route, const int32_t* expert_idx, uint16_t* q2,
                                float* pts2, int32_t* q2_bounds, int32_t* sw_done, cudaStream_t stream, bool* fused) {
  const double mean_rows = (double)g1.R / (double)g1.E;
  const bool fuse = grouped_gemm_reads_bounds(g1.R, g1.E) && !g1.gather_route && I <= kFusedSwigluMaxI &&
                    pair_grid_coresident();
  if (fused) *fused = fuse;
  if (fuse) {
    GroupedGemmProblem q = g1;
    q.split_rows = 0;
    if (mean_rows < kPairsOnlyRows) {
      // the small experts' GMM1 first: their rows are complete when the pairs start
      q.split_rows = kSplitRows;
      cudaError_t e = launch_warp_share(q, 0, kSplitRows, stream);
      if (e != cudaSuccess) return e;
    }
    q.topK = topK;  // a row's token is its route / topK
    q.sw_pts1 = pts1;
    q.sw_sorted = sorted_src_route;
    q.sw_q2 = q2;
    q.sw_pts2 = pts2;
    q.sw_bounds = q2_bounds;
    q.sw_done = sw_done;
    return launch_grouped_gemm_tc(q, stream);
  }
  cudaError_t e = launch_grouped_gemm(g1, stream);
  if (e != cudaSuccess) return e;
  return launch_swiglu_quant(g1.C, g1.R, I, g1.E, topK, pts1, sorted_src_route, g1.cumsum, nullptr, q2, pts2,
                             expert_idx, q2_bounds, stream);
}

}  // namespace moe
