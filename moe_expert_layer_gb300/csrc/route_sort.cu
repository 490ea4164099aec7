// FrontReorder on one rank: stable counting sort of the routes by expert id.
//
// PTO-ISA MegaMoE operator page, section "1. FrontReorder": phase 1 sorts
// (expertId[route], route) expert-major into sortedSrcRoute[dstRow], phase 2a
// counts routes per expert, phase 2b inverts the permutation into
// expandedRowIdx[srcRoute] = dstRow, phase 4 prefix-sums the counts (with one
// source rank cumsumMM collapses to the inclusive prefix over experts).
//
// The page's NPU merge sort (TSORT32 + TMRGSORT) is replaced by a counting sort,
// which is the natural GPU form for small integer keys: a per-block histogram,
// one scan over (expert, block), and a stable scatter in which each warp ranks
// its routes with __match_any_sync and a per-warp count table.  The order
// within an expert is the route order, so every output is unique (bit-exact).
// Bucket E collects routes with an expert id outside [0, E); they land after
// all valid routes with expandedRowIdx = -1.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kSortThreads = 1024;
constexpr int kSortWarps = kSortThreads / 32;

__device__ __forceinline__ int bucket_of(const int32_t* expert_idx, int r, int E) {
  const int e = __ldg(expert_idx + r);
  return (e >= 0 && e < E) ? e : E;
}

// Exclusive scan of one int per thread over a 1024-thread block.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    warp_sums[lane] = wi - w;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  __syncthreads();
  return r;
}

// Stable scatter of routes [r0, r1) given the first free expanded row of each
// bucket in `running` (smem, E+1 entries, advanced in place).
// `cnt` is a [kSortWarps][pitch] byte table in smem.
__device__ void scatter_chunk(const int32_t* expert_idx, int r0, int r1, int E, int* running,
                              uint8_t* cnt, int pitch, int32_t* sorted_src_route,
                              int32_t* expanded_row_idx) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  uint32_t* cnt32 = reinterpret_cast<uint32_t*>(cnt);
  const int table_words = kSortWarps * pitch / 4;
  for (int base = r0; base < r1; base += kSortThreads) {
    const int r = base + threadIdx.x;
    const bool live = r < r1;
    const int b = live ? bucket_of(expert_idx, r, E) : -1;
    for (int i = threadIdx.x; i < table_words; i += kSortThreads) cnt32[i] = 0u;
    __syncthreads();
    const unsigned same = __match_any_sync(0xffffffffu, b);
    const int rank_in_warp = __popc(same & lt_mask);
    if (live && rank_in_warp == 0) cnt[warp * pitch + b] = (uint8_t)__popc(same);
    __syncthreads();
    if (live) {
      int pos = running[b] + rank_in_warp;
      for (int w = 0; w < warp; ++w) pos += cnt[w * pitch + b];
      sorted_src_route[pos] = r;
      expanded_row_idx[r] = (b < E) ? pos : -1;
    }
    __syncthreads();
    for (int j = threadIdx.x; j <= E; j += kSortThreads) {
      int add = 0;
      for (int w = 0; w < kSortWarps; ++w) add += cnt[w * pitch + j];
      running[j] += add;
    }
    __syncthreads();
  }
}

__device__ __forceinline__ int table_pitch(int E) { return ((E + 1) + 3) & ~3; }

// Single-block sort for small route counts: histogram, scan and scatter in one launch.
__global__ void __launch_bounds__(kSortThreads) route_sort_single_kernel(
    const int32_t* __restrict__ expert_idx, int R, int E, int32_t* __restrict__ sorted_src_route,
    int32_t* __restrict__ expanded_row_idx, int32_t* __restrict__ tokens_per_expert,
    int32_t* __restrict__ cumsum) {
  extern __shared__ int smem_i[];
  int* hist = smem_i;                      // E+1
  int* warp_sums = hist + 1024;            // 32
  uint8_t* cnt = reinterpret_cast<uint8_t*>(warp_sums + 32);
  const int pitch = table_pitch(E);
  for (int j = threadIdx.x; j < 1024; j += kSortThreads) hist[j] = 0;
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += kSortThreads) atomicAdd(&hist[bucket_of(expert_idx, r, E)], 1);
  __syncthreads();
  const int j = threadIdx.x;
  const int total = (j <= E) ? hist[j] : 0;
  const int start = block_exclusive_scan(total, warp_sums);
  if (j < E) {
    tokens_per_expert[j] = total;
    cumsum[j] = start + total;
  }
  // hist becomes the running insertion point of each bucket
  if (j <= E) hist[j] = start;
  __syncthreads();
  scatter_chunk(expert_idx, 0, R, E, hist, cnt, pitch, sorted_src_route, expanded_row_idx);
}

__global__ void __launch_bounds__(kSortThreads) route_hist_kernel(const int32_t* __restrict__ expert_idx,
                                                                  int R, int E, int chunk,
                                                                  int32_t* __restrict__ block_hist) {
  extern __shared__ int smem_i[];
  int* hist = smem_i;
  for (int j = threadIdx.x; j <= E; j += kSortThreads) hist[j] = 0;
  __syncthreads();
  const int r0 = blockIdx.x * chunk, r1 = min(R, r0 + chunk);
  for (int r = r0 + threadIdx.x; r < r1; r += kSortThreads) atomicAdd(&hist[bucket_of(expert_idx, r, E)], 1);
  __syncthreads();
  for (int j = threadIdx.x; j <= E; j += kSortThreads) block_hist[blockIdx.x * (E + 1) + j] = hist[j];
}

__global__ void __launch_bounds__(kSortThreads) route_scan_kernel(const int32_t* __restrict__ block_hist,
                                                                  int nb, int E,
                                                                  int32_t* __restrict__ tokens_per_expert,
                                                                  int32_t* __restrict__ cumsum,
                                                                  int32_t* __restrict__ block_off) {
  __shared__ int warp_sums[32];
  const int j = threadIdx.x;
  int total = 0;
  if (j <= E)
    for (int b = 0; b < nb; ++b) total += block_hist[b * (E + 1) + j];
  const int start = block_exclusive_scan(total, warp_sums);
  if (j < E) {
    tokens_per_expert[j] = total;
    cumsum[j] = start + total;
  }
  if (j <= E) {
    int run = start;
    for (int b = 0; b < nb; ++b) {
      block_off[b * (E + 1) + j] = run;
      run += block_hist[b * (E + 1) + j];
    }
  }
}

__global__ void __launch_bounds__(kSortThreads) route_scatter_kernel(
    const int32_t* __restrict__ expert_idx, int R, int E, int chunk, const int32_t* __restrict__ block_off,
    int32_t* __restrict__ sorted_src_route, int32_t* __restrict__ expanded_row_idx) {
  extern __shared__ int smem_i[];
  int* running = smem_i;  // E+1 (padded to 1024)
  uint8_t* cnt = reinterpret_cast<uint8_t*>(running + 1024);
  for (int j = threadIdx.x; j <= E; j += kSortThreads) running[j] = block_off[blockIdx.x * (E + 1) + j];
  __syncthreads();
  const int r0 = blockIdx.x * chunk, r1 = min(R, r0 + chunk);
  scatter_chunk(expert_idx, r0, r1, E, running, cnt, table_pitch(E), sorted_src_route, expanded_row_idx);
}

constexpr int kSingleBlockMaxRoutes = 8192;
constexpr int kMultiBlockChunk = 8192;

size_t smem_single(int E) { return 1024 * 4 + 32 * 4 + (size_t)kSortWarps * (((E + 1) + 3) & ~3); }
size_t smem_scatter(int E) { return 1024 * 4 + (size_t)kSortWarps * (((E + 1) + 3) & ~3); }

}  // namespace

size_t route_sort_workspace_bytes(int R, int E) {
  if (R <= kSingleBlockMaxRoutes) return 0;
  const size_t nb = (size_t)((R + kMultiBlockChunk - 1) / kMultiBlockChunk);
  return 2 * nb * (size_t)(E + 1) * sizeof(int32_t);
}

cudaError_t launch_route_sort(const int32_t* expert_idx, int R, int E, int32_t* sorted_src_route,
                              int32_t* expanded_row_idx, int32_t* tokens_per_expert, int32_t* cumsum,
                              void* workspace, cudaStream_t stream) {
  if (R <= kSingleBlockMaxRoutes) {
    route_sort_single_kernel<<<1, kSortThreads, smem_single(E), stream>>>(
        expert_idx, R, E, sorted_src_route, expanded_row_idx, tokens_per_expert, cumsum);
    return cudaGetLastError();
  }
  const int nb = (R + kMultiBlockChunk - 1) / kMultiBlockChunk;
  int32_t* block_hist = static_cast<int32_t*>(workspace);
  int32_t* block_off = block_hist + (size_t)nb * (E + 1);
  route_hist_kernel<<<nb, kSortThreads, (size_t)(E + 1) * 4, stream>>>(expert_idx, R, E, kMultiBlockChunk,
                                                                       block_hist);
  route_scan_kernel<<<1, kSortThreads, 0, stream>>>(block_hist, nb, E, tokens_per_expert, cumsum, block_off);
  route_scatter_kernel<<<nb, kSortThreads, smem_scatter(E), stream>>>(expert_idx, R, E, kMultiBlockChunk,
                                                                      block_off, sorted_src_route,
                                                                      expanded_row_idx);
  return cudaGetLastError();
}

}  // namespace moe
