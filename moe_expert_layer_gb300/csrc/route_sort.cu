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
// a scan over (expert, block), and a stable scatter in which each warp ranks its
// routes with __match_any_sync and a per-warp count table.  Above one block's
// routes that is two launches: the histograms, then the scatter, each of whose
// blocks scans the histograms for its own offsets.  The order
// within an expert is the route order, so every output is unique (bit-exact).
// Bucket E collects routes with an expert id outside [0, E); they land after
// all valid routes with expandedRowIdx = -1.
#include "common.cuh"
#include "kernels.h"
#include "tensor_map.h"

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

// A block ranks up to kSortThreads * kMaxGroups routes [r0, r0 + n): warp w takes
// the consecutive range [r0 + w*rpw, r0 + (w+1)*rpw) (rpw a multiple of 32) and
// walks it 32 routes at a time, in order; __match_any_sync groups a step's routes by
// bucket, and the group's first lane advances the warp's own count of that bucket
// in `hist` (smem, [kSortWarps][pitch] uint16).  A route's rank among its range's
// routes of the same bucket is the count before its step plus the lanes below it
// in its group, so ranks follow route order (a stable sort) and no step needs a
// block-wide barrier.
constexpr int kMaxGroups = 8;

__device__ __forceinline__ void warp_rank(const int (&b)[kMaxGroups], int ng, uint16_t* hist_w,
                                          int (&rank)[kMaxGroups]) {
  const int lane = threadIdx.x & 31;
  const unsigned below = (1u << lane) - 1u;
#pragma unroll
  for (int g = 0; g < kMaxGroups; ++g) {
    if (g < ng) {  // warp-uniform
      const unsigned same = __match_any_sync(0xffffffffu, b[g]);
      const int leader = __ffs(same) - 1;
      int before = 0;
      if (lane == leader && b[g] >= 0) {
        before = hist_w[b[g]];
        hist_w[b[g]] = (uint16_t)(before + __popc(same));
      }
      before = __shfl_sync(0xffffffffu, before, leader);
      rank[g] = before + __popc(same & below);
      __syncwarp();  // the count is visible to the next step's leader
    }
  }
}

__device__ __forceinline__ int table_pitch(int E) { return ((E + 1) + 1) & ~1; }  // uint16 entries, even

// Shared memory of the sort kernels: two int arrays of 1024, 32 warp sums, the
// uint16 count table.
__host__ __device__ inline size_t sort_smem_bytes(int E) {
  return (1024 + 1024 + 32) * 4 + (size_t)kSortWarps * (size_t)(((E + 1) + 1) & ~1) * 2;
}

// Loads the buckets of this thread's routes (-1 past r1) and ranks them.
__device__ __forceinline__ void load_and_rank(const int32_t* expert_idx, int r0, int r1, int E, int rpw,
                                              uint16_t* hist, int pitch, int (&b)[kMaxGroups],
                                              int (&rank)[kMaxGroups]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = rpw / 32;
#pragma unroll
  for (int g = 0; g < kMaxGroups; ++g) {
    const int r = r0 + warp * rpw + g * 32 + lane;
    b[g] = (g < ng && r < r1) ? bucket_of(expert_idx, r, E) : -1;
  }
  uint32_t* h32 = reinterpret_cast<uint32_t*>(hist);
  for (int i = threadIdx.x; i < kSortWarps * pitch / 2; i += kSortThreads) h32[i] = 0u;
  __syncthreads();
  warp_rank(b, ng, hist + warp * pitch, rank);
  __syncthreads();
}

// Routes per warp range for n routes in one block: a multiple of 32.
__device__ __forceinline__ int range_per_warp(int n) { return ((n + kSortThreads - 1) / kSortThreads) * 32; }

// Single-block sort for small route counts (at most kSortThreads * kMaxGroups):
// ranking, histogram, scan and scatter in one launch.
__global__ void __launch_bounds__(kSortThreads) route_sort_single_kernel(
    const int32_t* __restrict__ expert_idx, int R, int E, int32_t* __restrict__ sorted_src_route,
    int32_t* __restrict__ expanded_row_idx, int32_t* __restrict__ tokens_per_expert,
    int32_t* __restrict__ cumsum) {
  extern __shared__ int smem_i[];
  int* warp_sums = smem_i + 2048;
  uint16_t* hist = reinterpret_cast<uint16_t*>(warp_sums + 32);
  const int pitch = table_pitch(E);
  const int rpw = range_per_warp(R);
  int b[kMaxGroups], rank[kMaxGroups];
  load_and_rank(expert_idx, 0, R, E, rpw, hist, pitch, b, rank);
  // bucket totals, their exclusive scan, and each warp's first row in every bucket
  const int j = threadIdx.x;
  int total = 0;
  if (j <= E)
    for (int w = 0; w < kSortWarps; ++w) total += hist[w * pitch + j];
  const int start = block_exclusive_scan(total, warp_sums);
  if (j < E) {
    tokens_per_expert[j] = total;
    cumsum[j] = start + total;
  }
  if (j <= E) {
    int run = start;  // <= R <= 8192: fits the table
    for (int w = 0; w < kSortWarps; ++w) {
      const int c = hist[w * pitch + j];
      hist[w * pitch + j] = (uint16_t)run;
      run += c;
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int g = 0; g < kMaxGroups; ++g) {
    if (b[g] >= 0) {
      const int r = warp * rpw + g * 32 + lane;
      const int pos = hist[warp * pitch + b[g]] + rank[g];
      sorted_src_route[pos] = r;
      expanded_row_idx[r] = (b[g] < E) ? pos : -1;
    }
  }
}

// Multi-block sort: `chunk` routes per block (at most kSortThreads * kMaxGroups).
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

// Every block scans the (bucket, block) histograms itself: bucket j's total over
// all blocks and its count in the blocks before this one, then the exclusive scan
// of the totals over buckets; block 0 also writes the counts and their prefix.
__global__ void __launch_bounds__(kSortThreads) route_scatter_kernel(
    const int32_t* __restrict__ expert_idx, int R, int E, int chunk, const int32_t* __restrict__ block_hist,
    int nb, int32_t* __restrict__ tokens_per_expert, int32_t* __restrict__ cumsum,
    int32_t* __restrict__ sorted_src_route, int32_t* __restrict__ expanded_row_idx) {
  extern __shared__ int smem_i[];
  int* base = smem_i;  // this block's first expanded row of each bucket
  int* warp_sums = smem_i + 2048;
  uint16_t* hist = reinterpret_cast<uint16_t*>(smem_i + 2048 + 32);
  const int pitch = table_pitch(E);
  const int r0 = blockIdx.x * chunk, r1 = min(R, r0 + chunk);
  {
    const int j = threadIdx.x;  // E + 1 <= kSortThreads buckets
    int total = 0, before = 0;
    if (j <= E)
      for (int b = 0; b < nb; ++b) {
        const int c = __ldg(block_hist + b * (E + 1) + j);
        total += c;
        before += b < (int)blockIdx.x ? c : 0;
      }
    const int start = block_exclusive_scan(total, warp_sums);
    if (j <= E) base[j] = start + before;
    if (blockIdx.x == 0 && j < E) {
      tokens_per_expert[j] = total;
      cumsum[j] = start + total;
    }
  }
  const int rpw = range_per_warp(chunk);
  int b[kMaxGroups], rank[kMaxGroups];
  load_and_rank(expert_idx, r0, r1, E, rpw, hist, pitch, b, rank);
  // each warp's offset within the block's routes of every bucket
  for (int j = threadIdx.x; j <= E; j += kSortThreads) {
    int run = 0;
    for (int w = 0; w < kSortWarps; ++w) {
      const int c = hist[w * pitch + j];
      hist[w * pitch + j] = (uint16_t)run;
      run += c;
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int g = 0; g < kMaxGroups; ++g) {
    if (b[g] >= 0) {
      const int r = r0 + warp * rpw + g * 32 + lane;
      const int pos = base[b[g]] + hist[warp * pitch + b[g]] + rank[g];
      sorted_src_route[pos] = r;
      expanded_row_idx[r] = (b[g] < E) ? pos : -1;
    }
  }
}

constexpr int kSingleBlockMaxRoutes = kSortThreads * kMaxGroups;

// Routes per block of the multi-block path: one pass of kSortThreads while that
// needs at most max_blocks blocks, more passes per block beyond (up to kMaxGroups),
// and more blocks only past max_blocks * kSingleBlockMaxRoutes routes.
int sort_chunk(int R, int max_blocks) {
  const int passes = (R + kSortThreads * max_blocks - 1) / (kSortThreads * max_blocks);
  return kSortThreads * (passes < 1 ? 1 : passes > kMaxGroups ? kMaxGroups : passes);
}

}  // namespace

size_t route_sort_workspace_bytes(int R, int E, int max_blocks) {
  if (R <= kSingleBlockMaxRoutes) return 0;
  const int chunk = sort_chunk(R, max_blocks);
  const size_t nb = (size_t)((R + chunk - 1) / chunk);
  return nb * (size_t)(E + 1) * sizeof(int32_t);  // the per-block histograms
}

cudaError_t launch_route_sort(const int32_t* expert_idx, int R, int E, int32_t* sorted_src_route,
                              int32_t* expanded_row_idx, int32_t* tokens_per_expert, int32_t* cumsum,
                              void* workspace, cudaStream_t stream, int max_blocks) {
  const size_t smem = sort_smem_bytes(E);  // 74 KB at E = 1023
  static PerContextOnce attr_set;
  const int dev = current_device();
  if (attr_set.needed(dev)) {
    const int most = (int)sort_smem_bytes(1023);
    cudaError_t e = cudaFuncSetAttribute(route_sort_single_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(route_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e != cudaSuccess) return e;
    attr_set.done(dev);
  }
  if (R <= kSingleBlockMaxRoutes) {
    route_sort_single_kernel<<<1, kSortThreads, smem, stream>>>(expert_idx, R, E, sorted_src_route,
                                                                expanded_row_idx, tokens_per_expert, cumsum);
    return cudaGetLastError();
  }
  const int chunk = sort_chunk(R, max_blocks);
  const int nb = (R + chunk - 1) / chunk;
  int32_t* block_hist = static_cast<int32_t*>(workspace);
  route_hist_kernel<<<nb, kSortThreads, (size_t)(E + 1) * 4, stream>>>(expert_idx, R, E, chunk, block_hist);
  route_scatter_kernel<<<nb, kSortThreads, smem, stream>>>(expert_idx, R, E, chunk, block_hist, nb,
                                                           tokens_per_expert, cumsum, sorted_src_route,
                                                           expanded_row_idx);
  return cudaGetLastError();
}

}  // namespace moe
