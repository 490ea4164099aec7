// The layer's row-wise, HBM-bound stages:
//   token quant (+ scatter of each token's codes to its expert-major rows)
//                      (PTO-ISA MegaMoE operator page, "1. FrontReorder", phase 2c)
//   SwiGLU + requant   (same page, "4. SwiGLU")
//   Combine+Unpermute  (same page, "6. Combine" and "7. Unpermute"), fused
// Rows are read with 16-byte vector loads kept in registers, so each input byte
// is read from HBM once; row maxima are warp-shuffle + shared-memory reductions.
// Arithmetic uses explicitly rounded fp32 intrinsics (no contraction), matching
// the rounding points the page defines.
#include "common.cuh"
#include "kernels.h"
#include "swiglu.cuh"

namespace moe {

namespace {

union Vec8h {
  int4 v;
  __half2 h2[4];
  __half h[8];
  uint32_t u[4];
};

constexpr int kRowThreads = 256;

// Integer-valued conversions without the conversion pipe (~16 per cycle per SM),
// all exact for the ranges used here:
//   rint_small(v):  round-half-even of |v| < 2^22, read off the mantissa of v + 1.5*2^23
//   codes_to_half2: two integers in [-127, 127] -> their binary16 pair, by placing
//                   q+128 in the mantissa of 1024 and subtracting 1152 (sub.f16x2)
__device__ __forceinline__ int rint_small(float v) {
  return __float_as_int(__fadd_rn(v, 12582912.0f)) - 0x4B400000;
}
// Adds a vector's sum of |code| to its 1024-deep segment's shared total.  The
// active lanes of a warp hold consecutive vectors starting at a multiple of 32,
// which never straddle a segment (128 vectors), so one atomic per warp suffices.
__device__ __forceinline__ void add_segment_l1(int* s_l1, int idx, int l1) {
  const unsigned mask = __activemask();
  const int sum = __reduce_add_sync(mask, l1);
  if ((int)(threadIdx.x & 31) == __ffs(mask) - 1) atomicAdd(&s_l1[(idx * 8) / kBoundSegment], sum);
}

__device__ __forceinline__ uint32_t codes_to_half2(int q0, int q1) {
  const uint32_t w = (uint32_t)(0x6400 + q0 + 128) | ((uint32_t)(0x6400 + q1 + 128) << 16);
  uint32_t r;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(0x64806480u));
  return r;
}

// --------------------------------------------------------------------------
// per-token dynamic quant: pts1 = amax / 127, q = round_half_away(x / pts1)
// --------------------------------------------------------------------------
// With `expanded_row_idx` set, the codes of token t are also written (as binary16)
// to row expanded_row_idx[t*topK + j] of `a1` for every valid route j: the
// expert-major GMM1 operand (FrontReorder's quant-scatter into offsetA).
// With `bounds` set, the token's sum of |code| over each 1024-deep segment of k is
// folded (atomic max) into bounds[e][segment] of every expert e it is routed to.
//
// SORT (the fused FrontReorder, R <= kFusedSortRoutes): the kernel also sorts the
// routes, without a kernel of its own.  Every CTA reads all R expert ids, counts the
// routes of each bucket (bucket E: invalid ids) and those that come before its own
// token's routes, and scans the counts: a route's expanded row is its bucket's start
// plus the number of earlier routes in the bucket (the stable order the sort
// defines).  Each CTA writes sorted_src_route and expanded_row_idx for its own
// routes; CTA 0 writes tokens_per_expert and cumsum.
constexpr int kFusedSortRoutes = 4096;

// Exclusive scan over the block of one value per thread (blockDim a multiple of 32).
__device__ __forceinline__ int block_scan_excl(int v, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < nw) warp_sums[lane] = wi - w;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  __syncthreads();
  return r;
}

template <int VPT, bool SORT>
__global__ void __launch_bounds__(kRowThreads) quant_tokens_kernel(const __half* __restrict__ x, int K,
                                                                   int8_t* __restrict__ xq_i8,
                                                                   __half* __restrict__ xq_f16,
                                                                   float* __restrict__ pts1,
                                                                   const int32_t* __restrict__ expanded_row_idx,
                                                                   int topK, __half* __restrict__ a1,
                                                                   const int32_t* __restrict__ expert_idx, int E,
                                                                   int32_t* __restrict__ bounds, int R,
                                                                   int32_t* __restrict__ sorted_src_route,
                                                                   int32_t* __restrict__ expanded_out,
                                                                   int32_t* __restrict__ tokens_per_expert,
                                                                   int32_t* __restrict__ cumsum) {
  __shared__ float red[kRowThreads / 32];
  __shared__ int s_l1[kBoundSegments];
  __shared__ int s_pos[SORT ? 1024 : 1];  // expanded row of each of the token's routes (-1: invalid)
  if (threadIdx.x < kBoundSegments) s_l1[threadIdx.x] = 0;  // visible after the row-max barriers
  const int t = blockIdx.x;
  const int nvec = K >> 3;
  const int4* row = reinterpret_cast<const int4*>(x + (size_t)t * K);
  Vec8h v[VPT];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = threadIdx.x + i * (int)blockDim.x;
    if (idx < nvec) {
      v[i].v = __ldg(row + idx);
      if constexpr (!SORT) {
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(__half2float(v[i].h[j])));
      }
    }
  }
  if constexpr (SORT) {
    // the row loads above are in flight while the routes are counted
    __shared__ int s_after[1024], s_before[1024], s_ws[32];
    const int nb = E + 1;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
      s_after[b] = 0;
      s_before[b] = 0;
    }
    __syncthreads();
    // each route counted once, in its bucket's count before or from this token's
    // routes; the ids come in 16-byte loads, several per thread in flight at once
    const int first = t * topK;
    auto count = [&](int r, int e) {
      const int b = (e >= 0 && e < E) ? e : E;
      atomicAdd(r < first ? &s_before[b] : &s_after[b], 1);
    };
    const int nq = R >> 2;  // whole groups of four routes
    const int4* ids4 = reinterpret_cast<const int4*>(expert_idx);
    constexpr int kBatch = 4;
    for (int q0 = threadIdx.x; q0 < nq; q0 += kBatch * (int)blockDim.x) {
      int4 v4[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int q = q0 + u * (int)blockDim.x;
        if (q < nq) v4[u] = __ldg(ids4 + q);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int q = q0 + u * (int)blockDim.x;
        if (q < nq) {
          count(4 * q, v4[u].x);
          count(4 * q + 1, v4[u].y);
          count(4 * q + 2, v4[u].z);
          count(4 * q + 3, v4[u].w);
        }
      }
    }
    for (int r = 4 * nq + threadIdx.x; r < R; r += blockDim.x) count(r, __ldg(expert_idx + r));
    __syncthreads();
    // exclusive scan of the bucket counts: thread i owns buckets [i*per, i*per + per)
    const int per = (nb + blockDim.x - 1) / blockDim.x;
    const int b0 = threadIdx.x * per, b1 = min(nb, b0 + per);
    int local = 0;
    for (int b = b0; b < b1; ++b) local += s_before[b] + s_after[b];
    int run = block_scan_excl(local, s_ws);
    for (int b = b0; b < b1; ++b) {
      const int c = s_before[b] + s_after[b];
      if (t == 0 && b < E) {
        tokens_per_expert[b] = c;
        cumsum[b] = run + c;
      }
      s_before[b] += run;  // first expanded row of this token's routes in bucket b
      run += c;
    }
    __syncthreads();
    for (int sl = threadIdx.x; sl < topK; sl += blockDim.x) {
      const int r = first + sl;
      const int e = __ldg(expert_idx + r);
      const int b = (e >= 0 && e < E) ? e : E;
      int pos = s_before[b];
      for (int s2 = 0; s2 < sl; ++s2) {  // this token's earlier routes in the same bucket
        const int e2 = __ldg(expert_idx + first + s2);
        pos += ((e2 >= 0 && e2 < E) ? e2 : E) == b ? 1 : 0;
      }
      sorted_src_route[pos] = r;
      const int d = b < E ? pos : -1;
      expanded_out[r] = d;
      s_pos[sl] = d;
    }
    __syncthreads();
  }
  if constexpr (SORT) {  // the row max once the routes are placed (the loads had that time to land)
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int idx = threadIdx.x + i * (int)blockDim.x;
      if (idx < nvec) {
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(__half2float(v[i].h[j])));
      }
    }
  }
  amax = block_max_nonneg(amax, red);
  const float scale = __fdiv_rn(amax, 127.0f);
  if (threadIdx.x == 0) pts1[t] = scale;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = threadIdx.x + i * (int)blockDim.x;
    if (idx < nvec) {
      int q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        q[j] = (amax > 0.0f) ? clamp127(rint_small(roundf(__fdiv_rn(__half2float(v[i].h[j]), scale)))) : 0;
      if (bounds) {
        int l1 = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) l1 += abs(q[j]);
        add_segment_l1(s_l1, idx, l1);
      }
      if (xq_i8) {
        uint2 packed;
        packed.x = (uint32_t)(q[0] & 0xff) | ((uint32_t)(q[1] & 0xff) << 8) | ((uint32_t)(q[2] & 0xff) << 16) |
                   ((uint32_t)(q[3] & 0xff) << 24);
        packed.y = (uint32_t)(q[4] & 0xff) | ((uint32_t)(q[5] & 0xff) << 8) | ((uint32_t)(q[6] & 0xff) << 16) |
                   ((uint32_t)(q[7] & 0xff) << 24);
        reinterpret_cast<uint2*>(xq_i8 + (size_t)t * K)[idx] = packed;
      }
      if (SORT || xq_f16 || expanded_row_idx) {
        int4 o;
        o.x = (int)codes_to_half2(q[0], q[1]);
        o.y = (int)codes_to_half2(q[2], q[3]);
        o.z = (int)codes_to_half2(q[4], q[5]);
        o.w = (int)codes_to_half2(q[6], q[7]);
        if (xq_f16) reinterpret_cast<int4*>(xq_f16 + (size_t)t * K)[idx] = o;
        if (SORT) {
          for (int s = 0; s < topK; ++s) {
            const int d = s_pos[s];
            if (d >= 0) reinterpret_cast<int4*>(a1 + (size_t)d * K)[idx] = o;
          }
        } else if (expanded_row_idx) {
          for (int s = 0; s < topK; ++s) {
            const int d = __ldg(expanded_row_idx + (size_t)t * topK + s);
            if (d >= 0) reinterpret_cast<int4*>(a1 + (size_t)d * K)[idx] = o;
          }
        }
      }
    }
  }
  if (bounds) {
    __syncthreads();
    const int nseg = (K + kBoundSegment - 1) / kBoundSegment;
    if (threadIdx.x < nseg) {
      for (int s = 0; s < topK; ++s) {
        const int e = __ldg(expert_idx + (size_t)t * topK + s);
        if (e >= 0 && e < E) atomicMax(bounds + (size_t)e * kBoundSegments + threadIdx.x, s_l1[threadIdx.x]);
      }
    }
  }
}

// --------------------------------------------------------------------------
// SwiGLU + requant over expanded rows d < cumsum[E-1]
// --------------------------------------------------------------------------
// With `bounds` set, the row's sum of |code| over each 1024-deep segment of I is
// folded (atomic max) into bounds[e][segment] of the row's expert e.
template <int VPT>
__global__ void __launch_bounds__(kRowThreads) swiglu_quant_kernel(
    const __half* __restrict__ c1, int I, int E, int topK, const float* __restrict__ pts1,
    const int32_t* __restrict__ sorted_src_route, const int32_t* __restrict__ cumsum,
    int8_t* __restrict__ q2_i8, __half* __restrict__ q2_f16, float* __restrict__ pts2,
    const int32_t* __restrict__ expert_idx, int32_t* __restrict__ bounds) {
  __shared__ float red[kRowThreads / 32];
  __shared__ int s_l1[kBoundSegments];
  const int d = blockIdx.x;
  const int nvec = I >> 3;
  const int4* gate = reinterpret_cast<const int4*>(c1 + (size_t)d * 2 * I);
  const int4* up = gate + nvec;
  // the row's loads go out before the validity check and the token-scale load, so the
  // CTA waits on one memory latency instead of three in a row (rows past the valid
  // ones exist, R in all, and their values are dropped)
  const int valid = __ldg(cumsum + E - 1);
  const int src = __ldg(sorted_src_route + d);
  Vec8h gv[VPT], uv[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = threadIdx.x + i * (int)blockDim.x;
    if (idx < nvec) {
      gv[i].v = __ldg(gate + idx);
      uv[i].v = __ldg(up + idx);
    }
  }
  if (d >= valid) return;
  if (threadIdx.x < kBoundSegments) s_l1[threadIdx.x] = 0;  // visible after the row-max barriers
  const float p1 = __ldg(pts1 + src / topK);
  const int e_row = bounds ? __ldg(expert_idx + src) : -1;
  float y[VPT][8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = threadIdx.x + i * (int)blockDim.x;
    if (idx < nvec) {
      const Vec8h& g = gv[i];
      const Vec8h& u = uv[i];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        y[i][j] = swiglu_y(g.h[j], u.h[j], p1);  // swiglu.cuh: fast exp, token scale on the gate only
        amax = fmaxf(amax, fabsf(y[i][j]));
      }
    }
  }
  amax = block_max_nonneg(amax, red);
  const float inv = swiglu_inv(amax);
  if (threadIdx.x == 0) pts2[d] = swiglu_pts2(amax, p1);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = threadIdx.x + i * (int)blockDim.x;
    if (idx < nvec) {
      // the codes as binary16 and their sum of |q| (swiglu.cuh); r keeps the code
      // floats, whose low bytes are the int8 codes with the top bit flipped
      float r[8];
      int l1 = 0;
      Vec8h hc;
      hc.v = swiglu_codes8(y[i], inv, bounds ? &l1 : nullptr, r);
      if (bounds) add_segment_l1(s_l1, idx, l1);
      if (q2_i8) {
        // the low bytes 0x80 + q, top bits flipped back: q's two's-complement bytes
        uint2 packed;
        packed.x = __byte_perm(__byte_perm(__float_as_uint(r[0]), __float_as_uint(r[1]), 0x0040),
                               __byte_perm(__float_as_uint(r[2]), __float_as_uint(r[3]), 0x0040), 0x5410) ^
                   0x80808080u;
        packed.y = __byte_perm(__byte_perm(__float_as_uint(r[4]), __float_as_uint(r[5]), 0x0040),
                               __byte_perm(__float_as_uint(r[6]), __float_as_uint(r[7]), 0x0040), 0x5410) ^
                   0x80808080u;
        reinterpret_cast<uint2*>(q2_i8 + (size_t)d * I)[idx] = packed;
      }
      if (q2_f16) reinterpret_cast<int4*>(q2_f16 + (size_t)d * I)[idx] = hc.v;
    }
  }
  if (bounds) {
    __syncthreads();
    const int nseg = (I + kBoundSegment - 1) / kBoundSegment;
    const int e = e_row;
    if (threadIdx.x < nseg && e >= 0 && e < E)
      atomicMax(bounds + (size_t)e * kBoundSegments + threadIdx.x, s_l1[threadIdx.x]);
  }
}

// --------------------------------------------------------------------------
// Combine (D = sat_f16(C2 * pts2)) fused with Unpermute (prob-weighted sum of
// the token's topK rows, fp32 accumulator, slot order, multiply then add).
// grid = (M, ceil(K / (8 * 128))); each thread owns 8 consecutive columns.
// --------------------------------------------------------------------------
constexpr int kCombineThreads = 128;

// The same for a compile-time topK (the common 1..8): every slot's loads are issued
// before any is used (invalid routes load row 0 and are skipped), so a thread keeps
// topK 16-byte row loads in flight instead of one.
template <int TK>
__global__ void __launch_bounds__(kCombineThreads) combine_unpermute_tk_kernel(
    const __half* __restrict__ c2, const float* __restrict__ pts2, const int32_t* __restrict__ expanded_row_idx,
    const float* __restrict__ probs, int K, __half* __restrict__ out) {
  const int t = blockIdx.x;
  const int vec = blockIdx.y * kCombineThreads + threadIdx.x;
  if (vec * 8 >= K) return;
  int d[TK];
  float p[TK], sc[TK];
  Vec8h c[TK];
#pragma unroll
  for (int u = 0; u < TK; ++u) d[u] = __ldg(expanded_row_idx + (size_t)t * TK + u);
#pragma unroll
  for (int u = 0; u < TK; ++u) {
    const int row = d[u] < 0 ? 0 : d[u];
    p[u] = __ldg(probs + (size_t)t * TK + u);
    sc[u] = __ldg(pts2 + row);
    c[u].v = __ldg(reinterpret_cast<const int4*>(c2 + (size_t)row * K) + vec);
  }
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
#pragma unroll
  for (int u = 0; u < TK; ++u) {
    if (d[u] < 0) continue;
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      // D = sat_f16(C2 * pts2), two at a time
      const __half2 dh = f2h2_sat(__fmul_rn(__half2float(c[u].h[j]), sc[u]),
                                  __fmul_rn(__half2float(c[u].h[j + 1]), sc[u]));
      acc[j] = __fadd_rn(acc[j], __fmul_rn(__low2float(dh), p[u]));
      acc[j + 1] = __fadd_rn(acc[j + 1], __fmul_rn(__high2float(dh), p[u]));
    }
  }
  Vec8h o;
#pragma unroll
  for (int j = 0; j < 4; ++j) o.h2[j] = f2h2_sat(acc[2 * j], acc[2 * j + 1]);
  reinterpret_cast<int4*>(out + (size_t)t * K)[vec] = o.v;
}

__global__ void __launch_bounds__(kCombineThreads) combine_unpermute_kernel(
    const __half* __restrict__ c2, const float* __restrict__ pts2, const int32_t* __restrict__ expanded_row_idx,
    const float* __restrict__ probs, int K, int topK, __half* __restrict__ out) {
  const int t = blockIdx.x;
  const int vec = blockIdx.y * kCombineThreads + threadIdx.x;
  if (vec * 8 >= K) return;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
  for (int s = 0; s < topK; ++s) {
    const int d = __ldg(expanded_row_idx + (size_t)t * topK + s);
    if (d < 0) continue;
    const float p = __ldg(probs + (size_t)t * topK + s);
    const float sc = __ldg(pts2 + d);
    Vec8h c;
    c.v = __ldg(reinterpret_cast<const int4*>(c2 + (size_t)d * K) + vec);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float dv = __half2float(f2h_sat(__fmul_rn(__half2float(c.h[j]), sc)));
      acc[j] = __fadd_rn(acc[j], __fmul_rn(dv, p));
    }
  }
  Vec8h o;
#pragma unroll
  for (int j = 0; j < 8; ++j) o.h[j] = f2h_sat(acc[j]);
  reinterpret_cast<int4*>(out + (size_t)t * K)[vec] = o.v;
}

// Threads for a row of nvec 16-byte vectors handled vpt per thread: whole warps,
// no more than the row needs (a 1408-wide SwiGLU row runs on 192 threads, not 256).
int row_threads(int nvec, int vpt) {
  const int t = (nvec + vpt - 1) / vpt;
  return (t + 31) / 32 * 32;
}

}  // namespace

namespace {

// One CTA per token, a 16-byte vector per thread and VPT vectors per thread at most.
template <bool SORT>
cudaError_t launch_quant(const uint16_t* x, int M, int K, int8_t* xq_i8, uint16_t* xq_f16, float* pts1,
                         const int32_t* expanded_row_idx, int topK, uint16_t* a1, const int32_t* expert_idx, int E,
                         int32_t* bounds, int32_t* sorted_src_route, int32_t* expanded_out,
                         int32_t* tokens_per_expert, int32_t* cumsum, cudaStream_t stream) {
  const int nvec = K / 8;
  const int vpt = (nvec + kRowThreads - 1) / kRowThreads;
  const int threads = row_threads(nvec, vpt);
  const __half* xh = reinterpret_cast<const __half*>(x);
  __half* qf = reinterpret_cast<__half*>(xq_f16);
  __half* ah = reinterpret_cast<__half*>(a1);
  const int R = M * topK;
#define MOE_QUANT(V)                                                                                            \
  quant_tokens_kernel<V, SORT><<<M, threads, 0, stream>>>(xh, K, xq_i8, qf, pts1, expanded_row_idx, topK, ah,  \
                                                          expert_idx, E, bounds, R, sorted_src_route,          \
                                                          expanded_out, tokens_per_expert, cumsum)
  if (vpt <= 1)
    MOE_QUANT(1);
  else if (vpt <= 2)
    MOE_QUANT(2);
  else if (vpt <= 4)
    MOE_QUANT(4);
  else if (vpt <= 8)
    MOE_QUANT(8);
  else
    return cudaErrorInvalidValue;
#undef MOE_QUANT
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_tokens(const uint16_t* x, int M, int K, int8_t* xq_i8, uint16_t* xq_f16, float* pts1,
                                const int32_t* expanded_row_idx, int topK, uint16_t* a1, const int32_t* expert_idx,
                                int E, int32_t* bounds, cudaStream_t stream) {
  return launch_quant<false>(x, M, K, xq_i8, xq_f16, pts1, expanded_row_idx, topK, a1, expert_idx, E, bounds,
                             nullptr, nullptr, nullptr, nullptr, stream);
}

cudaError_t launch_front_reorder(const uint16_t* x, int M, int K, const int32_t* expert_idx, int topK, int E,
                                 int32_t* sorted_src_route, int32_t* expanded_row_idx, int32_t* tokens_per_expert,
                                 int32_t* cumsum, uint16_t* a1, float* pts1, int32_t* bounds, void* sort_workspace,
                                 cudaStream_t stream) {
  const int R = M * topK;
  if (R <= kFusedSortRoutes)
    return launch_quant<true>(x, M, K, nullptr, nullptr, pts1, nullptr, topK, a1, expert_idx, E, bounds,
                              sorted_src_route, expanded_row_idx, tokens_per_expert, cumsum, stream);
  cudaError_t e = launch_route_sort(expert_idx, R, E, sorted_src_route, expanded_row_idx, tokens_per_expert, cumsum,
                                    sort_workspace, stream);
  if (e != cudaSuccess) return e;
  return launch_quant<false>(x, M, K, nullptr, nullptr, pts1, expanded_row_idx, topK, a1, expert_idx, E, bounds,
                             nullptr, nullptr, nullptr, nullptr, stream);
}

cudaError_t launch_swiglu_quant(const uint16_t* c1, int R, int I, int E, int topK, const float* pts1,
                                const int32_t* sorted_src_route, const int32_t* cumsum, int8_t* q2_i8,
                                uint16_t* q2_f16, float* pts2, const int32_t* expert_idx, int32_t* bounds,
                                cudaStream_t stream) {
  // Each row's CTA lives through a chain of dependent loads (route, token scale),
  // a block-wide max and the stores, so throughput comes from rows in flight: short
  // rows per thread-block (64 threads, up to 4 vectors each) once there are rows
  // enough to fill the GPU (I = 1408: 97 us instead of 115 at 49152 rows), 128
  // threads below 8192 rows (1024 rows: 64-thread blocks were 24% slower; 4096 rows
  // of I = 2048: 17.3 us with 128 threads, 19.2 with 64 or 256).
  const int nvec = I / 8;
  const int row_cap = R >= 8192 ? 64 : 128;
  const int vpt = min(8, (nvec + row_cap - 1) / row_cap);  // I <= 8192: at most 128 threads
  const int threads = row_threads(nvec, vpt);
  const __half* ch = reinterpret_cast<const __half*>(c1);
  __half* qf = reinterpret_cast<__half*>(q2_f16);
  if (vpt <= 1)
    swiglu_quant_kernel<1><<<R, threads, 0, stream>>>(ch, I, E, topK, pts1, sorted_src_route, cumsum, q2_i8,
                                                          qf, pts2, expert_idx, bounds);
  else if (vpt <= 2)
    swiglu_quant_kernel<2><<<R, threads, 0, stream>>>(ch, I, E, topK, pts1, sorted_src_route, cumsum, q2_i8,
                                                          qf, pts2, expert_idx, bounds);
  else if (vpt <= 4)
    swiglu_quant_kernel<4><<<R, threads, 0, stream>>>(ch, I, E, topK, pts1, sorted_src_route, cumsum, q2_i8,
                                                          qf, pts2, expert_idx, bounds);
  else if (vpt <= 8)
    swiglu_quant_kernel<8><<<R, threads, 0, stream>>>(ch, I, E, topK, pts1, sorted_src_route, cumsum, q2_i8,
                                                          qf, pts2, expert_idx, bounds);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_combine_unpermute(const uint16_t* c2, const float* pts2, const int32_t* expanded_row_idx,
                                     const float* probs, int M, int K, int topK, uint16_t* out,
                                     cudaStream_t stream) {
  dim3 grid(M, (K / 8 + kCombineThreads - 1) / kCombineThreads);
  const __half* ch = reinterpret_cast<const __half*>(c2);
  __half* oh = reinterpret_cast<__half*>(out);
  switch (topK) {
#define MOE_COMBINE_TK(TK)                                                                                   \
  case TK:                                                                                                   \
    combine_unpermute_tk_kernel<TK><<<grid, kCombineThreads, 0, stream>>>(ch, pts2, expanded_row_idx, probs, K, \
                                                                          oh);                               \
    break;
    MOE_COMBINE_TK(1)
    MOE_COMBINE_TK(2)
    MOE_COMBINE_TK(3)
    MOE_COMBINE_TK(4)
    MOE_COMBINE_TK(5)
    MOE_COMBINE_TK(6)
    MOE_COMBINE_TK(7)
    MOE_COMBINE_TK(8)
#undef MOE_COMBINE_TK
    default:
      combine_unpermute_kernel<<<grid, kCombineThreads, 0, stream>>>(ch, pts2, expanded_row_idx, probs, K, topK, oh);
  }
  return cudaGetLastError();
}

}  // namespace moe
