// Grouped W8A8 GEMM of the expert layer (PTO-ISA MegaMoE operator page,
// sections "3. GMM1" and "5. GMM2"), with the Dispatch gather of section
// "2. Dispatch" fused into the activation loads of GMM1.
//
// For expert e with rows [cumsum[e]-cnt_e, cumsum[e]) of the expert-major row
// space and every output channel n < N:
//     acc        = sum_k a[row][k] * W[e][n][k]          exact integer
//     C[row][n]  = sat_f16(float(acc) * scale[e][n])
//
// Engine.  GB300 runs int8 tensor-core and dp4a arithmetic at a small fraction
// of its binary16 rate, so the int8 operands are multiplied on the fp16 tensor
// path: every int8 value is exact in binary16, every product (|p| <= 127^2) is
// exact, and an fp32 accumulator is exact as long as all partial sums stay
// below 2^24 in magnitude.  The reduction is therefore split into chunks of 512
// (512 * 127^2 < 2^23); each chunk's fp32 sum is converted to int32 and added in
// integer registers, which makes the int32 accumulator bit-exact for any K.
//
// Data movement.  Weights stay int8 in HBM (they dominate the traffic): a TMA
// box of 128 channels x 64 k lands in shared memory and each thread converts its
// fragment to binary16 in registers (byte-permute into the 1024+v encoding, one
// subtract).  Activations are binary16-coded int8 (produced so by the quant and
// SwiGLU kernels), loaded by TMA with the 128-byte swizzle; for GMM1 each token
// row is fetched by its own 1-row TMA box at the token index taken from the sort,
// so no dispatched copy of the tokens is ever written.
//
// Tiling.  One CTA computes 128 channels x T rows of one expert.  The work list
// (expert, row tile) is derived by each CTA from cumsum; CTAs whose index lies
// beyond the number of row tiles exit at once.  The reduction is swapped so that
// weights are the MMA's M operand (16 channels per m16n8k16) and token rows its
// N operand, which keeps the tensor work proportional to the real row count for
// the 1-16 rows per expert of decode-sized batches.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kGemmThreads = 256;
constexpr int kBN = 128;        // channels per CTA
constexpr int kBK = 64;         // reduction depth per pipeline stage
constexpr int kStages = 6;
constexpr int kChunkBlocks = 8;  // 8 * 64 = 512-deep exact fp32 chunks

template <int T>
struct TileShape;
template <>
struct TileShape<16> { static constexpr int WM = 8, WN = 1; };
template <>
struct TileShape<32> { static constexpr int WM = 4, WN = 2; };
template <>
struct TileShape<64> { static constexpr int WM = 4, WN = 2; };

template <int T>
struct GemmCfg {
  static constexpr int WARPS_M = TileShape<T>::WM;
  static constexpr int WARPS_N = TileShape<T>::WN;
  static constexpr int MT = kBN / (16 * WARPS_M);  // m16 tiles per warp
  static constexpr int NT = T / (8 * WARPS_N);     // n8 tiles per warp
  static constexpr int X_BYTES = T * kBK * 2;      // binary16 activations, 128-B rows
  static constexpr int W_BYTES = kBN * kBK;        // int8 weights, 64-B rows
  static constexpr int STAGE_BYTES = X_BYTES + W_BYTES;
  static constexpr int SMEM_BYTES = kStages * STAGE_BYTES + 1024;
  static_assert(WARPS_M * WARPS_N == kGemmThreads / 32, "warp grid");
  static_assert(X_BYTES % 1024 == 0 && W_BYTES % 1024 == 0, "1024-B stage alignment (128-B swizzle)");
  static_assert(T * kBN * 2 <= STAGE_BYTES, "epilogue tile fits in one stage");
};

struct GemmArgs {
  const int32_t* cumsum;
  const int32_t* sorted_src_route;
  const float* scale;
  __half* C;
  int32_t* status;
  int E, N, Kd, topK;
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// 4 int8 (one 32-bit word) -> two half2 {b0,b1}, {b2,b3}, exactly.
// Byte v+128 placed in the mantissa of 0x6400 (=1024) gives 1024+v+128;
// subtracting 1152 leaves v.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a = __byte_perm(u, 0x6464u, 0x5140u);
  uint32_t b = __byte_perm(u, 0x6464u, 0x5342u);
  const uint32_t bias = 0x64806480u;  // half2(1152, 1152)
  asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Finds this CTA's (expert, first row, row count) from cumsum; returns false if
// the CTA index lies beyond the number of row tiles.  Uniform across the block.
template <int T>
__device__ bool find_tile(const int32_t* __restrict__ cumsum, int E, int tile, int& e_out, int& row0, int& rows,
                          int* s_scan) {
  // thread i owns experts [i*per, (i+1)*per): count their row tiles
  const int per = (E + kGemmThreads - 1) / kGemmThreads;
  const int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
  int local = 0;
  for (int e = e0; e < e1; ++e) {
    const int hi = __ldg(cumsum + e), lo = e ? __ldg(cumsum + e - 1) : 0;
    local += (hi - lo + T - 1) / T;
  }
  // exclusive prefix of `local` over the block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  int excl = incl - local, total = 0;
  for (int w = 0; w < kGemmThreads / 32; ++w) {
    if (w < warp) excl += s_scan[w];
    total += s_scan[w];
  }
  if (tile >= excl && tile < excl + local) {
    int acc = excl;
    for (int e = e0; e < e1; ++e) {
      const int hi = __ldg(cumsum + e), lo = e ? __ldg(cumsum + e - 1) : 0;
      const int nt = (hi - lo + T - 1) / T;
      if (tile < acc + nt) {
        const int j = tile - acc;
        s_scan[8] = e;
        s_scan[9] = lo + j * T;
        s_scan[10] = min(T, hi - lo - j * T);
        break;
      }
      acc += nt;
    }
  }
  __syncthreads();
  if (tile >= total) return false;
  e_out = s_scan[8];
  row0 = s_scan[9];
  rows = s_scan[10];
  return true;
}

template <int T, bool GATHER>
__global__ void __launch_bounds__(kGemmThreads) grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                                    const __grid_constant__ CUtensorMap tm_x,
                                                                    const GemmArgs args) {
  using Cfg = GemmCfg<T>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ int s_scan[16];
  __shared__ int s_tok[T];
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int e, row0, rows;
  if (!find_tile<T>(args.cumsum, args.E, blockIdx.x, e, row0, rows, s_scan)) return;
  const int ch0 = blockIdx.y * kBN;
  const int nk = args.Kd / kBK;

  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem_base - smem_u32(smem_raw));

  if (threadIdx.x == 0) {
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_x);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kGemmThreads / 32);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  if (GATHER) {
    for (int i = threadIdx.x; i < T; i += kGemmThreads)
      s_tok[i] = (i < rows) ? __ldg(args.sorted_src_route + row0 + i) / args.topK : -1;
    // rows beyond the tile's row count are never loaded: zero them once in every stage
    const int zero_words = (T - rows) * 32;  // 128-B rows
    for (int s = 0; s < kStages; ++s) {
      uint32_t* xs = reinterpret_cast<uint32_t*>(smem_gen + s * Cfg::STAGE_BYTES + rows * 128);
      for (int i = threadIdx.x; i < zero_words; i += kGemmThreads) xs[i] = 0u;
    }
  }
  __syncthreads();

  const uint32_t stage_tx = (uint32_t)Cfg::W_BYTES + (uint32_t)(GATHER ? rows : T) * 128u;
  const int w_row = e * args.N + ch0;

  // Producer (warp 0): issue the TMA loads of k-block kb into its stage.
  auto issue = [&](int kb) {
    const int s = kb % kStages;
    uint8_t* xs = smem_gen + s * Cfg::STAGE_BYTES;
    uint8_t* ws = xs + Cfg::X_BYTES;
    if (lane == 0) {
      mbar_arrive_expect_tx(&full_bar[s], stage_tx);
      tma_load_2d(ws, &tm_w, kb * kBK, w_row, &full_bar[s]);
      if (!GATHER) tma_load_2d(xs, &tm_x, kb * kBK, row0, &full_bar[s]);
    }
    __syncwarp();
    if (GATHER) {
      for (int i = lane; i < rows; i += 32) tma_load_2d(xs + i * 128, &tm_x, kb * kBK, s_tok[i], &full_bar[s]);
    }
  };

  if (warp == 0) {
    for (int kb = 0; kb < min(nk, kStages - 1); ++kb) issue(kb);
  }

  const int warp_m = warp % Cfg::WARPS_M, warp_n = warp / Cfg::WARPS_M;
  const int g = lane >> 2, tq = lane & 3;
  float accf[Cfg::MT][Cfg::NT][4];
  int acci[Cfg::MT][Cfg::NT][4];
#pragma unroll
  for (int mt = 0; mt < Cfg::MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < Cfg::NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        accf[mt][nt][i] = 0.0f;
        acci[mt][nt][i] = 0;
      }

  bool ok = true;
  for (int kb = 0; kb < nk; ++kb) {
    // producer: refill the stage freed by k-block kb-1
    if (warp == 0) {
      const int kn = kb + kStages - 1;
      if (kn < nk) {
        bool got = true;
        if (kn >= kStages) {
          if (lane == 0) got = mbar_wait_bounded(&empty_bar[kn % kStages], ((kn / kStages) - 1) & 1);
          got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
        }
        if (got && !*(volatile int*)&s_abort) {
          issue(kn);
        } else if (!got) {
          if (lane == 0) {
            s_abort = 1;
            record_status(args.status, MOE_ERR_TIMEOUT);
          }
        }
      }
    }
    const int s = kb % kStages;
    if (ok && !*(volatile int*)&s_abort) {
      ok = mbar_wait_bounded(&full_bar[s], (kb / kStages) & 1);
      if (!ok) {
        s_abort = 1;
        record_status(args.status, MOE_ERR_TIMEOUT);
      }
    }
    if (ok && !*(volatile int*)&s_abort) {
      const uint32_t xs = smem_base + s * Cfg::STAGE_BYTES;
      const uint32_t ws = xs + Cfg::X_BYTES;
      // B fragments (token rows): halves k = 16*tq .. 16*tq+15 of row n, 128-B swizzled
      uint4 bfrag[Cfg::NT][2];
#pragma unroll
      for (int nt = 0; nt < Cfg::NT; ++nt) {
        const int n = warp_n * Cfg::NT * 8 + nt * 8 + g;
        const uint32_t rb = xs + n * 128;
        bfrag[nt][0] = lds128(rb + (((2 * tq) ^ (n & 7)) << 4));
        bfrag[nt][1] = lds128(rb + (((2 * tq + 1) ^ (n & 7)) << 4));
      }
#pragma unroll
      for (int mt = 0; mt < Cfg::MT; ++mt) {
        const int m = warp_m * Cfg::MT * 16 + mt * 16 + g;
        const uint4 alo = lds128(ws + m * kBK + tq * 16);
        const uint4 ahi = lds128(ws + (m + 8) * kBK + tq * 16);
        const uint32_t aw_lo[4] = {alo.x, alo.y, alo.z, alo.w};
        const uint32_t aw_hi[4] = {ahi.x, ahi.y, ahi.z, ahi.w};
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
          uint32_t a0, a2, a1, a3;
          i8x4_to_f16x4(aw_lo[sl], a0, a2);  // row g:   k 4sl,4sl+1 | 4sl+2,4sl+3
          i8x4_to_f16x4(aw_hi[sl], a1, a3);  // row g+8
#pragma unroll
          for (int nt = 0; nt < Cfg::NT; ++nt) {
            const uint4& bv = bfrag[nt][sl >> 1];
            const uint32_t b0 = (sl & 1) ? bv.z : bv.x;
            const uint32_t b1 = (sl & 1) ? bv.w : bv.y;
            mma_f16_16816(accf[mt][nt], a0, a1, a2, a3, b0, b1);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[s]);
    // drain the exact fp32 chunk into the int32 accumulators
    if ((kb + 1) % kChunkBlocks == 0 || kb + 1 == nk) {
#pragma unroll
      for (int mt = 0; mt < Cfg::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < Cfg::NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acci[mt][nt][i] += __float2int_rn(accf[mt][nt][i]);
            accf[mt][nt][i] = 0.0f;
          }
    }
  }

  __syncthreads();
  if (s_abort) {
    // let any load still in flight land before the CTA's shared memory is released
    if (threadIdx.x == 0) {
      for (int kb = max(0, nk - kStages); kb < nk; ++kb) mbar_wait_bounded(&full_bar[kb % kStages], (kb / kStages) & 1);
    }
    return;
  }

  // epilogue: scale, convert, stage as [T][128] binary16 in stage 0, then coalesced stores
  __half* stile = reinterpret_cast<__half*>(smem_gen);
  const float* sc = args.scale + (size_t)e * args.N + ch0;
#pragma unroll
  for (int mt = 0; mt < Cfg::MT; ++mt) {
    const int m = warp_m * Cfg::MT * 16 + mt * 16 + g;
    const float s_lo = __ldg(sc + m), s_hi = __ldg(sc + m + 8);
#pragma unroll
    for (int nt = 0; nt < Cfg::NT; ++nt) {
      const int n = warp_n * Cfg::NT * 8 + nt * 8 + 2 * tq;
      stile[n * kBN + m] = f2h_sat(__fmul_rn(__int2float_rn(acci[mt][nt][0]), s_lo));
      stile[(n + 1) * kBN + m] = f2h_sat(__fmul_rn(__int2float_rn(acci[mt][nt][1]), s_lo));
      stile[n * kBN + m + 8] = f2h_sat(__fmul_rn(__int2float_rn(acci[mt][nt][2]), s_hi));
      stile[(n + 1) * kBN + m + 8] = f2h_sat(__fmul_rn(__int2float_rn(acci[mt][nt][3]), s_hi));
    }
  }
  __syncthreads();
  const int4* src = reinterpret_cast<const int4*>(stile);
  for (int i = threadIdx.x; i < rows * (kBN / 8); i += kGemmThreads) {
    const int r = i / (kBN / 8), c = i % (kBN / 8);
    reinterpret_cast<int4*>(args.C + (size_t)(row0 + r) * args.N + ch0)[c] = src[r * (kBN / 8) + c];
  }
}

// ------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------
typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PFN_encodeTiled get_encode_fn() {
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

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, size_t elem, const void* base, uint64_t inner,
               uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  PFN_encodeTiled fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * elem};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int T, bool GATHER>
cudaError_t launch_t(const GroupedGemmProblem& p, cudaStream_t stream) {
  using Cfg = GemmCfg<T>;
  CUtensorMap tw, tx;
  if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w, (uint64_t)p.Kd, (uint64_t)p.E * p.N, kBK, kBN,
                 CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (!encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.act, (uint64_t)p.Kd, (uint64_t)p.act_rows, kBK,
                 GATHER ? 1 : T, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<T, GATHER>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  GemmArgs a;
  a.cumsum = p.cumsum;
  a.sorted_src_route = p.sorted_src_route;
  a.scale = p.scale;
  a.C = reinterpret_cast<__half*>(p.C);
  a.status = p.status;
  a.E = p.E;
  a.N = p.N;
  a.Kd = p.Kd;
  a.topK = p.topK;
  // upper bound on row tiles: sum_e ceil(cnt_e / T) <= R / T + min(E, R)
  const int max_tiles = p.R / T + (p.E < p.R ? p.E : p.R) + 1;
  dim3 grid(max_tiles, p.N / kBN);
  grouped_gemm_kernel<T, GATHER><<<grid, kGemmThreads, Cfg::SMEM_BYTES, stream>>>(tw, tx, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm(const GroupedGemmProblem& p, cudaStream_t stream) {
  // row tile from the mean rows per expert (the host never reads device counts)
  const double mean_rows = (double)p.R / (double)p.E;
  if (p.gather) {
    if (mean_rows <= 12.0) return launch_t<16, true>(p, stream);
    if (mean_rows <= 24.0) return launch_t<32, true>(p, stream);
    return launch_t<64, true>(p, stream);
  }
  if (mean_rows <= 12.0) return launch_t<16, false>(p, stream);
  if (mean_rows <= 24.0) return launch_t<32, false>(p, stream);
  return launch_t<64, false>(p, stream);
}

}  // namespace moe
