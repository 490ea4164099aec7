// Grouped W8A8 GEMM of the expert layer on the 5th-generation tensor cores
// (tcgen05).  PTO-ISA MegaMoE operator page, sections "3. GMM1" and "5. GMM2".
//
// For expert e with rows [cumsum[e]-cnt_e, cumsum[e]) of the expert-major row
// space and every output channel n < N:
//     acc        = sum_k a[row][k] * W[e][n][k]          exact integer
//     C[row][n]  = sat_f16(float(acc) * scale[e][n])
//
// Exact integers on the fp16 tensor path.  GB300 executes int8 tensor MMAs
// and dp4a far below its binary16 rate, so the int8 operands are multiplied as
// binary16 (every int8 value, and every product |p| <= 127^2, is exact) with
// fp32 accumulation in tensor memory.  An fp32 sum of integers is exact while
// every partial sum stays below 2^24, so the reduction runs in chunks of 512
// (512 * 127^2 < 2^23); after each chunk the epilogue warps read the fp32
// accumulator, convert it to int32 and add it to a per-thread int32 sum.  The
// result is the exact integer dot product for any K.
//
// Operands.  The MMA is "swapped": weights are operand A (M = 128 output
// channels per work item) and token rows are operand B (N = T rows).
//   - Weights stay int8 in HBM (they are the dominant traffic).  A TMA box of
//     128 channels x 128 k lands in shared memory (128-byte swizzle); converter
//     warps read one channel row per thread, widen 4 int8 to 4 binary16 with a
//     byte permute into the 1024+v encoding and one subtract, and store the row
//     into a tensor-memory A buffer (tcgen05.st, 32x32b).
//   - Activations are binary16-coded int8 in expert-major rows (written so by the
//     quant-scatter and SwiGLU kernels), loaded by TMA as two [T][64] tiles per
//     stage in the canonical K-major 128-byte-swizzled layout the MMA reads
//     through a shared-memory descriptor.
//
// Roles (one persistent CTA per SM, work items strided over the CTAs):
//   warp 0      TMA producer of the weight ring (freed by the converters as soon
//               as they hold the stage in registers)
//   warp 2      TMA producer of the row-tile ring (freed when the stage's MMAs finish)
//   warp 1      tensor-memory allocation; one elected thread issues tcgen05.mma
//   warps 4-11  converters: group 0 widens the even stages, group 1 the odd
//               ones (warp w owns TMEM lanes 32*(w%4) .. +31)
//   warps 12-15 drain + epilogue: one thread per output channel
// Every wait on an mbarrier is bounded; a wait that gives up sets the status
// word to MOE_ERR_TIMEOUT and the CTA winds down (in-flight copies and MMAs
// are waited for, tensor memory is freed) before returning.
#include "common.cuh"
#include "kernels.h"
#include "tensor_map.h"

namespace moe {

namespace {

constexpr int kThreads = 640;
constexpr int kBN = 128;          // output channels per work item (MMA M)
constexpr int kBK = 128;          // reduction depth per stage
constexpr int kChunkStages = 4;   // 512-deep exact chunks
constexpr int kNumABuf = 4;       // tensor-memory A buffers (64 columns each)
constexpr int kTmemCols = 512;
constexpr int kAccCol0 = 0;       // accumulator buffers: columns [0,128) and [128,256)
constexpr int kAccStride = 128;
constexpr int kACol0 = 256;       // A buffers: columns 256 + 64*b
constexpr int kMaxExperts = 1024;
constexpr int kWProducerWarp = 0, kMmaWarp = 1, kXProducerWarp = 2, kConvWarp0 = 4, kNumConvWarps = 8,
              kDrainWarp0 = 12, kNumDrainWarps = 8;

template <int T>
struct Cfg {
  static constexpr int W_STAGES = 4;   // weight ring, freed after conversion
  static constexpr int X_STAGES = 4;   // token ring, freed by the MMA
  static constexpr int X_HALF_BYTES = T * 128;  // [T][64] binary16, 128-B swizzled rows
  static constexpr int X_BYTES = 2 * X_HALF_BYTES;
  static constexpr int W_BYTES = kBN * kBK;      // [128][128] int8, 128-B swizzled rows
  static constexpr int SMEM_BYTES = W_STAGES * W_BYTES + X_STAGES * X_BYTES + 1024;
  // kind::f16 instruction descriptor: D f32, A/B f16, both K-major, N = T, M = 128
  static constexpr uint32_t IDESC = (1u << 4) | ((uint32_t)(T >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  static_assert(T == 128, "row tile: N = 128 (the MMA costs the same for any N <= 128)");
  static_assert(X_HALF_BYTES % 1024 == 0, "1024-B alignment of swizzled tiles");
  static_assert(SMEM_BYTES + 10 * 1024 <= 227 * 1024, "shared memory");
};

struct Args {
  const int32_t* cumsum;
  const float* scale;
  __half* C;
  int32_t* status;
  int E, N, Kd;
};

// ------------------------------------------------------------------ tcgen05 helpers
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle layout:
// rows 128 B apart, groups of 8 rows 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);     // start address
  d |= (uint64_t)1 << 16;                        // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset: 8-row groups
  d |= (uint64_t)1 << 46;                        // descriptor version
  d |= (uint64_t)2 << 61;                        // swizzle: 128 B
  return d;
}

__device__ __forceinline__ void mma_f16_tmemA(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

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
  const uint32_t a = __byte_perm(u, 0x6464u, 0x5140u);
  const uint32_t b = __byte_perm(u, 0x6464u, 0x5342u);
  const uint32_t bias = 0x64806480u;  // half2(1152, 1152)
  asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

struct Item {
  int e, cb, row0, rows;
};

// Work item j -> (expert, channel block, first row, rows).  Items run expert-major,
// then channel block, then row tile: CTAs working at the same time share weight
// blocks (and token rows) through L2.
template <int T>
__device__ __forceinline__ Item decode_item(int j, const int* s_pref, const int* s_end, int E) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pref[mid] <= j) lo = mid; else hi = mid;
  }
  const int start = lo ? s_end[lo - 1] : 0;
  const int cnt = s_end[lo] - start;
  const int n_rt = (cnt + T - 1) / T;
  const int local = j - s_pref[lo];
  const int cb = local / n_rt, rt = local - cb * n_rt;
  Item it;
  it.e = lo;
  it.cb = cb;
  it.row0 = start + rt * T;
  it.rows = min(T, cnt - rt * T);
  return it;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* status) {
  if (*abort_flag) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  *abort_flag = 1;
  record_status(status, MOE_ERR_TIMEOUT);
  return false;
}

template <int T>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                                      const __grid_constant__ CUtensorMap tm_x,
                                                                      const Args args) {
  using C = Cfg<T>;
  constexpr int SW = C::W_STAGES, SX = C::X_STAGES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t wfull_bar[SW], wempty_bar[SW], xfull_bar[SX], xempty_bar[SX];
  __shared__ __align__(8) uint64_t afull_bar[kNumABuf], aempty_bar[kNumABuf];
  __shared__ __align__(8) uint64_t accfull_bar[2], accempty_bar[2], final_bar;
  __shared__ int s_pref[kMaxExperts + 1];
  __shared__ int s_end[kMaxExperts];
  __shared__ int s_wsum[16];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_w_issued, s_x_issued;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E, n_cb = args.N / kBN;
  const int nk = (args.Kd + kBK - 1) / kBK;  // a 64-deep tail reads TMA zero fill
  volatile int* abort_flag = &s_abort;

  // ---- work list (s_pref[e] = first work item of expert e), barriers, tensor memory
  {
    const int per = (E + kThreads - 1) / kThreads;
    const int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
    int local = 0;
    for (int e = e0; e < e1; ++e) {
      const int hi = __ldg(args.cumsum + e), lo = e ? __ldg(args.cumsum + e - 1) : 0;
      s_end[e] = hi;
      local += (hi - lo + T - 1) / T * n_cb;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) s_wsum[warp] = incl;
    if (threadIdx.x == 0) {
      s_abort = 0;
      s_w_issued = 0;
      s_x_issued = 0;
    }
    if (warp == kMmaWarp) {
      // all 512 tensor-memory columns (one CTA per SM)
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                   "n"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
      if (lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_x);
        for (int s = 0; s < SW; ++s) {
          mbar_init(&wfull_bar[s], 1);
          mbar_init(&wempty_bar[s], kNumConvWarps / 2);
        }
        for (int s = 0; s < SX; ++s) {
          mbar_init(&xfull_bar[s], 1);
          mbar_init(&xempty_bar[s], 1);
        }
        for (int b = 0; b < kNumABuf; ++b) {
          mbar_init(&afull_bar[b], kNumConvWarps / 2);
          mbar_init(&aempty_bar[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
          mbar_init(&accfull_bar[b], 1);
          mbar_init(&accempty_bar[b], kNumDrainWarps);
        }
        mbar_init(&final_bar, 1);
        fence_barrier_init();
      }
      tc_fence_before();
    }
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += s_wsum[w];
    for (int e = e0; e < e1; ++e) {
      s_pref[e] = run;
      const int lo = e ? s_end[e - 1] : 0;
      run += (s_end[e] - lo + T - 1) / T * n_cb;
    }
    if (e0 < E && e1 == E) s_pref[E] = run;
  }
  __syncthreads();
  tc_fence_after();
  const int total = s_pref[E];
  const uint32_t tmem = s_tmem;

  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem_base - smem_u32(smem_raw));
  const uint32_t w_ring = smem_base;                     // SW x [128][128] int8
  const uint32_t x_ring = smem_base + SW * C::W_BYTES;   // SX x 2 x [T][64] binary16

  if (warp == kWProducerWarp) {
    // ======================= weight producer (one lane) =======================
    if (lane == 0) {
      int n = 0;
      for (int j = blockIdx.x; j < total; j += gridDim.x) {
        const Item it = decode_item<T>(j, s_pref, s_end, E);
        const int w_row = it.e * args.N + it.cb * kBN;
        for (int kb = 0; kb < nk; ++kb, ++n) {
          const int slot = n % SW;
          if (!wait_or_abort(&wempty_bar[slot], ((n / SW) & 1) ^ 1, abort_flag, args.status)) goto w_done;
          mbar_arrive_expect_tx(&wfull_bar[slot], (uint32_t)C::W_BYTES);
          tma_load_2d(smem_gen + slot * C::W_BYTES, &tm_w, kb * kBK, w_row, &wfull_bar[slot]);
        }
      }
    w_done:
      s_w_issued = n;
    }
  } else if (warp == kXProducerWarp) {
    // ======================= token producer =======================
    int n = 0;
    for (int j = blockIdx.x; j < total; j += gridDim.x) {
      const Item it = decode_item<T>(j, s_pref, s_end, E);
      const uint32_t tx = (uint32_t)T * 256u;
      for (int kb = 0; kb < nk; ++kb, ++n) {
        const int slot = n % SX;
        bool ok = true;
        if (lane == 0) ok = wait_or_abort(&xempty_bar[slot], ((n / SX) & 1) ^ 1, abort_flag, args.status);
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) goto x_done;
        const uint32_t xs = x_ring + slot * C::X_BYTES;
        uint8_t* xs_g = smem_gen + (xs - smem_base);
        const int kx = kb * kBK;
        if (lane == 0) {
          mbar_arrive_expect_tx(&xfull_bar[slot], tx);
          tma_load_2d(xs_g, &tm_x, kx, it.row0, &xfull_bar[slot]);
          tma_load_2d(xs_g + C::X_HALF_BYTES, &tm_x, kx + 64, it.row0, &xfull_bar[slot]);
        }
        __syncwarp();
      }
    }
  x_done:
    if (lane == 0) s_x_issued = n;
  } else if (warp == kMmaWarp) {
    // ======================= MMA issuer (one thread) =======================
    if (lane == 0) {
      int n = 0, c = 0;
      bool ok = true;
      for (int j = blockIdx.x; j < total && ok; j += gridDim.x) {
        for (int kb = 0; kb < nk && ok; ++kb, ++n) {
          const int slot = n % SX, ab = n % kNumABuf, acc = c & 1;
          if (kb % kChunkStages == 0) {
            // a new exact chunk: the drain must have read this accumulator buffer
            ok = wait_or_abort(&accempty_bar[acc], ((c >> 1) & 1) ^ 1, abort_flag, args.status);
            if (!ok) break;
          }
          ok = wait_or_abort(&xfull_bar[slot], (n / SX) & 1, abort_flag, args.status) &&
               wait_or_abort(&afull_bar[ab], (n / kNumABuf) & 1, abort_flag, args.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t xs = x_ring + slot * C::X_BYTES;
          const uint32_t d_tmem = tmem + kAccCol0 + acc * kAccStride;
          const uint32_t a_tmem = tmem + kACol0 + ab * 64;
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const uint64_t bdesc = sw128_desc(xs + (s >> 2) * C::X_HALF_BYTES + (s & 3) * 32);
            mma_f16_tmemA(d_tmem, a_tmem + s * 8, bdesc, C::IDESC, (kb % kChunkStages != 0 || s != 0) ? 1u : 0u);
          }
          mma_commit(&xempty_bar[slot]);  // token stage free once these MMAs complete
          mma_commit(&aempty_bar[ab]);    // tensor-memory A buffer free
          if (kb % kChunkStages == kChunkStages - 1 || kb == nk - 1) {
            mma_commit(&accfull_bar[acc]);  // chunk accumulated: hand it to the drain
            ++c;
          }
        }
      }
      // every MMA issued by this thread has completed once final_bar fires
      mma_commit(&final_bar);
      mbar_wait_bounded(&final_bar, 0);
    }
    __syncwarp();
  } else if (warp >= kConvWarp0 && warp < kConvWarp0 + kNumConvWarps) {
    // ======================= converters =======================
    // Group g widens the stages n with n % 2 == g, a full 128-byte weight row per
    // thread, stores it into the stage's tensor-memory A buffer and hands it to the
    // MMA issuer.
    const int grp = (warp - kConvWarp0) >> 2;
    const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;         // weight channel row of this thread
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int n = 0;
    bool ok = true;
    for (int j = blockIdx.x; j < total && ok; j += gridDim.x) {
      for (int kb = 0; kb < nk; ++kb, ++n) {
        if ((n & 1) != grp) continue;
        const int slot = n % SW, ab = n % kNumABuf;
        ok = wait_or_abort(&wfull_bar[slot], (n / SW) & 1, abort_flag, args.status) &&
             wait_or_abort(&aempty_bar[ab], ((n / kNumABuf) & 1) ^ 1, abort_flag, args.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const uint32_t wrow = w_ring + slot * C::W_BYTES + r * kBK;
        uint32_t v[64];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 w4 = lds128(wrow + ((q ^ (r & 7)) << 4));
          i8x4_to_f16x4(w4.x, v[8 * q + 0], v[8 * q + 1]);
          i8x4_to_f16x4(w4.y, v[8 * q + 2], v[8 * q + 3]);
          i8x4_to_f16x4(w4.z, v[8 * q + 4], v[8 * q + 5]);
          i8x4_to_f16x4(w4.w, v[8 * q + 6], v[8 * q + 7]);
        }
        // the weight stage is in registers: hand it back to the producer
        __syncwarp();
        if (lane == 0) mbar_arrive(&wempty_bar[slot]);
        const uint32_t ta = tmem + lane_off + kACol0 + ab * 64;
        tmem_st32(ta, *reinterpret_cast<const uint32_t(*)[32]>(&v[0]));
        tmem_st32(ta + 32, *reinterpret_cast<const uint32_t(*)[32]>(&v[32]));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull_bar[ab]);
      }
    }
  } else if (warp >= kDrainWarp0) {
    // ======================= drain + epilogue =======================
    // warp w drains TMEM lanes 32*(w%4).. (output channels) and the 64 accumulator
    // columns (row-tile rows) of half (w-12)/4
    const int quarter = warp & 3;
    const int chalf = (warp - kDrainWarp0) >> 2;
    const int r = quarter * 32 + lane;  // output channel within the item
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16) + chalf * 64;
    const int nch = (nk + kChunkStages - 1) / kChunkStages;
    int c = 0;
    bool ok = true;
    for (int j = blockIdx.x; j < total && ok; j += gridDim.x) {
      const Item it = decode_item<T>(j, s_pref, s_end, E);
      const float sc = __ldg(args.scale + (size_t)it.e * args.N + it.cb * kBN + r);
      int acci[64];
#pragma unroll
      for (int t = 0; t < 64; ++t) acci[t] = 0;
      for (int ch = 0; ch < nch; ++ch, ++c) {
        const int acc = c & 1;
        ok = wait_or_abort(&accfull_bar[acc], (c >> 1) & 1, abort_flag, args.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int t0 = 0; t0 < 64; t0 += 16) {
          uint32_t v[16];
          tmem_ld16(lane_base + kAccCol0 + acc * kAccStride + t0, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) acci[t0 + i] += __float2int_rn(__uint_as_float(v[i]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty_bar[acc]);
      }
      if (!ok) break;
      // epilogue: channel r of rows row0 + 64*chalf + t (a warp writes 64 contiguous bytes per row)
      const int t_lo = chalf * 64;
      __half* dst = args.C + (size_t)(it.row0 + t_lo) * args.N + it.cb * kBN + r;
#pragma unroll
      for (int t = 0; t < 64; ++t)
        if (t_lo + t < it.rows) dst[(size_t)t * args.N] = f2h_sat(__fmul_rn(__int2float_rn(acci[t]), sc));
    }
  }

  __syncthreads();
  if (threadIdx.x == 0) {
    // copies still in flight (only after an abort) land before shared memory is released
    const int wi = s_w_issued, xi = s_x_issued;
    for (int n = max(0, wi - SW); n < wi; ++n) mbar_wait_bounded(&wfull_bar[n % SW], (n / SW) & 1);
    for (int n = max(0, xi - SX); n < xi; ++n) mbar_wait_bounded(&xfull_bar[n % SX], (n / SX) & 1);
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
  }
}

// ------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------
template <int T>
cudaError_t launch_t(const GroupedGemmProblem& p, cudaStream_t stream) {
  using Cf = Cfg<T>;
  CUtensorMap tw, tx;
  if (!encode_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w, (uint64_t)p.Kd, (uint64_t)p.E * p.N, kBK,
                            kBN))
    return cudaErrorInvalidValue;
  if (!encode_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.act, (uint64_t)p.Kd, (uint64_t)p.R, 64, T))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_tc_kernel<T>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  Args a;
  a.cumsum = p.cumsum;
  a.scale = p.scale;
  a.C = reinterpret_cast<__half*>(p.C);
  a.status = p.status;
  a.E = p.E;
  a.N = p.N;
  a.Kd = p.Kd;
  grouped_gemm_tc_kernel<T><<<sm_count(), kThreads, Cf::SMEM_BYTES, stream>>>(tw, tx, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm_tc(const GroupedGemmProblem& p, cudaStream_t stream) {
  return launch_t<128>(p, stream);
}

// Engine choice.  A tcgen05.mma of M=128, K=16 costs about the same for any N up to
// 128 (measured ~88 cycles on GB300), i.e. it consumes 2 KB of weights per issue
// slot: with few rows per expert that caps weight streaming at about the HBM rate.
// Warp-level HMMA (m16n8k16) consumes weights several times faster at N=8, so
// batches with at most 24 rows per expert on average run on it with 16-row tiles,
// larger ones on tcgen05 with 128-row tiles.  Measured at K=7168, I=2048, E=256:
// 16 rows per expert, GMM1 1.64 ms on the warp-MMA engine against 2.92 ms on
// tcgen05; 64 rows per expert, 4.97 ms against 3.73 ms.  The tile follows the mean
// rows per expert (the host never reads device counts).
cudaError_t launch_grouped_gemm(const GroupedGemmProblem& p, cudaStream_t stream) {
  const double mean_rows = (double)p.R / (double)p.E;
  if (mean_rows <= 24.0) return launch_grouped_gemm_hmma(p, 16, stream);
  return launch_grouped_gemm_tc(p, stream);
}

}  // namespace moe
