// Grouped W8A8 GEMM of the expert layer on warp-level tensor-core MMAs
// (PTO-ISA MegaMoE operator page, sections "3. GMM1" and "5. GMM2"): the engine
// for row tiles of up to 32 rows (decode-sized batches, a few rows per expert).
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
// Data movement.  Weights stay int8 in HBM (they dominate the traffic): each
// 256-deep pipeline stage brings two boxes of 128 channels x 128 k into shared
// memory (two tiled TMA copies in the row layout, one 32 KiB bulk copy in the
// tile layout) and each thread converts its fragment to binary16 in registers
// (byte-permute into the 1024+v encoding, one subtract).  Activations are
// binary16-coded int8 (produced so by the quant-scatter and SwiGLU kernels) in
// expert-major rows, loaded by tiled TMA boxes with the 128-byte swizzle.  The
// GATHER instantiation instead reads token-major codes, gathering each tile's
// token rows by index (tile::gather4, four rows per copy), so that the caller
// needs no dispatched copy of the tokens; the layer itself keeps the dispatched
// rows, which measured faster.
//
// Warps.  16 MMA warps in two groups of 8 (group g computes the stages in ring
// slots s % 2 == g), TMA producer warps (one per group for 16-row tiles, else one),
// and two epilogue warps that scale, convert and store each item from the int32
// sums both groups add into shared memory at the item's end, so that no MMA warp
// stops for an epilogue.
//
// Tiling.  One CTA computes 128 channels x T rows of one expert.  The work list
// (expert, row tile) is derived by each CTA from cumsum; CTAs whose index lies
// beyond the number of row tiles exit at once.  The reduction is swapped so that
// weights are the MMA's M operand (16 channels per m16n8k16) and token rows its
// N operand, which keeps the tensor work proportional to the real row count for
// the 1-16 rows per expert of decode-sized batches.
#include "common.cuh"
#include "kernels.h"
#include "tensor_map.h"

namespace moe {

namespace {

constexpr int kGroupWarps = 8;                        // MMA warps per group
constexpr int kGroups = 2;                            // group g computes the stages in slots s % kGroups == g
constexpr int kConsumerWarps = kGroups * kGroupWarps;
constexpr int kMaxProducerWarps = kGroups;  // TMA producer warps (per tile shape: 1 or kGroups)
// Epilogue warps (after the producers).  Two keep the CTA at 19-20 warps and the MMA
// warps at 96 registers; four epilogue warps (21-22 warps) would leave them 80 under
// the launch bound.
constexpr int kEpiWarps = 2;
constexpr int kBN = 128;         // channels per work item
constexpr int kBK = 256;         // reduction depth per pipeline stage
constexpr int kSubK = 128;       // weight sub-tile depth (one 128-byte swizzled TMA box)
constexpr int kQuarters = kBK / 64;  // 64-deep k quarters per stage
constexpr int kMaxExperts = 1024;

template <int T>
struct TileShape;
// P: independent fp32 partial accumulators per output fragment (k-slices are dealt
// round-robin to them). 16-row tiles have 2 fragments per warp and take 4 partials
// so that 8 MMA chains are in flight; 32-row tiles have 4 fragments and measure
// faster with a single partial (fewer registers, no fold in the epilogue).
// PRODUCERS: TMA producer warps.  With one per MMA group each fills only its group's
// ring slots, so a group that falls behind holds back its own stages' loads and not the
// other's: decode GMM1 / GMM2 1067 / 557 -> 1044 / 542 us on 16-row tiles; on 32-row
// tiles (mid: 1225 / 660 -> 1233 / 683 us, consumer-bound) one producer stays.
template <>
struct TileShape<16> { static constexpr int WM = 8, WN = 1, STAGES = 4, P = 4, PRODUCERS = 2; };
template <>
struct TileShape<32> { static constexpr int WM = 8, WN = 1, STAGES = 4, P = 1, PRODUCERS = 1; };

template <int T>
struct GemmCfg {
  static constexpr int WARPS_M = TileShape<T>::WM;
  static constexpr int WARPS_N = TileShape<T>::WN;
  static constexpr int STAGES = TileShape<T>::STAGES;
  static constexpr int MT = kBN / (16 * WARPS_M);  // m16 tiles per warp
  static constexpr int NT = T / (8 * WARPS_N);     // n8 tiles per warp
  static constexpr int P = TileShape<T>::P;
  static constexpr int PRODUCERS = TileShape<T>::PRODUCERS;
  static constexpr int THREADS = (kConsumerWarps + PRODUCERS + kEpiWarps) * 32;
  static_assert(PRODUCERS == 1 || PRODUCERS == kGroups, "one producer, or one per MMA group");
  static constexpr int X_HALF_BYTES = T * 128;     // one k quarter: [T][64] binary16, 128-B swizzled rows
  static constexpr int X_BYTES = kQuarters * X_HALF_BYTES;
  static constexpr int W_SUB_BYTES = kBN * kSubK;  // [128][128] int8, 128-B swizzled rows
  static constexpr int W_BYTES = (kBK / kSubK) * W_SUB_BYTES;
  static constexpr int STAGE_BYTES = X_BYTES + W_BYTES;
  static constexpr int EPI_BYTES = T * kBN * 2;
  static constexpr int PART_BYTES = kGroupWarps * MT * NT * 4 * 32 * 4;  // the item's int32 sums
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + PART_BYTES + 1024;
  static_assert(WARPS_M * WARPS_N == kGroupWarps, "warp grid");
  static_assert(T <= 32, "one lane per row of the epilogue's row copies");
  // stage n is computed by group n % kGroups: with STAGES a multiple of kGroups every
  // ring slot always belongs to the same group, which then waits on every phase of its
  // slots in order (a group never tests the parity of a phase it skipped)
  static_assert(STAGES % kGroups == 0, "ring slots per group");
  static_assert(X_HALF_BYTES % 1024 == 0, "1024-B alignment of swizzled tiles");
  static_assert(kBN == kWTileRows && kSubK == kWTileDepth && W_SUB_BYTES == kWTileBytes && kBK == 2 * kWTileDepth,
                "a stage is two adjacent weight tiles");
  static_assert(SMEM_BYTES + 9 * 1024 <= 227 * 1024, "shared memory");
};

struct GemmArgs {
  const int32_t* cumsum;
  const float* scale;
  __half* C;
  int32_t* status;
  int E, N, Kd;
  int split_rows;  // this engine serves the experts with at most split_rows rows
  int min_rows;    // ... and more than min_rows rows
  const int32_t* gather_route;  // null: tiled token boxes; else row d gathers token gather_route[d] / topK
  int topK;
  const uint8_t* w_tiles;  // null: weights through the tensor map; else the tile layout
  int w_kb;                // tiles per 128-channel block of the tile layout
};

// 4 int8 (one 32-bit word) -> two half2 {b0,b1}, {b2,b3}, exactly.
// Byte v+128 placed in the mantissa of 0x6400 (=1024) gives 1024+v+128;
// subtracting 1152 leaves v.  flip = 0x80808080 for two's-complement bytes
// (v+128 = v ^ 0x80), 0 for bytes stored as v+128 (the weight tiles).
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t flip, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ flip;
  uint32_t a = __byte_perm(u, 0x6464u, 0x5140u);
  uint32_t b = __byte_perm(u, 0x6464u, 0x5342u);
  const uint32_t bias = 0x64806480u;  // half2(1152, 1152)
  asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

// Not volatile: the compiler may reorder MMAs against independent loads and ALU work.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


// One 64-deep k-half of one stage for one warp: A fragments from the int8 weight tile
// (widened in registers), B fragments from the binary16 row tile, NTL live n8 tiles.
template <class Cfg, int NTL>
__device__ __forceinline__ void hmma_half_stage(const uint8_t* xh, const uint8_t* ws, uint32_t wflip, int half,
                                                int warp_m, int warp_n, int g, int tq, int pg,
                                                float (&accf)[Cfg::P][Cfg::MT][Cfg::NT][4]) {
  // Plain shared-memory reads (ordered after the stage's barrier wait by its memory
  // clobber) let the compiler issue every load of the stage before the first MMA.
  auto lds = [](const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); };
  // B fragments: binary16 k = 64half + 16tq .. +15 of row n (swizzled chunks 2tq, 2tq+1)
  uint4 bfrag[NTL][2];
#pragma unroll
  for (int nt = 0; nt < NTL; ++nt) {
    const int n = warp_n * Cfg::NT * 8 + nt * 8 + g;
    const uint8_t* rb = xh + n * 128;
    bfrag[nt][0] = lds(rb + (((2 * tq) ^ (n & 7)) << 4));
    bfrag[nt][1] = lds(rb + (((2 * tq + 1) ^ (n & 7)) << 4));
  }
#pragma unroll
  for (int mt = 0; mt < Cfg::MT; ++mt) {
    // A fragments: int8 k = 64half + 16tq .. +15 of channels perm(g) and 8 + perm(g)
    const int m = warp_m * Cfg::MT * 16 + mt * 16 + pg;
    const uint4 alo = lds(ws + m * kSubK + (((4 * half + tq) ^ (m & 7)) << 4));
    const uint4 ahi = lds(ws + (m + 8) * kSubK + (((4 * half + tq) ^ (m & 7)) << 4));
    const uint32_t aw_lo[4] = {alo.x, alo.y, alo.z, alo.w};
    const uint32_t aw_hi[4] = {ahi.x, ahi.y, ahi.z, ahi.w};
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
      uint32_t a0, a2, a1, a3;
      i8x4_to_f16x4(aw_lo[sl], wflip, a0, a2);  // row perm(g):   k 4sl,4sl+1 | 4sl+2,4sl+3
      i8x4_to_f16x4(aw_hi[sl], wflip, a1, a3);  // row 8+perm(g)
#pragma unroll
      for (int nt = 0; nt < NTL; ++nt) {
        const uint4& bv = bfrag[nt][sl >> 1];
        const uint32_t b0 = (sl & 1) ? bv.z : bv.x;
        const uint32_t b1 = (sl & 1) ? bv.w : bv.y;
        mma_f16_16816(accf[sl % Cfg::P][mt][nt], a0, a1, a2, a3, b0, b1);
      }
    }
  }
}

// A whole stage (all 64-deep k quarters) with NTL live n8 tiles.
template <class Cfg, int NTL>
__device__ __forceinline__ void hmma_stage(const uint8_t* xs, const uint8_t* ws, uint32_t wflip, int warp_m, int warp_n,
                                           int g, int tq, int pg, float (&accf)[Cfg::P][Cfg::MT][Cfg::NT][4]) {
#pragma unroll
  for (int q = 0; q < kQuarters; ++q)
    hmma_half_stage<Cfg, NTL>(xs + q * Cfg::X_HALF_BYTES, ws + (q >> 1) * Cfg::W_SUB_BYTES, wflip, q & 1, warp_m,
                              warp_n, g, tq, pg, accf);
}

// Dispatch on the live n8 tiles of the item (rows beyond the item's rows are
// skipped, so the MMA work follows the real row count).
template <class Cfg>
__device__ __forceinline__ void hmma_stage_live(int live_nt, const uint8_t* xs, const uint8_t* ws, uint32_t wflip,
                                                int warp_m, int warp_n, int g, int tq, int pg,
                                                float (&accf)[Cfg::P][Cfg::MT][Cfg::NT][4]) {
  if (Cfg::NT >= 4 && live_nt >= 4) {
    hmma_stage<Cfg, (Cfg::NT >= 4 ? 4 : 1)>(xs, ws, wflip, warp_m, warp_n, g, tq, pg, accf);
  } else if (Cfg::NT >= 3 && live_nt == 3) {
    hmma_stage<Cfg, (Cfg::NT >= 3 ? 3 : 1)>(xs, ws, wflip, warp_m, warp_n, g, tq, pg, accf);
  } else if (live_nt >= 2) {
    hmma_stage<Cfg, 2>(xs, ws, wflip, warp_m, warp_n, g, tq, pg, accf);
  } else if (live_nt == 1) {
    hmma_stage<Cfg, 1>(xs, ws, wflip, warp_m, warp_n, g, tq, pg, accf);
  }
}

// Exact fp32 chunk sums -> int32 accumulators; the fp32 partials restart at 0.
template <class Cfg>
__device__ __forceinline__ void drain_chunk(float (&accf)[Cfg::P][Cfg::MT][Cfg::NT][4], int (&acci)[Cfg::MT][Cfg::NT][4]) {
#pragma unroll
  for (int mt = 0; mt < Cfg::MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < Cfg::NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int q = 0; q < Cfg::P; ++q) {
          acci[mt][nt][i] += __float2int_rn(accf[q][mt][nt][i]);
          accf[q][mt][nt][i] = 0.0f;
        }
      }
}

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32)); }
__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 2, %0;" ::"n"(kEpiWarps * 32)); }
// The epilogue warps' barrier with an OR over their votes: the same answer in every
// epilogue warp, so they leave their loop together.
__device__ __forceinline__ bool epilogue_bar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 2, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "n"(kEpiWarps * 32)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ bool wait_part(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_wait_bounded(bar, parity)) return true;
  record_status(status, MOE_ERR_TIMEOUT);
  return false;
}

// MMA row i of an m16 tile reads weight channel perm(i) of the tile, chosen so
// that the two rows an 8-lane shared-memory phase reads differ in bit 2: with the
// 128-byte swizzle their 16-byte chunks then land in disjoint bank groups.
__device__ __forceinline__ int mrow_perm(int g) { return (g >> 1) + ((g & 1) << 2); }

struct Item {
  int e, cb, row0, rows;
};

// Work items of an expert with `cnt` rows on this engine: its row tiles x channel
// blocks, or none when the expert has more than split_rows rows (the tcgen05 pairs
// take it).  Experts without items leave the prefix flat, and the binary search in
// decode_item (last expert whose first item is <= j) skips them.
template <int T>
__device__ __forceinline__ int own_items(int cnt, int min_rows, int split_rows, int n_cb) {
  return cnt > min_rows && cnt <= split_rows ? (cnt + T - 1) / T * n_cb : 0;
}

// Work item j -> (expert, channel block, first row, rows).  Items are ordered
// expert-major, then channel block, then row tile, so CTAs that run at the
// same time share weight blocks through L2.  The expert is the last one whose
// first item is <= j; a CTA's items only move forward, so the search starts at the
// previous item's expert (e_hint): the next four prefixes are read at once (one
// shared-memory latency instead of a binary search's chain of eight, which cost
// 3.6% of GMM2's time at 8-stage items), and a binary search covers longer jumps.
__device__ __forceinline__ int find_expert(int j, const int* s_pref, int E, int e_hint) {
  int lo = e_hint, c = 0;
#pragma unroll
  for (int step = 1; step <= 4; ++step) c += s_pref[min(lo + step, E)] <= j ? 1 : 0;  // s_pref[E] > j
  lo += c;
  if (c == 4) {
    int hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pref[mid] <= j) lo = mid; else hi = mid;
    }
  }
  return lo;
}

template <int T>
__device__ __forceinline__ Item decode_item(int j, const int* s_pref, const int* s_end, int E, int n_cb,
                                            int& e_hint) {
  const int e = find_expert(j, s_pref, E, e_hint);
  e_hint = e;
  const int start = e ? s_end[e - 1] : 0;
  const int cnt = s_end[e] - start;
  const int n_rt = (cnt + T - 1) / T;
  const int local = j - s_pref[e];
  const int cb = local / n_rt, rt = local - cb * n_rt;
  Item it;
  it.e = e;
  it.cb = cb;
  it.row0 = start + rt * T;
  it.rows = min(T, cnt - rt * T);
  return it;
}

// GATHER: token rows gathered by index (args.gather_route) instead of tiled boxes of
// expert-major rows; a separate instantiation, so the tiled kernel carries none of it.
template <int T, bool GATHER, bool TILES>
__global__ void __launch_bounds__(GemmCfg<T>::THREADS, 1) grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                                       const __grid_constant__ CUtensorMap tm_x,
                                                                       const __grid_constant__ CUtensorMap tm_x8,
                                                                       const GemmArgs args) {
  using Cfg = GemmCfg<T>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[S];
  __shared__ __align__(8) uint64_t empty_bar[S];
  __shared__ __align__(8) uint64_t part_full_bar;   // both groups' partials are in the item's sums
  __shared__ __align__(8) uint64_t part_empty_bar;  // the epilogue warps have read (and cleared) them
  __shared__ int s_pref[kMaxExperts + 1];  // first work item of each expert
  __shared__ int s_end[kMaxExperts];       // cumsum
  __shared__ int s_wsum[kConsumerWarps];
  __shared__ int s_abort, s_issued[kMaxProducerWarps];  // per producer: 1 + its last stage issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E, n_cb = args.N / kBN;
  const int nk = (args.Kd + kBK - 1) / kBK;  // a ragged tail reads TMA zero fill

  // ---- work list: s_pref[e] = sum over e' < e of ceil(cnt_e' / T) * n_cb
  if (threadIdx.x < kConsumerWarps * 32) {
    const int per = (E + kConsumerWarps * 32 - 1) / (kConsumerWarps * 32);
    const int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
    int local = 0;
    for (int e = e0; e < e1; ++e) {
      const int hi = __ldg(args.cumsum + e), lo = e ? __ldg(args.cumsum + e - 1) : 0;
      s_end[e] = hi;
      local += own_items<T>(hi - lo, args.min_rows, args.split_rows, n_cb);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) s_wsum[warp] = incl;
    consumer_bar();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += s_wsum[w];
    for (int e = e0; e < e1; ++e) {
      s_pref[e] = run;
      const int lo = e ? s_end[e - 1] : 0;
      run += own_items<T>(s_end[e] - lo, args.min_rows, args.split_rows, n_cb);
    }
    if (e0 < E && e1 == E) s_pref[E] = run;
  } else if (warp == kConsumerWarps && lane == 0) {
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_x8);
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kGroupWarps);  // one group consumes each stage
    }
    mbar_init(&part_full_bar, kConsumerWarps);
    mbar_init(&part_empty_bar, kEpiWarps);
    s_abort = 0;
    for (int q = 0; q < kMaxProducerWarps; ++q) s_issued[q] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int total = s_pref[E];

  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem_base - smem_u32(smem_raw));
  __half* stile = reinterpret_cast<__half*>(smem_gen + S * Cfg::STAGE_BYTES);  // [T][kBN] output staging
  int* sums = reinterpret_cast<int*>(smem_gen + S * Cfg::STAGE_BYTES + Cfg::EPI_BYTES);  // fragment order
  constexpr int kPartWarp = Cfg::MT * Cfg::NT * 4 * 32;  // sums per consumer-warp slice
  for (int i = threadIdx.x; i < Cfg::PART_BYTES / 16; i += Cfg::THREADS)
    reinterpret_cast<int4*>(sums)[i] = make_int4(0, 0, 0, 0);  // the first item's sums start at zero

  if (GATHER) {
    // Gathered stages leave the rows past a tile's last 4-row group, and quarters
    // past K, unwritten.  Starting every token stage at zero keeps such rows finite
    // codes (zero, or a previous stage's), so their products with the zero-filled
    // weight columns past K vanish and the outputs of the extra rows, never stored,
    // cannot disturb anything.
    for (int s = 0; s < S; ++s) {
      int4* xz = reinterpret_cast<int4*>(smem_gen + s * Cfg::STAGE_BYTES);
      for (int i = threadIdx.x; i < Cfg::X_BYTES / 16; i += Cfg::THREADS) xz[i] = make_int4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  __syncthreads();

  if (warp >= kConsumerWarps && warp < kConsumerWarps + Cfg::PRODUCERS) {
    // ================= TMA producer warps =================
    // Producer q loads the stages n with n % PRODUCERS == q (with one per group, ring
    // slots s % kGroups == q, those of MMA group q) and walks past the others.
    const int q_own = warp - kConsumerWarps;
    constexpr bool gather = GATHER;
    int e_hint = 0;
    int slot = 0;
    uint32_t phase = 0;
    int issued = 0;  // stages issued (one producer), else 1 + the last one's global index
    int n = 0;       // global stage index (one producer per group)
    for (int j = blockIdx.x; j < total; j += gridDim.x) {
      const Item it = decode_item<T>(j, s_pref, s_end, E, n_cb, e_hint);
      const int w_row = it.e * args.N + it.cb * kBN;
      // Token rows.  Tiled: a box of T rows from the expert-major operand (tiles of at
      // most 8 rows, most decode tiles, load an 8-row box).  Gathered: the tile's rows
      // in 4-row groups, only the groups that hold real rows; lane l issues group
      // l % g4 of quarter l / g4, and its group's rows past the tile's last real row
      // repeat that row's token (their outputs are never stored).
      const bool small = (T > 8) && (it.rows <= 8);
      const void* tmx = small ? static_cast<const void*>(&tm_x8) : static_cast<const void*>(&tm_x);
      const int g4 = (it.rows + 3) >> 2;
      int4 tok = make_int4(0, 0, 0, 0);
      if (gather) {
        const int r0 = it.row0 + 4 * (lane % g4), last = it.row0 + it.rows - 1;
        tok.x = __ldg(args.gather_route + min(r0, last)) / args.topK;
        tok.y = __ldg(args.gather_route + min(r0 + 1, last)) / args.topK;
        tok.z = __ldg(args.gather_route + min(r0 + 2, last)) / args.topK;
        tok.w = __ldg(args.gather_route + min(r0 + 3, last)) / args.topK;
      }
      for (int kb = 0; kb < nk; ++kb) {
        if constexpr (Cfg::PRODUCERS > 1) {
          if (n++ % Cfg::PRODUCERS != q_own) {
            if (++slot == S) {
              slot = 0;
              phase ^= 1u;
            }
            continue;
          }
        }
        const int kx = kb * kBK;
        // quarters of this stage inside K (K % 128 == 0: a tail stage has 2); the
        // tiled boxes read zero fill past K, the gathers are not issued there
        const int nq = gather ? min(kQuarters, (args.Kd - kx) / 64) : kQuarters;
        const uint32_t tx = (uint32_t)Cfg::W_BYTES + (uint32_t)(gather ? 4 * g4 : (small ? 8 : T)) * 128u * nq;
        bool ok = true;
        if (lane == 0) {
          ok = !*(volatile int*)&s_abort && mbar_wait_bounded(&empty_bar[slot], phase ^ 1u);
          if (!ok) {
            s_abort = 1;
            record_status(args.status, MOE_ERR_TIMEOUT);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) goto producer_done;
        uint8_t* xs = smem_gen + slot * Cfg::STAGE_BYTES;
        uint8_t* ws = xs + Cfg::X_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full_bar[slot], tx);
          if (TILES) {
            // the stage's two 128-deep tiles are adjacent: one contiguous copy
            const size_t t0 = ((size_t)it.e * n_cb + it.cb) * args.w_kb + 2 * kb;
            bulk_load(ws, args.w_tiles + t0 * (size_t)Cfg::W_SUB_BYTES, (uint32_t)Cfg::W_BYTES, &full_bar[slot]);
          } else {
            tma_load_2d(ws, &tm_w, kx, w_row, &full_bar[slot]);
            tma_load_2d(ws + Cfg::W_SUB_BYTES, &tm_w, kx + kSubK, w_row, &full_bar[slot]);
          }
          if (!gather) {
#pragma unroll
            for (int q = 0; q < kQuarters; ++q)
              tma_load_2d(xs + q * Cfg::X_HALF_BYTES, tmx, kx + 64 * q, it.row0, &full_bar[slot]);
          }
        }
        if (gather) {
          __syncwarp();  // the stage's expected bytes are posted before any gather lands
          if (lane < g4 * nq) {
            const int q = lane / g4, r = lane - q * g4;
            tma_gather4(xs + q * Cfg::X_HALF_BYTES + r * 512, &tm_x, kx + 64 * q, tok, &full_bar[slot]);
          }
        }
        if constexpr (Cfg::PRODUCERS > 1) issued = n;  // n is already past this stage
        else ++issued;
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
  producer_done:
    if (lane == 0) s_issued[q_own] = issued;
  } else if (warp < kConsumerWarps) {
    // ================= MMA consumer warps =================
    // Group grp (8 warps) computes the stages held in ring slots s with
    // s % kGroups == grp (both 64-deep halves); at the item's end both groups add
    // their exact int32 partial sums into the item's sums (shared memory) and go on.
    const int grp = warp / kGroupWarps, wig = warp % kGroupWarps;
    const int warp_m = wig % Cfg::WARPS_M, warp_n = wig / Cfg::WARPS_M;
    const int g = lane >> 2, tq = lane & 3;
    const int pg = mrow_perm(g);
    constexpr uint32_t wflip = TILES ? 0u : 0x80808080u;  // tile bytes hold v + 128
    int* spart = sums + wig * kPartWarp + lane;
    int slot = 0;
    uint32_t phase = 0;
    int consumed = 0, n_items = 0, e_hint = 0;
    bool ok = true;
    for (int j = blockIdx.x; j < total && ok; j += gridDim.x) {
      const Item it = decode_item<T>(j, s_pref, s_end, E, n_cb, e_hint);
      float accf[Cfg::P][Cfg::MT][Cfg::NT][4];
      int acci[Cfg::MT][Cfg::NT][4];
#pragma unroll
      for (int mt = 0; mt < Cfg::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < Cfg::NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int q = 0; q < Cfg::P; ++q) accf[q][mt][nt][i] = 0.0f;
            acci[mt][nt][i] = 0;
          }
      // n8 tiles of this warp that hold real rows (the rest are skipped)
      const int live_nt = min(Cfg::NT, max(0, (it.rows - warp_n * Cfg::NT * 8 + 7) / 8));

      int own = 0;  // stages of this item computed by this group
      for (int kb = 0; kb < nk; ++kb) {
        if (slot % kGroups == grp) {
          ok = !*(volatile int*)&s_abort && mbar_wait_bounded(&full_bar[slot], phase);
          if (!ok) {
            s_abort = 1;
            record_status(args.status, MOE_ERR_TIMEOUT);
            break;
          }
          const uint8_t* xs = smem_gen + slot * Cfg::STAGE_BYTES;
          const uint8_t* ws = xs + Cfg::X_BYTES;
          // one uniform branch per stage on the number of live n8 tiles
          hmma_stage_live<Cfg>(live_nt, xs, ws, wflip, warp_m, warp_n, g, tq, pg, accf);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[slot]);
          ++consumed;
          // drain the exact fp32 chunk (2 own stages x 256 = 512 deep) into int32
          if (++own % 2 == 0) drain_chunk<Cfg>(accf, acci);
        }
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (own % 2 != 0) drain_chunk<Cfg>(accf, acci);
      // ---- hand-off: both groups add their partials into the item's sums
      // (shared-memory atomics, exact and in any order) once the epilogue warps have
      // read and cleared the previous item's, and go on to the next item at once.
      // (When the group that computed an item's last stage also ran its epilogue,
      // the other handing it the partials, an even stage count per item made that
      // the same group every time, and the in-order producer waited on it: the mid
      // workload's GMM1 / GMM2 took 1295 / 726 us, 1224 / 662 us with epilogue warps.)
      if (n_items > 0) {
        bool free = lane == 0 ? wait_part(&part_empty_bar, (n_items - 1) & 1, args.status) : true;
        free = __shfl_sync(0xffffffffu, free ? 1 : 0, 0) != 0;
        ok = ok && free;
      }
      if (ok) {
#pragma unroll
        for (int mt = 0; mt < Cfg::MT; ++mt)
#pragma unroll
          for (int nt = 0; nt < Cfg::NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) atomicAdd(spart + ((mt * Cfg::NT + nt) * 4 + i) * 32, acci[mt][nt][i]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&part_full_bar);
      ++n_items;
    }
    (void)consumed;
  } else {
    // ================= epilogue warps =================
    // Per item: the sums of consumer slices kSlices*ew .. kSlices*ew + kSlices - 1 (the
    // fragments those MMA warps hold) are read and cleared, scaled, converted and
    // staged as [T][128] binary16; then one warp hands each row (256 bytes) to an
    // asynchronous bulk copy to global memory and waits only until the copies have
    // read the staging tile.
    const int ew = warp - kConsumerWarps - Cfg::PRODUCERS;
    const int g = lane >> 2, tq = lane & 3;
    const int pg = mrow_perm(g);
    constexpr int kSlices = kGroupWarps / kEpiWarps;
    static_assert(kGroupWarps % kEpiWarps == 0, "consumer slices per epilogue warp");
    int n_items = 0, e_hint = 0;
    for (int j = blockIdx.x; j < total; j += gridDim.x) {
      const Item it = decode_item<T>(j, s_pref, s_end, E, n_cb, e_hint);
      const float* sc = args.scale + (size_t)it.e * args.N + it.cb * kBN;
      bool got = lane == 0 ? wait_part(&part_full_bar, n_items & 1, args.status) : true;
      got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      if (!got) s_abort = 1;
      // leave together on a failed wait or an abort (the previous item's row copies
      // have read the staging tile once every epilogue warp is past this barrier)
      if (epilogue_bar_or(!got || *(volatile int*)&s_abort)) break;
      __half h[kSlices][Cfg::MT][Cfg::NT][4];
#pragma unroll
      for (int sl = 0; sl < kSlices; ++sl) {
        const int wig = ew * kSlices + sl;
        const int warp_m = wig % Cfg::WARPS_M;
        int* sp = sums + wig * kPartWarp + lane;
#pragma unroll
        for (int mt = 0; mt < Cfg::MT; ++mt) {
          const int m = warp_m * Cfg::MT * 16 + mt * 16 + pg;
          const float s_lo = __ldg(sc + m), s_hi = __ldg(sc + m + 8);
#pragma unroll
          for (int nt = 0; nt < Cfg::NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              int* q = sp + ((mt * Cfg::NT + nt) * 4 + i) * 32;
              const int v = *q;
              *q = 0;
              h[sl][mt][nt][i] = f2h_sat(__fmul_rn(__int2float_rn(v), i < 2 ? s_lo : s_hi));
            }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&part_empty_bar);  // the sums are read and cleared
      {
#pragma unroll
        for (int sl = 0; sl < kSlices; ++sl) {
          const int wig = ew * kSlices + sl;
          const int warp_m = wig % Cfg::WARPS_M, warp_n = wig / Cfg::WARPS_M;
#pragma unroll
          for (int mt = 0; mt < Cfg::MT; ++mt) {
            const int m = warp_m * Cfg::MT * 16 + mt * 16 + pg;
#pragma unroll
            for (int nt = 0; nt < Cfg::NT; ++nt) {
              const int n = warp_n * Cfg::NT * 8 + nt * 8 + 2 * tq;
              stile[n * kBN + m] = h[sl][mt][nt][0];
              stile[(n + 1) * kBN + m] = h[sl][mt][nt][1];
              stile[n * kBN + m + 8] = h[sl][mt][nt][2];
              stile[(n + 1) * kBN + m + 8] = h[sl][mt][nt][3];
            }
          }
        }
      }
      fence_proxy_async_smem();  // the tile's writes before the bulk copies read it
      epilogue_bar();
      if (ew == 0) {
        // row r < rows (<= T <= 32) by lane r: N and the channel block are multiples
        // of 128, so both ends of every row copy are 16-byte aligned
        if (lane < it.rows)
          bulk_store(args.C + (size_t)(it.row0 + lane) * args.N + it.cb * kBN, stile + lane * kBN, kBN * 2);
        bulk_commit_group();
        bulk_wait_read_all();  // the tile is free for the next item
      }
      ++n_items;
    }
    bulk_wait_all();  // every row copy this thread issued has landed
  }

  __syncthreads();
  if (s_abort && threadIdx.x == kConsumerWarps * 32) {
    // let loads still in flight land before the CTA's shared memory is released: each
    // producer's last S / PRODUCERS issued stages are the latest phase of its slots
    // (with one producer, s_issued counts its stages, which are all of them in order)
    for (int q = 0; q < Cfg::PRODUCERS; ++q) {
      const int last = s_issued[q] - 1;  // -1: nothing issued
      for (int n = last; n >= 0 && n > last - S; n -= Cfg::PRODUCERS)
        mbar_wait_bounded(&full_bar[n % S], (uint32_t)((n / S) & 1));
    }
  }
}

// ------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------
template <int T, bool GATHER, bool TILES>
cudaError_t launch_t(const GroupedGemmProblem& p, cudaStream_t stream) {
  using Cfg = GemmCfg<T>;
  CUtensorMap tw, tx;
  if (!encode_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w, (uint64_t)p.Kd, (uint64_t)p.E * p.N, kSubK,
                            kBN))
    return cudaErrorInvalidValue;
  // token operand: tiled boxes of T and 8 rows, or (gathering) one-row boxes over the
  // token rows, passed in both slots
  CUtensorMap tx8;
  constexpr bool gather = GATHER;
  if (!encode_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.act, (uint64_t)p.Kd, (uint64_t)p.act_rows, 64,
                            gather ? 1 : T) ||
      !encode_tensor_map_2d(&tx8, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.act, (uint64_t)p.Kd, (uint64_t)p.act_rows, 64,
                            gather ? 1 : 8))
    return cudaErrorInvalidValue;
  static PerContextOnce attr_set;
  const int dev = current_device();
  if (attr_set.needed(dev)) {
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<T, GATHER, TILES>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    attr_set.done(dev);
  }
  GemmArgs a;
  a.cumsum = p.cumsum;
  a.scale = p.scale;
  a.C = reinterpret_cast<__half*>(p.C);
  a.status = p.status;
  a.E = p.E;
  a.N = p.N;
  a.Kd = p.Kd;
  a.split_rows = p.split_rows;
  a.min_rows = p.min_rows;
  a.gather_route = p.gather_route;
  a.topK = p.topK;
  a.w_tiles = TILES ? reinterpret_cast<const uint8_t*>(p.w) : nullptr;
  a.w_kb = p.w_kb;
  grouped_gemm_kernel<T, GATHER, TILES><<<sm_count(), Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(tw, tx, tx8, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm_hmma(const GroupedGemmProblem& p, int T, cudaStream_t stream) {
  const bool g = p.gather_route != nullptr;
  if (p.w_kb) {
    if (T == 32) return g ? launch_t<32, true, true>(p, stream) : launch_t<32, false, true>(p, stream);
    return g ? launch_t<16, true, true>(p, stream) : launch_t<16, false, true>(p, stream);
  }
  if (T == 32) return g ? launch_t<32, true, false>(p, stream) : launch_t<32, false, false>(p, stream);
  return g ? launch_t<16, true, false>(p, stream) : launch_t<16, false, false>(p, stream);
}

}  // namespace moe
