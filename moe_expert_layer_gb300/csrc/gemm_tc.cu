// Grouped W8A8 GEMM of the expert layer on the 5th-generation tensor cores
// (tcgen05), run by CTA pairs.  PTO-ISA MegaMoE operator page, sections "3. GMM1"
// and "5. GMM2".
//
// For expert e with rows [cumsum[e]-cnt_e, cumsum[e]) of the expert-major row
// space and every output channel n < N:
//     acc        = sum_k a[row][k] * W[e][n][k]          exact integer
//     C[row][n]  = sat_f16(float(acc) * scale[e][n])
//
// Exact integers on the fp16 tensor path.  GB300 executes int8 tensor MMAs
// and dp4a far below its binary16 rate, so the int8 operands are multiplied as
// binary16 (every int8 value, and every product |p| <= 128^2, is exact) with
// fp32 accumulation in tensor memory.  An fp32 sum of integers is exact while
// every partial sum stays within 2^24 in magnitude, so the reduction runs in
// chunks of 1024 (1024 * 128 * 128 = 2^24); after each chunk the drain warps read
// the fp32 accumulator, convert it to int32 and add it to per-thread int32 sums.
// The result is the exact integer dot product for any K.
//
// CTA pairs.  One tcgen05.mma of M = 256 costs ~92 cycles for any N <= 128 and
// 128 cycles at N = 256 (measured on GB300); at N = 256 changing the operand
// addresses between MMAs is free.  The issuing thread, however, is the limit:
// a tcgen05.commit holds it ~700 cycles while the MMA queue covers only ~500
// cycles of work, so with one commit per 8 MMAs a stage of 8 N = 256 MMAs took
// ~1210 cycles instead of 1024, and with one per 16 MMAs the pipe ran at its full
// 128 cycles per MMA (a one-thread issue loop measured on GB300).  So two CTAs of a
// cluster issue MMAs of M = 256, N = 256 (cta_group::2), one commit per 256-deep
// stage (16 MMAs): each CTA contributes 128 weight channels (operand A, in its own
// tensor memory) and half of the N token rows (operand B, in its own shared
// memory), and receives the 128 x N block of its channels in its tensor memory.
// A work item is (expert, 256-channel block, row tile of up to 256 rows); N is the
// tile's rows rounded up to 32 (the experts' rows are cut into balanced tiles).
//   - Weights stay int8 in HBM (they are the dominant traffic at small batches).
//     They arrive in k-blocks: a TMA box (or one 16 KiB tile) of 128 channels x
//     128 k in shared memory (128-byte swizzle), two per stage; converter warps read
//     one channel row per thread, widen 4 int8 to 4 binary16 with a byte permute
//     into the 1024+v encoding and one subtract, and store the row into the stage's
//     tensor-memory A buffer (tcgen05.st, 32x32b).
//   - Activations are binary16-coded int8 in expert-major rows (written so by the
//     quant-scatter and SwiGLU kernels), loaded by TMA as four [128][64] tiles per
//     stage in the canonical K-major 128-byte-swizzled layout the MMA reads
//     through a shared-memory descriptor.
//   - Tensor memory: the accumulator (256 columns) and two A buffers (128 columns
//     each).  The token ring and the A buffers have the same two slots, so one
//     commit per stage frees both; converters and the token producer refill a slot
//     while the MMAs of the other one (2048 cycles at N = 256) run.
//   - The MMA issuer cannot run far ahead of the tensor pipe (a stage completes
//     ~500 cycles after its last MMA is issued), so its per-stage work is kept to
//     one barrier wait and one commit: the stage's readiness (both CTAs' token
//     halves and A buffers) is gathered on one barrier in CTA 0, and the operand
//     descriptors of the stage's MMAs are one base plus constants.
//
// Roles (one persistent pair per two SMs, work items strided over the pairs):
//   warp 0      TMA producer of the weight ring (freed by the converters as soon
//               as they hold the stage in registers)
//   warp 1      tensor-memory allocation (both CTAs); in CTA 0 of the pair one
//               thread issues the pair's tcgen05.mma and commits
//   warp 2      TMA producer of the token ring
//   warp 3      relay: tells CTA 0's stage barrier when this CTA's token stage has landed
//   warps 4-7   converters (warp w owns TMEM lanes 32*(w%4) .. +31)
//   warps 8-23  drain + epilogue: warp w reads TMEM lanes 32*(w%4).. and the 64
//               accumulator columns 64*((w-8)/4) ..; each thread keeps 64 int32
//               sums, so the warpgroups rebalance registers (setmaxnreg) from the
//               single-lane roles and the converters to the drains.
// CTA 1 signals readiness of its A buffers, token stages and drained accumulator
// to barriers in CTA 0 (remote mbarrier arrives); the MMA commits arrive on the
// barriers of both CTAs (multicast).  Every wait on an mbarrier is bounded; a wait
// that gives up sets the status word to MOE_ERR_TIMEOUT and the CTA winds down
// (in-flight copies and MMAs are waited for, the pair synchronises, tensor memory
// is freed) before returning.
#include "common.cuh"
#include "kernels.h"
#include "swiglu.cuh"
#include "tensor_map.h"

namespace moe {

#ifdef MOE_GEMM_PROFILE
static unsigned long long* g_gemm_prof = nullptr;
extern "C" void moe_gemm_profile_set(void* p) { g_gemm_prof = static_cast<unsigned long long*>(p); }
#endif

namespace {

constexpr int kThreads = 768;
constexpr int kLaunchRegs = 80;     // registers per thread at launch (65536 / 768, rounded to 8)
constexpr int kRegsSingle = 40;     // warpgroup 0: producers, MMA issuer, relay
constexpr int kRegsConv = 56;       // warpgroup 1: converters
constexpr int kRegsDrain = 96;      // warpgroups 2-5: drains
static_assert(128 * kRegsSingle + 128 * kRegsConv + 512 * kRegsDrain <= kThreads * kLaunchRegs,
              "register split exceeds the registers the CTA is launched with");
constexpr int kBM = 128;            // weight channels per CTA
constexpr int kPairCh = 256;        // weight channels per pair (MMA M)
constexpr int kBK = 128;            // reduction depth of a k-block (one weight tile / TMA box pair)
constexpr int kKBlocks = 2;         // k-blocks per pipeline stage: one commit per 16 MMAs
constexpr int kTileRows = 256;      // token rows per work item (MMA N <= 256)
constexpr int kHalfRows = kTileRows / 2;  // token rows per CTA (TMA box height)
constexpr int kTmemCols = 512;      // accumulator [0, 256), A buffers 256 + 128*slot
constexpr int kACol0 = 256;
constexpr int kACols = kKBlocks * kBK / 2;  // binary16 pairs per 32-bit column: 128 columns per stage
constexpr int kMaxExperts = 1024;
constexpr int kStages = 2;          // token ring = A buffers (256-deep stages), freed by one commit per stage
constexpr int kWStages = 4;         // weight ring of k-blocks, freed after conversion
constexpr int kWBytes = kBM * kBK;  // [128][128] int8, 128-B swizzled rows
constexpr int kXHalfBytes = kHalfRows * 128;  // one token box: [128 rows][64] binary16, 128-B swizzled rows
constexpr int kXBlockBytes = 2 * kXHalfBytes;  // a k-block of tokens
constexpr int kXBytes = kKBlocks * kXBlockBytes;  // a stage of tokens (4 boxes)
static_assert(kXHalfBytes % 1024 == 0, "1024-B alignment of swizzled tiles");
static_assert(kBM == kWTileRows && kBK == kWTileDepth && kWBytes == kWTileBytes, "a weight stage is one tile");
constexpr int kSmemBytes = kWStages * kWBytes + kStages * kXBytes + 1024;
constexpr int kWProducerWarp = 0, kMmaWarp = 1, kXProducerWarp = 2, kRelayWarp = 3, kConvWarp0 = 4,
              kNumConvWarps = 4, kDrainWarp0 = 8, kNumDrainWarps = 16;
static_assert(kThreads == 32 * (kDrainWarp0 + kNumDrainWarps), "warp roles");
static_assert(kDrainWarp0 % 4 == 0 && kNumDrainWarps % 4 == 0, "drain warps: whole sets of the 4 SM sub-partitions");
static_assert(kSmemBytes + 15 * 1024 <= 227 * 1024, "shared memory (dynamic + ~14.3 KB static)");
static_assert(kACol0 + kStages * kACols == kTmemCols, "tensor memory: accumulator + A buffers");
// kind::f16 instruction descriptor: D f32, A/B f16, both K-major, M = 256; N is set per item
constexpr uint32_t kIdescBase = (1u << 4) | ((uint32_t)(256 >> 4) << 24);

struct Args {
  const int32_t* cumsum;
  const float* scale;
  __half* C;
  int32_t* status;
  int E, N, Kd;
  int split_rows;  // this engine serves the experts with more than split_rows rows
  const int32_t* bounds;  // [E][kBoundSegments] activation bounds, or null (1024-deep chunks)
  const int32_t* gather_route;  // null: tiled token boxes; else row d gathers token gather_route[d] / topK
  int topK;
  const uint8_t* w_tiles;  // null: weights through the tensor map; else the tile layout
  int w_kb;                // tiles per 128-channel block of the tile layout
  // SwiGLU fused into GMM1 (sw_q2 null: a plain grouped GEMM); see the drain role
  const float* sw_pts1;          // [M] token scales
  const int32_t* sw_sorted;      // [R] route of each expanded row
  __half* sw_q2;                 // [R][N/2] binary16 codes
  float* sw_pts2;                // [R]
  int32_t* sw_bounds;            // [E][kBoundSegments] or null
  int32_t* sw_done;              // [E] stored-item counters, zero at launch
#ifdef MOE_GEMM_PROFILE
  unsigned long long* prof;
#endif
};

// ------------------------------------------------------------------ SwiGLU fused into GMM1
// With args.sw_q2 set (GMM1 of a tiled operand) the drain warps also run SwiGLU +
// requant, one expanded row per warp at a time, on the rows of experts all of whose
// GMM1 items are stored.  Every drain warp counts each item it has finished (its
// epilogue stores fenced first) on the item's expert; an expert is complete at
// kSwigluCountPerItem * (its items), so the experts the warp-MMA engine served before
// this launch (no items here) are complete from the start.  Row warp gw of the grid
// owns rows gw, gw + W, ... (W = all row warps), taken in order: between items, while
// the next accumulator chunk is not ready, it requantises its next rows as far as
// their experts are complete; after its last item it finishes its rows, waiting
// (bounded) for their experts.  No wait ever depends on a CTA that is not already
// running: the pairs launch only when all of them can be resident at once (the host
// checks the occupancy).  The arithmetic is swiglu.cuh's, as in the SwiGLU kernel:
// the same bits.
constexpr int kSwigluMaxVpl = 6;                     // 16-byte vectors per lane of a row's half
constexpr int kSwigluRegI = kSwigluMaxVpl * 32 * 8;  // I <= 1536: the row stays in registers
constexpr int kSwigluCountPerItem = 2 * 16;          // drain warps of a pair

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// SwiGLU + requant of expanded row d (expert e) by one warp: the row's gate and up
// halves (C1, written by other CTAs: read through L2) in registers, max |y| across
// the warp, then the codes, pts2 and the row's segment sums of |q|.  y is computed
// twice from the loaded halves (for the max, then for the codes) rather than kept:
// the same instructions on the same inputs give the same values, and the drain warps'
// registers hold the row only once.
union SwVec {
  int4 v;
  __half h[8];
};

// Rows longer than the registers hold (I > 1536): the row is read twice (the second
// time from L2), 128 vectors at a time, one 1024-deep bound segment per pass.
__device__ __noinline__ void swiglu_long_row_warp(const Args& a, int d, int e, int lane, float p1) {
  const int I = a.N >> 1, nvec = I >> 3;
  const int4* gate = reinterpret_cast<const int4*>(a.C + (size_t)d * a.N);
  const int4* up = gate + nvec;
  constexpr int kVpl = kBoundSegment / 8 / 32;  // 4 vectors per lane: one segment
  float amax = 0.0f;
#pragma unroll 1
  for (int v0 = 0; v0 < nvec; v0 += 32 * kVpl) {
    SwVec g[kVpl], u[kVpl];
#pragma unroll
    for (int i = 0; i < kVpl; ++i) {
      const int v = v0 + lane + 32 * i;
      g[i].v = v < nvec ? __ldcg(gate + v) : make_int4(0, 0, 0, 0);
      u[i].v = v < nvec ? __ldcg(up + v) : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kVpl; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(swiglu_y(g[i].h[j], u[i].h[j], p1)));
  }
  amax = warp_max(amax);
  const float inv = swiglu_inv(amax);
  if (lane == 0) a.sw_pts2[d] = swiglu_pts2(amax, p1);
  int4* q2 = reinterpret_cast<int4*>(a.sw_q2 + (size_t)d * I);
#pragma unroll 1
  for (int v0 = 0, seg = 0; v0 < nvec; v0 += 32 * kVpl, ++seg) {
    SwVec g[kVpl], u[kVpl];
#pragma unroll
    for (int i = 0; i < kVpl; ++i) {
      const int v = v0 + lane + 32 * i;
      g[i].v = v < nvec ? __ldcg(gate + v) : make_int4(0, 0, 0, 0);
      u[i].v = v < nvec ? __ldcg(up + v) : make_int4(0, 0, 0, 0);
    }
    int l1 = 0;
#pragma unroll
    for (int i = 0; i < kVpl; ++i) {
      const int v = v0 + lane + 32 * i;
      if (v < nvec) {
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) y[j] = swiglu_y(g[i].h[j], u[i].h[j], p1);
        int l = 0;
        q2[v] = swiglu_codes8(y, inv, &l);
        l1 += l;
      }
    }
    if (a.sw_bounds) {
      const int sum = __reduce_add_sync(0xffffffffu, l1);
      if (lane == 0) atomicMax(a.sw_bounds + (size_t)e * kBoundSegments + seg, sum);
    }
  }
}

__device__ __forceinline__ void swiglu_row_warp(const Args& a, int d, int e, int lane) {
  const int I = a.N >> 1, nvec = I >> 3;
  const int4* gate = reinterpret_cast<const int4*>(a.C + (size_t)d * a.N);
  const int4* up = gate + nvec;
  const float p1 = __ldg(a.sw_pts1 + __ldg(a.sw_sorted + d) / a.topK);
  if (I > kSwigluRegI) {
    swiglu_long_row_warp(a, d, e, lane, p1);
    return;
  }
  using V = SwVec;
  V g[kSwigluMaxVpl], u[kSwigluMaxVpl];
#pragma unroll
  for (int i = 0; i < kSwigluMaxVpl; ++i) {
    const int v = lane + 32 * i;
    g[i].v = v < nvec ? __ldcg(gate + v) : make_int4(0, 0, 0, 0);
    u[i].v = v < nvec ? __ldcg(up + v) : make_int4(0, 0, 0, 0);
  }
  float amax = 0.0f;  // zero vectors past the row give y = 0
#pragma unroll
  for (int i = 0; i < kSwigluMaxVpl; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(swiglu_y(g[i].h[j], u[i].h[j], p1)));
  amax = warp_max(amax);
  const float inv = swiglu_inv(amax);
  if (lane == 0) a.sw_pts2[d] = swiglu_pts2(amax, p1);
  int4* q2 = reinterpret_cast<int4*>(a.sw_q2 + (size_t)d * I);
  int seg0 = 0, seg1 = 0;  // sums of |q| of the two 1024-deep segments I <= 1536 spans
#pragma unroll
  for (int i = 0; i < kSwigluMaxVpl; ++i) {
    const int v = lane + 32 * i;
    if (v < nvec) {
      float y[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) y[j] = swiglu_y(g[i].h[j], u[i].h[j], p1);
      int l1 = 0;
      q2[v] = swiglu_codes8(y, inv, &l1);
      if (v * 8 < kBoundSegment) seg0 += l1; else seg1 += l1;
    }
  }
  if (a.sw_bounds) {
    const int s0 = __reduce_add_sync(0xffffffffu, seg0), s1 = __reduce_add_sync(0xffffffffu, seg1);
    if (lane == 0) {
      atomicMax(a.sw_bounds + (size_t)e * kBoundSegments, s0);
      if (I > kBoundSegment) atomicMax(a.sw_bounds + (size_t)e * kBoundSegments + 1, s1);
    }
  }
}

// Role timing, compiled in only with -DMOE_GEMM_PROFILE: each role sums clock64()
// intervals (time in a wait, time doing its work) into registers and adds them to
// a 32-slot device buffer at the end.  Slot bases: weight producer 0, token producer
// 2, relay 4, MMA issuer 8 (8-15: accumulator wait, stage wait, issue, commit, stage
// body, set-up, item decode, final wait), converters 16, drains 24, issuer's total 31.
#ifdef MOE_GEMM_PROFILE
#define PROF_REGS unsigned long long _pf[8] = {0, 0, 0, 0, 0, 0, 0, 0}
#define PROF_WAIT(i, expr) ([&]() { const long long _t0 = clock64(); const bool _r = (expr); \
                                    _pf[i] += clock64() - _t0; return _r; }())
#define PROF_T0(v) const long long v = clock64()
#define PROF_ADD(i, t0) (_pf[i] += clock64() - (t0))
#define PROF_FLUSH(base) for (int _i = 0; _i < 8; ++_i) if (_pf[_i]) atomicAdd(args.prof + (base) + _i, _pf[_i])
#define PROF_TOTAL(t0) atomicAdd(args.prof + 31, (unsigned long long)(clock64() - (t0)))
#else
#define PROF_REGS
#define PROF_WAIT(i, expr) (expr)
#define PROF_T0(v)
#define PROF_ADD(i, t0)
#define PROF_FLUSH(base)
#define PROF_TOTAL(t0)
#endif

// ------------------------------------------------------------------ cluster / tcgen05 helpers
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Arrive on a barrier given by its shared::cluster address (either CTA of the pair).
// Default semantics: an arrive with cluster-scope release costs ~320 cycles on
// GB300, this one ~6; the data it publishes is tensor memory (ordered by
// tcgen05.wait + tcgen05.fence) or TMA-written shared memory whose barrier the
// signalling thread has already seen complete.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t caddr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}

template <uint32_t kRegs>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs)); }
template <uint32_t kRegs>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs)); }

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

// D[256 x N] (+)= A[256 x 16] * B[N x 16]^T over the pair: A rows 0-127 from this
// CTA's tensor memory, 128-255 from the peer's; B rows split N/2 + N/2 likewise.
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` in both CTAs of the pair once the MMAs issued so far complete.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void mma_commit_local(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
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
// subtracting 1152 leaves v.  kFlip = 0x80808080 takes two's-complement bytes
// (v+128 = v ^ 0x80); kFlip = 0 takes bytes already stored as v+128 (the weight
// tiles), one instruction less per word.
template <uint32_t kFlip>
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ kFlip;
  const uint32_t a = __byte_perm(u, 0x6464u, 0x5140u);
  const uint32_t b = __byte_perm(u, 0x6464u, 0x5342u);
  const uint32_t bias = 0x64806480u;  // half2(1152, 1152)
  asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

// Exact int32 of an integer-valued fp32 v with |v| <= 2^24, on the FMA and integer
// pipes: v = 4096*hi + lo with hi = rint(v / 4096) and |lo| <= 2048, each part
// read off the mantissa after adding 1.5 * 2^23 (all steps exact in fp32).  The
// drains convert two of every three values this way and the rest with cvt.rni
// (whose ~16 conversions per cycle per SM alone would set the drain time).
__device__ __forceinline__ int f2i_exact(float v) {
  const float kMagic = 12582912.0f;  // 1.5 * 2^23
  const float h = __fmaf_rn(v, 1.0f / 4096.0f, kMagic);
  const float hi = __fsub_rn(h, kMagic);
  const float lo = __fmaf_rn(-hi, 4096.0f, v);
  const float l = __fadd_rn(lo, kMagic);
  return (int)(((uint32_t)__float_as_int(h) << 12) + (uint32_t)__float_as_int(l) -
               ((0x4B400000u << 12) + 0x4B400000u));
}

struct Item {
  int e, cb, row0, rows, n_mma;
};

// Stages per exact chunk for expert e.  Without bounds 8 (1024 deep: every partial
// sum within 1024 * 128 * 128 = 2^24).  With bounds, the longest run of L whole
// 1024-deep segments such that every aligned run's bound sum B satisfies
// 128 * B <= 2^24, which keeps every partial sum of every row of the expert exact.
__device__ __forceinline__ int chunk_stages(const int32_t* bounds, int e, int nk) {
  constexpr int kStagesPerSegment = kBoundSegment / kBK;
  if (!bounds) return kStagesPerSegment;
  const int32_t* b = bounds + (size_t)e * kBoundSegments;
  const int nseg = (nk + kStagesPerSegment - 1) / kStagesPerSegment;
  for (int L = nseg; L > 1; --L) {
    bool ok = true;
    for (int s0 = 0; s0 < nseg && ok; s0 += L) {
      long long sum = 0;
      for (int s = s0; s < min(nseg, s0 + L); ++s) sum += __ldg(b + s);
      ok = sum * 128 <= (1ll << 24);
    }
    if (ok) return L * kStagesPerSegment;
  }
  return kStagesPerSegment;
}

// Work items on the pairs: (expert, channel block, row tile), for the experts with
// more than split_rows rows (the warp-MMA engine takes the others), expert-major,
// then channel block, then row tile, so that pairs working at the same time share
// each weight block through L2 and experts complete in order (the fused SwiGLU
// needs all of an expert's tiles).  An expert of cnt rows is cut into
// t = ceil(cnt / 256) row tiles of two sizes that are multiples of 32 rows, a and
// a + 32 (the larger ones first, as few as cover cnt), each run with MMA N = its rows
// rounded up to 32.  A tcgen05.mma costs about the same for any N up to 128 and grows
// with N above (96 cycles at N = 192, 128 at 256), so 795 rows as 224 + 192 + 192 +
// 187 take ~16% less tensor time than 256 + 256 + 256 + 27 (whose short tile costs
// nearly a full one); over the prefill and skewed routings, 6-7% less.
__device__ __forceinline__ int row_tiles(int cnt, int split_rows) {
  return cnt <= split_rows ? 0 : (cnt + kTileRows - 1) / kTileRows;
}

// Items of an expert with cnt rows on the pairs (all channel blocks).
__device__ __forceinline__ int expert_items(int cnt, int split_rows, int n_cb) {
  return n_cb * row_tiles(cnt, split_rows);
}

struct WorkList {
  const int* pref;  // first work item of each expert; pref[E] = their number
  const int* end;   // cumsum
  const int* tile;  // row tiles of each expert: a | k << 16 (k tiles of a + 32 rows, then a rows)
  int n_cb, E;
  bool pow2_n;      // MMA N a power of two (the gathering token producer deals 4-row groups
                    // of a half tile over the 32 lanes, which needs N / 8 to divide 32)
};

// The row tiling of an expert with cnt rows: t = row_tiles(cnt) tiles, a = 32 *
// floor(cnt / (32 t)) rows each, the first k of them 32 rows more (k < t unless a
// tile of a rows would leave rows out; the last tile holds what is left).
__device__ __forceinline__ int tile_plan(int cnt, int t) {
  if (t == 0) return 0;
  const int a = 32 * (cnt / (32 * t));
  const int k = (cnt - t * a + 31) / 32;
  return a | (k << 16);
}

// Work item j -> (expert, channel block, first row, rows, MMA N): the last expert
// whose first item is <= j (experts without items leave the prefix flat and are
// skipped).  A role's items only move forward, so the search starts at its previous
// item's expert (e_hint): the next four prefixes are read at once, and a binary
// search covers longer jumps.
__device__ __forceinline__ Item decode_item(int j, const WorkList& wl, int& e_hint) {
  Item it;
  int lo = e_hint, c = 0;
#pragma unroll
  for (int step = 1; step <= 4; ++step) c += wl.pref[min(lo + step, wl.E)] <= j ? 1 : 0;  // pref[E] > j
  lo += c;
  if (c == 4) {
    int hi = wl.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (wl.pref[mid] <= j) lo = mid; else hi = mid;
    }
  }
  e_hint = lo;
  const int start = lo ? wl.end[lo - 1] : 0;
  const int cnt = wl.end[lo] - start;
  const int n_rt = row_tiles(cnt, -1);
  const int a = wl.tile[lo] & 0xffff, k = wl.tile[lo] >> 16;
  const int local = j - wl.pref[lo];
  const int cb = local / n_rt, rt = local - cb * n_rt;
  const int row = rt < k ? rt * (a + 32) : k * (a + 32) + (rt - k) * a;
  it.e = lo;
  it.cb = cb;
  it.row0 = start + row;
  it.rows = min(rt < k ? a + 32 : a, cnt - row);
  it.n_mma = wl.pow2_n ? (it.rows <= 32 ? 32 : 1 << (32 - __clz(it.rows - 1)))  // 32, 64, 128 or 256
                      : (it.rows + 31) & ~31;                                  // N in steps of 32
  return it;
}

// try_wait that lets the warp sleep in hardware until the phase completes (up to
// `hint_ns`), instead of re-issuing probes that take issue slots from the MMA warp.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait: false after about two seconds of %globaltimer.
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint64_t* bar, uint32_t parity) {
  constexpr uint32_t kHintNs = 100000;
  if (mbar_try_wait_sleep(bar, parity, kHintNs)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait_sleep(bar, parity, kHintNs)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;  // fast path: one probe of a completed phase
  if (*abort_flag) return false;
  if (mbar_wait_sleep_bounded(bar, parity)) return true;
  *abort_flag = 1;
  record_status(status, MOE_ERR_TIMEOUT);
  return false;
}

// GATHER: token rows gathered by index (args.gather_route) instead of tiled boxes of
// expert-major rows; a separate instantiation, so the tiled kernel carries none of it.
// FUSE: kFuseNone, or kFuseSwiglu (GMM1 with SwiGLU: args.sw_*), each its own
// instantiation, so the plain kernel's drains carry none of the SwiGLU state (its
// register spills went from 28 to 4 bytes).
// TILES: the weights come as tiles (args.w_tiles), whose bytes hold v + 128; else
// through the tensor map as two's-complement int8.
enum { kFuseNone = 0, kFuseSwiglu = 1 };
template <bool GATHER, int FUSE, bool TILES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                             const Args args) {
  constexpr bool kSw = FUSE == kFuseSwiglu;
  constexpr uint32_t kWFlip = TILES ? 0u : 0x80808080u;
  static_assert(!(GATHER && FUSE != kFuseNone), "fusion runs on the tiled operand");
  constexpr int S = kStages, SW = kWStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t wfull_bar[SW], wempty_bar[SW], xfull_bar[S], ready_bar[S], sdone_bar[S];
  __shared__ __align__(8) uint64_t accfull_bar, accempty_bar, final_bar;
  __shared__ int s_pref[kMaxExperts + 1];
  __shared__ int s_end[kMaxExperts];
  __shared__ short s_chunk[kMaxExperts];  // stages per exact chunk of each expert
  __shared__ int s_tile[kMaxExperts];     // row tiling of each expert (WorkList::tile)
  __shared__ int s_wsum[kThreads / 32];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_w_issued, s_x_issued;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int E = args.E, n_cb = (args.N + kPairCh - 1) / kPairCh;
  const int nk = (args.Kd + kBK - 1) / kBK;  // k-blocks; a 64-deep tail reads TMA zero fill
  const int nst = (nk + kKBlocks - 1) / kKBlocks;  // pipeline stages per work item
  PROF_T0(t_start);
  PROF_REGS;
  volatile int* abort_flag = &s_abort;

  // ---- work list (s_pref[e] = first work item of expert e), barriers, tensor memory
  {
    const int per = (E + kThreads - 1) / kThreads;
    const int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
    int local = 0;  // work items of this thread's experts
    for (int e = e0; e < e1; ++e) {
      const int hi = __ldg(args.cumsum + e), lo = e ? __ldg(args.cumsum + e - 1) : 0;
      s_end[e] = hi;
      s_chunk[e] = (short)chunk_stages(args.bounds, e, nk);
      const int nt = row_tiles(hi - lo, args.split_rows);
      s_tile[e] = tile_plan(hi - lo, nt);
      local += nt * n_cb;
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
      // all 512 tensor-memory columns of both SMs (one pair per two SMs)
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                   "n"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
      if (lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_x);
        for (int s = 0; s < SW; ++s) {
          mbar_init(&wfull_bar[s], 1);
          mbar_init(&wempty_bar[s], kNumConvWarps);
        }
        for (int s = 0; s < S; ++s) {
          mbar_init(&xfull_bar[s], 1);
          mbar_init(&sdone_bar[s], 1);
          // CTA 0: both relays + both CTAs' converter warps
          mbar_init(&ready_bar[s], 2 + 2 * kNumConvWarps);
        }
        mbar_init(&accfull_bar, 1);
        mbar_init(&accempty_bar, 2 * kNumDrainWarps);
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
      run += row_tiles(s_end[e] - lo, args.split_rows) * n_cb;
    }
    if (e0 < E && e1 == E) s_pref[E] = run;
  }
  __syncthreads();
  cluster_sync_all();  // the peer's barriers and tensor memory are ready
  tc_fence_after();
  PROF_ADD(5, t_start);
  WorkList wl;
  wl.pref = s_pref;
  wl.end = s_end;
  wl.tile = s_tile;
  wl.n_cb = n_cb;
  wl.E = E;
  wl.pow2_n = GATHER;
  const int total = s_pref[E];
  const uint32_t tmem = s_tmem;

  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem_base - smem_u32(smem_raw));
  const uint32_t w_ring = smem_base;                  // SW x [128][128] int8
  const uint32_t x_ring = smem_base + SW * kWBytes;   // S x 4 x [128][64] binary16

  if (warp < kConvWarp0) {
    regs_dec<kRegsSingle>();
    if (warp == kWProducerWarp) {
      // ======================= weight producer (one lane) =======================
      if (lane == 0) {
        int n = 0;
        int e_hint = 0;
        for (int j = pair; j < total; j += npairs) {
          const Item it = decode_item(j, wl, e_hint);
          const int w_row = it.e * args.N + it.cb * kPairCh + (int)rank * kBM;
          // tile layout: this CTA's 128-channel block, its tiles in reduction order.  A
          // block past the expert's channels (N % 256 == 128, second CTA of the last
          // channel block) reads the expert's last block instead: finite int8 values
          // whose output channels are never stored, and never a tile past the buffer.
          const uint8_t* wt = nullptr;
          if (TILES) {
            const int nbk = args.N / kBM;
            const int nb = min(it.cb * (kPairCh / kBM) + (int)rank, nbk - 1);
            wt = args.w_tiles + ((size_t)it.e * nbk + nb) * (size_t)args.w_kb * kWBytes;
          }
          for (int kb = 0; kb < nk; ++kb, ++n) {
            const int slot = n % SW;
            if (!PROF_WAIT(0, wait_or_abort(&wempty_bar[slot], ((n / SW) & 1) ^ 1, abort_flag, args.status)))
              goto w_done;
            mbar_arrive_expect_tx(&wfull_bar[slot], (uint32_t)kWBytes);
            if (wt)
              bulk_load(smem_gen + slot * kWBytes, wt + (size_t)kb * kWBytes, (uint32_t)kWBytes, &wfull_bar[slot]);
            else
              tma_load_2d(smem_gen + slot * kWBytes, &tm_w, kb * kBK, w_row, &wfull_bar[slot]);
          }
        }
      w_done:
        s_w_issued = n;
        PROF_FLUSH(0);
      }
    } else if (warp == kXProducerWarp) {
      // ======================= token producer =======================
      // This CTA's half of the item's N rows (hr = N/2), as [hr][64] boxes: two per
      // k-block, up to four per stage.  Tiled: lane 0 loads 128-row boxes of the
      // expert-major operand.  Gathered: the half's 4-row groups (G = hr/4 of them)
      // are gathered by token index, lane l issuing group l % G of the boxes
      // (l / G) mod (32 / G) + 32 / G * i; rows past the item's last real row repeat
      // that row's token (their outputs are never stored).
      int n = 0;
      if (!GATHER) {
        if (lane == 0) {
          int e_hint = 0;
          for (int j = pair; j < total; j += npairs) {
            const Item it = decode_item(j, wl, e_hint);
            const int y = it.row0 + (int)rank * (it.n_mma >> 1);
            for (int st = 0; st < nst; ++st, ++n) {
              const int slot = n % S;
              const int nbox = 2 * min(kKBlocks, nk - st * kKBlocks);
              if (!PROF_WAIT(0, wait_or_abort(&sdone_bar[slot], ((n / S) & 1) ^ 1, abort_flag, args.status)))
                goto x_done;
              uint8_t* xs_g = smem_gen + SW * kWBytes + slot * kXBytes;
              mbar_arrive_expect_tx(&xfull_bar[slot], (uint32_t)(nbox * kXHalfBytes));
              for (int b = 0; b < nbox; ++b)
                tma_load_2d(xs_g + b * kXHalfBytes, &tm_x, st * kKBlocks * kBK + 64 * b, y, &xfull_bar[slot]);
            }
          }
        }
      } else {
        int e_hint = 0;
        for (int j = pair; j < total; j += npairs) {
          const Item it = decode_item(j, wl, e_hint);
          const int hr = it.n_mma >> 1;
          const int G = hr >> 2;
          const int r0 = it.row0 + (int)rank * hr + 4 * (lane % G), last = it.row0 + it.rows - 1;
          int4 tok;
          tok.x = __ldg(args.gather_route + min(r0, last)) / args.topK;
          tok.y = __ldg(args.gather_route + min(r0 + 1, last)) / args.topK;
          tok.z = __ldg(args.gather_route + min(r0 + 2, last)) / args.topK;
          tok.w = __ldg(args.gather_route + min(r0 + 3, last)) / args.topK;
          for (int st = 0; st < nst; ++st, ++n) {
            const int slot = n % S;
            const int nbox = 2 * min(kKBlocks, nk - st * kKBlocks);
            bool ok = true;
            if (lane == 0)
              ok = PROF_WAIT(0, wait_or_abort(&sdone_bar[slot], ((n / S) & 1) ^ 1, abort_flag, args.status));
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) goto x_done;
            uint8_t* xs_g = smem_gen + SW * kWBytes + slot * kXBytes;
            if (lane == 0) mbar_arrive_expect_tx(&xfull_bar[slot], (uint32_t)(hr * 128 * nbox));
            __syncwarp();  // the stage's expected bytes are posted before any gather lands
            for (int i = lane; i < nbox * G; i += 32) {
              const int box = i / G;
              tma_gather4(xs_g + box * kXHalfBytes + (i - box * G) * 512, &tm_x, st * kKBlocks * kBK + 64 * box,
                          tok, &xfull_bar[slot]);
            }
          }
        }
      }
    x_done:
      if (lane == 0) {
        s_x_issued = n;
        PROF_FLUSH(2);
      }
    } else if (warp == kRelayWarp) {
      // ======================= relay: token stage landed -> CTA 0's stage barrier =======================
      if (lane == 0) {
        const uint32_t ready_remote0 = cluster_addr(&ready_bar[0], 0);
        int n = 0;
        bool ok = true;
        for (int j = pair; j < total && ok; j += npairs) {
          for (int st = 0; st < nst; ++st, ++n) {
            const int slot = n % S;
            ok = PROF_WAIT(0, wait_or_abort(&xfull_bar[slot], (n / S) & 1, abort_flag, args.status));
            if (!ok) break;
            mbar_arrive_remote(ready_remote0 + slot * (uint32_t)sizeof(uint64_t));
          }
        }
        PROF_FLUSH(4);
      }
    } else {
      // ======================= MMA issuer (CTA 0, one thread) =======================
      if (rank == 0 && lane == 0) {
        int n = 0, c = 0;
        bool ok = true;
        int e_hint = 0;
        for (int j = pair; j < total && ok; j += npairs) {
          PROF_T0(t_item);
          const Item it = decode_item(j, wl, e_hint);
          const uint32_t idesc = kIdescBase | ((uint32_t)(it.n_mma >> 3) << 17);
          const int cs = s_chunk[it.e];
          PROF_ADD(6, t_item);
          int kc = 0;  // k-blocks done within the current exact chunk (cs is a whole number of stages)
          for (int st = 0; st < nst && ok; ++st, ++n) {
            PROF_T0(t_body);
            const int slot = n % S;
            const uint32_t ph = (n / S) & 1;
            const int nkb = min(kKBlocks, nk - st * kKBlocks);  // 1 only in an odd last stage
            if (kc == 0) {
              // a new exact chunk: both CTAs' drains must have read the accumulator
              ok = PROF_WAIT(0, wait_or_abort(&accempty_bar, (c & 1) ^ 1, abort_flag, args.status));
              if (!ok) break;
            }
            ok = PROF_WAIT(1, wait_or_abort(&ready_bar[slot], ph, abort_flag, args.status));
            if (!ok) break;
            PROF_T0(t_issue);
            tc_fence_after();
            // 16-deep step s of the stage: A columns 8s of the stage's buffer; token box
            // s/4 at byte 32*(s%4) of its 128-byte rows, i.e. the descriptor's start
            // address field advanced by that offset / 16 (no carry: shared addresses
            // stay below 256 KB)
            const uint64_t bdesc0 = sw128_desc(x_ring + slot * kXBytes);
            const uint32_t a0 = tmem + kACol0 + slot * kACols;
            mma_pair(tmem, a0, bdesc0, idesc, kc != 0 ? 1u : 0u);
#pragma unroll
            for (int s = 1; s < 8; ++s)
              mma_pair(tmem, a0 + s * 8, bdesc0 + (uint64_t)(((s >> 2) * kXHalfBytes + (s & 3) * 32) >> 4), idesc, 1u);
            if (nkb == kKBlocks) {
#pragma unroll
              for (int s = 8; s < 16; ++s)
                mma_pair(tmem, a0 + s * 8, bdesc0 + (uint64_t)(((s >> 2) * kXHalfBytes + (s & 3) * 32) >> 4), idesc,
                         1u);
            }
            PROF_ADD(2, t_issue);
            PROF_T0(t_commit);
            mma_commit_pair(&sdone_bar[slot]);  // token slot and A buffer free once these MMAs complete
            PROF_ADD(3, t_commit);
            kc += nkb;
            if (kc == cs || st == nst - 1) {
              mma_commit_pair(&accfull_bar);    // chunk accumulated: hand it to the drains
              ++c;
              kc = 0;
            }
            PROF_ADD(4, t_body);
          }
        }
        // every MMA issued by this thread has completed once final_bar fires
        PROF_T0(t_fin);
        mma_commit_local(&final_bar);
        mbar_wait_bounded(&final_bar, 0);
        PROF_ADD(7, t_fin);
        PROF_FLUSH(8);
        PROF_TOTAL(t_start);
      }
      __syncwarp();
    }
  } else if (warp < kDrainWarp0) {
    // ======================= converters =======================
    // A full 128-byte weight row of each k-block per thread, widened and stored into
    // the stage's tensor-memory A buffer in 64-k halves; once the stage's k-blocks
    // are stored it is handed to the MMA issuer.
    regs_dec<kRegsConv>();
    const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;         // weight channel row of this thread
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t ready_remote0 = cluster_addr(&ready_bar[0], 0);
    int n = 0, m = 0;  // stages, k-blocks (weight ring positions)
    bool ok = true;
    for (int j = pair; j < total && ok; j += npairs) {
      for (int st = 0; st < nst; ++st, ++n) {
        const int slot = n % S;
        const int nkb = min(kKBlocks, nk - st * kKBlocks);
        ok = PROF_WAIT(1, wait_or_abort(&sdone_bar[slot], ((n / S) & 1) ^ 1, abort_flag, args.status));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ta0 = tmem + lane_off + kACol0 + slot * kACols;
        for (int kbi = 0; kbi < nkb; ++kbi, ++m) {
          const int wslot = m % SW;
          ok = PROF_WAIT(0, wait_or_abort(&wfull_bar[wslot], (m / SW) & 1, abort_flag, args.status));
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          PROF_T0(t_conv);
          const uint32_t wrow = w_ring + wslot * kWBytes + r * kBK;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 w4 = lds128(wrow + (((4 * h + q) ^ (r & 7)) << 4));
              i8x4_to_f16x4<kWFlip>(w4.x, v[8 * q + 0], v[8 * q + 1]);
              i8x4_to_f16x4<kWFlip>(w4.y, v[8 * q + 2], v[8 * q + 3]);
              i8x4_to_f16x4<kWFlip>(w4.z, v[8 * q + 4], v[8 * q + 5]);
              i8x4_to_f16x4<kWFlip>(w4.w, v[8 * q + 6], v[8 * q + 7]);
            }
            if (h == 1) {
              // the weight k-block is in registers: hand it back to the producer
              __syncwarp();
              if (lane == 0) mbar_arrive(&wempty_bar[wslot]);
            }
            tmem_st32(ta0 + kbi * (kBK / 2) + 32 * h, v);
          }
          PROF_ADD(2, t_conv);
        }
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(ready_remote0 + slot * (uint32_t)sizeof(uint64_t));
      }
    }
    if (lane == 0) PROF_FLUSH(16);
  } else {
    // ======================= drain + epilogue =======================
    // warp w drains TMEM lanes 32*(w%4).. (output channels) and accumulator columns
    // 64*cg .. +63 (token rows of the item), cg = (w-8)/4
    regs_inc<kRegsDrain>();
    const int quarter = warp & 3;
    const int cg = (warp - kDrainWarp0) >> 2;
    const int r = quarter * 32 + lane;  // output channel within this CTA's 128
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16) + cg * 64;
    const uint32_t accempty_remote = cluster_addr(&accempty_bar, 0);
    int c = 0;
    // fused SwiGLU: this warp's rows gw, gw + stride, ... of the valid ones, and the
    // expert of the next one (rows only move forward).  The rows go to the drain warps
    // of the three SM sub-partitions (warp % 4) other than the MMA-issuing warp's: the
    // one thread that issues the MMAs sets the kernel's pace, and SwiGLU work beside it
    // slows its issue (prefill GMM1 + SwiGLU: 713 us with every drain warp on rows,
    // 696 us without the issuer's sub-partition; fewer sub-partitions lengthen the tail).
    // On those three, three of the four column groups take rows: the rows' issue slots
    // slow the converter warp of the same sub-partition, whose stages the MMAs wait for
    // (696 -> 690 us; two groups 701 us, one 775 us: the rows then pile up at the end).
    constexpr int kRowGroups = 3;
    static_assert(kRowGroups <= kNumDrainWarps / 4, "column groups of drain warps");
    constexpr int kRowWarps = 3 * kRowGroups;
    auto takes_rows = [](int w) { return (w & 3) != (kMmaWarp & 3) && ((w - kDrainWarp0) >> 2) < kRowGroups; };
    const bool row_warp = takes_rows(warp);
    int row_rank = 0;
    for (int w = kDrainWarp0; w < warp; ++w) row_rank += takes_rows(w) ? 1 : 0;
    const int sw_stride = (int)gridDim.x * kRowWarps;
    const int sw_valid = s_end[E - 1];
    int sw_row = row_warp ? (int)blockIdx.x * kRowWarps + row_rank : sw_valid;
    int sw_e = 0;
    bool ok = true;
    int e_hint = 0;
    for (int j = pair; j < total && ok; j += npairs) {
      const Item it = decode_item(j, wl, e_hint);
      const bool active = cg * 64 < it.n_mma;
      const int cs = s_chunk[it.e];
      const int nch = (nk + cs - 1) / cs;
      // One exact chunk for the whole reduction (activation bounds permitting): its
      // fp32 sums are the exact integers (|sum| <= 2^24), so the raw values are kept,
      // the accumulator is handed back to the MMAs right after the loads, and the
      // epilogue scales them as they are (float(acc) is the same value).  Two exact
      // chunks: the first is kept raw the same way, and the second is added to it in
      // fp32 as it is read -- one IEEE addition of two exact integers, i.e. the
      // correctly rounded float of their exact sum, which is what the epilogue
      // scales.  Either way the accumulator goes back to the MMAs after its loads
      // and additions alone.  Otherwise each chunk is converted to int32 and added
      // before the hand-back.
      const bool raw = nch <= 2;
      int acc[64];  // int32 sums, or (raw) the fp32 bits of the float total
#pragma unroll
      for (int t = 0; t < 64; ++t) acc[t] = 0;
      if (raw) {
        ok = PROF_WAIT(0, wait_or_abort(&accfull_bar, c & 1, abort_flag, args.status));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++c;
        tc_fence_after();
        if (active) {
          tmem_ld16(lane_base, *reinterpret_cast<uint32_t(*)[16]>(&acc[0]));
          tmem_ld16(lane_base + 16, *reinterpret_cast<uint32_t(*)[16]>(&acc[16]));
          tmem_ld16(lane_base + 32, *reinterpret_cast<uint32_t(*)[16]>(&acc[32]));
          tmem_ld16(lane_base + 48, *reinterpret_cast<uint32_t(*)[16]>(&acc[48]));
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(accempty_remote);
        if (nch == 2) {
          ok = PROF_WAIT(0, wait_or_abort(&accfull_bar, c & 1, abort_flag, args.status));
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          ++c;
          PROF_T0(t_drain);
          tc_fence_after();
          if (active) {
#pragma unroll
            for (int t0 = 0; t0 < 64; t0 += 16) {
              uint32_t v[16];
              tmem_ld16(lane_base + t0, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i)
                acc[t0 + i] = __float_as_int(__fadd_rn(__int_as_float(acc[t0 + i]), __uint_as_float(v[i])));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(accempty_remote);
          PROF_ADD(1, t_drain);
        }
      } else {
        for (int ch = 0; ch < nch; ++ch, ++c) {
          ok = PROF_WAIT(0, wait_or_abort(&accfull_bar, c & 1, abort_flag, args.status));
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          PROF_T0(t_drain);
          tc_fence_after();
          if (active) {
#pragma unroll
            for (int t0 = 0; t0 < 64; t0 += 16) {
              uint32_t v[16];
              tmem_ld16(lane_base + t0, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float f = __uint_as_float(v[i]);
                acc[t0 + i] += (i % 3 == 0) ? __float2int_rn(f) : f2i_exact(f);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(accempty_remote);
          PROF_ADD(1, t_drain);
        }
      }
      if (!ok) break;
      PROF_T0(t_epi);
      // epilogue: channel r of rows row0 + 64*cg + t (a warp writes 64 contiguous bytes per row)
      const int ch = it.cb * kPairCh + (int)rank * kBM + r;
      if (active && ch < args.N) {
        const float sc = __ldg(args.scale + (size_t)it.e * args.N + ch);
        const int t_lo = cg * 64;
        __half* dst = args.C + (size_t)(it.row0 + t_lo) * args.N + ch;
        if (raw) {
#pragma unroll
          for (int t = 0; t < 64; ++t)
            if (t_lo + t < it.rows) dst[(size_t)t * args.N] = f2h_sat(__fmul_rn(__int_as_float(acc[t]), sc));
        } else {
#pragma unroll
          for (int t = 0; t < 64; ++t)
            if (t_lo + t < it.rows) dst[(size_t)t * args.N] = f2h_sat(__fmul_rn(__int2float_rn(acc[t]), sc));
        }
      }
      PROF_ADD(2, t_epi);
      if (kSw) {
        // count this item on its expert once the warp's stores are visible GPU-wide, then
        // requantise own rows of complete experts while the next chunk is not ready
        __syncwarp();
        __threadfence();
        if (lane == 0) atomicAdd(args.sw_done + it.e, 1);
        while (sw_row < sw_valid && !mbar_test(&accfull_bar, c & 1)) {
          while (s_end[sw_e] <= sw_row) ++sw_e;
          const int lo = sw_e ? s_end[sw_e - 1] : 0;
          const int target = kSwigluCountPerItem * expert_items(s_end[sw_e] - lo, args.split_rows, n_cb);
          if (__shfl_sync(0xffffffffu, lane == 0 ? ld_acquire(args.sw_done + sw_e) : 0, 0) < target) break;
          swiglu_row_warp(args, sw_row, sw_e, lane);
          sw_row += sw_stride;
        }
      }
    }
    if (kSw && ok) {
      // the rest of this warp's rows, each once its expert is complete (bounded wait)
      while (sw_row < sw_valid) {
        while (s_end[sw_e] <= sw_row) ++sw_e;
        const int lo = sw_e ? s_end[sw_e - 1] : 0;
        const int target = kSwigluCountPerItem * expert_items(s_end[sw_e] - lo, args.split_rows, n_cb);
        const int done = lane == 0 ? (count_wait_bounded(args.sw_done + sw_e, target) ? 1 : 0) : 0;
        if (!__shfl_sync(0xffffffffu, done, 0)) {
          *abort_flag = 1;
          record_status(args.status, MOE_ERR_TIMEOUT);
          break;
        }
        swiglu_row_warp(args, sw_row, sw_e, lane);
        sw_row += sw_stride;
      }
    }
    if (lane == 0) PROF_FLUSH(24);
  }

  __syncthreads();
  if (threadIdx.x == 0) {
    // this CTA's copies still in flight (only after an abort) land before shared memory is released
    const int wi = s_w_issued, xi = s_x_issued;
    for (int n = max(0, wi - SW); n < wi; ++n) mbar_wait_bounded(&wfull_bar[n % SW], (n / SW) & 1);
    for (int n = max(0, xi - S); n < xi; ++n) mbar_wait_bounded(&xfull_bar[n % S], (n / S) & 1);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the pair's MMAs or remote arrivals may touch it
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
  }
}

template <bool GATHER, int FUSE, bool TILES>
cudaError_t launch_pair(const GroupedGemmProblem& p, cudaStream_t stream) {
  CUtensorMap tw, tx;
  if (!encode_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w, (uint64_t)p.Kd, (uint64_t)p.E * p.N, kBK,
                            kBM))
    return cudaErrorInvalidValue;
  // token operand: 128-row tiled boxes, or (gathering) one-row boxes over the token rows
  if (!encode_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.act, (uint64_t)p.Kd, (uint64_t)p.act_rows, 64,
                            GATHER ? 1 : kHalfRows))
    return cudaErrorInvalidValue;
  static PerContextOnce checked;
  const int dev = current_device();
  if (checked.needed(dev)) {
    // The warpgroups' register split (setmaxnreg) adds up to exactly the registers
    // the CTA is launched with; a build that launches with another count would
    // leave the drains' increase waiting forever, so it is refused here.
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, grouped_gemm_pair_kernel<GATHER, FUSE, TILES>);
    if (err != cudaSuccess) return err;
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidKernelImage;
    err = cudaFuncSetAttribute(grouped_gemm_pair_kernel<GATHER, FUSE, TILES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes);
    if (err != cudaSuccess) return err;
    checked.done(dev);
  }
  Args a;
  a.cumsum = p.cumsum;
  a.scale = p.scale;
  a.C = reinterpret_cast<__half*>(p.C);
  a.status = p.status;
  a.E = p.E;
  a.N = p.N;
  a.Kd = p.Kd;
  a.split_rows = p.split_rows;
  a.bounds = p.bounds;
  a.gather_route = p.gather_route;
  a.topK = p.topK;
  a.w_tiles = TILES ? reinterpret_cast<const uint8_t*>(p.w) : nullptr;
  a.w_kb = p.w_kb;
  a.sw_pts1 = p.sw_pts1;
  a.sw_sorted = p.sw_sorted;
  a.sw_q2 = reinterpret_cast<__half*>(p.sw_q2);
  a.sw_pts2 = p.sw_pts2;
  a.sw_bounds = p.sw_bounds;
  a.sw_done = p.sw_done;
  if (FUSE == kFuseSwiglu && (p.N / 2 > kFusedSwigluMaxI || p.topK < 1 || !a.sw_q2 || !a.sw_pts1 || !a.sw_sorted ||
                               !a.sw_pts2 || !a.sw_done))
    return cudaErrorInvalidValue;  // the fused SwiGLU runs on a tiled GMM1
#ifdef MOE_GEMM_PROFILE
  a.prof = g_gemm_prof;
  if (!a.prof) return cudaErrorInvalidValue;
#endif
  const int grid = sm_count() & ~1;  // whole pairs, one CTA per SM
  grouped_gemm_pair_kernel<GATHER, FUSE, TILES><<<grid, kThreads, kSmemBytes, stream>>>(tw, tx, a);
  return cudaGetLastError();
}

}  // namespace

static_assert(kFusedSwigluMaxI <= kBoundSegments * kBoundSegment, "fused SwiGLU: a bound segment per pass");

bool pair_grid_coresident() {
  static PerContextOnce queried;
  static bool ok[kMaxDevices] = {};
  const int dev = current_device();
  if (queried.needed(dev)) {
    // the kernel's attributes (dynamic shared memory) are set by its first launch; set
    // them here too so the query sees the launch's configuration
    if (cudaFuncSetAttribute(grouped_gemm_pair_kernel<false, kFuseSwiglu, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return false;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sm_count() & ~1));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_pair_kernel<false, kFuseSwiglu, true>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      clusters = 0;
    }
    ok[dev] = 2 * clusters >= (sm_count() & ~1);
    queried.done(dev);
  }
  return ok[dev];
}

template <bool TILES>
cudaError_t launch_pair_layout(const GroupedGemmProblem& p, cudaStream_t stream) {
  if (p.gather_route) {
    if (p.sw_q2) return cudaErrorInvalidValue;  // the fused SwiGLU runs on the tiled operand
    return launch_pair<true, kFuseNone, TILES>(p, stream);
  }
  return p.sw_q2 ? launch_pair<false, kFuseSwiglu, TILES>(p, stream) : launch_pair<false, kFuseNone, TILES>(p, stream);
}

cudaError_t launch_grouped_gemm_tc(const GroupedGemmProblem& p, cudaStream_t stream) {
  return p.w_kb ? launch_pair_layout<true>(p, stream) : launch_pair_layout<false>(p, stream);
}

}  // namespace moe
