/*
 * moe_layer.h -- C ABI of the GB300 (sm_103a) W8A8 mixture-of-experts expert layer.
 *
 * The layer follows the stage contract of the PTO-ISA MegaMoE operator page
 * ("pto-isa megamoe operator", kernels/manual/a2a3/dispatch_mega_combine/overview,
 * section "key implementation logic": FrontReorder -> Dispatch -> GMM1 -> SwiGLU ->
 * GMM2 -> Combine -> Unpermute) on a single GPU: the cross-rank count exchange,
 * dispatch pull and combine push of that page become gathers inside device memory.
 *
 * Conventions shared by every entry point
 *   - Shapes: M tokens, hidden size K, intermediate size I (GMM1 is 2I wide: the
 *     first I columns go through silu, the second I multiply it), E experts,
 *     topK routes per token, R = M * topK routes.  Route r = token * topK + slot.
 *   - binary16 values are passed as uint16_t bit patterns (IEEE half).
 *   - Every pointer argument is DEVICE memory owned by the caller, except where a
 *     parameter name ends in _host.  The library never allocates or frees device
 *     memory; scratch space comes from the caller's `workspace` (moe_route_sort_noalloc
 *     alone uses a fixed scratch array inside the library instead).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  No entry point synchronises, except moe_layer_fwd_host,
 *     moe_workspace_status and the pipeline's calls, which say so.
 *   - Arrays are dense row-major with the last index contiguous.  Every device
 *     pointer must be 16-byte aligned (the layer's workspace 256-byte aligned), and
 *     every entry point checks this for the pointers it is given (MOE_ERR_ALIGN);
 *     the host buffers of the _host entry points may have any alignment.
 *   - Preconditions checked on the host before anything is launched:
 *       M >= 1, 1 <= topK <= E <= 1023, K % 128 == 0, 128 <= K <= 16384,
 *       I % 64 == 0, 64 <= I <= 8192, M * topK < 2^24, current device sm_103.
 *     A violated precondition returns an error and launches nothing.
 *   - The route tables a stage entry point takes (sorted_src_route,
 *     expanded_row_idx, cumsum) must be what moe_route_sort (or moe_front_reorder)
 *     wrote for the same expert_idx and dimensions: the kernels use their entries
 *     as row indices without checking them, so other values read or write out of
 *     bounds.  moe_layer_fwd produces them itself.
 *   - Routes whose expert id lies outside [0, E) are dropped: sorted after all
 *     valid routes, counted in no expert, expandedRowIdx = -1, and they add
 *     nothing to the output.  Their number is R - cumsum[E-1].
 *   - Every fp32 -> binary16 conversion of a stage output (GMM epilogues, Combine,
 *     Unpermute) rounds to nearest even and saturates at +-65504.
 *   - Launch failures are reported as MOE_ERR_LAUNCH (cudaGetLastError after the
 *     launches).  A device-side wait that gives up (a pipeline barrier that never
 *     completes) makes the kernel record MOE_ERR_TIMEOUT in the workspace status
 *     word and return early; read it with moe_workspace_status.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t M;    /* tokens                         */
  int32_t K;    /* hidden size                    */
  int32_t I;    /* intermediate size (GMM1: 2I)   */
  int32_t E;    /* experts                        */
  int32_t topK; /* routes per token               */
  int32_t weight_layout; /* layout of the w1 / w2 arguments: MOE_WEIGHTS_ROWS (0, what a
                            zero-initialised field gives) or MOE_WEIGHTS_TILES (1); any
                            other value is MOE_ERR_SHAPE                              */
} moe_dims_t;

/*
 * Weight layouts.  A GEMM weight W has E experts, N output channels and a reduction
 * depth D (GMM1: N = 2I, D = K; GMM2: N = K, D = I).
 *   MOE_WEIGHTS_ROWS   W[E][N][D] int8, D contiguous.
 *   MOE_WEIGHTS_TILES  the same values as 16 KiB tiles of 128 channels x 128 reduction
 *                      steps, each tile one contiguous block, written by
 *                      moe_pack_weight_tiles: the GEMMs then stream every pipeline
 *                      stage of weights as one contiguous copy instead of 128 rows
 *                      7 KiB apart (a read stream of the decode weights measured
 *                      7.24 TB/s against 6.78 TB/s in the row order).  It plays the
 *                      part of the page's packed ("NZ") weight, laid out offline.
 *     Let NB = N / 128 and KB = 2 * ceil(D / 256) (tiles per channel block: the depth
 *     is padded with zeros to a multiple of 256).  Tile (e, nb, kb) starts at byte
 *     ((e * NB + nb) * KB + kb) * 16384; inside it, W[e][nb*128 + r][kb*128 + c]
 *     (r, c in [0, 128)) sits at byte r * 128 + (((c / 16) ^ (r % 8)) * 16) + c % 16,
 *     stored in excess-128 form: the byte is W + 128 (W's two's-complement byte with
 *     its top bit flipped), and the bytes of reduction steps kb*128 + c >= D hold
 *     0x80, the code of 0.  This is the image a 128-byte-swizzled tensor copy of the
 *     128 x 128 box leaves in shared memory, with the sign bits flipped so that the
 *     GEMMs widen four weights to binary16 with one instruction less.
 */
#define MOE_WEIGHTS_ROWS 0
#define MOE_WEIGHTS_TILES 1

typedef enum {
  MOE_OK = 0,
  MOE_ERR_NULL = -1,      /* a required pointer is NULL                      */
  MOE_ERR_SHAPE = -2,     /* dimensions outside the supported ranges         */
  MOE_ERR_ALIGN = -3,     /* a pointer is not 16-byte aligned                */
  MOE_ERR_ARCH = -4,      /* current device is not sm_103 / no device       */
  MOE_ERR_WORKSPACE = -5, /* workspace missing or smaller than required      */
  MOE_ERR_LAUNCH = -6,    /* a CUDA launch or copy failed                    */
  MOE_ERR_TIMEOUT = -8    /* a device-side pipeline wait gave up             */
} moe_status_t;

/* Human-readable name of a status code (static string). */
const char* moe_status_string(int32_t status);

/* ------------------------------------------------------------------------ */
/* Whole layer                                                               */
/* ------------------------------------------------------------------------ */

/* Bytes of device workspace moe_layer_fwd needs for these dimensions
 * (0 if the dimensions are invalid). */
size_t moe_layer_workspace_size(const moe_dims_t* d);

/*
 * out[t, :] = sum over the token's valid routes of probs[t, j] * FFN_e(x[t, :]),
 * the W8A8 expert layer of MegaMoe::Process() (all seven stages of the page).
 *
 *   x          [M][K]      binary16 tokens
 *   expert_idx [M][topK]   int32 expert of each route
 *   probs      [M][topK]   fp32 route weights (used as given, not renormalised)
 *   w1         [E][2I][K]  int8 GMM1 weights, K contiguous (the page's packed
 *                          weight1[e][k][n], transposed so the reduction runs along rows),
 *                          or their tiles (d->weight_layout, see "Weight layouts")
 *   s1         [E][2I]     fp32 GMM1 per-channel scales
 *   w2         [E][K][I]   int8 GMM2 weights, I contiguous, or their tiles
 *   s2         [E][K]      fp32 GMM2 per-channel scales
 *   out        [M][K]      binary16 result (written for every token; a token with
 *                          no valid route gets zeros)
 *   workspace  >= moe_layer_workspace_size(d) bytes of device memory, 256-byte
 *              aligned; its contents on entry do not matter.
 * The intermediates (route tables, quantised tokens, GMM outputs) live in the
 * workspace until the next call that uses it.
 */
int32_t moe_layer_fwd(const moe_dims_t* d, const uint16_t* x, const int32_t* expert_idx,
                      const float* probs, const int8_t* w1, const float* s1, const int8_t* w2,
                      const float* s2, uint16_t* out, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * The layer as a CUDA graph, for calls repeated on the same buffers (a serving
 * loop that writes each batch into fixed device buffers): moe_layer_graph_create
 * records exactly the launches of moe_layer_fwd with these arguments (same
 * preconditions and error codes) by stream capture on `stream`, which must not be
 * the legacy default stream (NULL: MOE_ERR_LAUNCH), and instantiates the graph;
 * nothing runs yet.  moe_layer_graph_launch runs it on `stream` (any stream of the
 * same device), asynchronously, with the same result as moe_layer_fwd on the
 * buffers' contents at that time; it saves part of the per-kernel launch gaps
 * (measured: 0.7% at decode, 1.7% at prefill).  The buffers must stay allocated
 * while the graph exists.  moe_layer_graph_destroy releases the graph (host
 * memory and CUDA graph objects; NULL is a no-op).
 */
typedef struct moe_layer_graph moe_layer_graph_t;
int32_t moe_layer_graph_create(const moe_dims_t* d, const uint16_t* x, const int32_t* expert_idx,
                               const float* probs, const int8_t* w1, const float* s1, const int8_t* w2,
                               const float* s2, uint16_t* out, void* workspace, size_t workspace_bytes,
                               void* stream, moe_layer_graph_t** graph);
/*
 * The same for moe_layer_fwd_host: the graph holds the copies of x_host,
 * expert_idx_host and probs_host into the workspace, the layer and the copy of the
 * output to out_host.  A launch does not synchronise: read out_host after the stream
 * has (cudaStreamSynchronize).  The host buffers must be page-locked (cudaHostAlloc,
 * cudaHostRegister); pageable memory cannot be captured (MOE_ERR_LAUNCH).
 */
int32_t moe_layer_graph_create_host(const moe_dims_t* d, const uint16_t* x_host, const int32_t* expert_idx_host,
                                    const float* probs_host, const int8_t* w1, const float* s1, const int8_t* w2,
                                    const float* s2, uint16_t* out_host, void* workspace, size_t workspace_bytes,
                                    void* stream, moe_layer_graph_t** graph);
int32_t moe_layer_graph_launch(moe_layer_graph_t* graph, void* stream);
int32_t moe_layer_graph_destroy(moe_layer_graph_t* graph);

/* Bytes of device workspace moe_layer_fwd_host needs (layer workspace plus
 * staging for the per-call host inputs and the output). */
size_t moe_layer_host_workspace_size(const moe_dims_t* d);

/*
 * moe_layer_fwd with the per-call tensors in HOST memory: copies x_host,
 * expert_idx_host and probs_host to the device (into the workspace), runs the
 * layer, copies the result to out_host, and synchronises `stream` before
 * returning.  Weights and scales stay device pointers (model parameters are
 * resident).  Host buffers should be page-locked for the copies to run at full
 * speed; pageable memory works but is slower.
 */
int32_t moe_layer_fwd_host(const moe_dims_t* d, const uint16_t* x_host,
                           const int32_t* expert_idx_host, const float* probs_host,
                           const int8_t* w1, const float* s1, const int8_t* w2, const float* s2,
                           uint16_t* out_host, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * A pipelined executor for a serving loop whose batches arrive and leave in HOST
 * memory: consecutive batches overlap their host->device copies, the layer and the
 * device->host copy of the result, on three streams the pipeline owns (the copies
 * of batch n+1 and n-1 run while the layer computes batch n).  Up to `depth` batches
 * (1..8) are in flight; each has its own staging buffers in the workspace, the
 * layer's own buffers are shared (the layer runs one batch at a time, as a CUDA
 * graph per staging slot).
 *   moe_layer_pipeline_workspace_size: device bytes for `depth` slots (0 for bad
 *     dimensions or depth).
 *   moe_layer_pipeline_create: checks as moe_layer_fwd (plus 1 <= depth <= 8:
 *     MOE_ERR_SHAPE), creates the streams, events and graphs (host objects; the
 *     only host memory it allocates is one page-locked status word per slot) on the
 *     current device; nothing runs yet.  Weights and workspace must stay allocated
 *     until moe_layer_pipeline_destroy.
 *   moe_layer_pipeline_submit: enqueues one batch (x_host [M][K], expert_idx_host
 *     [M][topK], probs_host [M][topK] in; out_host [M][K] out) and returns its ticket
 *     (0, 1, 2, ... in submission order).  When `depth` batches are in flight it
 *     first waits (host) until the oldest has completed.  The host buffers belong to
 *     the pipeline until their batch has completed: inputs must not change, out_host
 *     must not be read before then.  Page-locked host buffers (cudaHostAlloc,
 *     cudaHostRegister) let the copies overlap the layer; pageable ones work but
 *     serialise them.
 *   moe_layer_pipeline_wait: blocks until batch `ticket` and every earlier one have
 *     completed (out_host written).  Returns MOE_ERR_TIMEOUT if a device-side wait of
 *     any batch up to `ticket` gave up (that batch's output is then undefined),
 *     MOE_ERR_SHAPE for a ticket not yet submitted, MOE_ERR_LAUNCH if a copy or launch
 *     failed.
 *   moe_layer_pipeline_destroy: waits for every batch in flight, then releases the
 *     pipeline (NULL is a no-op).
 * A pipeline's calls must come from one host thread at a time (it keeps its ticket
 * counters without locks); separate pipelines are independent.
 */
typedef struct moe_layer_pipeline moe_layer_pipeline_t;
size_t moe_layer_pipeline_workspace_size(const moe_dims_t* d, int32_t depth);
int32_t moe_layer_pipeline_create(const moe_dims_t* d, const int8_t* w1, const float* s1, const int8_t* w2,
                                  const float* s2, void* workspace, size_t workspace_bytes, int32_t depth,
                                  moe_layer_pipeline_t** pipeline);
int32_t moe_layer_pipeline_submit(moe_layer_pipeline_t* pipeline, const uint16_t* x_host,
                                  const int32_t* expert_idx_host, const float* probs_host, uint16_t* out_host,
                                  uint64_t* ticket);
int32_t moe_layer_pipeline_wait(moe_layer_pipeline_t* pipeline, uint64_t ticket);
int32_t moe_layer_pipeline_destroy(moe_layer_pipeline_t* pipeline);

/* Reads the status word that kernels running on `workspace` (the layer's, or a
 * GEMM stage's) set when a device-side wait gives up.  Synchronises `stream`.
 * *host_status receives MOE_OK or MOE_ERR_TIMEOUT. */
int32_t moe_workspace_status(const void* workspace, int32_t* host_status, void* stream);

/* Clears that status word (asynchronous). */
int32_t moe_workspace_clear_status(void* workspace, void* stream);

/* ------------------------------------------------------------------------ */
/* Stages (same conventions).  Used by the parity tests and benchmarks; the */
/* layer runs the same kernels.                                              */
/* ------------------------------------------------------------------------ */

/* Workspace bytes of moe_route_sort (per-block histograms). */
size_t moe_route_sort_workspace_size(const moe_dims_t* d);

/*
 * FrontReorder phases 1, 2a, 2b and 4 on one rank (page section "1. FrontReorder"):
 * stable sort of the routes by expert id (ties by route id), the per-expert counts,
 * the inverse permutation and the prefix sum.
 *   sorted_src_route  [R]  out: route placed at expanded row d (the page's sortedSrcRoute)
 *   expanded_row_idx  [R]  out: expanded row of route r, -1 if r is invalid
 *   tokens_per_expert [E]  out: routes per expert
 *   cumsum            [E]  out: inclusive prefix sum of tokens_per_expert
 */
int32_t moe_route_sort(const moe_dims_t* d, const int32_t* expert_idx, int32_t* sorted_src_route,
                       int32_t* expanded_row_idx, int32_t* tokens_per_expert, int32_t* cumsum,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * FrontReorder phase 2c (page section "1. FrontReorder"): per-token dynamic int8
 * quantisation, once per token: pts1[t] = max_k |x[t,k]| / 127 and
 * q = round-half-away(x / pts1), clamped to [-127, 127]; an all-zero token gets
 * pts1 = 0 and zero codes.
 *   expert_idx [M][topK] (read only when a1_bounds is given)
 *   xq_i8  [M][K] int8 codes (may be NULL)
 *   xq_f16 [M][K] the same codes as binary16 integers (may be NULL; at least
 *          one of the two must be given): the operand GMM1 gathers from
 *   pts1   [M]    fp32 scales
 *   a1_bounds: NULL, or a zero-filled int32 [E][MOE_BOUND_SEGMENTS] that receives,
 *          for every expert, the segment maxima of sum |code| over the tokens routed
 *          to it (see "Activation bounds"; invalid routes contribute nothing)
 */
int32_t moe_quant_tokens(const moe_dims_t* d, const uint16_t* x, const int32_t* expert_idx, int8_t* xq_i8,
                         uint16_t* xq_f16, float* pts1, int32_t* a1_bounds, void* stream);

/*
 * Allocation-free route sort.  The paper has no counterpart: this entry point
 * exists for callers that cannot allocate device memory when they sort (an
 * engine plugin whose host engine owns all device memory, a server that
 * reserved the whole device up front, a loop where cudaMalloc's implicit
 * synchronisation is not allowed).  It computes exactly what moe_route_sort
 * computes, with the same checks and error codes, but takes no workspace: its
 * scratch is a fixed 256 KiB array in the library's own device memory, which
 * every GPU that loads the library holds until the process exits.
 *   - Supports M * topK <= MOE_ROUTE_SORT_NOALLOC_MAX_ROUTES (and the usual
 *     E <= 1023); larger sizes return MOE_ERR_SHAPE and launch nothing.
 *   - Allocates and frees nothing (no cudaMalloc/cudaFree, no library allocator).
 *   - The first call in each CUDA context of a device looks up the scratch
 *     array's device address (cudaGetSymbolAddress) with that device current and
 *     remembers it for that context: the first call on the device, and the first
 *     again after a cudaDeviceReset (or after the primary context was released
 *     and created anew), which loads the library's device code at a new address.
 *     Make that first call before any stream capture.
 *   - The multi-block sort it runs above 8192 routes uses at most 64 CTAs, as
 *     moe_route_sort does, sized to the fixed scratch.
 *   - All calls share the one scratch array: calls that may overlap on the GPU
 *     (different streams without ordering between them) race and must not be
 *     issued.  Calls ordered on one stream are safe; nothing in the scratch needs
 *     clearing between them.
 * Arguments as for moe_route_sort, minus the workspace.
 */
#define MOE_ROUTE_SORT_NOALLOC_MAX_ROUTES 524288
int32_t moe_route_sort_noalloc(const moe_dims_t* d, const int32_t* expert_idx, int32_t* sorted_src_route,
                               int32_t* expanded_row_idx, int32_t* tokens_per_expert, int32_t* cumsum,
                               void* stream);

/*
 * Activation bounds.  The grouped GEMMs accumulate exact integers in fp32 in
 * chunks whose every partial sum stays within 2^24.  Without further knowledge
 * a chunk is 1024 deep (1024 * 128 * 128 = 2^24).  A bounds array
 *   int32_t bounds[E][MOE_BOUND_SEGMENTS]
 * holds, for expert e and the s-th MOE_BOUND_SEGMENT-deep segment of the
 * reduction dimension (k in [1024 s, 1024 s + 1024)), an upper bound of
 *   sum over k in the segment of |a[row][k]|      for every row of expert e,
 * so a chunk of consecutive segments S is exact when 128 * sum_{s in S} bound[e][s]
 * <= 2^24 (|w| <= 128); the GEMMs then use the longest such uniform chunk per
 * expert.  moe_quant_tokens, moe_quant_dispatch and moe_swiglu_quant produce exact maxima when
 * given a zero-filled array (atomic max); a bound that is too small makes the
 * GEMM results inexact.  Passing NULL everywhere keeps the 1024-deep chunks.
 */
#define MOE_BOUND_SEGMENT 1024
#define MOE_BOUND_SEGMENTS 16

/*
 * FrontReorder phase 2c with the quant-scatter (page section "1. FrontReorder"):
 * quantise every token once (as moe_quant_tokens) and write its codes, as
 * binary16 integers, to each of its expanded rows:
 *   a1_f16[expanded_row_idx[t*topK + j]][k] = q[t][k]   for every valid route j
 * giving the expert-major GMM1 operand (rows of invalid routes are not written).
 *   expert_idx [M][topK] (read only when a1_bounds is given); expanded_row_idx [R]
 *   from moe_route_sort; a1_f16 [R][K]; pts1 [M];
 *   a1_bounds: NULL, or a zero-filled int32 [E][MOE_BOUND_SEGMENTS] that receives
 *   the per-expert segment maxima of sum |code| (see "Activation bounds").
 */
int32_t moe_quant_dispatch(const moe_dims_t* d, const uint16_t* x, const int32_t* expert_idx,
                           const int32_t* expanded_row_idx, uint16_t* a1_f16, float* pts1, int32_t* a1_bounds,
                           void* stream);

/*
 * FrontReorder in one call (page section "1. FrontReorder", phases 1-2c and 4, with
 * "2. Dispatch"): exactly moe_route_sort followed by moe_quant_dispatch, with the
 * same outputs.  Up to 4096 routes no sort kernel runs: each token's quant CTA
 * counts all routes' expert ids itself and places its own routes (one launch
 * instead of two); above that the route-sort kernels run first.
 *   workspace: moe_route_sort_workspace_size(d) bytes (0 up to 8192 routes)
 *   other arguments as for moe_route_sort and moe_quant_dispatch
 *   (expert_idx is read in any case; a1_bounds may be NULL)
 */
int32_t moe_front_reorder(const moe_dims_t* d, const uint16_t* x, const int32_t* expert_idx,
                          int32_t* sorted_src_route, int32_t* expanded_row_idx, int32_t* tokens_per_expert,
                          int32_t* cumsum, uint16_t* a1_f16, float* pts1, int32_t* a1_bounds, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Workspace bytes of moe_gmm1 / moe_gmm1_swiglu / moe_gmm2 (status word and E counters). */
size_t moe_gmm_workspace_size(const moe_dims_t* d);

/*
 * Bytes of the MOE_WEIGHTS_TILES form of GMM `gemm`'s weights (1: w1, N = 2I, D = K;
 * 2: w2, N = K, D = I): E * (N / 128) * KB * 16384 with KB = 2 * ceil(D / 256).
 * 0 if the dimensions are invalid or gemm is neither 1 nor 2 (d->weight_layout is
 * not read).
 */
size_t moe_weight_tiles_bytes(const moe_dims_t* d, int32_t gemm);

/*
 * Writes the tiles of a row-layout weight (see "Weight layouts"): w [E][N][D] int8
 * (MOE_WEIGHTS_ROWS), tiles >= moe_weight_tiles_bytes(d, gemm) bytes, both device
 * memory, 16-byte aligned, not overlapping.  Done once when the weights are loaded;
 * the layer then runs with d->weight_layout = MOE_WEIGHTS_TILES on the tile buffers.
 * d->weight_layout is not read.  Asynchronous on `stream`; errors as the other
 * entry points (MOE_ERR_SHAPE also for gemm outside {1, 2}).
 */
int32_t moe_pack_weight_tiles(const moe_dims_t* d, int32_t gemm, const int8_t* w, int8_t* tiles, void* stream);

/*
 * GMM1 (page section "3. GMM1", with "2. Dispatch" fused as a gather): for each
 * valid expanded row d of expert e (rows cumsum[e]-count_e .. cumsum[e]-1):
 *   acc[n]   = sum_k a1[d][k] * w1[e][n][k]                (exact integer)
 *   c1[d][n] = binary16(float(acc[n]) * s1[e][n])          n < 2I
 * where a1[d] is
 *   a1_f16[d]  when sorted_src_route is NULL: a1_f16 is [R][K] expert-major
 *          (moe_quant_dispatch; the layer's path);
 *   a1_f16[sorted_src_route[d] / topK]  when sorted_src_route is given: a1_f16 is
 *          [M][K] token-major binary16-coded codes (moe_quant_tokens), gathered by
 *          TMA in 4-row groups.  This needs topK times less activation memory but
 *          runs GMM1 1.2x (16-row tiles) to 3.2x (tcgen05 pairs) slower on GB300:
 *          a gather moves 512 B per TMA instruction, a tiled box up to 16 KB.
 *   a1_bounds: NULL or the activation bounds of the rows a1[d] (see "Activation bounds");
 *   w1: in the layout d->weight_layout names (w1[e][n][k] above is the row form's value);
 *   c1 [R][2I] (rows >= cumsum[E-1] untouched)
 */
int32_t moe_gmm1(const moe_dims_t* d, const uint16_t* a1_f16, const int32_t* sorted_src_route, const int32_t* cumsum,
                 const int32_t* a1_bounds, const int8_t* w1, const float* s1, uint16_t* c1, void* workspace,
                 size_t workspace_bytes, void* stream);

/*
 * SwiGLU + dynamic requant (page section "4. SwiGLU"), per valid expanded row d
 * with token t = sorted_src_route[d] / topK:
 *   h = float(c1[d]) * pts1[t];  y_j = silu(h_j) * h_{j+I},  silu(v) = v / (1 + exp(-v))
 *   pts2[d] = max_j |y_j| / 127;  q_j = round-half-even(y_j * (127 / max|y|)), clamped
 *   q2_i8 [R][I] int8 (may be NULL); q2_f16 [R][I] binary16-coded (may be NULL); pts2 [R];
 *   q2_bounds: NULL, or a zero-filled int32 [E][MOE_BOUND_SEGMENTS] that receives the
 *   per-expert segment maxima of sum |q| (see "Activation bounds"); expert_idx
 *   [M][topK] is read only then (the expert of row d is expert_idx[sorted_src_route[d]])
 */
int32_t moe_swiglu_quant(const moe_dims_t* d, const uint16_t* c1, const float* pts1,
                         const int32_t* sorted_src_route, const int32_t* cumsum, const int32_t* expert_idx,
                         int8_t* q2_i8, uint16_t* q2_f16, float* pts2, int32_t* q2_bounds, void* stream);

/*
 * GMM1 followed by SwiGLU + dynamic requant (page sections "3. GMM1" and "4. SwiGLU"):
 * c1 exactly as moe_gmm1 writes it (the dispatched operand: a1_f16 [R][K] expert-major),
 * then q2_f16, pts2 and q2_bounds exactly as moe_swiglu_quant writes them from c1 (q2
 * only in the binary16-coded form the GMM2 reads; expert_idx is read only for the
 * bounds).  When the tcgen05 CTA pairs run (more than 24 routes per expert on
 * average; below 256 the warp-MMA engine first takes the experts of at most 32 rows),
 * the SwiGLU runs inside the pairs' GMM1 kernel: their drain warps requantise the rows
 * of each expert as soon as all of the expert's GMM1 tiles are stored, between the
 * tensor-core work items, so the SwiGLU kernel's pass over c1 leaves the critical path
 * (the overlap of GMM1 and SwiGLU the page builds with its per-expert flags).
 * Otherwise GMM1 and the SwiGLU kernel run one after the other.  The results are the
 * same bits either way.
 *   workspace: moe_gmm_workspace_size(d) bytes (status word and per-expert counters).
 */
int32_t moe_gmm1_swiglu(const moe_dims_t* d, const uint16_t* a1_f16, const int32_t* cumsum, const int32_t* a1_bounds,
                        const int8_t* w1, const float* s1, uint16_t* c1, const float* pts1,
                        const int32_t* sorted_src_route, const int32_t* expert_idx, uint16_t* q2_f16, float* pts2,
                        int32_t* q2_bounds, void* workspace, size_t workspace_bytes, void* stream);

/*
 * GMM2 (page section "5. GMM2"): for each valid expanded row d of expert e,
 *   c2[d][k] = binary16(float(sum_i q2[d,i] * w2[e][k][i]) * s2[e][k])
 *   q2_f16 [R][I] binary16-coded int8 codes; q2_bounds: NULL or their activation
 *   bounds (see "Activation bounds"); w2 in the layout d->weight_layout names; c2 [R][K]
 */
int32_t moe_gmm2(const moe_dims_t* d, const uint16_t* q2_f16, const int32_t* cumsum, const int32_t* q2_bounds,
                 const int8_t* w2, const float* s2, uint16_t* c2, void* workspace, size_t workspace_bytes,
                 void* stream);

/*
 * Combine + Unpermute (page sections "6. Combine" and "7. Unpermute"), fused:
 *   D = binary16(float(c2[d][k]) * pts2[d])
 *   out[t][k] = binary16(sum_{j=0..topK-1, route valid} float(D[expanded_row_idx[t*topK+j]][k]) * probs[t][j])
 * with an fp32 accumulator, slots in order, multiply then add.
 */
int32_t moe_combine_unpermute(const moe_dims_t* d, const uint16_t* c2, const float* pts2,
                              const int32_t* expanded_row_idx, const float* probs, uint16_t* out,
                              void* stream);

/* ------------------------------------------------------------------------ */
/* Diagnostics                                                               */
/* ------------------------------------------------------------------------ */

/*
 * Exercises the bounded device-side wait every pipeline kernel uses (failure
 * detection): a one-warp kernel waits on a barrier phase that nothing completes,
 * gives up after limit_us microseconds (1 .. 2,000,000) and writes MOE_ERR_TIMEOUT
 * to *status (device memory, cleared first).  The kernel returns normally; the
 * context stays usable.  Asynchronous on `stream`.
 */
int32_t moe_selftest_wait_timeout(int32_t* status, uint32_t limit_us, void* stream);

/*
 * The same for the bounded wait on a count raised by other CTAs (the per-expert item
 * counters the SwiGLU fused into GMM1 waits on, see moe_gmm1_swiglu): a one-warp kernel
 * clears *count (device int32), waits for it to reach 1, which nothing does, gives up
 * after limit_us microseconds (1 .. 2,000,000) and writes MOE_ERR_TIMEOUT to *status
 * (device memory, cleared first).  Asynchronous on `stream`.
 */
int32_t moe_selftest_count_timeout(int32_t* status, int32_t* count, uint32_t limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYER_H */
