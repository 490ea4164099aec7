// C ABI of the expert layer: host-side validation, workspace carving and the
// launch sequence of MegaMoe::Process() on one GPU (PTO-ISA MegaMoE operator
// page, section "key implementation logic").  See include/moe_layer.h for the
// contract of every entry point.
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include <cuda_runtime.h>

#include "../../include/moe_layer.h"
#include "abi_checks.h"
#include "kernels.h"

struct moe_layer_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

// The pipelined executor (include/moe_layer.h): per staging slot the inputs and
// output of one batch, its layer graph, and the events that order the three streams.
constexpr int kPipeMaxDepth = 8;
struct moe_layer_pipeline {
  int depth, device;
  size_t x_bytes, ei_bytes, pr_bytes, out_bytes;
  cudaStream_t copy_in, run, copy_out;
  cudaEvent_t in_done[kPipeMaxDepth], run_done[kPipeMaxDepth], out_done[kPipeMaxDepth];
  moe_layer_graph* graph[kPipeMaxDepth];
  uint16_t* x[kPipeMaxDepth];
  int32_t* ei[kPipeMaxDepth];
  float* pr[kPipeMaxDepth];
  uint16_t* out[kPipeMaxDepth];
  int32_t* status_dev[kPipeMaxDepth];  // the layer's status word, copied after each batch
  int32_t* status_host;                // page-locked, one word per slot
  uint64_t submitted, completed;       // batches submitted; batches known complete
  int32_t error;                       // first failure seen, and its batch
  uint64_t error_ticket;
};

namespace {

using moe::aligned16;
using moe::all_aligned16;
using moe::check_device;
using moe::check_dims;
using moe::check_shape;
using moe::launch_status;

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

// Tiles per 128-channel block of a GEMM's weights in the layout d names (0: rows).
int weight_kb(const moe_dims_t* d, int D) {
  return d->weight_layout == MOE_WEIGHTS_TILES ? moe::weight_tile_kb(D) : 0;
}

// Layout of the layer workspace.
struct Layout {
  size_t status, bounds1, bounds2, sw_done, zeroed, sorted, expanded, tpe, cumsum, sort_ws, a1, pts1, c1, q2, pts2, c2,
      total;
  // host-variant staging
  size_t hx, hei, hprobs, hout, host_total;
};

Layout layout_of(const moe_dims_t* d) {
  const size_t M = d->M, K = d->K, I = d->I, E = d->E, R = M * d->topK;
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  // status word, both bounds arrays and the fused SwiGLU's per-expert counters are
  // contiguous: one memset clears them
  L.status = 0;
  L.bounds1 = 16;
  L.bounds2 = L.bounds1 + E * moe::kBoundSegments * 4;
  L.sw_done = L.bounds2 + E * moe::kBoundSegments * 4;
  L.zeroed = L.sw_done + E * 4;
  take(L.zeroed);
  L.sorted = take(R * 4);
  L.expanded = take(R * 4);
  L.tpe = take(E * 4);
  L.cumsum = take(E * 4);
  L.sort_ws = take(moe::route_sort_workspace_bytes((int)R, (int)E));
  L.a1 = take(R * K * 2);
  L.pts1 = take(M * 4);
  L.c1 = take(R * 2 * I * 2);
  L.q2 = take(R * I * 2);
  L.pts2 = take(R * 4);
  L.c2 = take(R * K * 2);
  L.total = off;
  L.hx = take(M * K * 2);
  L.hei = take(R * 4);
  L.hprobs = take(R * 4);
  L.hout = take(M * K * 2);
  L.host_total = off;
  return L;
}

template <typename P>
P* at(void* base, size_t off) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(base) + off);
}

// The pipeline's workspace: the layer's, then `depth` staging slots (x, expert_idx,
// probs, out, status word), each part 256-byte aligned.
size_t pipeline_slot_bytes(const moe_dims_t* d) {
  const size_t M = d->M, K = d->K, R = M * d->topK;
  return align_up(M * K * 2) + align_up(R * 4) + align_up(R * 4) + align_up(M * K * 2) + align_up(16);
}

int32_t run_layer(const moe_dims_t* d, const uint16_t* x, const int32_t* expert_idx, const float* probs,
                  const int8_t* w1, const float* s1, const int8_t* w2, const float* s2, uint16_t* out,
                  void* ws, const Layout& L, cudaStream_t st) {
  const int M = d->M, K = d->K, I = d->I, E = d->E, topK = d->topK, R = M * topK;
  int32_t* status = at<int32_t>(ws, L.status);
  int32_t* sorted = at<int32_t>(ws, L.sorted);
  int32_t* expanded = at<int32_t>(ws, L.expanded);
  int32_t* tpe = at<int32_t>(ws, L.tpe);
  int32_t* cumsum = at<int32_t>(ws, L.cumsum);
  uint16_t* a1 = at<uint16_t>(ws, L.a1);
  float* pts1 = at<float>(ws, L.pts1);
  uint16_t* c1 = at<uint16_t>(ws, L.c1);
  uint16_t* q2 = at<uint16_t>(ws, L.q2);
  float* pts2 = at<float>(ws, L.pts2);
  uint16_t* c2 = at<uint16_t>(ws, L.c2);

  // activation bounds only where the GEMM engine reads them (above 24 rows per expert)
  const bool use_bounds = moe::grouped_gemm_reads_bounds(R, E);
  int32_t* bounds1 = use_bounds ? at<int32_t>(ws, L.bounds1) : nullptr;
  int32_t* bounds2 = use_bounds ? at<int32_t>(ws, L.bounds2) : nullptr;
  cudaError_t e;
  if ((e = cudaMemsetAsync(status, 0, L.zeroed, st)) != cudaSuccess) return launch_status(e);
  // FrontReorder: sort the routes, quantise each token once and scatter its codes to
  // its expert-major rows (a TMA gather of token rows inside GMM1 measured 1.2-3.2x
  // slower GMM1 on GB300: one gather4 moves 512 B, a tiled box up to 16 KB)
  if ((e = moe::launch_front_reorder(x, M, K, expert_idx, topK, E, sorted, expanded, tpe, cumsum, a1, pts1, bounds1,
                                     at<void>(ws, L.sort_ws), st)) != cudaSuccess)
    return launch_status(e);

  moe::GroupedGemmProblem g1{};
  g1.act = a1;
  g1.topK = topK;
  g1.act_rows = R;
  g1.cumsum = cumsum;
  g1.w = w1;
  g1.w_kb = weight_kb(d, K);
  g1.scale = s1;
  g1.C = c1;
  g1.R = R;
  g1.E = E;
  g1.N = 2 * I;
  g1.Kd = K;
  g1.status = status;
  g1.bounds = bounds1;
  // GMM1 and SwiGLU: the SwiGLU inside the GMM1 kernel when the tcgen05 pairs run
  if ((e = moe::launch_gemm1_swiglu(g1, I, topK, pts1, sorted, expert_idx, q2, pts2, bounds2,
                                    at<int32_t>(ws, L.sw_done), st)) != cudaSuccess)
    return launch_status(e);

  moe::GroupedGemmProblem g2{};
  g2.act = q2;
  g2.act_rows = R;
  g2.cumsum = cumsum;
  g2.w = w2;
  g2.w_kb = weight_kb(d, I);
  g2.scale = s2;
  g2.C = c2;
  g2.R = R;
  g2.E = E;
  g2.N = K;
  g2.Kd = I;
  g2.status = status;
  g2.bounds = bounds2;
  if ((e = moe::launch_grouped_gemm(g2, st)) != cudaSuccess) return launch_status(e);

  e = moe::launch_combine_unpermute(c2, pts2, expanded, probs, M, K, topK, out, st);
  return launch_status(e);
}

// moe_layer_fwd_host's work, enqueued on st without the final synchronisation:
// the per-call inputs copied into the workspace's staging, the layer, the output
// copied back.
int32_t enqueue_layer_host(const moe_dims_t* d, const uint16_t* x_host, const int32_t* expert_idx_host,
                           const float* probs_host, const int8_t* w1, const float* s1, const int8_t* w2,
                           const float* s2, uint16_t* out_host, void* workspace, size_t workspace_bytes,
                           cudaStream_t st) {
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!x_host || !expert_idx_host || !probs_host || !w1 || !s1 || !w2 || !s2 || !out_host || !workspace)
    return MOE_ERR_NULL;
  if (!aligned16(w1) || !aligned16(s1) || !aligned16(w2) || !aligned16(s2) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MOE_ERR_ALIGN;
  const Layout L = layout_of(d);
  if (workspace_bytes < L.host_total) return MOE_ERR_WORKSPACE;
  if ((rc = check_device()) != MOE_OK) return rc;
  const size_t M = d->M, K = d->K, R = M * d->topK;
  uint16_t* dx = at<uint16_t>(workspace, L.hx);
  int32_t* dei = at<int32_t>(workspace, L.hei);
  float* dpr = at<float>(workspace, L.hprobs);
  uint16_t* dout = at<uint16_t>(workspace, L.hout);
  if (cudaMemcpyAsync(dx, x_host, M * K * 2, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(dei, expert_idx_host, R * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(dpr, probs_host, R * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_ERR_LAUNCH;
  rc = run_layer(d, dx, dei, dpr, w1, s1, w2, s2, dout, workspace, L, st);
  if (rc != MOE_OK) return rc;
  if (cudaMemcpyAsync(out_host, dout, M * K * 2, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_LAUNCH;
  return MOE_OK;
}

// Records what `enqueue` puts on st (stream capture) and instantiates it.
template <class F>
int32_t capture_graph(cudaStream_t st, F enqueue, moe_layer_graph_t** graph) {
  if (!st) return MOE_ERR_LAUNCH;  // the legacy default stream cannot be captured
  if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return MOE_ERR_LAUNCH;
  const int32_t rc = enqueue();
  cudaGraph_t g = nullptr;
  const cudaError_t e_end = cudaStreamEndCapture(st, &g);
  if (rc != MOE_OK || e_end != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();  // a failed capture leaves no sticky error behind
    return rc != MOE_OK ? rc : MOE_ERR_LAUNCH;
  }
  cudaGraphExec_t exec = nullptr;
  if (cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    return MOE_ERR_LAUNCH;
  }
  moe_layer_graph_t* h = static_cast<moe_layer_graph_t*>(std::malloc(sizeof(moe_layer_graph_t)));
  if (!h) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(g);
    return MOE_ERR_LAUNCH;
  }
  h->graph = g;
  h->exec = exec;
  *graph = h;
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(int32_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "null pointer";
    case MOE_ERR_SHAPE: return "unsupported dimensions";
    case MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
    case MOE_ERR_ARCH: return "current device is not sm_103";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_LAUNCH: return "CUDA launch or copy failed";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

size_t moe_layer_workspace_size(const moe_dims_t* d) {
  if (check_dims(d) != MOE_OK) return 0;
  return layout_of(d).total;
}

size_t moe_layer_host_workspace_size(const moe_dims_t* d) {
  if (check_dims(d) != MOE_OK) return 0;
  return layout_of(d).host_total;
}

int32_t moe_layer_fwd(const moe_dims_t* d, const uint16_t* x, const int32_t* expert_idx, const float* probs,
                      const int8_t* w1, const float* s1, const int8_t* w2, const float* s2, uint16_t* out,
                      void* workspace, size_t workspace_bytes, void* stream) {
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!x || !expert_idx || !probs || !w1 || !s1 || !w2 || !s2 || !out || !workspace) return MOE_ERR_NULL;
  if (!aligned16(x) || !aligned16(expert_idx) || !aligned16(probs) || !aligned16(w1) || !aligned16(s1) ||
      !aligned16(w2) || !aligned16(s2) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MOE_ERR_ALIGN;
  const Layout L = layout_of(d);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  if ((rc = check_device()) != MOE_OK) return rc;
  return run_layer(d, x, expert_idx, probs, w1, s1, w2, s2, out, workspace, L, static_cast<cudaStream_t>(stream));
}

int32_t moe_layer_graph_create(const moe_dims_t* d, const uint16_t* x, const int32_t* expert_idx,
                               const float* probs, const int8_t* w1, const float* s1, const int8_t* w2,
                               const float* s2, uint16_t* out, void* workspace, size_t workspace_bytes,
                               void* stream, moe_layer_graph_t** graph) {
  if (!graph) return MOE_ERR_NULL;
  *graph = nullptr;
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!x || !expert_idx || !probs || !w1 || !s1 || !w2 || !s2 || !out || !workspace) return MOE_ERR_NULL;
  if (!aligned16(x) || !aligned16(expert_idx) || !aligned16(probs) || !aligned16(w1) || !aligned16(s1) ||
      !aligned16(w2) || !aligned16(s2) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MOE_ERR_ALIGN;
  const Layout L = layout_of(d);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (!stream) return MOE_ERR_LAUNCH;  // the legacy default stream cannot be captured
  if ((rc = check_device()) != MOE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return capture_graph(st, [&]() { return run_layer(d, x, expert_idx, probs, w1, s1, w2, s2, out, workspace, L, st); },
                       graph);
}

int32_t moe_layer_graph_launch(moe_layer_graph_t* graph, void* stream) {
  if (!graph) return MOE_ERR_NULL;
  return launch_status(cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)));
}

int32_t moe_layer_graph_destroy(moe_layer_graph_t* graph) {
  if (!graph) return MOE_OK;
  const cudaError_t a = cudaGraphExecDestroy(graph->exec);
  const cudaError_t b = cudaGraphDestroy(graph->graph);
  std::free(graph);
  return (a == cudaSuccess && b == cudaSuccess) ? MOE_OK : MOE_ERR_LAUNCH;
}

int32_t moe_layer_fwd_host(const moe_dims_t* d, const uint16_t* x_host, const int32_t* expert_idx_host,
                           const float* probs_host, const int8_t* w1, const float* s1, const int8_t* w2,
                           const float* s2, uint16_t* out_host, void* workspace, size_t workspace_bytes,
                           void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int32_t rc = enqueue_layer_host(d, x_host, expert_idx_host, probs_host, w1, s1, w2, s2, out_host, workspace,
                                        workspace_bytes, st);
  if (rc != MOE_OK) return rc;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_LAUNCH;
  return MOE_OK;
}

int32_t moe_layer_graph_create_host(const moe_dims_t* d, const uint16_t* x_host, const int32_t* expert_idx_host,
                                    const float* probs_host, const int8_t* w1, const float* s1, const int8_t* w2,
                                    const float* s2, uint16_t* out_host, void* workspace, size_t workspace_bytes,
                                    void* stream, moe_layer_graph_t** graph) {
  if (!graph) return MOE_ERR_NULL;
  *graph = nullptr;
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!x_host || !expert_idx_host || !probs_host || !w1 || !s1 || !w2 || !s2 || !out_host || !workspace)
    return MOE_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return capture_graph(st, [&]() {
    return enqueue_layer_host(d, x_host, expert_idx_host, probs_host, w1, s1, w2, s2, out_host, workspace,
                              workspace_bytes, st);
  }, graph);
}

size_t moe_layer_pipeline_workspace_size(const moe_dims_t* d, int32_t depth) {
  if (check_dims(d) != MOE_OK || depth < 1 || depth > kPipeMaxDepth) return 0;
  return layout_of(d).total + (size_t)depth * pipeline_slot_bytes(d);
}

namespace {

// Waits for batch t (the oldest not yet known complete) and folds in its status.
int32_t pipeline_retire(moe_layer_pipeline_t* p, uint64_t t) {
  const int s = (int)(t % (uint64_t)p->depth);
  int32_t rc = MOE_OK;
  if (cudaEventSynchronize(p->out_done[s]) != cudaSuccess)
    rc = MOE_ERR_LAUNCH;
  else if (p->status_host[s] != MOE_OK)
    rc = p->status_host[s];
  if (rc != MOE_OK && p->error == MOE_OK) {
    p->error = rc;
    p->error_ticket = t;
  }
  p->completed = t + 1;
  return rc;
}

void pipeline_release(moe_layer_pipeline_t* p) {
  if (p->run) {
    cudaStreamSynchronize(p->copy_in);
    cudaStreamSynchronize(p->run);
    cudaStreamSynchronize(p->copy_out);
  }
  for (int s = 0; s < kPipeMaxDepth; ++s) {
    moe_layer_graph_destroy(p->graph[s]);
    if (p->in_done[s]) cudaEventDestroy(p->in_done[s]);
    if (p->run_done[s]) cudaEventDestroy(p->run_done[s]);
    if (p->out_done[s]) cudaEventDestroy(p->out_done[s]);
  }
  if (p->copy_in) cudaStreamDestroy(p->copy_in);
  if (p->run) cudaStreamDestroy(p->run);
  if (p->copy_out) cudaStreamDestroy(p->copy_out);
  if (p->status_host) cudaFreeHost(p->status_host);
  std::free(p);
}

}  // namespace

int32_t moe_layer_pipeline_create(const moe_dims_t* d, const int8_t* w1, const float* s1, const int8_t* w2,
                                  const float* s2, void* workspace, size_t workspace_bytes, int32_t depth,
                                  moe_layer_pipeline_t** pipeline) {
  if (!pipeline) return MOE_ERR_NULL;
  *pipeline = nullptr;
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (depth < 1 || depth > kPipeMaxDepth) return MOE_ERR_SHAPE;
  if (!w1 || !s1 || !w2 || !s2 || !workspace) return MOE_ERR_NULL;
  if (!aligned16(w1) || !aligned16(s1) || !aligned16(w2) || !aligned16(s2) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MOE_ERR_ALIGN;
  const Layout L = layout_of(d);
  if (workspace_bytes < L.total + (size_t)depth * pipeline_slot_bytes(d)) return MOE_ERR_WORKSPACE;
  if ((rc = check_device()) != MOE_OK) return rc;
  moe_layer_pipeline_t* p = static_cast<moe_layer_pipeline_t*>(std::calloc(1, sizeof(moe_layer_pipeline_t)));
  if (!p) return MOE_ERR_LAUNCH;
  const size_t M = d->M, K = d->K, R = M * d->topK;
  p->depth = depth;
  p->x_bytes = M * K * 2;
  p->ei_bytes = R * 4;
  p->pr_bytes = R * 4;
  p->out_bytes = M * K * 2;
  bool ok = cudaGetDevice(&p->device) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->copy_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->run, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->copy_out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaHostAlloc(reinterpret_cast<void**>(&p->status_host), kPipeMaxDepth * sizeof(int32_t),
                          cudaHostAllocDefault) == cudaSuccess;
  size_t off = L.total;
  for (int s = 0; ok && s < depth; ++s) {
    p->x[s] = at<uint16_t>(workspace, off);
    off += align_up(p->x_bytes);
    p->ei[s] = at<int32_t>(workspace, off);
    off += align_up(p->ei_bytes);
    p->pr[s] = at<float>(workspace, off);
    off += align_up(p->pr_bytes);
    p->out[s] = at<uint16_t>(workspace, off);
    off += align_up(p->out_bytes);
    p->status_dev[s] = at<int32_t>(workspace, off);
    off += align_up(16);
    p->status_host[s] = MOE_OK;
    ok = cudaEventCreateWithFlags(&p->in_done[s], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->run_done[s], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->out_done[s], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) break;
    // the slot's layer graph: the layer on the slot's buffers, then its status word
    // copied out of the shared layer workspace
    const int32_t* ws_status = at<int32_t>(workspace, L.status);
    rc = capture_graph(p->run, [&]() {
      const int32_t r = run_layer(d, p->x[s], p->ei[s], p->pr[s], w1, s1, w2, s2, p->out[s], workspace, L, p->run);
      if (r != MOE_OK) return r;
      return launch_status(cudaMemcpyAsync(p->status_dev[s], ws_status, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                           p->run));
    }, &p->graph[s]);
    ok = rc == MOE_OK;
  }
  if (!ok) {
    pipeline_release(p);
    return rc != MOE_OK ? rc : MOE_ERR_LAUNCH;
  }
  *pipeline = p;
  return MOE_OK;
}

int32_t moe_layer_pipeline_submit(moe_layer_pipeline_t* p, const uint16_t* x_host, const int32_t* expert_idx_host,
                                  const float* probs_host, uint16_t* out_host, uint64_t* ticket) {
  if (!p || !x_host || !expert_idx_host || !probs_host || !out_host || !ticket) return MOE_ERR_NULL;
  if (cudaSetDevice(p->device) != cudaSuccess) return MOE_ERR_LAUNCH;
  const uint64_t n = p->submitted;
  const int s = (int)(n % (uint64_t)p->depth);
  // the slot's previous batch must be complete before its buffers and events are reused
  while (p->completed + (uint64_t)p->depth <= n) pipeline_retire(p, p->completed);
  bool ok = cudaMemcpyAsync(p->x[s], x_host, p->x_bytes, cudaMemcpyHostToDevice, p->copy_in) == cudaSuccess &&
            cudaMemcpyAsync(p->ei[s], expert_idx_host, p->ei_bytes, cudaMemcpyHostToDevice, p->copy_in) ==
                cudaSuccess &&
            cudaMemcpyAsync(p->pr[s], probs_host, p->pr_bytes, cudaMemcpyHostToDevice, p->copy_in) == cudaSuccess &&
            cudaEventRecord(p->in_done[s], p->copy_in) == cudaSuccess;
  ok = ok && cudaStreamWaitEvent(p->run, p->in_done[s], 0) == cudaSuccess &&
       cudaGraphLaunch(p->graph[s]->exec, p->run) == cudaSuccess &&
       cudaEventRecord(p->run_done[s], p->run) == cudaSuccess;
  ok = ok && cudaStreamWaitEvent(p->copy_out, p->run_done[s], 0) == cudaSuccess &&
       cudaMemcpyAsync(out_host, p->out[s], p->out_bytes, cudaMemcpyDeviceToHost, p->copy_out) == cudaSuccess &&
       cudaMemcpyAsync(p->status_host + s, p->status_dev[s], sizeof(int32_t), cudaMemcpyDeviceToHost,
                       p->copy_out) == cudaSuccess &&
       cudaEventRecord(p->out_done[s], p->copy_out) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return MOE_ERR_LAUNCH;
  }
  p->submitted = n + 1;
  *ticket = n;
  return MOE_OK;
}

int32_t moe_layer_pipeline_wait(moe_layer_pipeline_t* p, uint64_t ticket) {
  if (!p) return MOE_ERR_NULL;
  if (ticket >= p->submitted) return MOE_ERR_SHAPE;
  if (cudaSetDevice(p->device) != cudaSuccess) return MOE_ERR_LAUNCH;
  while (p->completed <= ticket) pipeline_retire(p, p->completed);
  return (p->error != MOE_OK && p->error_ticket <= ticket) ? p->error : MOE_OK;
}

int32_t moe_layer_pipeline_destroy(moe_layer_pipeline_t* p) {
  if (!p) return MOE_OK;
  cudaSetDevice(p->device);
  pipeline_release(p);
  return MOE_OK;
}

int32_t moe_workspace_status(const void* workspace, int32_t* host_status, void* stream) {
  if (!workspace || !host_status) return MOE_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_status, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_LAUNCH;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_LAUNCH;
  return MOE_OK;
}

int32_t moe_workspace_clear_status(void* workspace, void* stream) {
  if (!workspace) return MOE_ERR_NULL;
  return launch_status(cudaMemsetAsync(workspace, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)));
}

// ----------------------------------------------------------------------------- stages

size_t moe_route_sort_workspace_size(const moe_dims_t* d) {
  if (check_dims(d) != MOE_OK) return 0;
  return moe::route_sort_workspace_bytes(d->M * d->topK, d->E);
}

int32_t moe_route_sort(const moe_dims_t* d, const int32_t* expert_idx, int32_t* sorted_src_route,
                       int32_t* expanded_row_idx, int32_t* tokens_per_expert, int32_t* cumsum, void* workspace,
                       size_t workspace_bytes, void* stream) {
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!expert_idx || !sorted_src_route || !expanded_row_idx || !tokens_per_expert || !cumsum) return MOE_ERR_NULL;
  if (!all_aligned16({expert_idx, sorted_src_route, expanded_row_idx, tokens_per_expert, cumsum, workspace}))
    return MOE_ERR_ALIGN;
  const size_t need = moe::route_sort_workspace_bytes(d->M * d->topK, d->E);
  if (need && (!workspace || workspace_bytes < need)) return MOE_ERR_WORKSPACE;
  if ((rc = check_device()) != MOE_OK) return rc;
  return launch_status(moe::launch_route_sort(expert_idx, d->M * d->topK, d->E, sorted_src_route, expanded_row_idx,
                                              tokens_per_expert, cumsum, workspace,
                                              static_cast<cudaStream_t>(stream)));
}

int32_t moe_quant_tokens(const moe_dims_t* d, const uint16_t* x, const int32_t* expert_idx, int8_t* xq_i8,
                         uint16_t* xq_f16, float* pts1, int32_t* a1_bounds, void* stream) {
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!x || !pts1 || (!xq_i8 && !xq_f16) || (a1_bounds && !expert_idx)) return MOE_ERR_NULL;
  if (!all_aligned16({x, expert_idx, xq_i8, xq_f16, pts1, a1_bounds})) return MOE_ERR_ALIGN;
  if ((rc = check_device()) != MOE_OK) return rc;
  return launch_status(moe::launch_quant_tokens(x, d->M, d->K, xq_i8, xq_f16, pts1, nullptr, d->topK, nullptr,
                                                expert_idx, d->E, a1_bounds, static_cast<cudaStream_t>(stream)));
}

int32_t moe_quant_dispatch(const moe_dims_t* d, const uint16_t* x, const int32_t* expert_idx,
                           const int32_t* expanded_row_idx, uint16_t* a1_f16, float* pts1, int32_t* a1_bounds,
                           void* stream) {
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!x || !expanded_row_idx || !a1_f16 || !pts1 || (a1_bounds && !expert_idx)) return MOE_ERR_NULL;
  if (!all_aligned16({x, expert_idx, expanded_row_idx, a1_f16, pts1, a1_bounds})) return MOE_ERR_ALIGN;
  if ((rc = check_device()) != MOE_OK) return rc;
  return launch_status(moe::launch_quant_tokens(x, d->M, d->K, nullptr, nullptr, pts1, expanded_row_idx, d->topK,
                                                a1_f16, expert_idx, d->E, a1_bounds,
                                                static_cast<cudaStream_t>(stream)));
}

int32_t moe_front_reorder(const moe_dims_t* d, const uint16_t* x, const int32_t* expert_idx,
                          int32_t* sorted_src_route, int32_t* expanded_row_idx, int32_t* tokens_per_expert,
                          int32_t* cumsum, uint16_t* a1_f16, float* pts1, int32_t* a1_bounds, void* workspace,
                          size_t workspace_bytes, void* stream) {
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!x || !expert_idx || !sorted_src_route || !expanded_row_idx || !tokens_per_expert || !cumsum || !a1_f16 ||
      !pts1)
    return MOE_ERR_NULL;
  if (!all_aligned16({x, expert_idx, sorted_src_route, expanded_row_idx, tokens_per_expert, cumsum, a1_f16, pts1,
                      a1_bounds, workspace}))
    return MOE_ERR_ALIGN;
  const size_t need = moe::route_sort_workspace_bytes(d->M * d->topK, d->E);
  if (need && (!workspace || workspace_bytes < need)) return MOE_ERR_WORKSPACE;
  if ((rc = check_device()) != MOE_OK) return rc;
  return launch_status(moe::launch_front_reorder(x, d->M, d->K, expert_idx, d->topK, d->E, sorted_src_route,
                                                 expanded_row_idx, tokens_per_expert, cumsum, a1_f16, pts1, a1_bounds,
                                                 workspace, static_cast<cudaStream_t>(stream)));
}

// GEMM stage workspace: the status word, then (moe_gmm1_swiglu) E int32 counters.
constexpr size_t kGmmCounters = 16;
size_t moe_gmm_workspace_size(const moe_dims_t* d) {
  if (check_dims(d) != MOE_OK) return 0;
  return align_up(kGmmCounters + (size_t)d->E * 4);
}

size_t moe_weight_tiles_bytes(const moe_dims_t* d, int32_t gemm) {
  if (check_shape(d) != MOE_OK || (gemm != 1 && gemm != 2)) return 0;
  return gemm == 1 ? moe::weight_tiles_bytes(d->E, 2 * d->I, d->K) : moe::weight_tiles_bytes(d->E, d->K, d->I);
}

int32_t moe_pack_weight_tiles(const moe_dims_t* d, int32_t gemm, const int8_t* w, int8_t* tiles, void* stream) {
  int32_t rc = check_shape(d);
  if (rc != MOE_OK) return rc;
  if (gemm != 1 && gemm != 2) return MOE_ERR_SHAPE;
  if (!w || !tiles) return MOE_ERR_NULL;
  if (!aligned16(w) || !aligned16(tiles)) return MOE_ERR_ALIGN;
  if ((rc = check_device()) != MOE_OK) return rc;
  const int N = gemm == 1 ? 2 * d->I : d->K, D = gemm == 1 ? d->K : d->I;
  return launch_status(moe::launch_pack_weight_tiles(w, d->E, N, D, tiles, static_cast<cudaStream_t>(stream)));
}

int32_t moe_gmm1(const moe_dims_t* d, const uint16_t* a1_f16, const int32_t* sorted_src_route, const int32_t* cumsum,
                 const int32_t* a1_bounds, const int8_t* w1, const float* s1, uint16_t* c1, void* workspace,
                 size_t workspace_bytes, void* stream) {
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!a1_f16 || !cumsum || !w1 || !s1 || !c1 || !workspace) return MOE_ERR_NULL;
  if (!all_aligned16({a1_f16, sorted_src_route, cumsum, a1_bounds, w1, s1, c1, workspace})) return MOE_ERR_ALIGN;
  if (workspace_bytes < moe_gmm_workspace_size(d)) return MOE_ERR_WORKSPACE;
  if ((rc = check_device()) != MOE_OK) return rc;
  moe::GroupedGemmProblem g{};
  g.act = a1_f16;
  g.gather_route = sorted_src_route;
  g.topK = d->topK;
  g.act_rows = sorted_src_route ? d->M : d->M * d->topK;
  g.cumsum = cumsum;
  g.w = w1;
  g.w_kb = weight_kb(d, d->K);
  g.scale = s1;
  g.C = c1;
  g.R = d->M * d->topK;
  g.E = d->E;
  g.N = 2 * d->I;
  g.Kd = d->K;
  g.status = static_cast<int32_t*>(workspace);
  g.bounds = a1_bounds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_LAUNCH;
  return launch_status(moe::launch_grouped_gemm(g, st));
}

int32_t moe_swiglu_quant(const moe_dims_t* d, const uint16_t* c1, const float* pts1, const int32_t* sorted_src_route,
                         const int32_t* cumsum, const int32_t* expert_idx, int8_t* q2_i8, uint16_t* q2_f16,
                         float* pts2, int32_t* q2_bounds, void* stream) {
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!c1 || !pts1 || !sorted_src_route || !cumsum || !pts2 || (!q2_i8 && !q2_f16) || (q2_bounds && !expert_idx))
    return MOE_ERR_NULL;
  if (!all_aligned16({c1, pts1, sorted_src_route, cumsum, expert_idx, q2_i8, q2_f16, pts2, q2_bounds}))
    return MOE_ERR_ALIGN;
  if ((rc = check_device()) != MOE_OK) return rc;
  return launch_status(moe::launch_swiglu_quant(c1, d->M * d->topK, d->I, d->E, d->topK, pts1, sorted_src_route,
                                                cumsum, q2_i8, q2_f16, pts2, expert_idx, q2_bounds,
                                                static_cast<cudaStream_t>(stream)));
}

int32_t moe_gmm1_swiglu(const moe_dims_t* d, const uint16_t* a1_f16, const int32_t* cumsum, const int32_t* a1_bounds,
                        const int8_t* w1, const float* s1, uint16_t* c1, const float* pts1,
                        const int32_t* sorted_src_route, const int32_t* expert_idx, uint16_t* q2_f16, float* pts2,
                        int32_t* q2_bounds, void* workspace, size_t workspace_bytes, void* stream) {
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!a1_f16 || !cumsum || !w1 || !s1 || !c1 || !pts1 || !sorted_src_route || !q2_f16 || !pts2 || !workspace ||
      (q2_bounds && !expert_idx))
    return MOE_ERR_NULL;
  if (!all_aligned16({a1_f16, cumsum, a1_bounds, w1, s1, c1, pts1, sorted_src_route, expert_idx, q2_f16, pts2,
                      q2_bounds, workspace}))
    return MOE_ERR_ALIGN;
  if (workspace_bytes < moe_gmm_workspace_size(d)) return MOE_ERR_WORKSPACE;
  if ((rc = check_device()) != MOE_OK) return rc;
  moe::GroupedGemmProblem g{};
  g.act = a1_f16;
  g.topK = d->topK;
  g.act_rows = d->M * d->topK;
  g.cumsum = cumsum;
  g.w = w1;
  g.w_kb = weight_kb(d, d->K);
  g.scale = s1;
  g.C = c1;
  g.R = d->M * d->topK;
  g.E = d->E;
  g.N = 2 * d->I;
  g.Kd = d->K;
  g.status = static_cast<int32_t*>(workspace);
  g.bounds = a1_bounds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, kGmmCounters + (size_t)d->E * 4, st) != cudaSuccess) return MOE_ERR_LAUNCH;
  int32_t* counters = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + kGmmCounters);
  return launch_status(moe::launch_gemm1_swiglu(g, d->I, d->topK, pts1, sorted_src_route, expert_idx, q2_f16, pts2,
                                                q2_bounds, counters, st));
}

int32_t moe_gmm2(const moe_dims_t* d, const uint16_t* q2_f16, const int32_t* cumsum, const int32_t* q2_bounds,
                 const int8_t* w2, const float* s2, uint16_t* c2, void* workspace, size_t workspace_bytes,
                 void* stream) {
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!q2_f16 || !cumsum || !w2 || !s2 || !c2 || !workspace) return MOE_ERR_NULL;
  if (!all_aligned16({q2_f16, cumsum, q2_bounds, w2, s2, c2, workspace})) return MOE_ERR_ALIGN;
  if (workspace_bytes < moe_gmm_workspace_size(d)) return MOE_ERR_WORKSPACE;
  if ((rc = check_device()) != MOE_OK) return rc;
  moe::GroupedGemmProblem g{};
  g.act = q2_f16;
  g.act_rows = d->M * d->topK;
  g.cumsum = cumsum;
  g.w = w2;
  g.w_kb = weight_kb(d, d->I);
  g.scale = s2;
  g.C = c2;
  g.R = d->M * d->topK;
  g.E = d->E;
  g.N = d->K;
  g.Kd = d->I;
  g.status = static_cast<int32_t*>(workspace);
  g.bounds = q2_bounds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_LAUNCH;
  return launch_status(moe::launch_grouped_gemm(g, st));
}

int32_t moe_combine_unpermute(const moe_dims_t* d, const uint16_t* c2, const float* pts2,
                              const int32_t* expanded_row_idx, const float* probs, uint16_t* out, void* stream) {
  int32_t rc = check_dims(d);
  if (rc != MOE_OK) return rc;
  if (!c2 || !pts2 || !expanded_row_idx || !probs || !out) return MOE_ERR_NULL;
  if (!all_aligned16({c2, pts2, expanded_row_idx, probs, out})) return MOE_ERR_ALIGN;
  if ((rc = check_device()) != MOE_OK) return rc;
  return launch_status(moe::launch_combine_unpermute(c2, pts2, expanded_row_idx, probs, d->M, d->K, d->topK, out,
                                                     static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
