"""GB300 (sm_103a) W8A8 mixture-of-experts expert layer.

Thin Python binding over the C ABI in ``include/moe_layer.h`` (library
``_build/libmoe_layer.so``, built by ``moe_expert_layer_gb300.build``).  The
functions below carry the ABI's names and only marshal arguments: torch
tensors (device memory) become raw pointers, the stream defaults to torch's
current stream, and a non-zero status raises ``MoeError``.  Every stage of the
layer runs in the library's CUDA kernels; there is no other code path, and
importing the binding fails loudly when the library is missing.
"""
import ctypes
import os

from . import build as _build

LIB_PATH = _build.LIB_PATH

STATUS = {0: "MOE_OK", -1: "MOE_ERR_NULL", -2: "MOE_ERR_SHAPE", -3: "MOE_ERR_ALIGN",
          -4: "MOE_ERR_ARCH", -5: "MOE_ERR_WORKSPACE", -6: "MOE_ERR_LAUNCH",
          -8: "MOE_ERR_TIMEOUT"}

# every entry point declared in include/moe_layer.h
EXPORTS = [
    "moe_status_string", "moe_layer_workspace_size", "moe_layer_fwd",
    "moe_layer_host_workspace_size", "moe_layer_fwd_host", "moe_workspace_status",
    "moe_workspace_clear_status", "moe_route_sort_workspace_size", "moe_route_sort",
    "moe_quant_tokens", "moe_quant_dispatch", "moe_front_reorder", "moe_gmm_workspace_size", "moe_gmm1",
    "moe_swiglu_quant", "moe_gmm1_swiglu", "moe_gmm2", "moe_combine_unpermute", "moe_route_sort_noalloc",
    "moe_selftest_wait_timeout", "moe_selftest_count_timeout",
    "moe_layer_graph_create", "moe_layer_graph_create_host", "moe_layer_graph_launch", "moe_layer_graph_destroy",
    "moe_layer_pipeline_workspace_size", "moe_layer_pipeline_create", "moe_layer_pipeline_submit",
    "moe_layer_pipeline_wait", "moe_layer_pipeline_destroy",
    "moe_weight_tiles_bytes", "moe_pack_weight_tiles",
]

# weight layouts (moe_dims_t.weight_layout)
WEIGHTS_ROWS = 0
WEIGHTS_TILES = 1


class MoeError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (fn, STATUS.get(code, "unknown"), code))


class moe_dims_t(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int32), ("K", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("topK", ctypes.c_int32), ("weight_layout", ctypes.c_int32)]


def dims(M, K, I, E, topK, weight_layout=WEIGHTS_ROWS):
    return moe_dims_t(M, K, I, E, topK, weight_layout)


_lib = None


def load_library(path=None):
    """Loads the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise ImportError("libmoe_layer.so not built (run moe_expert_layer_gb300.build.build())")
    lib = ctypes.CDLL(path)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    D = ctypes.POINTER(moe_dims_t)
    sigs = {
        "moe_status_string": ([i32], ctypes.c_char_p),
        "moe_layer_workspace_size": ([D], sz),
        "moe_layer_host_workspace_size": ([D], sz),
        "moe_layer_fwd": ([D] + [vp] * 9 + [sz, vp], i32),
        "moe_layer_fwd_host": ([D] + [vp] * 9 + [sz, vp], i32),
        "moe_layer_graph_create": ([D] + [vp] * 9 + [sz, vp, ctypes.POINTER(vp)], i32),
        "moe_layer_graph_create_host": ([D] + [vp] * 9 + [sz, vp, ctypes.POINTER(vp)], i32),
        "moe_layer_graph_launch": ([vp, vp], i32),
        "moe_layer_graph_destroy": ([vp], i32),
        "moe_layer_pipeline_workspace_size": ([D, i32], sz),
        "moe_layer_pipeline_create": ([D] + [vp] * 5 + [sz, i32, ctypes.POINTER(vp)], i32),
        "moe_layer_pipeline_submit": ([vp] * 5 + [ctypes.POINTER(ctypes.c_uint64)], i32),
        "moe_layer_pipeline_wait": ([vp, ctypes.c_uint64], i32),
        "moe_layer_pipeline_destroy": ([vp], i32),
        "moe_workspace_status": ([vp, ctypes.POINTER(i32), vp], i32),
        "moe_workspace_clear_status": ([vp, vp], i32),
        "moe_route_sort_workspace_size": ([D], sz),
        "moe_route_sort": ([D] + [vp] * 6 + [sz, vp], i32),
        "moe_quant_tokens": ([D] + [vp] * 7, i32),
        "moe_gmm_workspace_size": ([D], sz),
        "moe_quant_dispatch": ([D] + [vp] * 7, i32),
        "moe_front_reorder": ([D] + [vp] * 10 + [sz, vp], i32),
        "moe_gmm1": ([D] + [vp] * 8 + [sz, vp], i32),
        "moe_swiglu_quant": ([D] + [vp] * 10, i32),
        "moe_gmm1_swiglu": ([D] + [vp] * 13 + [sz, vp], i32),
        "moe_gmm2": ([D] + [vp] * 7 + [sz, vp], i32),
        "moe_combine_unpermute": ([D] + [vp] * 6, i32),
        "moe_route_sort_noalloc": ([D] + [vp] * 6, i32),
        "moe_selftest_wait_timeout": ([vp, ctypes.c_uint32, vp], i32),
        "moe_selftest_count_timeout": ([vp, vp, ctypes.c_uint32, vp], i32),
        "moe_weight_tiles_bytes": ([D, i32], sz),
        "moe_pack_weight_tiles": ([D, i32, vp, vp, vp], i32),
    }
    for name, (args, res) in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _p(t):
    """Raw pointer of a tensor (device or host), or None.  The ABI takes dense
    row-major arrays, so a tensor with any other strides (a transpose, a column
    slice, an expanded view) is refused rather than read with the wrong layout."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("the C ABI takes dense row-major arrays; got a tensor with shape %s and strides %s"
                         % (tuple(t.shape), tuple(t.stride())))
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, code):
    if code != 0:
        raise MoeError(fn, code)


def moe_layer_workspace_size(d):
    return load_library().moe_layer_workspace_size(ctypes.byref(d))


def moe_layer_host_workspace_size(d):
    return load_library().moe_layer_host_workspace_size(ctypes.byref(d))


def moe_route_sort_workspace_size(d):
    return load_library().moe_route_sort_workspace_size(ctypes.byref(d))


def moe_gmm_workspace_size(d):
    return load_library().moe_gmm_workspace_size(ctypes.byref(d))


def moe_weight_tiles_bytes(d, gemm):
    return load_library().moe_weight_tiles_bytes(ctypes.byref(d), gemm)


def moe_pack_weight_tiles(d, gemm, w, tiles, stream=None):
    _check("moe_pack_weight_tiles", load_library().moe_pack_weight_tiles(
        ctypes.byref(d), gemm, _p(w), _p(tiles), _stream(stream)))


def moe_layer_fwd(d, x, expert_idx, probs, w1, s1, w2, s2, out, workspace, stream=None):
    _check("moe_layer_fwd", load_library().moe_layer_fwd(
        ctypes.byref(d), _p(x), _p(expert_idx), _p(probs), _p(w1), _p(s1), _p(w2), _p(s2), _p(out),
        _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_layer_graph_create(d, x, expert_idx, probs, w1, s1, w2, s2, out, workspace, stream):
    """Records moe_layer_fwd on these buffers as a CUDA graph; returns the handle."""
    h = ctypes.c_void_p()
    _check("moe_layer_graph_create", load_library().moe_layer_graph_create(
        ctypes.byref(d), _p(x), _p(expert_idx), _p(probs), _p(w1), _p(s1), _p(w2), _p(s2), _p(out),
        _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream), ctypes.byref(h)))
    return h


def moe_layer_graph_create_host(d, x_host, expert_idx_host, probs_host, w1, s1, w2, s2, out_host, workspace,
                                stream):
    """Records moe_layer_fwd_host (copies included, no synchronisation) as a CUDA graph."""
    h = ctypes.c_void_p()
    _check("moe_layer_graph_create_host", load_library().moe_layer_graph_create_host(
        ctypes.byref(d), _p(x_host), _p(expert_idx_host), _p(probs_host), _p(w1), _p(s1), _p(w2), _p(s2),
        _p(out_host), _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream),
        ctypes.byref(h)))
    return h


def moe_layer_graph_launch(graph, stream=None):
    _check("moe_layer_graph_launch", load_library().moe_layer_graph_launch(graph, _stream(stream)))


def moe_layer_graph_destroy(graph):
    _check("moe_layer_graph_destroy", load_library().moe_layer_graph_destroy(graph))


def moe_layer_pipeline_workspace_size(d, depth):
    return load_library().moe_layer_pipeline_workspace_size(ctypes.byref(d), depth)


def moe_layer_pipeline_create(d, w1, s1, w2, s2, workspace, depth=2):
    """The pipelined host-memory executor; returns its handle."""
    h = ctypes.c_void_p()
    _check("moe_layer_pipeline_create", load_library().moe_layer_pipeline_create(
        ctypes.byref(d), _p(w1), _p(s1), _p(w2), _p(s2), _p(workspace),
        workspace.numel() * workspace.element_size(), depth, ctypes.byref(h)))
    return h


def moe_layer_pipeline_submit(pipeline, x_host, expert_idx_host, probs_host, out_host):
    """Enqueues one batch (host tensors); returns its ticket."""
    t = ctypes.c_uint64()
    _check("moe_layer_pipeline_submit", load_library().moe_layer_pipeline_submit(
        pipeline, _p(x_host), _p(expert_idx_host), _p(probs_host), _p(out_host), ctypes.byref(t)))
    return t.value


def moe_layer_pipeline_wait(pipeline, ticket):
    _check("moe_layer_pipeline_wait", load_library().moe_layer_pipeline_wait(pipeline, ticket))


def moe_layer_pipeline_destroy(pipeline):
    _check("moe_layer_pipeline_destroy", load_library().moe_layer_pipeline_destroy(pipeline))


def moe_layer_fwd_host(d, x_host, expert_idx_host, probs_host, w1, s1, w2, s2, out_host, workspace,
                       stream=None):
    _check("moe_layer_fwd_host", load_library().moe_layer_fwd_host(
        ctypes.byref(d), _p(x_host), _p(expert_idx_host), _p(probs_host), _p(w1), _p(s1), _p(w2),
        _p(s2), _p(out_host), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def moe_workspace_status(workspace, stream=None):
    st = ctypes.c_int32(0)
    _check("moe_workspace_status",
           load_library().moe_workspace_status(_p(workspace), ctypes.byref(st), _stream(stream)))
    return st.value


def moe_workspace_clear_status(workspace, stream=None):
    _check("moe_workspace_clear_status",
           load_library().moe_workspace_clear_status(_p(workspace), _stream(stream)))


def moe_route_sort(d, expert_idx, sorted_src_route, expanded_row_idx, tokens_per_expert, cumsum,
                   workspace=None, stream=None):
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("moe_route_sort", load_library().moe_route_sort(
        ctypes.byref(d), _p(expert_idx), _p(sorted_src_route), _p(expanded_row_idx),
        _p(tokens_per_expert), _p(cumsum), _p(workspace), nbytes, _stream(stream)))


def moe_quant_tokens(d, x, expert_idx, xq_i8, xq_f16, pts1, a1_bounds, stream=None):
    _check("moe_quant_tokens", load_library().moe_quant_tokens(
        ctypes.byref(d), _p(x), _p(expert_idx), _p(xq_i8), _p(xq_f16), _p(pts1), _p(a1_bounds), _stream(stream)))


def moe_quant_dispatch(d, x, expert_idx, expanded_row_idx, a1_f16, pts1, a1_bounds, stream=None):
    _check("moe_quant_dispatch", load_library().moe_quant_dispatch(
        ctypes.byref(d), _p(x), _p(expert_idx), _p(expanded_row_idx), _p(a1_f16), _p(pts1), _p(a1_bounds),
        _stream(stream)))


def moe_front_reorder(d, x, expert_idx, sorted_src_route, expanded_row_idx, tokens_per_expert, cumsum, a1_f16,
                      pts1, a1_bounds, workspace=None, stream=None):
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("moe_front_reorder", load_library().moe_front_reorder(
        ctypes.byref(d), _p(x), _p(expert_idx), _p(sorted_src_route), _p(expanded_row_idx), _p(tokens_per_expert),
        _p(cumsum), _p(a1_f16), _p(pts1), _p(a1_bounds), _p(workspace), nbytes, _stream(stream)))


def moe_gmm1(d, a1_f16, sorted_src_route, cumsum, a1_bounds, w1, s1, c1, workspace, stream=None):
    _check("moe_gmm1", load_library().moe_gmm1(
        ctypes.byref(d), _p(a1_f16), _p(sorted_src_route), _p(cumsum), _p(a1_bounds), _p(w1), _p(s1), _p(c1),
        _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_swiglu_quant(d, c1, pts1, sorted_src_route, cumsum, expert_idx, q2_i8, q2_f16, pts2, q2_bounds,
                     stream=None):
    _check("moe_swiglu_quant", load_library().moe_swiglu_quant(
        ctypes.byref(d), _p(c1), _p(pts1), _p(sorted_src_route), _p(cumsum), _p(expert_idx), _p(q2_i8),
        _p(q2_f16), _p(pts2), _p(q2_bounds), _stream(stream)))


def moe_gmm1_swiglu(d, a1_f16, cumsum, a1_bounds, w1, s1, c1, pts1, sorted_src_route, expert_idx, q2_f16, pts2,
                    q2_bounds, workspace, stream=None):
    _check("moe_gmm1_swiglu", load_library().moe_gmm1_swiglu(
        ctypes.byref(d), _p(a1_f16), _p(cumsum), _p(a1_bounds), _p(w1), _p(s1), _p(c1), _p(pts1),
        _p(sorted_src_route), _p(expert_idx), _p(q2_f16), _p(pts2), _p(q2_bounds), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_gmm2(d, q2_f16, cumsum, q2_bounds, w2, s2, c2, workspace, stream=None):
    _check("moe_gmm2", load_library().moe_gmm2(
        ctypes.byref(d), _p(q2_f16), _p(cumsum), _p(q2_bounds), _p(w2), _p(s2), _p(c2), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_combine_unpermute(d, c2, pts2, expanded_row_idx, probs, out, stream=None):
    _check("moe_combine_unpermute", load_library().moe_combine_unpermute(
        ctypes.byref(d), _p(c2), _p(pts2), _p(expanded_row_idx), _p(probs), _p(out),
        _stream(stream)))


def moe_selftest_wait_timeout(status, limit_us, stream=None):
    """Runs the bounded-wait self-test; status (int32 device tensor) receives the code."""
    _check("moe_selftest_wait_timeout", load_library().moe_selftest_wait_timeout(
        _p(status), limit_us, _stream(stream)))


def moe_selftest_count_timeout(status, count, limit_us, stream=None):
    """Runs the bounded count-wait self-test; status and count are int32 device tensors."""
    _check("moe_selftest_count_timeout", load_library().moe_selftest_count_timeout(
        _p(status), _p(count), limit_us, _stream(stream)))


# Largest route count (M * topK) moe_route_sort_noalloc accepts (its fixed scratch).
ROUTE_SORT_NOALLOC_MAX_ROUTES = 524288

# Activation bounds arrays: int32 [E][BOUND_SEGMENTS], one entry per BOUND_SEGMENT-deep
# segment of the reduction dimension (include/moe_layer.h, "Activation bounds").
BOUND_SEGMENT = 1024
BOUND_SEGMENTS = 16


def moe_route_sort_noalloc(d, expert_idx, sorted_src_route, expanded_row_idx, tokens_per_expert,
                           cumsum, stream=None):
    """moe_route_sort without a workspace, for callers that cannot allocate device
    memory; its scratch is a fixed array inside the library (see the header)."""
    _check("moe_route_sort_noalloc", load_library().moe_route_sort_noalloc(
        ctypes.byref(d), _p(expert_idx), _p(sorted_src_route), _p(expanded_row_idx),
        _p(tokens_per_expert), _p(cumsum), _stream(stream)))
