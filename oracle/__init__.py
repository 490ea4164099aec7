"""CPU oracle of the W8A8 MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product (the CUDA library
in ``moe_expert_layer_gb300``) never calls it.

The arithmetic lives in ``moe_oracle.c`` (plain C, scalar IEEE fp32, built
with ``-ffp-contract=off``), which restates the seven stages of the PTO-ISA
MegaMoE operator page on one rank.  This module compiles it and wraps each
entry point for numpy arrays.  Pins: ``tests/test_oracle.py``.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lib = None

CFLAGS = ["-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
          "-shared"]


def build(force=False):
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc"] + CFLAGS + [_SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        ci, vp, i64 = ctypes.c_int, ctypes.c_void_p, ctypes.c_int64
        sig = {
            "oracle_f16_to_f32": ([i64, vp, vp], None),
            "oracle_f32_to_f16": ([i64, vp, vp], None),
            "oracle_f32_to_f16_sat": ([i64, vp, vp], None),
            "oracle_route_sort": ([ci, ci, ci, vp, vp, vp, vp, vp], ci),
            "oracle_quant_tokens": ([ci, ci, vp, vp, vp], None),
            "oracle_gmm1": ([ci, ci, ci, ci, ci, vp, vp, vp, vp, vp, ci, vp, vp], None),
            "oracle_swiglu_quant": ([ci, ci, ci, vp, vp, vp, vp, vp], None),
            "oracle_gmm2": ([ci, ci, ci, vp, vp, vp, vp, vp, ci, vp, vp], None),
            "oracle_combine": ([ci, ci, vp, vp, vp], None),
            "oracle_unpermute": ([ci, ci, ci, vp, vp, vp, vp], None),
            "oracle_layer_fwd": ([ci] * 5 + [vp] * 18, ci),
            "oracle_layer_tokens": ([ci] * 5 + [vp] * 7 + [ci, vp, vp], None),
            "oracle_max_threads": ([], ci),
            "oracle_set_threads": ([ci], None),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _h(a):
    """float16 array -> contiguous uint16 bit view"""
    return np.ascontiguousarray(a, dtype=np.float16).view(np.uint16)


def f16_to_f32(bits):
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float32)
    _load().oracle_f16_to_f32(bits.size, _p(bits), _p(out))
    return out


def f32_to_f16(vals):
    vals = _c(vals, np.float32)
    out = np.empty(vals.shape, np.uint16)
    _load().oracle_f32_to_f16(vals.size, _p(vals), _p(out))
    return out.view(np.float16)


def f32_to_f16_sat(vals):
    """Stage-output conversion: RNE, saturating at +-65504."""
    vals = _c(vals, np.float32)
    out = np.empty(vals.shape, np.uint16)
    _load().oracle_f32_to_f16_sat(vals.size, _p(vals), _p(out))
    return out.view(np.float16)


def route_sort(expert_idx, E):
    """FrontReorder sort/count/invert/prefix.  Returns dict with
    sorted_src_route[R], expanded_row_idx[R], tokens_per_expert[E], cumsum[E],
    invalid (number of routes with an expert id outside [0, E))."""
    ei = _c(expert_idx, np.int32)
    M, topK = ei.shape
    R = M * topK
    s = np.empty(R, np.int32)
    x = np.empty(R, np.int32)
    tpe = np.empty(E, np.int32)
    cs = np.empty(E, np.int32)
    inv = _load().oracle_route_sort(M, topK, E, _p(ei), _p(s), _p(x), _p(tpe), _p(cs))
    return {"sorted_src_route": s, "expanded_row_idx": x, "tokens_per_expert": tpe,
            "cumsum": cs, "invalid": int(inv)}


def quant_tokens(x):
    """FrontReorder per-token quant: (xq int8[M,K], pts1 fp32[M])."""
    xb = _h(x)
    M, K = xb.shape
    xq = np.empty((M, K), np.int8)
    pts1 = np.empty(M, np.float32)
    _load().oracle_quant_tokens(M, K, _p(xb), _p(xq), _p(pts1))
    return xq, pts1


def gmm1(xq, sorted_src_route, expert_idx, w1, s1, R_valid, want_acc=False):
    """GMM1 over expanded rows [0, R_valid): (acc1 int32 or None, c1 float16[R_valid, 2I])."""
    xq = _c(xq, np.int8)
    ei = _c(expert_idx, np.int32)
    M, K = xq.shape
    topK = ei.shape[1]
    E, N, _ = w1.shape
    I = N // 2
    acc = np.empty((R_valid, N), np.int32) if want_acc else None
    c1 = np.empty((R_valid, N), np.uint16)
    _load().oracle_gmm1(M, K, I, E, topK, _p(xq), _p(_c(sorted_src_route, np.int32)), _p(ei),
                        _p(_c(w1, np.int8)), _p(_c(s1, np.float32)), R_valid, _p(acc), _p(c1))
    return acc, c1.view(np.float16)


def swiglu_quant(c1, pts1, sorted_src_route, topK):
    """SwiGLU + requant: (q2 int8[R_valid, I], pts2 fp32[R_valid])."""
    c1b = _h(c1)
    R_valid, N = c1b.shape
    I = N // 2
    q2 = np.empty((R_valid, I), np.int8)
    pts2 = np.empty(R_valid, np.float32)
    _load().oracle_swiglu_quant(R_valid, I, topK, _p(c1b), _p(_c(pts1, np.float32)),
                                _p(_c(sorted_src_route, np.int32)), _p(q2), _p(pts2))
    return q2, pts2


def gmm2(q2, sorted_src_route, expert_idx, w2, s2, want_acc=False):
    """GMM2: (acc2 int32 or None, c2 float16[R_valid, K])."""
    q2 = _c(q2, np.int8)
    R_valid, I = q2.shape
    E, K, _ = w2.shape
    ei = _c(expert_idx, np.int32)
    topK = ei.shape[1]
    acc = np.empty((R_valid, K), np.int32) if want_acc else None
    c2 = np.empty((R_valid, K), np.uint16)
    _load().oracle_gmm2(K, I, topK, _p(q2), _p(_c(sorted_src_route, np.int32)), _p(ei),
                        _p(_c(w2, np.int8)), _p(_c(s2, np.float32)), R_valid, _p(acc), _p(c2))
    return acc, c2.view(np.float16)


def combine(c2, pts2):
    c2b = _h(c2)
    R_valid, K = c2b.shape
    d = np.empty((R_valid, K), np.uint16)
    _load().oracle_combine(R_valid, K, _p(c2b), _p(_c(pts2, np.float32)), _p(d))
    return d.view(np.float16)


def unpermute(dmat, expanded_row_idx, probs):
    db = _h(dmat)
    pr = _c(probs, np.float32)
    M, topK = pr.shape
    K = db.shape[1]
    out = np.empty((M, K), np.uint16)
    _load().oracle_unpermute(M, K, topK, _p(db), _p(_c(expanded_row_idx, np.int32)), _p(pr),
                             _p(out))
    return out.view(np.float16)


def layer_fwd(inp, intermediates=False):
    """Whole layer.  inp: dict from synth.make_inputs.  Returns out float16[M,K],
    or (out, dict of intermediates) when intermediates=True."""
    x = _h(inp["x"])
    M, K = x.shape
    ei = _c(inp["expert_idx"], np.int32)
    topK = ei.shape[1]
    w1 = _c(inp["w1"], np.int8)
    E, N, _ = w1.shape
    I = N // 2
    R = M * topK
    out = np.empty((M, K), np.uint16)
    it = None
    ptrs = [None] * 10
    if intermediates:
        it = {"sorted_src_route": np.empty(R, np.int32), "expanded_row_idx": np.empty(R, np.int32),
              "tokens_per_expert": np.empty(E, np.int32), "cumsum": np.empty(E, np.int32),
              "xq": np.empty((M, K), np.int8), "pts1": np.empty(M, np.float32),
              "c1": np.empty((R, N), np.uint16), "q2": np.empty((R, I), np.int8),
              "pts2": np.empty(R, np.float32), "c2": np.empty((R, K), np.uint16)}
        ptrs = [_p(it[k]) for k in ("sorted_src_route", "expanded_row_idx", "tokens_per_expert",
                                    "cumsum", "xq", "pts1", "c1", "q2", "pts2", "c2")]
    inv = _load().oracle_layer_fwd(M, K, I, E, topK, _p(x), _p(ei),
                                   _p(_c(inp["probs"], np.float32)), _p(w1),
                                   _p(_c(inp["s1"], np.float32)), _p(_c(inp["w2"], np.int8)),
                                   _p(_c(inp["s2"], np.float32)), _p(out), *ptrs)
    out = out.view(np.float16)
    if not intermediates:
        return out
    Rv = R - inv
    it["invalid"] = int(inv)
    for k in ("c1", "q2", "pts2", "c2"):
        it[k] = it[k][:Rv]
    it["c1"] = it["c1"].view(np.float16)
    it["c2"] = it["c2"].view(np.float16)
    return out, it


def layer_tokens(inp, tokens):
    """Output rows of the layer for the given token indices (float16[n, K])."""
    x = _h(inp["x"])
    M, K = x.shape
    ei = _c(inp["expert_idx"], np.int32)
    topK = ei.shape[1]
    w1 = _c(inp["w1"], np.int8)
    E, N, _ = w1.shape
    I = N // 2
    tok = _c(tokens, np.int32)
    out = np.empty((tok.size, K), np.uint16)
    _load().oracle_layer_tokens(M, K, I, E, topK, _p(x), _p(ei), _p(_c(inp["probs"], np.float32)),
                                _p(w1), _p(_c(inp["s1"], np.float32)), _p(_c(inp["w2"], np.int8)),
                                _p(_c(inp["s2"], np.float32)), tok.size, _p(tok), _p(out))
    return out.view(np.float16)


def max_threads():
    """Threads the oracle's OpenMP regions run on (omp_get_max_threads)."""
    return int(_load().oracle_max_threads())


def set_threads(n):
    """Threads the oracle's OpenMP regions use from now on (diagnostics; no arithmetic)."""
    _load().oracle_set_threads(int(n))
