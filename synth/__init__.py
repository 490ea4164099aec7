"""Seeded synthetic inputs for the W8A8 MoE expert layer.

The draws come from ``synth.c`` (counter-based SplitMix64, compiled on first
use into ``synth/_build/libsynth.so``).  Nothing here computes any part of
the layer: this module only produces its inputs, and both the CPU oracle and
the CUDA path are fed the same bytes from it.

Workloads (tokens ``M``, hidden ``K``, intermediate ``I`` with the gate|up
projection ``2I`` wide, experts ``E``, routes per token ``topK``):

========  =====  =====  =====  ===  ====  =======  ====
name          M      K      I    E  topK  routing  seed
========  =====  =====  =====  ===  ====  =======  ====
tiny         16    256    256    8     2  uniform     0
decode      128   7168   2048  256     8  uniform     1
mid         512   7168   2048  256     8  biased      2
skewed     2048   7168   2048  256     8  zipf1.2     3
prefill    8192   4096   1408   64     6  uniform     4
decode16      8   7168   2048   16     8  uniform     5
mid16       512   7168   2048   16     8  biased      6
midrows16    32   7168   2048   16     8  biased      7
========  =====  =====  =====  ===  ====  =======  ====

``decode16`` keeps decode's shapes and rows per expert (about 4) with 16
experts, so that its weights (0.7 GB) stay above the L2 size while a
counter capture of one GEMM launch remains small.  ``mid16`` keeps mid's
token count (the quant and combine shapes) and ``midrows16`` mid's rows per
expert (about 16, the 32-row warp-MMA tiles), both with 16 experts.

x is binary16 N(0,1); w1/w2 are int8 uniform over [-127, 127]; s1/s2 are
fp32 uniform on [1e-3, 1e-2).  Weight layout: w1[E][2I][K] and w2[E][K][I]
(reduction dimension contiguous), s1[E][2I], s2[E][K].
"""
import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None

ROUTING_MODES = {"uniform": 0, "biased": 1, "zipf": 2}

# stream ids (one per drawn tensor); routing streams 6-10 live in synth.c
_S_X, _S_W1, _S_S1, _S_W2, _S_S2 = 1, 2, 3, 4, 5


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    I: int
    E: int
    topK: int
    routing: str
    seed: int
    zipf_s: float = 1.2

    @property
    def R(self):
        return self.M * self.topK


CONFIGS = {
    "tiny": Workload("tiny", 16, 256, 256, 8, 2, "uniform", 0),
    "decode": Workload("decode", 128, 7168, 2048, 256, 8, "uniform", 1),
    "mid": Workload("mid", 512, 7168, 2048, 256, 8, "biased", 2),
    "skewed": Workload("skewed", 2048, 7168, 2048, 256, 8, "zipf", 3),
    "prefill": Workload("prefill", 8192, 4096, 1408, 64, 6, "uniform", 4),
    "decode16": Workload("decode16", 8, 7168, 2048, 16, 8, "uniform", 5),
    "mid16": Workload("mid16", 512, 7168, 2048, 16, 8, "biased", 6),
    "midrows16": Workload("midrows16", 32, 7168, 2048, 16, 8, "biased", 7),
}


def build(force=False):
    """Compile synth.c into synth/_build/libsynth.so (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fopenmp", "-fPIC", "-shared",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, vp, ci, cd = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p,
                                ctypes.c_int, ctypes.c_double)
        lib.synth_normal_f16.argtypes = [u64, u64, i64, vp]
        lib.synth_int8_sym127.argtypes = [u64, u64, i64, vp]
        lib.synth_uniform_f32.argtypes = [u64, u64, i64, cd, cd, vp]
        lib.synth_routing.argtypes = [u64, ci, ci, ci, ci, cd, vp, vp]
        for f in (lib.synth_normal_f16, lib.synth_int8_sym127, lib.synth_uniform_f32,
                  lib.synth_routing):
            f.restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def normal_f16(seed, stream, shape):
    """binary16 N(0,1) draws, returned as a float16 array."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_f16(seed, stream, out.size, _ptr(out))
    return out.view(np.float16)


def int8_sym127(seed, stream, shape):
    out = np.empty(shape, dtype=np.int8)
    _load().synth_int8_sym127(seed, stream, out.size, _ptr(out))
    return out


def uniform_f32(seed, stream, shape, lo, hi):
    out = np.empty(shape, dtype=np.float32)
    _load().synth_uniform_f32(seed, stream, out.size, lo, hi, _ptr(out))
    return out


def routing(seed, M, E, topK, mode="uniform", zipf_s=1.2):
    """(expert_idx int32[M,topK], probs fp32[M,topK]); distinct experts per token."""
    if not (1 <= topK <= min(E, 64)):
        raise ValueError("need 1 <= topK <= min(E, 64)")
    ei = np.empty((M, topK), dtype=np.int32)
    pr = np.empty((M, topK), dtype=np.float32)
    _load().synth_routing(seed, M, E, topK, ROUTING_MODES[mode], zipf_s, _ptr(ei), _ptr(pr))
    return ei, pr


def make_inputs(cfg, with_weights=True):
    """All layer inputs of a workload (a name from CONFIGS or a Workload).

    Returns a dict of numpy arrays: x float16[M,K], expert_idx int32[M,topK],
    probs float32[M,topK], w1 int8[E,2I,K], s1 float32[E,2I],
    w2 int8[E,K,I], s2 float32[E,K].
    """
    w = CONFIGS[cfg] if isinstance(cfg, str) else cfg
    s = w.seed
    out = {"x": normal_f16(s, _S_X, (w.M, w.K))}
    out["expert_idx"], out["probs"] = routing(s, w.M, w.E, w.topK, w.routing, w.zipf_s)
    if with_weights:
        out["w1"] = int8_sym127(s, _S_W1, (w.E, 2 * w.I, w.K))
        out["s1"] = uniform_f32(s, _S_S1, (w.E, 2 * w.I), 1e-3, 1e-2)
        out["w2"] = int8_sym127(s, _S_W2, (w.E, w.K, w.I))
        out["s2"] = uniform_f32(s, _S_S2, (w.E, w.K), 1e-3, 1e-2)
    return out
