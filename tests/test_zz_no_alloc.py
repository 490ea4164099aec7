"""The allocation-free route sort (moe_route_sort_noalloc) against the regular one.

moe_route_sort_noalloc serves callers that cannot allocate device memory (an
engine plugin whose host engine owns all device memory, a server that reserved
the device up front, a loop where cudaMalloc's synchronisation is not allowed):
its scratch is a fixed array inside the library instead of a caller workspace.
It must produce exactly what moe_route_sort produces.  This file is collected
last on purpose (its name), and passes alone in a fresh process as well as
after the other tests.
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import moe_expert_layer_gb300 as moe
    from gpu_util import assert_bits_equal, dev, empty, host


def _outputs(R, E):
    return (empty(R, torch.int32), empty(R, torch.int32), empty(E, torch.int32), empty(E, torch.int32))


def _regular(d, ei_dev, R, E):
    outs = _outputs(R, E)
    ws = empty(max(16, moe.moe_route_sort_workspace_size(d)), torch.uint8)
    moe.moe_route_sort(d, ei_dev, *outs, ws)
    return [host(t) for t in outs]


def _noalloc(d, ei_dev, R, E):
    outs = _outputs(R, E)
    moe.moe_route_sort_noalloc(d, ei_dev, *outs)
    return [host(t) for t in outs]


CASES = [
    # (M, topK, E, routing, seed): large route counts take the multi-block path whose
    # scratch is the fixed array; the last case is a small single-block sort
    (8192, 6, 64, "uniform", 4),
    (2048, 8, 256, "zipf", 3),
    (20000, 7, 1023, "biased", 9),
    (128, 8, 256, "uniform", 1),
]


def test_noalloc_matches_regular_sort_on_consecutive_calls():
    names = ["sorted_src_route", "expanded_row_idx", "tokens_per_expert", "cumsum"]
    for M, topK, E, routing, seed in CASES:
        ei, _ = synth.routing(seed, M, E, topK, routing)
        ei[::13, 0] = -1  # invalid routes exercise the extra bucket
        d = moe.dims(M, 128, 64, E, topK)
        ei_dev = dev(ei)
        ref = _regular(d, ei_dev, M * topK, E)
        for call in range(2):  # two calls in a row share the scratch array
            got = _noalloc(d, ei_dev, M * topK, E)
            for n, g, r in zip(names, got, ref):
                assert_bits_equal(g, r, "%s (M=%d E=%d, call %d)" % (n, M, E, call))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    M = moe.ROUTE_SORT_NOALLOC_MAX_ROUTES // 8 + 1
    d = moe.dims(M, 128, 64, 16, 8)
    t = empty(1, torch.int32)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route_sort_noalloc(d, t, t, t, t, t)
    assert e.value.code == -2
