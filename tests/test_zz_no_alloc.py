"""The allocation-free route sort (moe_route_sort_noalloc) against the oracle and the
regular sort.

moe_route_sort_noalloc serves callers that cannot allocate device memory (an
engine plugin whose host engine owns all device memory, a server that reserved
the device up front, a loop where cudaMalloc's synchronisation is not allowed):
its scratch is a fixed array inside the library instead of a caller workspace.
It must produce exactly what the route sort defines (the oracle) and what
moe_route_sort produces, and it must not allocate.  This file is collected last
on purpose (its name), and passes alone in a fresh process as well as after the
other tests.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import moe_expert_layer_gb300 as moe
    from gpu_util import assert_bits_equal, dev, empty, host

NAMES = ["sorted_src_route", "expanded_row_idx", "tokens_per_expert", "cumsum"]


def _outputs(R, E):
    return (empty(R, torch.int32), empty(R, torch.int32), empty(E, torch.int32), empty(E, torch.int32))


def _regular(d, ei_dev, R, E):
    outs = _outputs(R, E)
    ws = empty(max(16, moe.moe_route_sort_workspace_size(d)), torch.uint8)
    moe.moe_route_sort(d, ei_dev, *outs, ws)
    return [host(t) for t in outs]


def _noalloc(d, ei_dev, outs):
    moe.moe_route_sort_noalloc(d, ei_dev, *outs)
    return [host(t) for t in outs]


def _oracle(ei, E):
    rs = oracle.route_sort(ei, E)
    return [rs[n] for n in NAMES]


CASES = [
    # (M, topK, E, routing, seed): large route counts take the multi-block path whose
    # scratch is the fixed array; the largest case fills it exactly (R at the limit,
    # E = 1023: 64 blocks of 8192 routes, 64 * 1024 scratch entries), the next one
    # sits one route below the limit; the last case is a small single-block sort
    (8192, 6, 64, "uniform", 4),
    (2048, 8, 256, "zipf", 3),
    (20000, 7, 1023, "biased", 9),
    (65536, 8, 1023, "uniform", 12),
    (524287, 1, 1023, "uniform", 13),
    (128, 8, 256, "uniform", 1),
]


@pytest.mark.parametrize("M,topK,E,routing,seed", CASES)
def test_noalloc_matches_oracle_and_regular_sort_on_consecutive_calls(M, topK, E, routing, seed):
    ei, _ = synth.routing(seed, M, E, topK, routing)
    ei[::13, 0] = -1  # invalid routes exercise the extra bucket
    R = M * topK
    assert R <= moe.ROUTE_SORT_NOALLOC_MAX_ROUTES
    d = moe.dims(M, 128, 64, E, topK)
    ei_dev = dev(ei)
    want = _oracle(ei, E)
    regular = _regular(d, ei_dev, R, E)
    for n, g, r in zip(NAMES, regular, want):
        assert_bits_equal(g, r, "regular %s (M=%d E=%d)" % (n, M, E))
    for call in range(2):  # two calls in a row share the scratch array
        got = _noalloc(d, ei_dev, _outputs(R, E))
        for n, g, r in zip(NAMES, got, want):
            assert_bits_equal(g, r, "%s (M=%d E=%d, call %d)" % (n, M, E, call))


def test_noalloc_allocates_no_device_memory():
    """After a first call (which loads the sort kernels and looks up the scratch
    address), further calls leave the device's free memory unchanged."""
    M, topK, E = 65536, 8, 1023
    ei, _ = synth.routing(14, M, E, topK, "uniform")
    d = moe.dims(M, 128, 64, E, topK)
    ei_dev = dev(ei)
    outs = _outputs(M * topK, E)
    moe.moe_route_sort_noalloc(d, ei_dev, *outs)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        moe.moe_route_sort_noalloc(d, ei_dev, *outs)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    for n, g, r in zip(NAMES, [host(t) for t in outs], _oracle(ei, E)):
        assert_bits_equal(g, r, n)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    M = moe.ROUTE_SORT_NOALLOC_MAX_ROUTES // 8 + 1
    d = moe.dims(M, 128, 64, 16, 8)
    t = empty(1, torch.int32)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route_sort_noalloc(d, t, t, t, t, t)
    assert e.value.code == -2
