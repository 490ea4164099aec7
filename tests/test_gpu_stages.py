"""GPU parity of each stage against the CPU oracle, through the C ABI.

Each stage is fed the oracle's own inputs for that stage, so a mismatch points
at one kernel.  Index, sort and quant outputs are compared bit for bit; GEMM
outputs too (identical int8 operands give identical int32 accumulators, and the
epilogue's rounding points are fixed); SwiGLU's codes within 1 LSB on <= 0.1%
of elements (exp is evaluated by different libraries on the two sides).
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import moe_expert_layer_gb300 as moe
    from gpu_util import assert_bits_equal, assert_q2_close, dev, empty, host


def _dims(w, layout=0):
    return moe.dims(w.M, w.K, w.I, w.E, w.topK, layout)


def tiles_ref(w):
    """The weight-tile layout of include/moe_layer.h written out with numpy: w [E][N][D]
    int8 -> tiles (e, nb, kb) of 128 channels x 128 reduction bytes, depth zero-padded to
    a multiple of 256, 16-byte chunk c of tile row r stored at chunk c ^ (r % 8), every
    byte in excess-128 form (w + 128, the padding's zeros as 0x80)."""
    E, N, D = w.shape
    KB = 2 * ((D + 255) // 256)
    pad = np.zeros((E, N, KB * 128), np.int8)
    pad[:, :, :D] = w
    pad = (pad.view(np.uint8) ^ 0x80).view(np.int8)
    t = pad.reshape(E, N // 128, 128, KB, 8, 16).transpose(0, 1, 3, 2, 4, 5)  # e, nb, kb, r, chunk, byte
    out = np.empty_like(t)
    r = np.arange(128)
    for c in range(8):
        out[:, :, :, r, c ^ (r % 8), :] = t[:, :, :, r, c, :]
    return out.reshape(-1)


def _weights(d, gemm, w, layout):
    """The GEMM weight on the device in the given layout (tiles packed by the library)."""
    if layout == 0:
        return dev(w)
    tiles = empty(moe.moe_weight_tiles_bytes(d, gemm), torch.int8)
    moe.moe_pack_weight_tiles(d, gemm, dev(w), tiles)
    return tiles


def _sort_on_gpu(w, expert_idx):
    d = _dims(w)
    R = w.M * w.topK
    s, x = empty(R, torch.int32), empty(R, torch.int32)
    tpe, cs = empty(w.E, torch.int32), empty(w.E, torch.int32)
    nws = moe.moe_route_sort_workspace_size(d)
    ws = empty(max(nws, 16), torch.uint8)
    moe.moe_route_sort(d, dev(expert_idx), s, x, tpe, cs, ws)
    torch.cuda.synchronize()
    return host(s), host(x), host(tpe), host(cs)


# ------------------------------------------------------------------ route sort
SORT_CASES = [
    ("tiny", None), ("decode", None), ("mid", None), ("skewed", None), ("prefill", None),
    ("M1", synth.Workload("M1", 1, 128, 64, 4, 1, "uniform", 21)),
    ("topk1", synth.Workload("topk1", 333, 128, 64, 7, 1, "uniform", 22)),
    ("E1", synth.Workload("E1", 100, 128, 64, 1, 1, "uniform", 23)),
    ("E1023", synth.Workload("E1023", 3000, 128, 64, 1023, 8, "zipf", 24)),
    ("bigR", synth.Workload("bigR", 20000, 128, 64, 300, 5, "biased", 25)),
    # past 64 blocks of 8192 routes: blocks of 8192, as many as it takes
    ("R600k", synth.Workload("R600k", 75000, 128, 64, 1023, 8, "uniform", 26)),
]


@pytest.mark.parametrize("name,w", SORT_CASES, ids=[c[0] for c in SORT_CASES])
def test_route_sort_bit_exact(name, w):
    w = w or synth.CONFIGS[name]
    ei, _ = synth.routing(w.seed, w.M, w.E, w.topK, w.routing)
    ref = oracle.route_sort(ei, w.E)
    s, x, tpe, cs = _sort_on_gpu(w, ei)
    assert_bits_equal(s, ref["sorted_src_route"], "sorted_src_route")
    assert_bits_equal(x, ref["expanded_row_idx"], "expanded_row_idx")
    assert_bits_equal(tpe, ref["tokens_per_expert"], "tokens_per_expert")
    assert_bits_equal(cs, ref["cumsum"], "cumsum")


@pytest.mark.parametrize("M", [40, 9000])
def test_route_sort_invalid_ids_and_hot_expert(M):
    w = synth.Workload("inv", M, 128, 64, 16, 4, "uniform", 31)
    ei, _ = synth.routing(w.seed, w.M, w.E, w.topK, "uniform")
    ei[::7, 0] = -3
    ei[::11, 1] = 16  # == E: out of range
    ei[1::5, 2] = 5   # hot expert
    ref = oracle.route_sort(ei, w.E)
    assert ref["invalid"] > 0
    s, x, tpe, cs = _sort_on_gpu(w, ei)
    assert_bits_equal(s, ref["sorted_src_route"], "sorted_src_route")
    assert_bits_equal(x, ref["expanded_row_idx"], "expanded_row_idx")
    assert_bits_equal(tpe, ref["tokens_per_expert"], "tokens_per_expert")
    assert_bits_equal(cs, ref["cumsum"], "cumsum")


# ------------------------------------------------------------------ token quant
@pytest.mark.parametrize("M,K", [(16, 256), (128, 7168), (37, 4096), (5, 16384), (3, 128)])
def test_quant_tokens_bit_exact(M, K):
    x = synth.normal_f16(41, 1, (M, K))
    x[min(2, M - 1)] = 0  # an all-zero token
    xq_ref, pts_ref = oracle.quant_tokens(x)
    d = moe.dims(M, K, 64, 4, 1)
    xq8, xq16, pts = empty((M, K), torch.int8), empty((M, K), torch.float16), empty(M, torch.float32)
    moe.moe_quant_tokens(d, dev(x), None, xq8, xq16, pts, None)
    torch.cuda.synchronize()
    assert_bits_equal(host(xq8), xq_ref, "xq")
    assert_bits_equal(host(pts), pts_ref, "pts1")
    assert_bits_equal(host(xq16), xq_ref.astype(np.float16), "xq as binary16")


# ------------------------------------------------------------------ quant + scatter to expert-major rows
@pytest.mark.parametrize("cfg", ["tiny", "decode", "prefill"])
def test_quant_dispatch_bit_exact(cfg):
    w = synth.CONFIGS[cfg]
    x = synth.normal_f16(w.seed, 1, (w.M, w.K))
    ei, _ = synth.routing(w.seed, w.M, w.E, w.topK, w.routing)
    ei[1, 0] = -1  # an invalid route: its row is not written
    rs = oracle.route_sort(ei, w.E)
    xq_ref, pts_ref = oracle.quant_tokens(x)
    Rv = w.R - rs["invalid"]
    a1_ref = xq_ref[rs["sorted_src_route"][:Rv] // w.topK].astype(np.float16)
    d = _dims(w)
    a1 = torch.full((w.R, w.K), 7.0, dtype=torch.float16, device="cuda")
    pts = empty(w.M, torch.float32)
    moe.moe_quant_dispatch(d, dev(x), None, dev(rs["expanded_row_idx"]), a1, pts, None)
    torch.cuda.synchronize()
    got = host(a1)
    assert_bits_equal(got[:Rv], a1_ref, "a1")
    assert np.all(got[Rv:].astype(np.float32) == 7.0)  # rows past the valid ones untouched
    assert_bits_equal(host(pts), pts_ref, "pts1")


FRONT_CASES = [
    ("tiny", None), ("decode", None), ("mid", None),
    ("r4096", synth.Workload("r4096", 1024, 256, 64, 64, 4, "zipf", 31)),      # the largest fused sort
    ("r4100", synth.Workload("r4100", 1025, 256, 64, 64, 4, "zipf", 32)),      # the route-sort kernels first
    ("skewed", None),
    ("e1023", synth.Workload("e1023", 300, 128, 64, 1023, 8, "biased", 33)),
    ("topk64", synth.Workload("topk64", 40, 128, 64, 96, 64, "uniform", 34)),  # more routes than threads
    ("m1", synth.Workload("m1", 1, 384, 64, 4, 3, "uniform", 35)),
]


@pytest.mark.parametrize("name,w", FRONT_CASES, ids=[c[0] for c in FRONT_CASES])
def test_front_reorder_bit_exact(name, w):
    """FrontReorder in one call equals the sort and the quant-scatter done apart: the
    same route tables, codes, scales and activation bounds, bit for bit (invalid
    routes and an expert repeated within a token included)."""
    w = w or synth.CONFIGS[name]
    x = synth.normal_f16(w.seed, 1, (w.M, w.K))
    ei, _ = synth.routing(w.seed, w.M, w.E, w.topK, w.routing)
    ei[0, 0] = -1          # invalid routes: sorted last, no row written
    if w.M > 2:
        ei[2, -1] = w.E + 5
    if w.topK > 1:
        ei[-1, 1] = ei[-1, 0]  # the same expert twice in one token: slot order decides
    ref = oracle.route_sort(ei, w.E)
    xq_ref, pts_ref = oracle.quant_tokens(x)
    Rv = w.R - ref["invalid"]
    a1_ref = xq_ref[ref["sorted_src_route"][:Rv] // w.topK]
    d = _dims(w)
    s, xr = empty(w.R, torch.int32), empty(w.R, torch.int32)
    tpe, cs = empty(w.E, torch.int32), empty(w.E, torch.int32)
    ws = empty(max(16, moe.moe_route_sort_workspace_size(d)), torch.uint8)
    a1 = torch.full((w.R, w.K), 7.0, dtype=torch.float16, device="cuda")
    pts = empty(w.M, torch.float32)
    bounds = torch.zeros((w.E, moe.BOUND_SEGMENTS), dtype=torch.int32, device="cuda")
    moe.moe_front_reorder(d, dev(x), dev(ei), s, xr, tpe, cs, a1, pts, bounds, ws)
    torch.cuda.synchronize()
    assert_bits_equal(host(s), ref["sorted_src_route"], "sorted_src_route")
    assert_bits_equal(host(xr), ref["expanded_row_idx"], "expanded_row_idx")
    assert_bits_equal(host(tpe), ref["tokens_per_expert"], "tokens_per_expert")
    assert_bits_equal(host(cs), ref["cumsum"], "cumsum")
    got = host(a1)
    assert_bits_equal(got[:Rv], a1_ref.astype(np.float16), "a1")
    assert np.all(got[Rv:].astype(np.float32) == 7.0)
    assert_bits_equal(host(pts), pts_ref, "pts1")
    assert_bits_equal(host(bounds), _bounds_ref(a1_ref, ref["cumsum"], w.E), "a1 bounds")


def _bounds_ref(codes, cumsum, E):
    """Per-expert, per-1024-deep-segment maxima of sum |code| over the expert's rows."""
    S = moe.BOUND_SEGMENTS
    b = np.zeros((E, S), np.int32)
    l1 = np.abs(codes.astype(np.int64))
    nseg = (codes.shape[1] + moe.BOUND_SEGMENT - 1) // moe.BOUND_SEGMENT
    seg = np.stack([l1[:, s * moe.BOUND_SEGMENT:(s + 1) * moe.BOUND_SEGMENT].sum(1) for s in range(nseg)], 1)
    lo = 0
    for e in range(E):
        hi = int(cumsum[e])
        if hi > lo:
            b[e, :nseg] = seg[lo:hi].max(0)
        lo = hi
    return b


@pytest.mark.parametrize("cfg", ["decode", "prefill", "mid"])
def test_quant_tokens_bounds(cfg):
    """The token quant's activation bounds (the layer's path: codes stay token-major,
    GMM1 gathers them) are the exact per-expert segment maxima of sum |code| over the
    expert's routed tokens, as if the codes had been dispatched to expert-major rows."""
    w = synth.CONFIGS[cfg]
    x = synth.normal_f16(w.seed, 1, (w.M, w.K))
    ei, _ = synth.routing(w.seed, w.M, w.E, w.topK, w.routing)
    ei[1, 0] = -1
    rs = oracle.route_sort(ei, w.E)
    xq_ref, pts_ref = oracle.quant_tokens(x)
    Rv = w.R - rs["invalid"]
    a1_ref = xq_ref[rs["sorted_src_route"][:Rv] // w.topK]
    d = _dims(w)
    xq16, pts = empty((w.M, w.K), torch.float16), empty(w.M, torch.float32)
    bounds = torch.zeros((w.E, moe.BOUND_SEGMENTS), dtype=torch.int32, device="cuda")
    moe.moe_quant_tokens(d, dev(x), dev(ei), None, xq16, pts, bounds)
    torch.cuda.synchronize()
    assert_bits_equal(host(xq16), xq_ref.astype(np.float16), "xq as binary16")
    assert_bits_equal(host(pts), pts_ref, "pts1")
    assert_bits_equal(host(bounds), _bounds_ref(a1_ref, rs["cumsum"], w.E), "a1 bounds")


@pytest.mark.parametrize("cfg", ["decode", "prefill", "mid"])
def test_quant_dispatch_bounds(cfg):
    """The activation bounds the quant-scatter produces are the exact per-expert
    segment maxima of sum |code| (invalid routes contribute nothing)."""
    w = synth.CONFIGS[cfg]
    x = synth.normal_f16(w.seed, 1, (w.M, w.K))
    ei, _ = synth.routing(w.seed, w.M, w.E, w.topK, w.routing)
    ei[1, 0] = -1
    rs = oracle.route_sort(ei, w.E)
    xq_ref, _ = oracle.quant_tokens(x)
    Rv = w.R - rs["invalid"]
    a1_ref = xq_ref[rs["sorted_src_route"][:Rv] // w.topK]
    d = _dims(w)
    a1 = empty((w.R, w.K), torch.float16)
    pts = empty(w.M, torch.float32)
    bounds = torch.zeros((w.E, moe.BOUND_SEGMENTS), dtype=torch.int32, device="cuda")
    moe.moe_quant_dispatch(d, dev(x), dev(ei), dev(rs["expanded_row_idx"]), a1, pts, bounds)
    torch.cuda.synchronize()
    assert_bits_equal(host(bounds), _bounds_ref(a1_ref, rs["cumsum"], w.E), "a1 bounds")


# ------------------------------------------------------------------ GEMMs
def _a1(xq, rs, topK, R):
    """Expert-major GMM1 operand built from the oracle's per-token codes."""
    Rv = R - rs["invalid"]
    a1 = np.zeros((R, xq.shape[1]), np.float16)
    a1[:Rv] = xq[rs["sorted_src_route"][:Rv] // topK]
    return a1


def _stage_inputs(w):
    inp = synth.make_inputs(w)
    rs = oracle.route_sort(inp["expert_idx"], w.E)
    xq, pts1 = oracle.quant_tokens(inp["x"])
    return inp, rs, xq, pts1


GEMM_CASES = [
    synth.Workload("g_dec", 60, 512, 128, 16, 2, "uniform", 59),            # warp-MMA engine, 16-row tiles
    synth.Workload("g_dec_odd", 60, 768, 64, 16, 2, "uniform", 60),         # 16-row tiles, odd stage counts (3, 1):
                                                                            # the two producers' stages alternate across items
    synth.Workload("g_small", 40, 256, 128, 8, 2, "uniform", 51),           # warp-MMA engine, 32-row tiles
    synth.Workload("g_mid", 160, 512, 192, 16, 2, "biased", 52),            # warp-MMA engine, 32-row tiles, ragged
    synth.Workload("g_mid_tc", 320, 512, 192, 16, 2, "biased", 57),         # tcgen05 pairs, small N tiles, 128-channel tail
    synth.Workload("g_big", 384, 1024, 256, 4, 2, "zipf", 53),              # tcgen05 pairs, N=256 tiles, hot expert
    synth.Workload("g_kchunks", 64, 2560, 64, 2, 1, "uniform", 54),         # tcgen05 pairs, three 1024-deep chunks
    synth.Workload("g_tiles", 700, 512, 192, 3, 2, "zipf", 55),             # several balanced row tiles per expert, 64-deep tail
    synth.Workload("g_odd", 48, 384, 192, 8, 2, "uniform", 56),             # warp-MMA engine, 3 stages per item
    synth.Workload("g_hybrid", 400, 512, 192, 32, 2, "zipf", 58),           # both engines: small experts on warp MMA
]


def _gmm1(d, xq, rs, topK, R, gather, bounds, w1, s1, c1, ws):
    """GMM1 on the oracle's token codes: gathered from token rows by the kernel
    (the layer's path), or from expert-major rows dispatched here.  w1 is on the
    device already, in d's weight layout."""
    if gather:
        moe.moe_gmm1(d, dev(xq.astype(np.float16)), dev(rs["sorted_src_route"]), dev(rs["cumsum"]), bounds,
                     w1, dev(s1), c1, ws)
    else:
        moe.moe_gmm1(d, dev(_a1(xq, rs, topK, R)), None, dev(rs["cumsum"]), bounds, w1, dev(s1), c1, ws)


LAYOUTS = [0, 1]
LAYOUT_IDS = ["wrows", "wtiles"]


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("gather", [True, False], ids=["gather", "rows"])
@pytest.mark.parametrize("bounded", [False, True], ids=["chunk1024", "bounds"])
@pytest.mark.parametrize("w", GEMM_CASES, ids=[w.name for w in GEMM_CASES])
def test_gmm1_bit_exact(w, bounded, gather, layout):
    inp, rs, xq, pts1 = _stage_inputs(w)
    Rv = w.R - rs["invalid"]
    _, c1_ref = oracle.gmm1(xq, rs["sorted_src_route"], inp["expert_idx"], inp["w1"], inp["s1"], Rv)
    d = _dims(w, layout)
    c1 = torch.full((w.R, 2 * w.I), float("nan"), dtype=torch.float16, device="cuda")
    ws = empty(moe.moe_gmm_workspace_size(d), torch.uint8)
    bounds = dev(_bounds_ref(_a1(xq, rs, w.topK, w.R), rs["cumsum"], w.E)) if bounded else None
    _gmm1(d, xq, rs, w.topK, w.R, gather, bounds, _weights(d, 1, inp["w1"], layout), inp["s1"], c1, ws)
    assert moe.moe_workspace_status(ws) == 0
    assert_bits_equal(host(c1)[:Rv], c1_ref, "c1")


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("bounded", [False, True], ids=["chunk1024", "bounds"])
@pytest.mark.parametrize("w", GEMM_CASES, ids=[w.name for w in GEMM_CASES])
def test_gmm2_bit_exact(w, bounded, layout):
    inp, rs, xq, pts1 = _stage_inputs(w)
    Rv = w.R - rs["invalid"]
    q2 = synth.int8_sym127(w.seed, 77, (Rv, w.I))
    _, c2_ref = oracle.gmm2(q2, rs["sorted_src_route"], inp["expert_idx"], inp["w2"], inp["s2"])
    d = _dims(w, layout)
    c2 = empty((w.R, w.K), torch.float16)
    ws = empty(moe.moe_gmm_workspace_size(d), torch.uint8)
    q2f = np.zeros((w.R, w.I), np.float16)
    q2f[:Rv] = q2
    bounds = dev(_bounds_ref(q2f, rs["cumsum"], w.E)) if bounded else None
    moe.moe_gmm2(d, dev(q2f), dev(rs["cumsum"]), bounds, _weights(d, 2, inp["w2"], layout), dev(inp["s2"]), c2, ws)
    assert moe.moe_workspace_status(ws) == 0
    assert_bits_equal(host(c2)[:Rv], c2_ref, "c2")


@pytest.mark.parametrize("bounded", [False, True], ids=["chunk1024", "bounds"])
def test_gmm_pairs_only_with_small_experts(bounded):
    """Above 256 rows per expert on average the tcgen05 pairs take every expert, the
    small ones (here 20, 10 and 0 rows beside 1200 and 70) as single small-N tiles."""
    w = synth.Workload("pairs_only", 1300, 512, 192, 5, 1, "uniform", 81)
    inp = synth.make_inputs(w)
    ei = np.zeros((w.M, 1), np.int32)
    ei[1200:1270] = 1
    ei[1270:1290] = 2
    ei[1290:] = 3
    inp["expert_idx"] = ei[np.random.default_rng(81).permutation(w.M)]  # the tokens of each expert spread out
    rs = oracle.route_sort(inp["expert_idx"], w.E)
    assert list(rs["tokens_per_expert"]) == [1200, 70, 20, 10, 0] and w.R / w.E >= 256
    xq, _ = oracle.quant_tokens(inp["x"])
    _, c1_ref = oracle.gmm1(xq, rs["sorted_src_route"], inp["expert_idx"], inp["w1"], inp["s1"], w.R)
    d = _dims(w, 1)
    ws = empty(moe.moe_gmm_workspace_size(d), torch.uint8)
    a1 = _a1(xq, rs, 1, w.R)
    c1 = torch.full((w.R, 2 * w.I), float("nan"), dtype=torch.float16, device="cuda")
    b1 = dev(_bounds_ref(a1, rs["cumsum"], w.E)) if bounded else None
    moe.moe_gmm1(d, dev(a1), None, dev(rs["cumsum"]), b1, _weights(d, 1, inp["w1"], 1), dev(inp["s1"]), c1, ws)
    assert moe.moe_workspace_status(ws) == 0
    assert_bits_equal(host(c1), c1_ref, "c1")
    q2 = synth.int8_sym127(w.seed, 77, (w.R, w.I))
    _, c2_ref = oracle.gmm2(q2, rs["sorted_src_route"], inp["expert_idx"], inp["w2"], inp["s2"])
    c2 = empty((w.R, w.K), torch.float16)
    q2f = q2.astype(np.float16)
    b2 = dev(_bounds_ref(q2f, rs["cumsum"], w.E)) if bounded else None
    moe.moe_gmm2(d, dev(q2f), dev(rs["cumsum"]), b2, _weights(d, 2, inp["w2"], 1), dev(inp["s2"]), c2, ws)
    assert moe.moe_workspace_status(ws) == 0
    assert_bits_equal(host(c2), c2_ref, "c2")


FUSED_CASES = [
    # every expert on the tcgen05 pairs (>= 256 routes per expert): SwiGLU inside GMM1
    synth.Workload("f_prefill_i", 2048, 512, 1408, 8, 1, "uniform", 91),   # the prefill I, 6 vectors per lane
    synth.Workload("f_i64", 1024, 1024, 64, 2, 2, "biased", 92),           # a row half of one vector
    synth.Workload("f_i1536", 600, 256, 1536, 2, 1, "zipf", 93),            # the largest row held in registers
    synth.Workload("f_tiles", 1800, 256, 320, 6, 1, "zipf", 94),            # uneven experts, small and balanced tiles
    synth.Workload("f_i2048", 600, 256, 2048, 2, 1, "uniform", 96),         # rows read twice, 1024 deep at a time
    synth.Workload("f_i2496", 512, 256, 2496, 2, 1, "biased", 99),          # ... with a partial last pass
    # both engines (25-255 routes per expert): experts of <= 32 rows on the warp-MMA
    # engine first, the rest on the pairs with the SwiGLU of every row inside
    synth.Workload("f_hybrid", 400, 512, 192, 32, 2, "zipf", 95),
    synth.Workload("f_hybrid_long", 400, 256, 2048, 16, 2, "zipf", 97),
    # not fused: the warp-MMA engine alone (<= 24 routes per expert)
    synth.Workload("f_warp_only", 128, 256, 192, 16, 2, "uniform", 98),
]


def _fused_vs_separate(w, bounded, inp=None):
    """moe_gmm1_swiglu against moe_gmm1 then moe_swiglu_quant on w's inputs (or the
    given ones), bit for bit, on two calls in a row."""
    if inp is None:
        inp = synth.make_inputs(w)
    rs = oracle.route_sort(inp["expert_idx"], w.E)
    xq, pts1 = oracle.quant_tokens(inp["x"])
    d = _dims(w, 1)
    a1 = dev(_a1(xq, rs, w.topK, w.R))
    cs, srt, ei = dev(rs["cumsum"]), dev(rs["sorted_src_route"]), dev(inp["expert_idx"])
    w1, s1, p1 = _weights(d, 1, inp["w1"], 1), dev(inp["s1"]), dev(pts1)
    b1 = dev(_bounds_ref(_a1(xq, rs, w.topK, w.R), rs["cumsum"], w.E)) if bounded else None
    ws = empty(moe.moe_gmm_workspace_size(d), torch.uint8)
    Rv = w.R - rs["invalid"]

    def run(fused):
        c1 = torch.full((w.R, 2 * w.I), float("nan"), dtype=torch.float16, device="cuda")
        q2 = torch.full((w.R, w.I), float("nan"), dtype=torch.float16, device="cuda")
        pts2 = torch.full((w.R,), float("nan"), dtype=torch.float32, device="cuda")
        b2 = torch.zeros((w.E, moe.BOUND_SEGMENTS), dtype=torch.int32, device="cuda")
        if fused:
            moe.moe_gmm1_swiglu(d, a1, cs, b1, w1, s1, c1, p1, srt, ei, q2, pts2, b2, ws)
        else:
            moe.moe_gmm1(d, a1, None, cs, b1, w1, s1, c1, ws)
            moe.moe_swiglu_quant(d, c1, p1, srt, cs, ei, None, q2, pts2, b2)
        assert moe.moe_workspace_status(ws) == 0
        return [host(t) for t in (c1[:Rv], q2[:Rv], pts2[:Rv], b2)]

    ref = run(False)
    for call in range(2):
        got = run(True)
        for n, g, r in zip(["c1", "q2", "pts2", "q2 bounds"], got, ref):
            assert_bits_equal(g, r, "%s (%s, call %d)" % (n, w.name, call))


@pytest.mark.parametrize("bounded", [False, True], ids=["chunk1024", "bounds"])
@pytest.mark.parametrize("w", FUSED_CASES, ids=[w.name for w in FUSED_CASES])
def test_gmm1_swiglu_matches_the_separate_kernels(w, bounded):
    """moe_gmm1_swiglu (SwiGLU fused into the tcgen05 GMM1 where it applies) writes the
    same c1, q2, pts2 and q2 bounds as moe_gmm1 followed by moe_swiglu_quant, bit for
    bit, on two calls in a row."""
    _fused_vs_separate(w, bounded)


def test_gmm1_swiglu_no_expert_on_the_pairs():
    """28 routes per expert, none above 32: the warp-MMA engine serves every expert,
    the pairs launch with no work item and their drain warps requantise every row
    (each expert complete from the start)."""
    w = synth.Workload("f_none_on_pairs", 56, 256, 320, 2, 1, "uniform", 90)
    inp = synth.make_inputs(w)
    inp["expert_idx"] = (np.arange(w.M, dtype=np.int32) % w.E).reshape(w.M, 1)
    _fused_vs_separate(w, True, inp)


@pytest.mark.parametrize("E,N,D", [(3, 128, 128), (2, 384, 192), (2, 256, 64), (1, 128, 1408), (2, 128, 7168),
                                   (3, 256, 320)])
def test_pack_weight_tiles_layout(E, N, D):
    """moe_pack_weight_tiles writes exactly the documented tile layout (bit for bit),
    the excess-128 bytes and the depth padding's 0x80 included."""
    w = synth.int8_sym127(E * N + D, 5, (E, N, D))
    # GMM2 form: N = K (multiple of 128), D = I (multiple of 64)
    d = moe.dims(1, N, D, E, 1)
    tiles = torch.full((moe.moe_weight_tiles_bytes(d, 2),), 99, dtype=torch.int8, device="cuda")
    moe.moe_pack_weight_tiles(d, 2, dev(w), tiles)
    torch.cuda.synchronize()
    assert tiles.numel() == tiles_ref(w).size
    assert_bits_equal(host(tiles), tiles_ref(w), "tiles")


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("M,wv", [(8, 127), (40, 127), (40, -128)])
def test_gmm_accumulator_exact_beyond_fp32_mantissa(M, wv, layout):
    """Partial sums far above 2^24 that cancel to a small integer.  The reduction
    runs +127*wv terms, then small terms, then -127*wv terms: a single fp32
    accumulator would reach ~5.6e7 (ulp 4) while adding the small terms and lose
    them; the exact chunked accumulation must return them bit for bit (scale 1,
    |acc| < 2048, so binary16 holds the integer exactly).  M=8 runs on the
    warp-MMA engine, M=40 on the tcgen05 pairs, whose 1024-deep chunks reach
    1024*127*128 < 2^24 with wv = -128."""
    K, I, E = 7168, 64, 1
    mid = 168
    h = (K - mid) // 2
    rng = np.random.default_rng(5)
    xq = np.empty((M, K), np.int8)
    xq[:, :h], xq[:, h + mid:] = 127, -127
    xq[:, h:h + mid] = rng.integers(-2, 3, (M, mid))
    w1 = np.empty((E, 2 * I, K), np.int8)
    w1[0, :, :h], w1[0, :, h + mid:] = wv, wv
    w1[0, :, h:h + mid] = rng.integers(-3, 4, (2 * I, mid))
    s1 = np.ones((E, 2 * I), np.float32)
    ei = np.zeros((M, 1), np.int32)
    rs = oracle.route_sort(ei, E)
    acc_ref, c1_ref = oracle.gmm1(xq, rs["sorted_src_route"], ei, w1, s1, M, want_acc=True)
    assert np.abs(acc_ref).max() < 2048 and np.count_nonzero(acc_ref) > acc_ref.size // 2
    d = moe.dims(M, K, I, E, 1, layout)
    c1 = empty((M, 2 * I), torch.float16)
    ws = empty(moe.moe_gmm_workspace_size(d), torch.uint8)
    _gmm1(d, xq, rs, 1, M, True, None, _weights(d, 1, w1, layout), s1, c1, ws)
    got = host(c1).astype(np.float64)
    assert np.array_equal(got, acc_ref.astype(np.float64))


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("K", [2048, 4096, 7168])
def test_gmm_bounds_at_the_limit(K, layout):
    """Chunks merged by the activation bounds, with partial sums reaching 2^24 (at
    K=2048 the merged chunk is the whole reduction: the single-chunk epilogue).
    Every row has sum |code| = 131072 = 2^24 / 128 over the first 2048 k (so those
    two segments form one chunk only when their bounds allow it) and small codes
    after; weights are -128 where the codes are large, so the fp32 partial sums of
    the merged chunk reach -2^24 exactly before the small terms are added."""
    M, I, E = 40, 64, 1
    rng = np.random.default_rng(K)
    xq = rng.integers(-1, 2, (M, K)).astype(np.int8)
    xq[:, :1024] = 64
    xq[:, 1024:2048] = 64           # 2048 * 64 = 131072 in the first two segments
    xq[:, 2048:] = 0                # nothing after: one merged chunk holds the whole sum
    if K > 3010:
        xq[:, 3000:3010] = rng.integers(-3, 4, (M, 10))
    w1 = rng.integers(-2, 3, (E, 2 * I, K)).astype(np.int8)
    w1[0, :, :2048] = -128
    s1 = np.ones((E, 2 * I), np.float32) / 4096
    ei = np.zeros((M, 1), np.int32)
    rs = oracle.route_sort(ei, E)
    acc_ref, c1_ref = oracle.gmm1(xq, rs["sorted_src_route"], ei, w1, s1, M, want_acc=True)
    assert acc_ref.min() <= -(1 << 24) + 100
    a1 = _a1(xq, rs, 1, M)
    b = _bounds_ref(a1, rs["cumsum"], E)
    assert b[0, :2].sum() * 128 <= (1 << 24) and b[0, :3].sum() * 128 > (1 << 24) - (1 << 17)
    d = moe.dims(M, K, I, E, 1, layout)
    c1 = empty((M, 2 * I), torch.float16)
    ws = empty(moe.moe_gmm_workspace_size(d), torch.uint8)
    _gmm1(d, xq, rs, 1, M, True, dev(b), _weights(d, 1, w1, layout), s1, c1, ws)
    assert moe.moe_workspace_status(ws) == 0
    assert_bits_equal(host(c1), c1_ref, "c1")


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("gather", [True, False], ids=["gather", "rows"])
def test_gmm_empty_experts_and_single_rows(gather, layout):
    """Experts with 0 and 1 rows, and a row tile tail of every length."""
    w = synth.Workload("sparse", 23, 256, 64, 12, 1, "uniform", 61)
    inp, rs, xq, pts1 = _stage_inputs(w)
    inp["expert_idx"][:, 0] = np.array([0, 3, 3, 5, 5, 5] + [7] * 17, np.int32)
    rs = oracle.route_sort(inp["expert_idx"], w.E)
    _, c1_ref = oracle.gmm1(xq, rs["sorted_src_route"], inp["expert_idx"], inp["w1"], inp["s1"], w.R)
    d = _dims(w, layout)
    c1 = empty((w.R, 2 * w.I), torch.float16)
    ws = empty(moe.moe_gmm_workspace_size(d), torch.uint8)
    _gmm1(d, xq, rs, 1, w.R, gather, None, _weights(d, 1, inp["w1"], layout), inp["s1"], c1, ws)
    assert_bits_equal(host(c1), c1_ref, "c1")


# ------------------------------------------------------------------ SwiGLU
@pytest.mark.parametrize("R,I,spread", [(64, 256, 1500), (300, 2048, 1500), (77, 1408, 1500), (5, 8192, 1500),
                                         (2000, 1408, 100), (300, 2048, 30), (4096, 1408, 1500), (4101, 2048, 30),
                                         (4096, 8192, 100)])
def test_swiglu_quant(R, I, spread):
    """spread 1500 puts the SwiGLU inputs h at |h| ~ 45 (as the workloads do);
    100 and 30 at |h| ~ 3 and ~1, where exp(-h) and the division shape every value."""
    rng = np.random.default_rng(R + I)
    c1 = (rng.standard_normal((R, 2 * I)) * spread).astype(np.float16)
    c1[1] = 0
    topK = 1
    M = R
    pts1 = rng.uniform(0.02, 0.05, M).astype(np.float32)
    sorted_src = rng.permutation(R).astype(np.int32)
    cumsum = np.array([R], np.int32)
    q2_ref, pts2_ref = oracle.swiglu_quant(c1, pts1, sorted_src, topK)
    d = moe.dims(M, 128, I, 1, 1)
    q8, q16, p2 = empty((R, I), torch.int8), empty((R, I), torch.float16), empty(R, torch.float32)
    moe.moe_swiglu_quant(d, dev(c1), dev(pts1), dev(sorted_src), dev(cumsum), None, q8, q16, p2, None)
    torch.cuda.synchronize()
    assert_q2_close(host(q8), q2_ref)
    assert np.array_equal(host(q16).astype(np.int8), host(q8))
    np.testing.assert_allclose(host(p2), pts2_ref, rtol=1e-6, atol=0)


@pytest.mark.parametrize("R,I,E", [(300, 2048, 5), (2000, 1408, 16)])
def test_swiglu_quant_bounds(R, I, E):
    """The requant's activation bounds are the exact per-expert segment maxima of
    sum |q2| of the codes it writes (row d belongs to expert expert_idx[src])."""
    rng = np.random.default_rng(R * I)
    c1 = (rng.standard_normal((R, 2 * I)) * 200).astype(np.float16)
    pts1 = rng.uniform(0.02, 0.05, R).astype(np.float32)
    ei = np.sort(rng.integers(0, E, R)).astype(np.int32).reshape(R, 1)   # expert-major rows, topK = 1
    sorted_src = np.arange(R, dtype=np.int32)
    cumsum = np.cumsum(np.bincount(ei.ravel(), minlength=E)).astype(np.int32)
    d = moe.dims(R, 128, I, E, 1)
    q8, q16, p2 = empty((R, I), torch.int8), empty((R, I), torch.float16), empty(R, torch.float32)
    bounds = torch.zeros((E, moe.BOUND_SEGMENTS), dtype=torch.int32, device="cuda")
    moe.moe_swiglu_quant(d, dev(c1), dev(pts1), dev(sorted_src), dev(cumsum), dev(ei), q8, q16, p2, bounds)
    torch.cuda.synchronize()
    assert_bits_equal(host(bounds), _bounds_ref(host(q8), cumsum, E), "q2 bounds")


# ------------------------------------------------------------------ Combine + Unpermute
COMBINE_CASES = ["tiny", "decode", "prefill",
                 synth.Workload("topk12", 37, 512, 64, 20, 12, "uniform", 71),   # slots beyond the unrolled 8
                 synth.Workload("topk3", 45, 384, 64, 7, 3, "biased", 72)]


@pytest.mark.parametrize("cfg", COMBINE_CASES, ids=[c if isinstance(c, str) else c.name for c in COMBINE_CASES])
def test_combine_unpermute_bit_exact(cfg):
    w = synth.CONFIGS[cfg] if isinstance(cfg, str) else cfg
    ei, probs = synth.routing(w.seed, w.M, w.E, w.topK, w.routing)
    ei[0, 0] = -1  # one invalid route
    rs = oracle.route_sort(ei, w.E)
    Rv = w.R - rs["invalid"]
    rng = np.random.default_rng(7)
    c2 = (rng.standard_normal((w.R, w.K)) * 400).astype(np.float16)
    pts2 = rng.uniform(20, 200, w.R).astype(np.float32)
    dmat = oracle.combine(c2[:Rv], pts2[:Rv])
    out_ref = oracle.unpermute(dmat, rs["expanded_row_idx"], probs)
    d = _dims(w)
    out = empty((w.M, w.K), torch.float16)
    moe.moe_combine_unpermute(d, dev(c2), dev(pts2), dev(rs["expanded_row_idx"]), dev(probs), out)
    torch.cuda.synchronize()
    assert_bits_equal(host(out), out_ref, "out")
