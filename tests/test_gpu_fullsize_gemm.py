"""Full-size GMM1 / SwiGLU / GMM2 parity on the path the layer takes.

For the decode, mid, skewed and prefill workloads the GEMM stages run exactly as
inside moe_layer_fwd: the tile weight layout the benchmark uses, the activation
bounds the layer computes (above 24 rows per expert), and the engine choice and
split (warp-MMA tiles for experts of at most 32 rows, tcgen05 pairs for the
rest).  The stages are fed the oracle's own quantised tokens, so the comparison
isolates each GEMM:

  - GMM1's binary16 outputs equal the oracle's bit for bit on: a middle row of
    every active expert, the first and last row of every work tile (the pairs'
    balanced row tiles of up to 256 rows, 16/32-row warp-MMA tiles), and every row
    of the most loaded expert;
  - SwiGLU's codes on those rows are within 1 LSB on at most 0.1% of elements of
    the oracle's, its scales within 1e-6 relative;
  - GMM2, given the same int8 codes on both sides, equals the oracle bit for bit
    on the same rows;
  - above 24 rows per expert (skewed, prefill), the fused GMM1 + SwiGLU stage the
    layer runs there writes the same c1, q2, pts2 and q2 bounds as the two kernels,
    bit for bit, on every row.
The reference rows are evaluated one at a time by the oracle (its GEMM over a
list of expanded rows), so the CPU cost stays bounded at full size.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

if torch.cuda.is_available():
    import moe_expert_layer_gb300 as moe
    from gpu_util import assert_bits_equal, assert_q2_close, dev, empty, host

SPLIT_ROWS = 32    # experts with at most this many rows run on the warp-MMA engine (when split)
PAIR_ROWS = 256    # token rows per tcgen05 pair tile


def pair_row_tiles(cnt):
    """Row tiles of an expert on the tcgen05 pairs: t = ceil(cnt / 256) tiles of
    a = 32 * floor(cnt / (32 t)) rows, the first k of them a + 32 rows (k the fewest
    that cover cnt), the last holding what is left; (first, rows) each."""
    t = (cnt + PAIR_ROWS - 1) // PAIR_ROWS
    a = 32 * (cnt // (32 * t))
    k = (cnt - t * a + 31) // 32
    out, row = [], 0
    for rt in range(t):
        n = min(a + 32 if rt < k else a, cnt - row)
        out.append((row, n))
        row += n
    assert row == cnt and all(0 < n <= PAIR_ROWS for _, n in out)
    return out


def work_tiles(cumsum, R, E):
    """(first row, last row) of every work tile of the grouped GEMM, as the engines
    cut them: everything on warp-MMA tiles of 16 (up to 8 rows per expert on
    average) or 32 rows up to 24 rows per expert; above, experts of at most 32 rows
    on 32-row warp-MMA tiles (all experts on the pairs from 256 rows per expert on
    average) and the others on the pairs' balanced row tiles."""
    mean = R / E
    tiles = []
    lo = 0
    for e in range(E):
        hi = int(cumsum[e])
        cnt = hi - lo
        if cnt:
            if mean <= 24.0:
                step = 16 if mean <= 8.0 else 32
                tiles += [(t0, min(hi, t0 + step) - 1) for t0 in range(lo, hi, step)]
            elif cnt <= SPLIT_ROWS and mean < 256.0:
                tiles += [(lo, hi - 1)]
            else:
                tiles += [(lo + r0, lo + r0 + n - 1) for r0, n in pair_row_tiles(cnt)]
        lo = hi
    return tiles


def selected_rows(cumsum, R, E):
    rows = set()
    for a, b in work_tiles(cumsum, R, E):
        rows.update((a, b))
    lo = 0
    counts = []
    for e in range(E):
        hi = int(cumsum[e])
        if hi > lo:
            rows.add((lo + hi - 1) // 2)
        counts.append(hi - lo)
        lo = hi
    e_hot = int(np.argmax(counts))
    hot_lo = int(cumsum[e_hot - 1]) if e_hot else 0
    rows.update(range(hot_lo, int(cumsum[e_hot])))
    return np.array(sorted(rows), np.int64)


def segment_bounds(codes, cumsum, E, depth):
    """The activation bounds of include/moe_layer.h written out in numpy: for each
    expert and 1024-deep segment, the largest sum of |code| over the expert's rows."""
    nseg = (depth + moe.BOUND_SEGMENT - 1) // moe.BOUND_SEGMENT
    b = np.zeros((E, moe.BOUND_SEGMENTS), np.int32)
    lo = 0
    for e in range(E):
        hi = int(cumsum[e])
        if hi > lo:
            a = np.abs(codes[lo:hi].astype(np.int32))
            for s in range(nseg):
                b[e, s] = a[:, s * moe.BOUND_SEGMENT:(s + 1) * moe.BOUND_SEGMENT].sum(axis=1).max()
        lo = hi
    return b


@pytest.mark.parametrize("cfg", ["decode", "mid", "skewed", "prefill"])
def test_gemm_stages_bit_exact_at_full_size(cfg):
    w = synth.CONFIGS[cfg]
    inp = synth.make_inputs(cfg)
    R, E, K, I, topK = w.R, w.E, w.K, w.I, w.topK
    rs = oracle.route_sort(inp["expert_idx"], E)
    assert rs["invalid"] == 0
    sorted_src, cumsum = rs["sorted_src_route"], rs["cumsum"]
    xq, pts1 = oracle.quant_tokens(inp["x"])
    a1 = xq[sorted_src // topK]  # the dispatched expert-major operand, from the oracle's codes
    use_bounds = R / E > 24.0    # where the layer computes activation bounds

    d = moe.dims(w.M, K, I, E, topK, moe.WEIGHTS_TILES)
    w_t = {}
    for g, k in ((1, "w1"), (2, "w2")):
        t = empty(moe.moe_weight_tiles_bytes(d, g), torch.int8)
        moe.moe_pack_weight_tiles(d, g, dev(inp[k]), t)
        w_t[k] = t
    s1, s2 = dev(inp["s1"]), dev(inp["s2"])
    cs_dev, sorted_dev, ei_dev = dev(cumsum), dev(sorted_src), dev(inp["expert_idx"])
    gws = empty(moe.moe_gmm_workspace_size(d), torch.uint8)

    # the layer's own producer of the GEMM1 operand and its bounds, checked at full size
    a1_gpu = empty((R, K), torch.float16)
    b1_gpu = torch.zeros((E, moe.BOUND_SEGMENTS), dtype=torch.int32, device="cuda")
    pts1_gpu = empty(w.M, torch.float32)
    moe.moe_quant_dispatch(d, dev(inp["x"]), ei_dev, dev(rs["expanded_row_idx"]), a1_gpu, pts1_gpu,
                           b1_gpu if use_bounds else None)
    assert_bits_equal(host(a1_gpu), a1.astype(np.float16), "a1 (quant-scatter)")
    assert_bits_equal(host(pts1_gpu), pts1, "pts1")
    b1 = segment_bounds(a1, cumsum, E, K) if use_bounds else None
    if use_bounds:
        assert_bits_equal(host(b1_gpu), b1, "a1 activation bounds")

    rows = selected_rows(cumsum, R, E)
    sub = sorted_src[rows].astype(np.int32)

    # GMM1 on the oracle's codes
    c1 = empty((R, 2 * I), torch.float16)
    moe.moe_gmm1(d, dev(a1.astype(np.float16)), None, cs_dev, dev(b1) if use_bounds else None,
                 w_t["w1"], s1, c1, gws)
    assert moe.moe_workspace_status(gws) == 0
    c1_h = host(c1)
    _, ref_c1 = oracle.gmm1(xq, sub, inp["expert_idx"], inp["w1"], inp["s1"], rows.size)
    assert_bits_equal(c1_h[rows], ref_c1, "%s GMM1 (%d rows)" % (cfg, rows.size))

    # SwiGLU + requant on GMM1's output (equal to the oracle's on the checked rows)
    q2_i8 = empty((R, I), torch.int8)
    q2_f16 = empty((R, I), torch.float16)
    pts2 = empty(R, torch.float32)
    b2_gpu = torch.zeros((E, moe.BOUND_SEGMENTS), dtype=torch.int32, device="cuda")
    moe.moe_swiglu_quant(d, c1, dev(pts1), sorted_dev, cs_dev, ei_dev, q2_i8, q2_f16, pts2,
                         b2_gpu if use_bounds else None)
    q2_h, pts2_h = host(q2_i8), host(pts2)
    assert_bits_equal(host(q2_f16), q2_h.astype(np.float16), "q2 binary16 form")
    ref_q2, ref_pts2 = oracle.swiglu_quant(ref_c1, pts1, sub, topK)
    assert_q2_close(q2_h[rows], ref_q2, "%s q2" % cfg)
    np.testing.assert_allclose(pts2_h[rows], ref_pts2, rtol=1e-6)
    if use_bounds:
        assert_bits_equal(host(b2_gpu), segment_bounds(q2_h, cumsum, E, I), "q2 activation bounds")

    if use_bounds:
        # the layer's path above 24 rows per expert: SwiGLU inside the pairs' GMM1
        # kernel; the same bits as the two kernels above, on every row
        c1f = torch.full_like(c1, float("nan"))
        q2f = torch.full_like(q2_f16, float("nan"))
        pts2f = torch.full_like(pts2, float("nan"))
        b2f = torch.zeros_like(b2_gpu)
        moe.moe_gmm1_swiglu(d, dev(a1.astype(np.float16)), cs_dev, dev(b1), w_t["w1"], s1, c1f, dev(pts1),
                            sorted_dev, ei_dev, q2f, pts2f, b2f, gws)
        assert moe.moe_workspace_status(gws) == 0
        Rv = int(cumsum[-1])
        assert_bits_equal(host(c1f)[:Rv], c1_h[:Rv], "%s fused c1" % cfg)
        assert_bits_equal(host(q2f)[:Rv], host(q2_f16)[:Rv], "%s fused q2" % cfg)
        assert_bits_equal(host(pts2f)[:Rv], pts2_h[:Rv], "%s fused pts2" % cfg)
        assert_bits_equal(host(b2f), host(b2_gpu), "%s fused q2 bounds" % cfg)

    # GMM2 on the same int8 codes on both sides (the GPU's q2)
    c2 = empty((R, K), torch.float16)
    moe.moe_gmm2(d, q2_f16, cs_dev, b2_gpu if use_bounds else None, w_t["w2"], s2, c2, gws)
    assert moe.moe_workspace_status(gws) == 0
    _, ref_c2 = oracle.gmm2(q2_h[rows], sub, inp["expert_idx"], inp["w2"], inp["s2"])
    assert_bits_equal(host(c2)[rows], ref_c2, "%s GMM2 (%d rows)" % (cfg, rows.size))


def test_row_selection_covers_every_tile_and_expert():
    """Host check of the selection itself on the skewed routing: every active
    expert and every tile end is in it, the hottest expert whole."""
    w = synth.CONFIGS["skewed"]
    ei, _ = synth.routing(w.seed, w.M, w.E, w.topK, w.routing)
    rs = oracle.route_sort(ei, w.E)
    cs = rs["cumsum"]
    rows = set(selected_rows(cs, w.R, w.E).tolist())
    tiles = work_tiles(cs, w.R, w.E)
    assert all(a in rows and b in rows for a, b in tiles)
    lo = 0
    for e in range(w.E):
        hi = int(cs[e])
        assert hi == lo or any(lo <= r < hi for r in rows)
        lo = hi
    counts = rs["tokens_per_expert"]
    e_hot = int(np.argmax(counts))
    hot = range(int(cs[e_hot]) - int(counts[e_hot]), int(cs[e_hot]))
    assert set(hot) <= rows and counts[e_hot] > 0.1 * w.R
