"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: numpy/scipy library
routines (int64 matmul, float16 casts, expit), brute force on tiny inputs,
closed forms, hand-worked fixtures under tests/golden/, and invariants of the
route sort.  A plausible slip in the oracle (a swapped SwiGLU half, a wrong
rounding mode, a dropped scale, an unstable sort, an off-by-one in cumsum)
fails at least one of them.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth
from conftest import read_golden

F16_MAX = 65504.0


def sat_f16(v):
    """Reference stage conversion built from numpy's own float16 cast."""
    return np.clip(np.asarray(v, np.float32), -F16_MAX, F16_MAX).astype(np.float16)


# ---------------------------------------------------------------- binary16 conversions
def test_f16_to_f32_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.f16_to_f32(bits)
    ref = bits.view(np.float16).astype(np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_f32_to_f16_matches_numpy_rne():
    rng = np.random.default_rng(0)
    halves = np.arange(0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)
    nxt = np.arange(1, 0x7C01, dtype=np.uint16).view(np.float16).astype(np.float32)
    mids = ((halves.astype(np.float64) + nxt.astype(np.float64)) / 2).astype(np.float32)  # ties
    vals = np.concatenate([halves, mids, -mids, rng.standard_normal(100000).astype(np.float32) * 1000,
                           np.array([65519.0, 65520.0, 1e6, -1e6, 6e-8, 3e-8, 2.9e-8], np.float32)])
    got = oracle.f32_to_f16(vals).view(np.uint16)
    with np.errstate(over="ignore"):  # 65520 and +-1e6 overflow to +-inf on purpose (IEEE cast)
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_f32_to_f16_saturates():
    vals = np.array([65504.0, 65519.0, 65520.0, 70000.0, 1e30, -65520.0, -1e30, 1.0], np.float32)
    got = oracle.f32_to_f16_sat(vals).astype(np.float32)
    assert np.array_equal(got, [65504, 65504, 65504, 65504, 65504, -65504, -65504, 1.0])


# ---------------------------------------------------------------- FrontReorder sort
def brute_sort(expert_idx, E):
    """O(R^2) rank of each route under the key (valid?0:1, expert, route)."""
    ei = expert_idx.ravel()
    R = ei.size
    valid = (ei >= 0) & (ei < E)
    key = [(0 if valid[r] else 1, int(ei[r]) if valid[r] else 0, r) for r in range(R)]
    rank = np.array([sum(1 for q in range(R) if key[q] < key[r]) for r in range(R)])
    sorted_src = np.empty(R, np.int64)
    sorted_src[rank] = np.arange(R)
    expanded = np.where(valid, rank, -1)
    tpe = np.array([(ei == e).sum() for e in range(E)])
    return sorted_src, expanded, tpe, np.cumsum(tpe)


@pytest.mark.parametrize("M,topK,E,seed", [(16, 2, 8, 0), (7, 3, 5, 1), (33, 4, 16, 2), (1, 1, 1, 3)])
def test_route_sort_brute_force(M, topK, E, seed):
    ei, _ = synth.routing(seed, M, E, topK, "uniform")
    got = oracle.route_sort(ei, E)
    s, x, tpe, cs = brute_sort(ei, E)
    assert np.array_equal(got["sorted_src_route"], s)
    assert np.array_equal(got["expanded_row_idx"], x)
    assert np.array_equal(got["tokens_per_expert"], tpe)
    assert np.array_equal(got["cumsum"], cs)
    assert got["invalid"] == 0


def test_route_sort_invalid_and_duplicates():
    ei = np.array([[3, -1], [0, 3], [7, 0], [3, 3], [2, 99]], np.int32)  # E = 4
    got = oracle.route_sort(ei, 4)
    s, x, tpe, cs = brute_sort(ei, 4)
    assert np.array_equal(got["sorted_src_route"], s)
    assert np.array_equal(got["expanded_row_idx"], x)
    assert np.array_equal(got["tokens_per_expert"], tpe)
    assert got["invalid"] == 3
    assert list(got["sorted_src_route"][-3:]) == [1, 4, 9]  # invalid routes last, ascending
    assert all(got["expanded_row_idx"][r] == -1 for r in (1, 4, 9))


@pytest.mark.parametrize("mode", ["uniform", "biased", "zipf"])
def test_route_sort_invariants(mode):
    M, E, topK = 300, 64, 6
    ei, _ = synth.routing(5, M, E, topK, mode)
    g = oracle.route_sort(ei, E)
    R = M * topK
    s, x, tpe, cs = g["sorted_src_route"], g["expanded_row_idx"], g["tokens_per_expert"], g["cumsum"]
    assert tpe.sum() == R and cs[-1] == R
    assert np.array_equal(np.sort(x), np.arange(R))  # a permutation
    assert np.array_equal(x[s], np.arange(R))  # inverse of the sort
    sorted_expert = ei.ravel()[s]
    assert np.all(np.diff(sorted_expert) >= 0)
    same = np.diff(sorted_expert) == 0
    assert np.all(np.diff(s)[same] > 0)  # stable: routes ascending inside an expert
    assert np.array_equal(np.bincount(ei.ravel(), minlength=E), tpe)
    assert np.array_equal(np.cumsum(tpe), cs)


def test_route_sort_one_hot_and_empty_experts():
    ei = np.full((10, 1), 3, np.int32)
    g = oracle.route_sort(ei, 6)
    assert list(g["tokens_per_expert"]) == [0, 0, 0, 10, 0, 0]
    assert list(g["cumsum"]) == [0, 0, 0, 10, 10, 10]
    assert np.array_equal(g["sorted_src_route"], np.arange(10))


# ---------------------------------------------------------------- token quant
def test_quant_golden_round_half_away():
    x, q, s = read_golden("quant_round_half_away.txt")
    xq, pts1 = oracle.quant_tokens(np.array([x], np.float16))
    assert list(xq[0]) == [int(v) for v in q]
    assert pts1[0] == np.float32(s[0])


def test_quant_golden_divides_by_the_rounded_scale():
    """Phase 2c divides each element by the binary32 scale (pinned where that
    differs from multiplying by 127/amax or dividing x*127 by amax)."""
    rows = read_golden("quant_divide_inexact_scale.txt")
    for i in range(0, len(rows), 3):
        x, q, s = rows[i:i + 3]
        xq, pts1 = oracle.quant_tokens(np.array([x], np.float16))
        assert list(xq[0]) == [int(v) for v in q], "row with amax %g" % max(abs(v) for v in x)
        assert pts1[0] == np.float32(s[0])


def test_quant_properties():
    x = synth.normal_f16(11, 1, (64, 512))
    x[5] = 0  # all-zero row
    x[6, :] = np.float16(-3.0)  # constant row
    xq, pts1 = oracle.quant_tokens(x)
    xf = x.astype(np.float32)
    amax = np.abs(xf).max(1)
    assert np.array_equal(pts1, (amax / np.float32(127)).astype(np.float32))
    assert pts1[5] == 0 and not xq[5].any()
    assert np.all(xq[6] == -127)
    nz = amax > 0
    # the element of largest magnitude maps to +-127
    arg = np.abs(xf).argmax(1)
    assert np.all(np.abs(xq[np.arange(64), arg][nz]) == 127)
    # |x - q*s| <= s/2 (plus fp32 rounding slack)
    err = np.abs(xf - xq.astype(np.float32) * pts1[:, None])
    assert np.all(err[nz] <= pts1[nz, None] * (0.5 + 1e-5))
    assert xq.min() >= -127


# ---------------------------------------------------------------- grouped GEMMs
def _gmm_setup(seed=3, M=24, K=256, I=128, E=5, topK=2):
    w = synth.Workload("t", M, K, I, E, topK, "uniform", seed)
    d = synth.make_inputs(w)
    rs = oracle.route_sort(d["expert_idx"], E)
    xq, pts1 = oracle.quant_tokens(d["x"])
    return d, rs, xq, pts1


def test_gmm1_matches_int64_matmul():
    d, rs, xq, pts1 = _gmm_setup()
    R = rs["sorted_src_route"].size
    acc, c1 = oracle.gmm1(xq, rs["sorted_src_route"], d["expert_idx"], d["w1"], d["s1"], R, True)
    tok = rs["sorted_src_route"] // d["expert_idx"].shape[1]
    exp = d["expert_idx"].ravel()[rs["sorted_src_route"]]
    for row in range(R):
        ref = d["w1"][exp[row]].astype(np.int64) @ xq[tok[row]].astype(np.int64)
        assert np.array_equal(acc[row], ref)
        ref_c = sat_f16(ref.astype(np.float32) * d["s1"][exp[row]])
        assert np.array_equal(c1[row].view(np.uint16), ref_c.view(np.uint16))


def test_gmm_adversarial_accumulator_range():
    """All-+-127 operands: |acc| = K * 16129 (the largest magnitude), exact in int32."""
    K, I, E = 7168, 64, 1
    xq = np.full((2, K), 127, np.int8)
    xq[1, ::2] = -127
    w1 = np.full((E, 2 * I, K), 127, np.int8)
    w1[0, 1::2, :] = -127
    s1 = np.full((E, 2 * I), 1e-3, np.float32)
    ei = np.zeros((2, 1), np.int32)
    rs = oracle.route_sort(ei, E)
    acc, c1 = oracle.gmm1(xq, rs["sorted_src_route"], ei, w1, s1, 2, True)
    assert acc[0, 0] == K * 16129 and acc[0, 1] == -K * 16129
    assert acc[1, 0] == 0
    assert np.all(np.abs(c1.astype(np.float32)) <= F16_MAX)


def test_gmm2_matches_int64_matmul():
    d, rs, xq, pts1 = _gmm_setup(seed=4)
    R = rs["sorted_src_route"].size
    I = d["w2"].shape[2]
    q2 = synth.int8_sym127(9, 1, (R, I))
    acc, c2 = oracle.gmm2(q2, rs["sorted_src_route"], d["expert_idx"], d["w2"], d["s2"], True)
    exp = d["expert_idx"].ravel()[rs["sorted_src_route"]]
    for row in range(R):
        ref = d["w2"][exp[row]].astype(np.int64) @ q2[row].astype(np.int64)
        assert np.array_equal(acc[row], ref)
        ref_c = sat_f16(ref.astype(np.float32) * d["s2"][exp[row]])
        assert np.array_equal(c2[row].view(np.uint16), ref_c.view(np.uint16))


# ---------------------------------------------------------------- SwiGLU + requant
def test_swiglu_golden_round_half_even():
    up, q, s = read_golden("requant_round_half_even.txt")
    I = len(up)
    c1 = np.array([[64.0] * I + up], np.float16)
    q2, pts2 = oracle.swiglu_quant(c1, np.ones(1, np.float32), np.zeros(1, np.int32), 1)
    assert list(q2[0]) == [int(v) for v in q]
    assert pts2[0] == np.float32(s[0])


def test_swiglu_matches_expit():
    """silu acts on the FIRST half: y = h1 * sigmoid(h1) * h2 (scipy's expit)."""
    rng = np.random.default_rng(1)
    R, I = 40, 96
    c1 = (rng.standard_normal((R, 2 * I)) * 300).astype(np.float16)
    c1[3] = 0  # all-zero row -> scale 0, codes 0
    pts1 = rng.uniform(0.01, 0.05, R).astype(np.float32)
    sorted_src = np.arange(R, dtype=np.int32)  # topK = 1, row d <-> token d
    q2, pts2 = oracle.swiglu_quant(c1, pts1, sorted_src, 1)
    h = c1.astype(np.float64) * pts1[:, None].astype(np.float64)
    y = h[:, :I] * expit(h[:, :I]) * h[:, I:]
    amax = np.abs(y).max(1)
    assert pts2[3] == 0 and not q2[3].any()
    nz = amax > 0
    np.testing.assert_allclose(pts2[nz], amax[nz] / 127, rtol=1e-5)
    qref = np.rint(y[nz] * (127 / amax[nz, None]))
    diff = np.abs(q2[nz].astype(np.int64) - qref)
    assert diff.max() <= 1 and (diff > 0).mean() < 1e-3
    # swapping the halves gives a different answer (the pin is sensitive to it)
    ysw = h[:, I:] * expit(h[:, I:]) * h[:, :I]
    qsw = np.rint(ysw[nz] * (127 / np.abs(ysw[nz]).max(1, keepdims=True)))
    assert (np.abs(q2[nz] - qsw) > 1).mean() > 0.3


# ---------------------------------------------------------------- Combine + Unpermute
def test_combine_unpermute_closed_form():
    # two tokens, topK = 2; row values and probs chosen so every product is exact
    c2 = np.array([[1.0, -2.0, 4.0], [3.0, 0.5, -1.0], [8.0, 1.0, 2.0], [0.0, 0.0, 6.0]], np.float16)
    pts2 = np.array([2.0, 0.5, 0.25, 1.0], np.float32)
    dmat = oracle.combine(c2, pts2)
    assert np.array_equal(dmat.astype(np.float32),
                          [[2, -4, 8], [1.5, 0.25, -0.5], [2, 0.25, 0.5], [0, 0, 6]])
    expanded = np.array([2, 0, 1, -1], np.int32)  # token 1 slot 1 invalid
    probs = np.array([[0.25, 0.75], [0.5, 0.5]], np.float32)
    out = oracle.unpermute(dmat, expanded, probs).astype(np.float32)
    assert np.array_equal(out, [[0.25 * 2 + 0.75 * 2, 0.25 * 0.25 - 0.75 * 4, 0.25 * 0.5 + 0.75 * 8],
                                [0.5 * 1.5, 0.5 * 0.25, -0.5 * 0.5]])


def test_unpermute_golden_slot_order_multiply_then_add():
    """Unpermute: fp32 accumulator from zero, slots in order, a rounded multiply then a
    rounded add (pinned on cancelling sums where a fused multiply-add, a binary16
    accumulator or the reverse slot order give other binary16 outputs)."""
    rows = read_golden("unpermute_slot_order_fp32.txt")
    n_tok = len(rows) // 3
    topK = len(rows[0])
    R = n_tok * topK
    # expanded rows in an order other than the route order, so the gather is pinned too
    expanded = np.array([(5 * r + 2) % R for r in range(R)], np.int32)
    assert sorted(expanded) == list(range(R))
    dmat = np.zeros((R, 1), np.float16)
    probs = np.zeros((n_tok, topK), np.float32)
    want = []
    for t in range(n_tok):
        dvals, p, out = rows[3 * t:3 * t + 3]
        for j in range(topK):
            dmat[expanded[t * topK + j], 0] = dvals[j]
        probs[t] = np.array(p, np.float64).astype(np.float32)
        want.append(out[0])
    got = oracle.unpermute(dmat, expanded, probs).astype(np.float64)[:, 0]
    assert list(got) == want


def test_combine_saturates():
    c2 = np.array([[60000.0, -60000.0, 1.0]], np.float16)
    dmat = oracle.combine(c2, np.array([4.0], np.float32))
    assert np.array_equal(dmat.astype(np.float32), [[65504, -65504, 4]])


# ---------------------------------------------------------------- whole layer
def _dense_ffn_ref(x, w1, s1, w2, s2):
    """Independent float64 restatement of one expert's W8A8 FFN on one token,
    built from numpy/scipy library routines (tolerance check, not bit-exact)."""
    xf = x.astype(np.float64)
    amax = np.abs(xf).max()
    xq = np.clip(np.sign(xf) * np.floor(np.abs(xf) / (amax / 127) + 0.5), -127, 127)
    c1 = (w1.astype(np.int64) @ xq.astype(np.int64)) * s1.astype(np.float64)
    h = c1 * (amax / 127)
    I = w1.shape[0] // 2
    y = h[:I] * expit(h[:I]) * h[I:]
    a2 = np.abs(y).max()
    q2 = np.clip(np.rint(y * 127 / a2), -127, 127)
    c2 = (w2.astype(np.int64) @ q2.astype(np.int64)) * s2.astype(np.float64)
    return c2 * (a2 / 127)


def test_layer_one_hot_is_dense_ffn():
    """topK = 1, prob 1, every token to one expert: the layer is a dense W8A8 FFN."""
    w = synth.Workload("t", 12, 256, 128, 3, 1, "uniform", 7)
    d = synth.make_inputs(w)
    d["expert_idx"][:] = 1
    d["probs"][:] = 1.0
    out = oracle.layer_fwd(d).astype(np.float64)
    for t in range(12):
        ref = _dense_ffn_ref(d["x"][t], d["w1"][1], d["s1"][1], d["w2"][1], d["s2"][1])
        assert np.abs(out[t] - ref).max() <= 1e-2 * np.abs(ref).max()


def test_layer_identical_experts_convex_probs():
    """All experts equal and probs summing to 1: out = the expert's FFN of the token."""
    w = synth.Workload("t", 10, 256, 128, 4, 3, "uniform", 8)
    d = synth.make_inputs(w)
    for e in range(1, 4):
        d["w1"][e], d["s1"][e], d["w2"][e], d["s2"][e] = d["w1"][0], d["s1"][0], d["w2"][0], d["s2"][0]
    out = oracle.layer_fwd(d).astype(np.float64)
    for t in range(10):
        ref = _dense_ffn_ref(d["x"][t], d["w1"][0], d["s1"][0], d["w2"][0], d["s2"][0])
        assert np.abs(out[t] - ref).max() <= 1e-2 * np.abs(ref).max()


def test_layer_zero_token_rows():
    d = synth.make_inputs("tiny")
    d["x"][[2, 9]] = 0
    out = oracle.layer_fwd(d)
    assert not out[[2, 9]].astype(np.float32).any()


@pytest.mark.parametrize("cfg", ["tiny"])
def test_layer_permuted_equals_per_token(cfg):
    """The permuted pipeline (sort, grouped GEMMs over expert-major rows,
    unpermute) equals the per-token evaluation bit for bit."""
    d = synth.make_inputs(cfg)
    out, it = oracle.layer_fwd(d, intermediates=True)
    per_tok = oracle.layer_tokens(d, np.arange(d["x"].shape[0]))
    assert np.array_equal(out.view(np.uint16), per_tok.view(np.uint16))
    assert np.isfinite(out.astype(np.float32)).all()


def test_layer_invalid_routes_skipped():
    d = synth.make_inputs("tiny")
    ref = d["expert_idx"].copy()
    d["expert_idx"][4, 1] = -5
    d["expert_idx"][7, 0] = 100
    out, it = oracle.layer_fwd(d, intermediates=True)
    assert it["invalid"] == 2
    # token 4 equals a layer where slot 1's probability is 0
    d2 = dict(d)
    d2["expert_idx"] = ref
    d2["probs"] = d["probs"].copy()
    d2["probs"][4, 1] = 0.0
    d2["probs"][7, 0] = 0.0
    out2 = oracle.layer_fwd(d2)
    assert np.array_equal(out.view(np.uint16), out2.view(np.uint16))
