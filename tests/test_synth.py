"""The seeded input generator (synth/) draws what its recipe says: the value
distributions, ranges and routing structure of the workloads.  These checks pin
the generator against its own definition (counter-based SplitMix64 streams,
Box-Muller normals, Gumbel-top-k routing) and against closed forms of those
distributions; none of them touches the layer's arithmetic."""
import numpy as np
import pytest

import synth


def binomial_bound(p, n, sigmas=5.0):
    return sigmas * np.sqrt(p * (1.0 - p) / n)


def test_streams_are_deterministic_and_seed_dependent():
    a = synth.make_inputs("tiny")
    b = synth.make_inputs("tiny")
    for k in a:
        assert a[k].tobytes() == b[k].tobytes(), k
    other = synth.make_inputs(synth.Workload("tiny", 16, 256, 256, 8, 2, "uniform", 1))
    for k in a:
        assert a[k].tobytes() != other[k].tobytes(), k


def test_draw_is_independent_of_the_tensor_length():
    # counter-based: element i of a stream does not depend on how many are drawn
    long = synth.normal_f16(5, 1, (4096,))
    short = synth.normal_f16(5, 1, (1000,))
    assert long[:1000].tobytes() == short.tobytes()
    w_long = synth.int8_sym127(5, 2, (999,))
    w_short = synth.int8_sym127(5, 2, (500,))
    assert w_long[:500].tobytes() == w_short.tobytes()


def test_tokens_are_standard_normal_in_binary16():
    x = synth.normal_f16(11, 1, (1 << 20,)).astype(np.float64)
    n = x.size
    assert abs(x.mean()) < 5.0 / np.sqrt(n)
    assert abs(x.var() - 1.0) < 5.0 * np.sqrt(2.0 / n)
    # tails of N(0,1): P(|x| > 2) = 0.0455, P(|x| > 3) = 0.0027
    for t, p in [(2.0, 0.04550026), (3.0, 0.00269980)]:
        assert abs((np.abs(x) > t).mean() - p) < binomial_bound(p, n)
    assert np.isfinite(x).all()


def test_weights_uniform_over_the_255_symmetric_codes():
    w = synth.int8_sym127(12, 2, (255 * 4000 + 1,))  # odd length: the last pair is half used
    assert w.min() == -127 and w.max() == 127  # -128 never drawn
    counts = np.bincount(w.astype(np.int64) + 127, minlength=255)
    assert counts.size == 255
    n, p = w.size, 1.0 / 255
    assert np.all(np.abs(counts / n - p) < binomial_bound(p, n))


def test_scales_uniform_on_the_stated_interval():
    s = synth.uniform_f32(13, 3, (1 << 18,), 1e-3, 1e-2)
    assert s.dtype == np.float32
    assert s.min() >= np.float32(1e-3) and s.max() <= np.float32(1e-2)
    u = (s.astype(np.float64) - 1e-3) / 9e-3
    n = u.size
    assert abs(u.mean() - 0.5) < 5.0 * np.sqrt(1.0 / 12.0 / n)
    hist = np.histogram(u, bins=10, range=(0.0, 1.0))[0] / n
    assert np.all(np.abs(hist - 0.1) < binomial_bound(0.1, n))


@pytest.mark.parametrize("mode", ["uniform", "biased", "zipf"])
def test_routes_are_distinct_valid_experts_with_softmax_probs(mode):
    M, E, topK = 3000, 64, 6
    ei, pr = synth.routing(21, M, E, topK, mode)
    assert ei.shape == (M, topK) and pr.shape == (M, topK)
    assert ei.min() >= 0 and ei.max() < E
    srt = np.sort(ei, axis=1)
    assert np.all(srt[:, 1:] != srt[:, :-1])  # no expert twice in a token
    assert np.all(pr > 0)
    np.testing.assert_allclose(pr.astype(np.float64).sum(axis=1), 1.0, atol=4e-7)


def test_uniform_routing_gives_every_expert_the_same_share():
    M, E, topK = 20000, 32, 4
    ei, _ = synth.routing(22, M, E, topK, "uniform")
    freq = np.bincount(ei.ravel(), minlength=E) / (M * topK)
    # each expert is in a token's k-subset with probability k/E, independently per token
    p = 1.0 / E
    assert np.all(np.abs(freq - p) < 5.0 * np.sqrt(topK / E * (1 - topK / E) / M) / topK)


def test_uniform_routing_probs_are_softmax_of_standard_normals():
    # log p_i - log p_j = z_i - z_j with z ~ N(0,1) independent: N(0, 2)
    _, pr = synth.routing(23, 50000, 16, 3, "uniform")
    d = np.log(pr[:, 0].astype(np.float64)) - np.log(pr[:, 1].astype(np.float64))
    n = d.size
    assert abs(d.mean()) < 5.0 * np.sqrt(2.0 / n)
    assert abs(d.var() - 2.0) < 5.0 * 2.0 * np.sqrt(2.0 / n)


def test_zipf_first_pick_follows_the_zipf_law():
    # Gumbel-top-k with k = 1 draws one expert from softmax(logit) = the Zipf law
    # over a seeded permutation: the sorted first-pick frequencies are (i+1)^-s / H
    M, E, s = 200000, 16, 1.2
    ei, _ = synth.routing(24, M, E, 1, "zipf", s)
    freq = np.sort(np.bincount(ei.ravel(), minlength=E) / M)[::-1]
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    p /= p.sum()
    assert np.all(np.abs(freq - p) < binomial_bound(p, M))


def test_zipf_top_k_draws_without_replacement():
    # k = 2 of 3 experts with Zipf weights w.  Gumbel-top-k is sequential sampling
    # without replacement, so j is left out when the pair is the other two, drawn in
    # either order: P(j excluded) = sum over i != j of w_i * w_l / (1 - w_i), with l
    # the third expert
    M, E, s = 200000, 3, 1.2
    ei, _ = synth.routing(25, M, E, 2, "zipf", s)
    freq = np.sort(np.bincount(ei.ravel(), minlength=E) / M)[::-1]
    w = np.arange(1, E + 1, dtype=np.float64) ** -s
    w /= w.sum()
    incl = []
    for j in range(E):
        others = [i for i in range(E) if i != j]
        excl = sum(w[i] * w[[o for o in others if o != i][0]] / (1.0 - w[i]) for i in others)
        incl.append(1.0 - excl)
    incl = np.array(incl)
    assert abs(incl.sum() - 2.0) < 1e-12
    assert np.all(np.abs(freq - incl) < binomial_bound(incl, M))


def test_skewed_workload_top_expert_share():
    # Zipf s = 1.2 over 256 experts, 8 distinct per token: the hottest expert takes
    # about 11.7% of the 16384 routes (it is in almost every token's set, capped at 1/8)
    w = synth.CONFIGS["skewed"]
    ei, _ = synth.routing(w.seed, w.M, w.E, w.topK, w.routing, w.zipf_s)
    counts = np.bincount(ei.ravel(), minlength=w.E)
    share = counts.max() / ei.size
    assert 0.10 < share <= 0.125
    assert (counts > 0.05 * ei.size).sum() >= 2  # more than one expert above 5%


def test_biased_routing_is_skewed_by_the_expert_bias():
    # b ~ N(0, 0.25) per expert shifts the experts' shares: the spread of the
    # counts is far above the multinomial spread of uniform routing
    w = synth.CONFIGS["mid"]
    ei, _ = synth.routing(w.seed, w.M, w.E, w.topK, w.routing)
    counts = np.bincount(ei.ravel(), minlength=w.E)
    mean = ei.size / w.E
    assert counts.std() > 1.5 * np.sqrt(mean)
    eu, _ = synth.routing(w.seed, w.M, w.E, w.topK, "uniform")
    assert np.bincount(eu.ravel(), minlength=w.E).std() < 1.3 * np.sqrt(mean)
