"""Helpers for the GPU parity tests: numpy <-> torch device tensors and the
comparison rules the layer is held to."""
import numpy as np
import torch


def dev(a):
    """numpy array -> contiguous CUDA tensor with the same bytes (float16 stays float16)."""
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.cpu().numpy()


def empty(shape, dtype):
    return torch.empty(shape, dtype=dtype, device="cuda")


def upload_inputs(inp):
    return {k: dev(v) for k, v in inp.items()}


def assert_bits_equal(got, ref, what):
    g = np.ascontiguousarray(got).view(np.uint16 if got.dtype == np.float16 else got.dtype)
    r = np.ascontiguousarray(ref).view(np.uint16 if ref.dtype == np.float16 else ref.dtype)
    if not np.array_equal(g, r):
        bad = np.argwhere(g != r)
        raise AssertionError("%s: %d of %d elements differ; first at %s: got %s ref %s" % (
            what, len(bad), g.size, tuple(bad[0]), got[tuple(bad[0])], ref[tuple(bad[0])]))


def assert_q2_close(got, ref, what="q2"):
    """Requantised activations: at most 1 LSB apart, on at most 0.1% of elements."""
    d = np.abs(got.astype(np.int32) - ref.astype(np.int32))
    assert d.max(initial=0) <= 1, "%s: max LSB difference %d" % (what, d.max())
    frac = (d > 0).mean() if d.size else 0.0
    assert frac <= 1e-3, "%s: %.4f%% of elements differ by 1 LSB" % (what, 100 * frac)


def assert_out_close(got, ref, what="out"):
    """Final output: per row, max |got - ref| <= 1e-2 * max |ref row|, no NaN/Inf."""
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    assert np.isfinite(g).all(), "%s: NaN/Inf in the output" % what
    err = np.abs(g - r).max(axis=1)
    lim = 1e-2 * np.abs(r).max(axis=1)
    bad = np.nonzero(err > lim)[0]
    assert bad.size == 0, "%s: %d rows out of tolerance, e.g. row %d err %g lim %g" % (
        what, bad.size, bad[0], err[bad[0]], lim[bad[0]])
