"""Failure detection on the GPU without a fault: a device-side wait that can never
complete must give up, report MOE_ERR_TIMEOUT through the status word, and leave
the context usable for the next launches."""
import time

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import moe_expert_layer_gb300 as moe
    from gpu_util import assert_out_close, empty, host, upload_inputs


def test_bounded_wait_times_out_and_reports():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    moe.moe_selftest_wait_timeout(status, 50000)  # 50 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) == -8  # MOE_ERR_TIMEOUT
    assert 0.04 < dt < 5.0


def test_context_usable_after_timeout():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_selftest_wait_timeout(status, 10000)
    torch.cuda.synchronize()
    assert int(status.item()) == -8
    w = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(w)
    dev = upload_inputs(inp)
    d = moe.dims(w.M, w.K, w.I, w.E, w.topK)
    ws = empty(moe.moe_layer_workspace_size(d), torch.uint8)
    out = empty((w.M, w.K), torch.float16)
    moe.moe_layer_fwd(d, dev["x"], dev["expert_idx"], dev["probs"], dev["w1"], dev["s1"], dev["w2"],
                      dev["s2"], out, ws)
    assert moe.moe_workspace_status(ws) == 0
    assert_out_close(host(out), oracle.layer_fwd(inp))


def test_selftest_rejects_bad_limits():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_wait_timeout(status, 0)
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_wait_timeout(status, 3000000)


def test_bounded_count_wait_times_out_and_reports():
    """The wait the SwiGLU fused into GMM1 uses on other CTAs' item counts gives up on a
    count nothing raises, reports MOE_ERR_TIMEOUT, and the context then runs a layer
    whose GMM1 fuses SwiGLU (every expert on the tcgen05 pairs) correctly."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    count = torch.ones(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    moe.moe_selftest_count_timeout(status, count, 50000)  # 50 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) == -8 and int(count.item()) == 0
    assert 0.04 < dt < 5.0
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_count_timeout(status, count, 0)
    w = synth.Workload("fused_after_timeout", 1024, 256, 128, 4, 1, "uniform", 115)
    inp = synth.make_inputs(w)
    dev = upload_inputs(inp)
    d = moe.dims(w.M, w.K, w.I, w.E, w.topK)
    ws = empty(moe.moe_layer_workspace_size(d), torch.uint8)
    out = empty((w.M, w.K), torch.float16)
    moe.moe_layer_fwd(d, dev["x"], dev["expert_idx"], dev["probs"], dev["w1"], dev["s1"], dev["w2"],
                      dev["s2"], out, ws)
    assert moe.moe_workspace_status(ws) == 0
    assert_out_close(host(out), oracle.layer_fwd(inp))
