"""The benchmark's N > 1 host logic on CPU: world_size-2 `gloo` process groups.

The layer has no exchange step between GPUs: with N ranks every rank runs its own
replica of the layer (same weights, its own token batch), and the job's time is the
slowest rank's.  These tests run that host logic (replica inputs, the max over
ranks, the job throughput) in two CPU processes, and the reference arm under
torchrun with two ranks (rank 0 alone reports).
"""
import hashlib
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _digest(a):
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).digest()


def _rank_main(rank, world, port, result_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import bench
    import oracle
    import synth

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.CONFIGS["tiny"]
        inp = bench.replica_inputs(w, rank)
        names = sorted(inp)
        mine = torch.tensor(np.frombuffer(b"".join(_digest(inp[n]) for n in names), dtype=np.uint8))
        every = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(every, mine)
        per_rank = [{n: bytes(e[32 * i:32 * (i + 1)].tolist()) for i, n in enumerate(names)} for e in every]

        # each rank's replica output from its own batch (the oracle stands in for the layer)
        out = oracle.layer_tokens(inp, np.arange(w.M, dtype=np.int32))
        step_ms = 1.0 + 0.5 * rank  # the slower rank decides the job's time
        ms = bench.max_over_ranks(step_ms, world, "cpu")
        res = {
            "names": names,
            "same": {n: all(p[n] == per_rank[0][n] for p in per_rank) for n in names},
            "ms": ms,
            "value": bench.job_tokens_per_s(world, w.M, ms),
            "out_digest": _digest(out).hex(),
            "out_finite": bool(np.isfinite(out.view(np.float16)).all()),
        }
        with open(os.path.join(result_dir, "rank%d.json" % rank), "w") as f:
            json.dump(res, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replicas_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp

    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    same = res[0]["same"]
    for n in ("w1", "s1", "w2", "s2"):
        assert same[n], "weights differ between replicas: " + n
    for n in ("x", "expert_idx", "probs"):
        assert not same[n], "replicas share their token batch: " + n
    for r in res:
        assert r["ms"] == 1.5  # max over the ranks' 1.0 and 1.5 ms
        assert r["value"] == world * 16 / 1.5e-3
        assert r["out_finite"]
    assert res[0]["out_digest"] != res[1]["out_digest"]


def test_rank0_inputs_are_the_workload_itself():
    sys.path.insert(0, ROOT)
    import bench
    import synth

    w = synth.CONFIGS["tiny"]
    a, b = bench.replica_inputs(w, 0), synth.make_inputs(w)
    assert sorted(a) == sorted(b)
    for n in a:
        assert np.array_equal(a[n], b[n])


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(2.25, 1, "cpu") == 2.25
    assert bench.job_tokens_per_s(1, 128, 2.0) == 64000.0


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched like the N = 2 run: one JSON line (rank 0),
    both ranks exit 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--workload", "tiny", "--steps", "2", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=280)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
