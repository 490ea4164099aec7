"""Benchmark of the W8A8 MoE expert layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill] [--also tiny,decode,mid,skewed]
                    [--impl reference]

One step = one pass of the whole layer (FrontReorder: route sort and token quant
with the scatter to expert-major rows, GMM1, SwiGLU + requant, GMM2, Combine + Unpermute) over one
batch of the workload's seeded synthetic inputs.  With N > 1 (torchrun, one process per GPU)
every rank runs an independent replica of the layer on its own batch: the path
has no exchange step, so there is no collective on the data path (weak scaling).

Prints one JSON line on rank 0.  `value` is tokens/s of the whole job with the
inputs resident in device memory on the headline workload (prefill, the largest
configuration); `e2e` repeats the measurement with the batches in host memory,
host<->device copies included, through the pipelined executor (moe_layer_pipeline_*;
`e2e.serial`: one batch at a time through the host-buffer graph); `workloads` carries the same
step, stage and roofline figures for the other configurations, measured in the
same run.  `--impl reference` times the CPU oracle instead (on the host cores,
rank 0 only).
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="prefill", choices=sorted(synth.CONFIGS),
                    help="the headline workload (the JSON line's value, roofline, e2e)")
    ap.add_argument("--also", default="tiny,decode,mid,skewed",
                    help="comma-separated workloads measured in the same run and reported under "
                         "`workloads` (single GPU only; 'none' for none)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time moe_layer_fwd stream launches instead of the layer's CUDA graph")
    ap.add_argument("--weights", default="tiles", choices=["tiles", "rows"],
                    help="weight layout the layer reads: 16 KiB tiles packed once before timing "
                         "(moe_pack_weight_tiles), or the [E][N][D] rows as given")
    return ap.parse_args()


def workload_desc(w):
    return "%s MoE layer: M=%d K=%d I=%d (GMM1 2I=%d) E=%d topK=%d, %s routing, seed %d" % (
        w.name, w.M, w.K, w.I, 2 * w.I, w.E, w.topK, w.routing, w.seed)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------------------- algorithmic work
def algorithmic(w, expert_idx):
    """Bytes and ops each stage must move / perform for one step: the algorithmic
    work of each stage of the layer, counted from the shapes and the active experts."""
    R = w.M * w.topK
    active = int(np.unique(expert_idx[(expert_idx >= 0) & (expert_idx < w.E)]).size)
    K, I, M = w.K, w.I, w.M
    st = {}
    # FrontReorder: the route sort (expert ids in, two route tables and the counts out)
    # and the token quant with the scatter (read x, write the expert-major codes); one
    # kernel up to 4096 routes, where the stage is timed whole
    st["route_sort"] = {"bytes": 4 * R + 8 * R + 8 * w.E}
    st["quant"] = {"bytes": 2 * M * K + 2 * R * K + 4 * M}
    st["front_reorder"] = {"bytes": st["route_sort"]["bytes"] + st["quant"]["bytes"]}
    st["gmm1"] = {"bytes": active * 2 * I * K + active * 2 * I * 4 + R * K * 2 + R * 2 * I * 2,
                  "ops": 2 * R * K * 2 * I}
    st["swiglu"] = {"bytes": R * 2 * I * 2 + R * I * 2 + 8 * R}
    st["gmm2"] = {"bytes": active * K * I + active * K * 4 + R * I * 2 + R * K * 2,
                  "ops": 2 * R * I * K}
    # GMM1 with SwiGLU fused in (every expert on the tcgen05 pairs): both stages' bytes
    st["gmm1_swiglu"] = {"bytes": st["gmm1"]["bytes"] + st["swiglu"]["bytes"], "ops": st["gmm1"]["ops"]}
    st["combine"] = {"bytes": R * K * 2 + 12 * R + M * K * 2}
    return st, active


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.lines = []
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        # the busiest half of the samples (the sampler also sees the idle edges)
        top = sorted(sm)[len(sm) // 2:]
        return {"sm_mhz": statistics.median(top), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- reference arm
REFERENCE_BUDGET_S = 150.0


def run_reference(args, rank, world):
    """The CPU oracle, as it stands, on the host cores: each step evaluates a
    bounded sample of the workload's tokens (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    w = synth.CONFIGS[args.workload]
    inp = synth.make_inputs(w)
    # first call pages in the weights; the second estimates the cost of one token
    oracle.layer_tokens(inp, np.arange(min(w.M, 2), dtype=np.int32))
    t0 = time.perf_counter()
    oracle.layer_tokens(inp, np.arange(min(w.M, 2), dtype=np.int32))
    t_tok = (time.perf_counter() - t0) / min(w.M, 2)
    # tokens per step: at most 16, and few enough that the warm-up and timed steps
    # together stay near REFERENCE_BUDGET_S of host time for any --steps / --warmup
    n_tok = int(max(1, min(w.M, 16, REFERENCE_BUDGET_S / (max(1, args.steps + args.warmup) * t_tok))))
    toks = np.arange(n_tok, dtype=np.int32)
    cores = min(n_tok, oracle.max_threads())  # the per-token loop runs one token per thread
    for _ in range(args.warmup):
        oracle.layer_tokens(inp, toks)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.layer_tokens(inp, toks)
    dt = time.perf_counter() - t0
    value = n_tok * args.steps / dt
    sample = "%d of the %d tokens of the %s workload per step (per-token oracle evaluation)" % (
        n_tok, w.M, w.name)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic", "config": {"workload": workload_desc(w), "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(w, inp):
    """The oracle on the host cores over a bounded sample of the workload."""
    import oracle
    n_tok = min(w.M, 32)
    toks = np.arange(n_tok, dtype=np.int32)
    oracle.layer_tokens(inp, toks[:1])
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.layer_tokens(inp, toks)
        reps += 1
        if time.perf_counter() - t0 > 12.0:
            break
    dt = time.perf_counter() - t0
    return {"value": n_tok * reps / dt, "unit": UNIT, "cores": min(n_tok, oracle.max_threads()), "kind": "oracle",
            "sample": "%d x %d tokens of the %s workload (per-token oracle evaluation, %.1f s)" % (
                reps, n_tok, w.name, dt)}


# ----------------------------------------------------------------------------- ncu traffic record
def engine_source(w):
    """Source file of the GEMM engine the library picks for this workload."""
    name = "gemm_hmma.cu" if w.R / w.E <= 24.0 else "gemm_tc.cu"
    return os.path.join(ROOT, "moe_expert_layer_gb300", "csrc", name)


def traffic_record(stage, workload, kernel_file):
    """dram bytes per launch of the dominant kernel from the committed ncu summary
    (profiles/<stage>_<workload>_ncu.md), valid only while the kernel source is
    unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "%s_%s_ncu.md" % (stage, workload))
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m1 = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    m2 = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not (m1 and m2):
        return None
    src = open(kernel_file, "rb").read()
    if hashlib.sha256(src).hexdigest() != m2.group(1):
        return None
    return int(m1.group(1))


# ----------------------------------------------------------------------------- replicas (N > 1)
def replica_inputs(w, rank):
    """The inputs rank `rank` runs: every rank the same weights and scales, its own
    token batch and routing (rank 0 the workload's own seed, rank r seed + 1000 r)."""
    inp = synth.make_inputs(w)
    if rank:
        r = synth.Workload(w.name, w.M, w.K, w.I, w.E, w.topK, w.routing, w.seed + 1000 * rank)
        inp.update(synth.make_inputs(r, with_weights=False))
    return inp


def max_over_ranks(v, world, device):
    """The largest of the ranks' values (every rank gets it); `device` is where the
    process group's backend reduces (cuda for NCCL, cpu for gloo)."""
    if world <= 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, M, ms):
    """Whole-job throughput: every rank's M tokens over the slowest rank's step time."""
    return world * M / (ms * 1e-3)


# ----------------------------------------------------------------------------- GPU arm
class Gpu:
    """What every workload measurement shares: the modules, the launching stream, the
    L2 flush buffer, the process group."""

    def __init__(self, world, rank, local_rank):
        import torch
        import torch.distributed as dist
        import moe_expert_layer_gb300 as moe
        self.torch, self.dist, self.moe = torch, dist, moe
        self.world, self.rank, self.local_rank = world, rank, local_rank
        torch.cuda.set_device(local_rank)
        if world > 1:
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        self.stream = torch.cuda.Stream()  # a capturable stream (not the legacy default stream)
        self.flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")  # > L2 (126 MB)

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()
        self.torch.cuda.synchronize()


def step_stats(step_ms):
    return {"mean": statistics.mean(step_ms), "median": statistics.median(step_ms), "min": min(step_ms)}


def fused_swiglu(w):
    """Whether the layer runs SwiGLU inside the GMM1 kernel for this workload: the
    tcgen05 pairs run (more than 24 routes per expert on average)."""
    return w.R / w.E > 24.0


def roofline_of(w, stage_ms, alg, peaks):
    """The dominant GEMM stage against its bound: HBM when its bytes take longer at the
    measured copy rate than its MACs at the measured dense 16-bit tensor rate, tensor
    otherwise.  Both engines multiply the int8 codes as binary16 (kind::f16 / HMMA
    f16), whose dense rate equals the bf16 rate the peak was measured with."""
    dom = max([n for n in stage_ms if "ops" in alg[n]], key=lambda n: stage_ms[n])
    src = engine_source(w)
    mean_rows = w.R / w.E
    kernel = ("grouped_gemm_kernel" if mean_rows <= 24.0 else
              "grouped_gemm_pair_kernel" if mean_rows >= 256.0 else
              "grouped_gemm_kernel (experts <= 32 rows) + grouped_gemm_pair_kernel (the rest)")
    t_dom = stage_ms[dom] * 1e-3
    t_hbm = alg[dom]["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg[dom]["ops"] / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        ach = alg[dom]["bytes"] / t_dom / 1e9
        r = {"kernel": "%s (%s)" % (kernel, dom.upper()), "bound": "hbm", "achieved": round(ach, 1),
             "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 3),
             "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, a copy's read + write rate)",
             "algorithmic_bytes_per_launch": alg[dom]["bytes"]}
    else:
        ach = alg[dom]["ops"] / t_dom / 1e12
        r = {"kernel": "%s (%s)" % (kernel, dom.upper()), "bound": "tensor", "achieved": round(ach, 1),
             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 3),
             "peak_source": peaks["source"] + " (MEASURED_PEAKS.json bf16_tflops, burst; the int8 "
                            "codes run on the binary16 tensor path at the same rate)",
             "algorithmic_ops_per_launch": alg[dom]["ops"]}
    r["us_per_launch"] = round(stage_ms[dom] * 1e3, 2)
    r["traffic"] = traffic_record(dom, w.name, src)
    if r["frac"] > 1.0:
        # the denominators are a plain copy and cuBLAS: a kernel that streams reads
        # (no writes) or packed tiles can pass them; far above 1 would mean missing work
        r["above_peak"] = True
    return r


def launches_per_step(w):
    """Our kernels per layer call: the sort (fused into the quant kernel up to 4096
    routes, one kernel up to 8192, two above), the quant, each GEMM (one engine up
    to 24 rows per expert on average and from 256 on; between, the warp-MMA engine on
    16-row and on 32-row tiles, then the tcgen05 pairs), SwiGLU (inside GMM1 when
    fused_swiglu), combine."""
    sort_launches = 0 if w.R <= 4096 else (1 if w.R <= 8192 else 2)
    gemm_launches = 1 if (w.R / w.E <= 24.0 or w.R / w.E >= 256.0) else 3
    return sort_launches + 1 + 2 * gemm_launches + (0 if fused_swiglu(w) else 1) + 1


def measure_workload(g, w, args, headline, keep_host=False):
    """One workload: the layer step timed over args.steps steps (L2 flushed before
    each), the stages timed apart through the stage entry points, and, for the
    headline workload, the end-to-end host-buffer path.  Returns the report and the
    host inputs (with the weights only if keep_host)."""
    torch, moe, stream = g.torch, g.moe, g.stream
    inp = replica_inputs(w, g.rank)  # each rank its own batch, the same weights
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in inp.items()}
    host_inp = inp if keep_host else {k: inp[k] for k in ("x", "expert_idx", "probs")}
    del inp
    layout = moe.WEIGHTS_TILES if args.weights == "tiles" else moe.WEIGHTS_ROWS
    d = moe.dims(w.M, w.K, w.I, w.E, w.topK, layout)
    if layout == moe.WEIGHTS_TILES:
        # once, at weight-load time (outside every timed region): the row-layout
        # weights rewritten as tiles, which the layer then reads instead
        for gi, k in ((1, "w1"), (2, "w2")):
            t = torch.empty(moe.moe_weight_tiles_bytes(d, gi), dtype=torch.int8, device="cuda")
            moe.moe_pack_weight_tiles(d, gi, dev[k], t)
            dev[k] = t
        torch.cuda.synchronize()
    ws = torch.empty(moe.moe_layer_workspace_size(d), dtype=torch.uint8, device="cuda")
    out = torch.empty((w.M, w.K), dtype=torch.float16, device="cuda")
    graph = None
    if not args.no_graph:  # the layer's launches recorded once, replayed every step
        graph = moe.moe_layer_graph_create(d, dev["x"], dev["expert_idx"], dev["probs"], dev["w1"], dev["s1"],
                                           dev["w2"], dev["s2"], out, ws, stream)

    def step():
        if graph is not None:
            moe.moe_layer_graph_launch(graph, stream)
        else:
            moe.moe_layer_fwd(d, dev["x"], dev["expert_idx"], dev["probs"], dev["w1"], dev["s1"],
                              dev["w2"], dev["s2"], out, ws, stream)

    for _ in range(max(3, args.warmup)):
        step()
    g.barrier()
    if moe.moe_workspace_status(ws) != 0:
        raise RuntimeError("device status after warm-up: %d" % moe.moe_workspace_status(ws))

    # ---- timed region: K layer steps, L2 flushed before each, CUDA events on the stream
    clocks = ClockSampler(g.local_rank)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    g.barrier()
    t_wall = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            g.flush.fill_(i & 0xff)
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
    g.barrier()
    t_wall = time.perf_counter() - t_wall
    clocks.stop()
    if graph is not None:
        moe.moe_layer_graph_destroy(graph)
    st = step_stats([a.elapsed_time(b) for a, b in ev])
    ms = max_over_ranks(st["mean"], g.world, "cuda")
    st = {k: max_over_ranks(v, g.world, "cuda") for k, v in st.items()}

    # ---- per-stage timing through the stage entry points (same kernels), for the roofline
    R = w.R
    i32, f16, f32 = torch.int32, torch.float16, torch.float32
    sorted_, expanded = torch.empty(R, dtype=i32, device="cuda"), torch.empty(R, dtype=i32, device="cuda")
    tpe, cs = torch.empty(w.E, dtype=i32, device="cuda"), torch.empty(w.E, dtype=i32, device="cuda")
    sws = torch.empty(max(16, moe.moe_route_sort_workspace_size(d)), dtype=torch.uint8, device="cuda")
    a1, pts1 = torch.empty((R, w.K), dtype=f16, device="cuda"), torch.empty(w.M, dtype=f32, device="cuda")
    c1 = torch.empty((R, 2 * w.I), dtype=f16, device="cuda")
    q2, pts2 = torch.empty((R, w.I), dtype=f16, device="cuda"), torch.empty(R, dtype=f32, device="cuda")
    c2 = torch.empty((R, w.K), dtype=f16, device="cuda")
    gws = torch.empty(moe.moe_gmm_workspace_size(d), dtype=torch.uint8, device="cuda")
    bounds = torch.zeros((2, w.E, moe.BOUND_SEGMENTS), dtype=i32, device="cuda")  # activation bounds of a1, q2
    # the layer computes them only where its GEMM engine reads them (above 24 rows per expert)
    b1, b2 = (bounds[0], bounds[1]) if w.R / w.E > 24.0 else (None, None)
    fused_front = w.R <= 4096  # the layer's FrontReorder is one kernel
    fused_sw = fused_swiglu(w)  # the layer's GMM1 runs SwiGLU too
    names = ((["front_reorder"] if fused_front else ["route_sort", "quant"]) +
             (["gmm1_swiglu"] if fused_sw else ["gmm1", "swiglu"]) + ["gmm2", "combine"])
    nev = len(names) + 1

    def stages(evs):
        with torch.cuda.stream(stream):
            bounds.zero_()  # the layer clears them with its status word
        it = iter(evs)
        next(it).record(stream)
        if fused_front:
            moe.moe_front_reorder(d, dev["x"], dev["expert_idx"], sorted_, expanded, tpe, cs, a1, pts1, b1, sws,
                                  stream)
        else:  # what moe_front_reorder launches above 4096 routes, timed apart
            moe.moe_route_sort(d, dev["expert_idx"], sorted_, expanded, tpe, cs, sws, stream)
            next(it).record(stream)
            moe.moe_quant_dispatch(d, dev["x"], dev["expert_idx"], expanded, a1, pts1, b1, stream)
        next(it).record(stream)
        if fused_sw:
            moe.moe_gmm1_swiglu(d, a1, cs, b1, dev["w1"], dev["s1"], c1, pts1, sorted_, dev["expert_idx"], q2, pts2,
                                b2, gws, stream)
        else:
            moe.moe_gmm1(d, a1, None, cs, b1, dev["w1"], dev["s1"], c1, gws, stream)
            next(it).record(stream)
            moe.moe_swiglu_quant(d, c1, pts1, sorted_, cs, dev["expert_idx"], None, q2, pts2, b2, stream)
        next(it).record(stream)
        moe.moe_gmm2(d, q2, cs, b2, dev["w2"], dev["s2"], c2, gws, stream)
        next(it).record(stream)
        moe.moe_combine_unpermute(d, c2, pts2, expanded, dev["probs"], out, stream)
        next(it).record(stream)

    for _ in range(3):
        stages([torch.cuda.Event(enable_timing=True) for _ in range(nev)])
    n_stage_steps = max(3, min(args.steps, 50))
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(n_stage_steps)]
    g.barrier()
    with torch.cuda.stream(stream):
        for i in range(n_stage_steps):
            g.flush.fill_(i & 0xff)
            stages(sev[i])
    g.barrier()
    stage_ms = {n: statistics.mean(s[j].elapsed_time(s[j + 1]) for s in sev) for j, n in enumerate(names)}

    alg, active = algorithmic(w, host_inp["expert_idx"])
    peaks = load_peaks()
    stage_report = {}
    for n in names:
        t = stage_ms[n] * 1e-3
        rep = {"us": round(stage_ms[n] * 1e3, 2), "GBps": round(alg[n]["bytes"] / t / 1e9, 1),
               "hbm_frac": round(alg[n]["bytes"] / t / 1e9 / peaks["hbm_gbs"], 3)}
        if "ops" in alg[n]:
            rep["TOPS"] = round(alg[n]["ops"] / t / 1e12, 2)
            rep["tensor_frac"] = round(alg[n]["ops"] / t / 1e12 / peaks["bf16_tflops"], 3)
        stage_report[n] = rep
    layer_ops = alg["gmm1"]["ops"] + alg["gmm2"]["ops"]
    rep = {
        "fused_gmm1_swiglu": fused_sw,
        "workload": workload_desc(w), "ms_per_step": round(ms, 4),
        "ms_per_step_median": round(st["median"], 4), "ms_per_step_min": round(st["min"], 4),
        "value": round(job_tokens_per_s(g.world, w.M, ms), 1), "unit": UNIT,
        "int8_TOPS": round(layer_ops / (ms * 1e-3) / 1e12, 2),
        "roofline": roofline_of(w, stage_ms, alg, peaks), "stages": stage_report,
        "gpu_launches_per_step": launches_per_step(w), "clocks": clocks.summary(),
        "wall_s_timed_region": round(t_wall, 3), "active_experts": active,
        "gemm_bytes": alg["gmm1"]["bytes"] + alg["gmm2"]["bytes"], "weight_bytes": active * 3 * w.K * w.I,
        "launch": ("CUDA graph of the layer's launches (moe_layer_graph_launch)" if not args.no_graph
                   else "stream launches (moe_layer_fwd)"),
    }

    # ---- end to end through the host-buffer entry point (headline workload)
    if headline and not args.no_e2e:
        hws = torch.empty(moe.moe_layer_host_workspace_size(d), dtype=torch.uint8, device="cuda")
        xh = torch.from_numpy(host_inp["x"]).pin_memory()
        eih = torch.from_numpy(host_inp["expert_idx"]).pin_memory()
        prh = torch.from_numpy(host_inp["probs"]).pin_memory()
        outh = torch.empty((w.M, w.K), dtype=torch.float16).pin_memory()
        hgraph = None
        if not args.no_graph:  # copies in, layer, copy out: recorded once
            hgraph = moe.moe_layer_graph_create_host(d, xh, eih, prh, dev["w1"], dev["s1"], dev["w2"], dev["s2"],
                                                     outh, hws, stream)

        def host_step():
            if hgraph is not None:
                moe.moe_layer_graph_launch(hgraph, stream)
                stream.synchronize()
            else:
                moe.moe_layer_fwd_host(d, xh, eih, prh, dev["w1"], dev["s1"], dev["w2"], dev["s2"], outh,
                                       hws, stream)

        for _ in range(3):
            host_step()
        n_e2e = max(3, min(args.steps, 100))
        tot = 0.0
        g.barrier()
        for i in range(n_e2e):
            g.flush.fill_(i & 0xff)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            host_step()  # synchronises the stream before returning
            tot += time.perf_counter() - t0
        g.barrier()
        serial_ms = 1e3 * tot / n_e2e
        if hgraph is not None:
            moe.moe_layer_graph_destroy(hgraph)
        del hws
        serial_ms = max_over_ranks(serial_ms, g.world, "cuda")

        # the serving loop's form: the pipelined executor overlaps each batch's copies
        # with its neighbours' layer (two staging slots); every step still copies its
        # inputs in and its result out inside the timed region
        depth = 2
        pws = torch.empty(moe.moe_layer_pipeline_workspace_size(d, depth), dtype=torch.uint8, device="cuda")
        pipe = moe.moe_layer_pipeline_create(d, dev["w1"], dev["s1"], dev["w2"], dev["s2"], pws, depth)
        outs = [outh] + [torch.empty_like(outh).pin_memory() for _ in range(depth - 1)]
        try:
            for i in range(3):
                moe.moe_layer_pipeline_wait(pipe, moe.moe_layer_pipeline_submit(pipe, xh, eih, prh, outs[i % depth]))
            g.barrier()
            t0 = time.perf_counter()
            for i in range(n_e2e):
                ticket = moe.moe_layer_pipeline_submit(pipe, xh, eih, prh, outs[i % depth])
            moe.moe_layer_pipeline_wait(pipe, ticket)
            tot = time.perf_counter() - t0
            g.barrier()
        finally:
            moe.moe_layer_pipeline_destroy(pipe)
        e_ms = max_over_ranks(1e3 * tot / n_e2e, g.world, "cuda")
        rep["e2e"] = {"value": job_tokens_per_s(g.world, w.M, e_ms), "unit": UNIT,
                      "h2d_bytes_per_step": int(host_inp["x"].nbytes + host_inp["expert_idx"].nbytes
                                                + host_inp["probs"].nbytes),
                      "d2h_bytes_per_step": int(w.M * w.K * 2), "ms_per_step": round(e_ms, 4), "steps": n_e2e,
                      "path": ("moe_layer_pipeline_submit for each of the steps (pinned host buffers; %d staging "
                               "slots: the copies of one batch overlap the layer of its neighbours), then "
                               "moe_layer_pipeline_wait on the last; host wall clock" % depth),
                      "l2": "no flush between pipelined steps: each step streams its weights and activations "
                            "(%.2f GB) through HBM, far more than the 126 MB L2" % (
                                (alg["gmm1"]["bytes"] + alg["gmm2"]["bytes"]) / 1e9),
                      "serial": {"value": job_tokens_per_s(g.world, w.M, serial_ms), "ms_per_step": round(serial_ms, 4),
                                 "path": ("moe_layer_graph_create_host + moe_layer_graph_launch, then a stream "
                                          "synchronise, L2 flushed before each step" if not args.no_graph
                                          else "moe_layer_fwd_host, L2 flushed before each step")}}
    return rep, host_inp


def single_thread_oracle(inputs):
    """The oracle on ONE host thread over a few tokens of each workload given
    ({name: its host inputs}), next to the all-cores figure of cpu_baseline."""
    import oracle
    res = {}
    prev = oracle.max_threads()
    oracle.set_threads(1)
    try:
        for name, inp in inputs.items():
            w = synth.CONFIGS[name]
            oracle.layer_tokens(inp, np.arange(1, dtype=np.int32))  # page in
            n_tok = min(w.M, 4)
            toks = np.arange(n_tok, dtype=np.int32)
            t0 = time.perf_counter()
            reps = 0
            while True:
                oracle.layer_tokens(inp, toks)
                reps += 1
                if time.perf_counter() - t0 > 3.0:
                    break
            dt = time.perf_counter() - t0
            res[name] = {"value": n_tok * reps / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "%d x %d tokens of the %s workload (per-token oracle evaluation, %.1f s)"
                                   % (reps, n_tok, name, dt)}
    finally:
        oracle.set_threads(prev)
    return res


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    g = Gpu(world, rank, local_rank)
    w = synth.CONFIGS[args.workload]
    head, host_inp = measure_workload(g, w, args, headline=True)
    g.torch.cuda.empty_cache()

    # the other configurations, measured in the same run (one GPU only: under
    # torchrun every rank would repeat them)
    others, kept = {}, {}
    extra = [n for n in args.also.split(",") if n and n != "none" and n != w.name] if world == 1 else []
    one_thread = [] if args.no_cpu_baseline or world > 1 else ["tiny", "decode"]
    for name in extra:
        rep, hinp = measure_workload(g, synth.CONFIGS[name], args, headline=False, keep_host=name in one_thread)
        rep.pop("launch", None)
        others[name] = rep
        if name in one_thread:
            kept[name] = hinp
        del hinp
        g.torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            g.dist.barrier()
            g.dist.destroy_process_group()
        return

    cpu = cpu1 = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(w, synth.make_inputs(w))
        for name in one_thread:
            if name not in kept:
                kept[name] = synth.make_inputs(name)
        cpu1 = single_thread_oracle(kept)

    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "ms_per_step_median": head["ms_per_step_median"], "ms_per_step_min": head["ms_per_step_min"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic",
        "config": {"workload": head["workload"], "parallelism": "replicas" if world > 1 else "single GPU",
                   "launch": head["launch"],
                   "weights": ("16 KiB tiles (MOE_WEIGHTS_TILES), packed once before timing" if args.weights == "tiles"
                               else "[E][N][D] rows (MOE_WEIGHTS_ROWS)"),
                   "l2": "flushed before every timed step (512 MB write); the GEMMs move %.2f GB per "
                         "step, %.2f GB of them int8 weights"
                         % (head["gemm_bytes"] / 1e9, head["weight_bytes"] / 1e9),
                   "active_experts": head["active_experts"]},
        "int8_TOPS": head["int8_TOPS"],
        "roofline": head["roofline"],
        "stages": head["stages"],
        "cpu_baseline": cpu,
        "cpu_baseline_1thread": cpu1,
        "e2e": head.get("e2e"),
        "gpu_launches": head["gpu_launches_per_step"] * args.steps,
        "clocks": head["clocks"],
        "wall_s_timed_region": head["wall_s_timed_region"],
        "workloads": others,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        g.dist.barrier()
        g.dist.destroy_process_group()


if __name__ == "__main__":
    main()
