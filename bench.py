"""Benchmark: one hybrid optimizer step (Muon on every view-split matrix of
the 1.23B-parameter OMN-shaped set + global-norm clip + AdamW on the
262M-parameter embedding and gains), timed on the GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  ``value`` is optimizer steps per second over all
ranks (each rank runs a full replica: the step has no cross-device exchange
on one node here), inputs resident in HBM.  ``e2e`` is the same metric
with each step's gradients copied in from pinned host memory and the step's
gradient norm read back.  ``--impl reference`` times the fp64 CPU oracle on
a bounded sample of the same workload.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "optimizer steps/sec (1.24B-param Muon set); NS TFLOP/s and % BF16 peak"
WORKLOAD = 3


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="keep only the first N layers of the workload (small cases for ncu captures)")
    ap.add_argument("--precision", default="bf16", choices=["bf16", "f32"],
                    help="Newton-Schulz operands: bf16 (the benchmark) or the fp32 mode (three TF32 products)")
    ap.add_argument("--overlap", action="store_true",
                    help="run clip + AdamW on a side stream that starts after the momentum phase")
    ap.add_argument("--separate-gram", action="store_true",
                    help="A/B: run the Gram of the on-chip chain's matrices (p <= 128) as a tile-kernel "
                         "launch of its own instead of inside the chain launch (workload 4)")
    ap.add_argument("--fused-momentum", action="store_true",
                    help="A/B: run the momentum pass of the chain's wide p <= 128 matrices inside the chain launch "
                         "instead of in the momentum kernel (workload 4; measured slower)")
    ap.add_argument("--pdl", choices=["graph", "always", "never"], default="graph",
                    help="A/B: when launches carry the programmatic-dependent-launch attribute (the library's "
                         "default: in CUDA graph capture only)")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch the timed steps directly instead of replaying one step (Muon, clip, AdamW "
                         "with the step count on the device) captured in a CUDA graph")
    ap.add_argument("--e2e-buffers", type=int, default=3,
                    help="gradient buffer sets of the end-to-end run (each with its plan): uploads run up to "
                         "this many steps minus one ahead of the step that uses them")
    ap.add_argument("--e2e-copy", choices=["kernel", "engine"], default="engine",
                    help="e2e uploads by the copy engine, or by the library's copy kernel (gbo_h2d_copy) on "
                         "--e2e-copy-sms SMs the plans leave free")
    ap.add_argument("--e2e-copy-sms", type=int, default=4,
                    help="SMs of the e2e copy kernel, left free of the Newton-Schulz kernels during e2e steps")
    ap.add_argument("--no-tail-split", action="store_true",
                    help="A/B: run a CTA-pair launch's last partial wave as whole 256 x 256 tiles instead of "
                         "256 x 128 halves")
    ap.add_argument("--no-momentum-stream", action="store_true",
                    help="A/B: run the momentum pass as the register kernel (several blocks per SM) instead of "
                         "streaming its tiles through shared memory by bulk copies")
    ap.add_argument("--workspace-cap-frac", type=float, default=0.0,
                    help="cap the Muon workspace at this fraction of what the whole table needs (0: no cap); "
                         "the step then runs in groups of weights on the smaller workspace")
    ap.add_argument("--extra", default="2,4,5",
                    help="after the headline run, time these other workloads in the same process "
                         "(comma-separated indices, or 'none'); reported under extra_workloads")
    ap.add_argument("--workload", type=int, default=WORKLOAD,
                    help="synthetic set: 3 = the 1.23B OMN-shaped set (the benchmark); 2 = one "
                         "d=2048 layer, 4 = many small MLA/KDA matrices, 5 = 7B NorMuon (profiling)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world):
    """Largest value over all ranks (identity on one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(steps, seconds_max, world):
    """Whole-job steps/s: every rank ran ``steps`` steps of a full replica."""
    return world * steps / seconds_max


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    """nvidia-smi samples (100 ms) kept only inside [t0, t1] of the host clock."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        import datetime
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if t0 <= ts <= t1:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in the timed region"]}
        num = lambda x: float(x) if x.replace(".", "", 1).isdigit() else None  # noqa: E731
        sm = sorted(v for v in (num(r[1]) for r in rows) if v is not None)
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# the fp64 oracle on a bounded sample (CPU baseline and the reference arm)

def oracle_sample_time(wl, budget_elems=4_000_000):
    """Time the oracle on one matrix of every distinct oriented shape plus
    AdamW on ``budget_elems`` elements (all of them with ``budget_elems=None``,
    in slices of 16M), and extrapolate to the whole step.  Returns (seconds
    per full step, description)."""
    import numpy as np
    import torch

    import oracle
    from adamw_optimizer_step_gb300 import workloads as wk
    from oracle.views import sub_matrices

    counts = {}
    first = {}
    for i, t in enumerate(wl.muon):
        for r0, m, n in sub_matrices(t.rows, t.cols, t.view, t.split):
            counts[(m, n)] = counts.get((m, n), 0) + 1
            first.setdefault((m, n), (i, r0))
    total = 0.0
    parts = []
    for (m, n), c in counts.items():
        i, r0 = first[(m, n)]
        t = wl.muon[i]
        W, G, Bm, _ = wk.muon_tensor_inputs(wl, i)
        W, G, Bm = (x[r0:r0 + m].double().numpy() for x in (W, G, Bm))
        t0 = time.perf_counter()
        oracle.muon_step_tensor(W, G, Bm, lr=wl.lr)
        dt = time.perf_counter() - t0
        total += c * dt
        parts.append("%dx%d x%d" % (m, n, c))
    n_adam = wl.adamw_params
    if n_adam:
        k = n_adam if budget_elems is None else min(budget_elems, n_adam)
        # the AdamW oracle is elementwise: a full pass runs slice by slice
        # (the clip norm over all slices first, as the step does)
        piece = min(k, 16 * 1024 * 1024)
        g = torch.Generator().manual_seed(7)
        p, gr, mm, vv = (torch.randn(piece, generator=g).double().numpy() for _ in range(4))
        vv = np.abs(vv)
        slices = [piece] * (k // piece) + ([k % piece] if k % piece else [])
        t0 = time.perf_counter()
        N = oracle.global_grad_norm([gr[:n] for n in slices])
        c = oracle.clip_coefficient(N, 1.0)
        for n in slices:
            oracle.adamw_update(p[:n], gr[:n], mm[:n], vv[:n], coef=c, lr=3e-4, t=1)
        dt = time.perf_counter() - t0
        total += dt * n_adam / k
        parts.append("AdamW %s %d of %d elements" % ("all" if k == n_adam else "sampled,", k, n_adam))
    return total, "one matrix per shape (%s), scaled by count; %s" % (", ".join(parts[:-1]), parts[-1])


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from adamw_optimizer_step_gb300 import workloads as wk
    wl = wk.workload(WORKLOAD)
    for _ in range(args.warmup):
        oracle_sample_time(wl, budget_elems=1_000_000)
    times = []
    desc = ""
    for _ in range(args.steps):
        t, desc = oracle_sample_time(wl)
        times.append(t)
    times.sort()
    per_step = times[len(times) // 2]
    value = 1.0 / per_step
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "ms_per_step_extrapolated": True,
        "ms_per_step_basis": "extrapolated, not wall time: each timed step runs the oracle on one matrix of "
                             "every shape and a 4M-element AdamW slice and scales each part by its count to "
                             "the full step (steps x ms_per_step is far above this run's wall time)",
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "description": wl.description, "muon_params": wl.muon_params,
                   "adamw_params": wl.adamw_params},
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------
# ours

# the sources of ns_gemm_tc_kernel, whose DRAM traffic profiles/traffic.json records
TC_KERNEL_SOURCES = ["ns_gemm_tc.cu", "tc_common.cuh"]


def traffic_record(kernel_files):
    """DRAM bytes per unit from the committed ncu summary, or None when the
    kernel's sources changed since the counters were taken (sha256 over the
    listed files, concatenated in order)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    if rec.get("source_files") != list(kernel_files):
        return None
    h = hashlib.sha256()
    for f in kernel_files:
        h.update(open(os.path.join(ROOT, "adamw_optimizer_step_gb300", "csrc", f), "rb").read())
    if rec.get("source_sha256") != h.hexdigest():
        return None
    return rec


def run_e2e(n_steps, world, bufs, step, total, after_momentum, copy_blocks=0):
    """Steps/s with each step's gradients copied in from pinned host memory
    and the step's gradient norm read back on the host.  ``bufs`` holds K
    (Muon, AdamW) flat gradient buffer sets, each bound to its own plan:
    uploads run on a copy stream, in step order, up to K - 1 steps ahead of
    the step that computes, as a trainer prefetches its inputs: the Muon
    gradients first, which a step needs at its start, then the AdamW
    gradients, which it needs only for its clip and AdamW after its GEMMs.
    The upload enqueued with step n starts once step n's momentum pass is
    done (``after_momentum[b]``, recorded by buffer set b's plan), so it
    runs under the Newton-Schulz GEMMs, which leave most of the HBM
    bandwidth free, rather than under the memory-bound momentum pass; with
    K > 2 a copy that stalls is absorbed by the lead the uploads have built
    up (each upload is shorter than a step).  Every step's
    copy and read stay inside the timed region.  Returns (steps/s over all
    ranks, bytes copied in per step, the upload's GB/s when it runs
    alone, each step's host wall time in ms up to its norm read).  A single
    step has been seen to stall for ~150 ms on a host whose previous process
    had just exited (the upload's wait, not the GPU's work): the per-step
    times show such a stall, and the default 40 steps bound its weight in
    the mean.  ``copy_blocks`` > 0: the uploads are made by the library's
    copy kernel on that many SMs, which the plans leave free (gbo_h2d_copy:
    SM loads of the page-locked host buffers); 0: by the copy engine
    (cudaMemcpyAsync through torch)."""
    import torch
    from adamw_optimizer_step_gb300 import _binding, hostmem
    g_flat, ag_flat = bufs[0]
    # page-locked host buffers on huge pages (hostmem: fewer and shorter
    # copy stalls than the driver's small-page pinned memory)
    h_g = hostmem.pinned_empty(g_flat.numel(), g_flat.dtype)
    h_ag = hostmem.pinned_empty(ag_flat.numel(), ag_flat.dtype)
    assert h_g.is_pinned() and h_ag.is_pinned()
    h_g.copy_(g_flat)
    h_ag.copy_(ag_flat)
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    nb = len(bufs)
    copied = [torch.cuda.Event() for _ in range(nb)]       # Muon gradients in
    copied_adam = [torch.cuda.Event() for _ in range(nb)]  # AdamW gradients in
    done = [torch.cuda.Event() for _ in range(nb)]

    def upload(b, after=None, timed=None):
        # the Muon gradients first: a step needs them at its start, its AdamW
        # gradients only after the Newton-Schulz GEMMs
        copy.wait_event(done[b])  # the step that last read buffer pair b has finished
        if after is not None:
            copy.wait_event(after)
        if timed is not None:  # the copies' own duration on the copy stream
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(copy)
        if copy_blocks:
            _binding.gbo_h2d_copy(bufs[b][0], h_g, blocks=copy_blocks, stream=copy)
            copied[b].record(copy)
            _binding.gbo_h2d_copy(bufs[b][1], h_ag, blocks=copy_blocks, stream=copy)
        else:
            with torch.cuda.stream(copy):
                bufs[b][0].copy_(h_g, non_blocking=True)
                copied[b].record(copy)
                bufs[b][1].copy_(h_ag, non_blocking=True)
        copied_adam[b].record(copy)
        if timed is not None:
            ev1.record(copy)
            timed.append((ev0, ev1))

    # the step's result comes back through a pinned buffer (no pageable copy)
    h_total = torch.empty(total.shape, dtype=total.dtype, pin_memory=True)
    read = torch.cuda.Event()

    def read_result():
        h_total.copy_(total, non_blocking=True)
        read.record(compute)
        read.synchronize()
        return float(h_total[0])

    # the upload alone (after one untimed copy), to tell a copy-bound host
    # from a compute-bound one: the host side of this path varies between hosts
    h2d = h_g.numel() * h_g.element_size() + h_ag.numel() * h_ag.element_size()
    upload(0)
    torch.cuda.synchronize()
    alone = []  # three uploads on their own (host wall time each)
    for _ in range(3):
        t_up = time.perf_counter()
        upload(0)
        torch.cuda.synchronize()
        alone.append(time.perf_counter() - t_up)
    up_gbs = h2d / statistics.median(alone) / 1e9

    def run(n_run, wall=None, timed=None, enqueue=None):
        # the uploads of steps 0 .. nb - 2 first; then, as step n is
        # enqueued, the upload of step n + nb - 1 into the buffer set step
        # n - 1 used (it starts once step n - 1 is done and step n's
        # momentum pass is, and after the uploads before it)
        for m in range(min(nb - 1, n_run)):
            upload(m, timed=timed)
        t_prev = time.perf_counter()
        for n in range(n_run):
            b = n % nb
            t_q = time.perf_counter()
            compute.wait_event(copied[b])
            step(buf=b, before_adamw=copied_adam[b])
            done[b].record(compute)
            if n + nb - 1 < n_run:
                upload((n + nb - 1) % nb, after_momentum[b], timed=timed)
            if enqueue is not None:
                enqueue.append((time.perf_counter() - t_q) * 1e3)
            _ = read_result()  # the step's result on the host
            if wall is not None:
                t_now = time.perf_counter()
                wall.append((t_now - t_prev) * 1e3)
                t_prev = t_now
        torch.cuda.synchronize()

    run(nb)  # untimed: each buffer set's plan runs once (its first step sets it up on the device)
    barrier(world)
    wall, timed, enqueue = [], [], []
    t0 = time.perf_counter()
    run(n_steps, wall, timed, enqueue)
    e2e_t = max_over_ranks(time.perf_counter() - t0, world)
    up_ms = [a.elapsed_time(b) for a, b in timed]
    diag = {"upload_alone_ms": [x * 1e3 for x in alone],
            "upload_copy_ms": {"median": statistics.median(up_ms), "max": max(up_ms),
                               "over_2x_median": sum(u > 2 * statistics.median(up_ms) for u in up_ms),
                               "basis": "each upload's own duration on the copy stream (CUDA events after its "
                                        "waits)"},
            "enqueue_ms": {"median": statistics.median(enqueue), "max": max(enqueue),
                           "basis": "host time to enqueue a step and the next upload"}}
    return aggregate(n_steps, e2e_t, world), h2d, up_gbs, wall, diag


# nominal GB300 figures (NVIDIA's datasheet: dense bf16 without sparsity,
# HBM3e bandwidth), reported beside the measured denominators
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 7900.0


def load_peaks():
    """The measured roofline denominators (MEASURED_PEAKS.json), else the
    fallbacks, and where each came from."""
    measured = {}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        measured = json.load(open(path))
    burst = measured.get("bf16_tflops")
    sustained = measured.get("bf16_tflops_sustained")
    hbm = measured.get("hbm_gbs")
    src = "measured (MEASURED_PEAKS.json)"
    if burst is None or hbm is None:
        burst, sustained, hbm, src = 1900.0, 1700.0, 6800.0, "fallback"
    return {"burst": burst, "sustained": sustained or burst, "hbm": hbm, "source": src}


def step_floor(flops, floor_bytes, peaks):
    """(tensor ms, HBM ms): executed tensor FLOPs at the burst bf16 rate and
    the algorithmic bytes at the HBM copy rate; the floor is the larger."""
    tensor_ms = flops / (peaks["burst"] * 1e12) * 1e3
    hbm_ms = floor_bytes / (peaks["hbm"] * 1e9) * 1e3
    return tensor_ms, hbm_ms


def floor_bytes_of(wl, torch):
    """Per Muon parameter G read, B read and written, W read and written;
    32 B per AdamW parameter (the clip pass and the update)."""
    w_es = torch.empty(0, dtype=wl.w_dtype).element_size()
    g_es = torch.empty(0, dtype=wl.g_dtype).element_size()
    return (g_es + 8 + 2 * w_es) * wl.muon_params + 32.0 * wl.adamw_params


EXTRA_STEPS = {2: 200, 4: 30, 5: 5}  # about 0.2 to 1 s of timed work each


def run_extra_workload(index, peaks, local, warmup=3, use_graph=True):
    """Steps/s of another synthetic set, timed like the headline run (CUDA
    events on the launching stream, inputs resident in HBM, clocks sampled
    during the timed region).  The step is Muon on every matrix, plus clip +
    AdamW when the set has AdamW parameters."""
    import torch
    import adamw_optimizer_step_gb300 as gbo
    from adamw_optimizer_step_gb300 import workloads as wk

    wl = wk.workload(index)
    dev = "cuda"
    entries = []
    for i, t in enumerate(wl.muon):
        W, G, Bm, v = wk.muon_tensor_inputs(wl, i, device=dev)
        entries.append(dict(w=W, g=G, mom=Bm, row_v=v, view=t.view, split=t.split))
    params = [wk.adamw_tensor_inputs(wl, i, device=dev) for i in range(len(wl.adamw))]
    plan = gbo.gbo_muon_plan_create(entries, normuon=wl.normuon)
    info = gbo.gbo_muon_plan_info(plan)
    ws = torch.empty(gbo.gbo_muon_workspace_bytes(plan), dtype=torch.uint8, device=dev)
    cws = torch.empty(gbo.gbo_clip_norm_workspace_bytes(), dtype=torch.uint8, device=dev)
    total = torch.zeros(1, device=dev)
    coef = torch.zeros(1, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    n = [0]

    def step():
        n[0] += 1
        gbo.gbo_muon_step(plan, wl.lr, ws, dev_status=status, stream=stream)
        if params:
            gbo.gbo_clip_norm([p[1] for p in params], 1.0, total, coef, cws, dev_status=status, stream=stream)
            gbo.gbo_adamw_step(params, lr=wl.adamw_lr, step=n[0], coef=coef, dev_status=status, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    steps = EXTRA_STEPS.get(index, 10)
    graph = None
    if use_graph:  # one step captured in a CUDA graph, the step count on the device
        dev_step = torch.full((1,), n[0], dtype=torch.int32, device=dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cs = torch.cuda.current_stream()
            gbo.gbo_muon_step(plan, wl.lr, ws, dev_status=status, stream=cs)
            if params:
                dev_step.add_(1)
                gbo.gbo_clip_norm([p[1] for p in params], 1.0, total, coef, cws, dev_status=status, stream=cs)
                gbo.gbo_adamw_step(params, lr=wl.adamw_lr, coef=coef, dev_status=status, stream=cs,
                                   dev_step=dev_step)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)  # let the sampler start
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    start, end = ev(), ev()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    l0 = gbo.gbo_launch_count()
    start.record(stream)  # the steps as a user runs them, without phase events
    for _ in range(steps):
        if graph is not None:
            graph.replay()
        else:
            step()
    end.record(stream)
    torch.cuda.synchronize()
    launches = gbo.gbo_launch_count() - l0
    clk = clocks.stop(t_wall0, time.time())
    if graph is not None:
        n[0] += steps + 2  # the replays advanced the device's step count
    # the phase times from a second run of as many steps, with the plan's
    # phase events
    gbo.gbo_muon_plan_set_timing(plan, True)
    gbo.gbo_muon_plan_phase_times(plan)  # reset
    lp0 = gbo.gbo_launch_count()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    phases = gbo.gbo_muon_plan_phase_times(plan)
    gbo.gbo_muon_plan_set_timing(plan, False)
    if graph is not None:  # the graph replays the kernels of one direct step
        launches = gbo.gbo_launch_count() - lp0
    if int(status.item()) != 0:
        raise RuntimeError("device status %d during workload %d" % (int(status.item()), index))
    ms = start.elapsed_time(end) / steps
    gemm_ms = sum(phases[k][0] for k in ("gram", "product", "square", "final")) / steps
    flops = info["ns_flops_executed"]
    tensor_ms, hbm_ms = step_floor(flops, floor_bytes_of(wl, torch), peaks)
    ns_tf = flops / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None
    return {
        "workload": wl.name, "description": wl.description, "muon_params": wl.muon_params,
        "adamw_params": wl.adamw_params, "matrices": info["n_matrices"], "normuon": wl.normuon,
        "steps": steps, "warmup": warmup, "value": 1e3 / ms, "unit": "steps/s", "ms_per_step": ms,
        "step_floor": {"ms": max(tensor_ms, hbm_ms), "frac": max(tensor_ms, hbm_ms) / ms, "tensor_ms": tensor_ms,
                       "hbm_ms": hbm_ms},
        "ns_tflops_executed": ns_tf,
        "ns_frac_of_burst": None if ns_tf is None else ns_tf / peaks["burst"],
        "phases_ms_per_step": {k: v[0] / steps for k, v in phases.items()},
        "gpu_launches_per_step": launches / steps,
        "clocks": clk,
    }


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import adamw_optimizer_step_gb300 as gbo
    from adamw_optimizer_step_gb300 import workloads as wk

    gbo.lib()
    if args.separate_gram:
        from adamw_optimizer_step_gb300 import _binding
        _binding.gbo_testing_set_fused_gram(False)
    if args.fused_momentum:
        from adamw_optimizer_step_gb300 import _binding
        _binding.gbo_testing_set_fused_momentum(True)
    if args.no_tail_split:
        from adamw_optimizer_step_gb300 import _binding
        _binding.gbo_testing_set_tail_split(False)
    if args.no_momentum_stream:
        from adamw_optimizer_step_gb300 import _binding
        _binding.gbo_testing_set_momentum_stream(False)
    if args.pdl != "graph":
        from adamw_optimizer_step_gb300 import _binding
        _binding.gbo_testing_set_pdl({"never": 0, "always": 1}[args.pdl])
    wl = wk.workload(args.workload)
    if args.layers:
        wl = wk.first_layers(wl, args.layers)
    dev = "cuda"
    # Muon gradients live in one flat buffer so the end-to-end run can copy
    # a step's gradients in with one transfer; likewise the AdamW gradients.
    n_muon = wl.muon_params
    g_flat = torch.empty(n_muon, dtype=wl.g_dtype, device=dev)
    entries = []
    off = 0
    for i, t in enumerate(wl.muon):
        W, G, Bm, v = wk.muon_tensor_inputs(wl, i, device=dev)
        g = g_flat[off:off + t.numel].view(t.rows, t.cols)
        g.copy_(G)
        del G
        off += t.numel
        entries.append(dict(w=W, g=g, mom=Bm, row_v=v, view=t.view, split=t.split))
    n_adam = wl.adamw_params
    ag_flat = torch.empty(n_adam, dtype=torch.float32, device=dev)
    params = []
    off = 0
    for i, t in enumerate(wl.adamw):
        p, g, m, v = wk.adamw_tensor_inputs(wl, i, device=dev)
        gv = ag_flat[off:off + t.numel].view(t.shape)
        gv.copy_(g)
        del g
        off += t.numel
        params.append((p, gv, m, v))
    f32 = args.precision == "f32"
    prec = gbo.GBO_NS_F32 if f32 else gbo.GBO_NS_BF16
    plan = gbo.gbo_muon_plan_create(entries, precision=prec, normuon=wl.normuon)
    ws_whole = gbo.gbo_muon_workspace_bytes(plan)
    cap = int(ws_whole * args.workspace_cap_frac) if args.workspace_cap_frac > 0 else 0
    if cap:
        plan = gbo.gbo_muon_plan_create(entries, precision=prec, normuon=wl.normuon, workspace_cap=cap)
    info = gbo.gbo_muon_plan_info(plan)
    ws = torch.empty(gbo.gbo_muon_workspace_bytes(plan), dtype=torch.uint8, device=dev)
    cws = torch.empty(gbo.gbo_clip_norm_workspace_bytes(), dtype=torch.uint8, device=dev)
    total = torch.zeros(1, device=dev)
    coef = torch.zeros(1, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # plans and AdamW tables bound to gradient buffer pairs (the end-to-end
    # run adds a second pair)
    bound = [(plan, params, [p[1] for p in params])]
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    step_no = [0]
    overlap = args.overlap

    # recorded by each buffer pair's plan right after its momentum pass
    after_momentum = [torch.cuda.Event()]
    gbo.gbo_muon_plan_set_event(plan, 0, after_momentum[0])

    def step(record=None, buf=0, before_adamw=None):
        """One optimizer step: Muon, then clip + AdamW, on one stream.  With
        --overlap the AdamW path (independent of the Muon path) runs on a side
        stream that starts once the momentum kernel is done, overlapping the
        Newton-Schulz GEMMs; the main stream joins it before the step ends.
        Measured on GB300 the overlap saves nothing: the memory-bound AdamW
        slows the concurrent Gram products by about as much as it hides."""
        step_no[0] += 1
        plan_b, params_b, adam_grads = bound[buf]
        if overlap:
            side.wait_stream(stream)
        gbo.gbo_muon_step(plan_b, wl.lr, ws, dev_status=status, stream=stream)
        adam_stream = side if overlap else stream
        if overlap:
            side.wait_event(after_momentum[buf])
        if before_adamw is not None:  # this step's AdamW gradients have landed
            adam_stream.wait_event(before_adamw)
        if record is not None:
            record[0].record(adam_stream)
        gbo.gbo_clip_norm(adam_grads, 1.0, total, coef, cws, dev_status=status, stream=adam_stream)
        gbo.gbo_adamw_step(params_b, lr=wl.adamw_lr, step=step_no[0], coef=coef, dev_status=status,
                           stream=adam_stream)
        if record is not None:
            record[1].record(adam_stream)
        if overlap:
            stream.wait_stream(side)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # --graph: the step (Muon, clip, AdamW with the step count on the device)
    # captured once in a CUDA graph and replayed
    graph = None
    if args.graph and not overlap:
        dev_step = torch.full((1,), step_no[0], dtype=torch.int32, device=dev)
        plan0, params0, adam_grads0 = bound[0]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cs = torch.cuda.current_stream()
            dev_step.add_(1)
            gbo.gbo_muon_step(plan0, wl.lr, ws, dev_status=status, stream=cs)
            gbo.gbo_clip_norm(adam_grads0, 1.0, total, coef, cws, dev_status=status, stream=cs)
            gbo.gbo_adamw_step(params0, lr=wl.adamw_lr, coef=coef, dev_status=status, stream=cs, dev_step=dev_step)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()

    # timed region: inputs resident in HBM (the working set is ~20 GB, far
    # above the 129 MB L2, so every step streams from HBM).  The step runs
    # as a user runs it, without the plan's phase events: recording events
    # between launches costs a few us each (~50 us a step on the one-layer
    # set), so the phase times come from a second run of as many steps
    # right after it.
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)  # let the sampler start
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    l0 = gbo.gbo_launch_count()
    start, end = ev(), ev()
    marks = [ev() for _ in range(args.steps)]  # after each step: per-step times
    start.record(stream)
    for k in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step()
        marks[k].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = gbo.gbo_launch_count() - l0  # a graph's replays launch without the library counting them
    if graph is not None:
        step_no[0] += args.steps + 2  # the replays advanced the device's step count
    clk = clocks.stop(t_wall0, time.time())
    # the phase run: the same steps with the plan's phase events and the
    # AdamW path bracketed by events
    gbo.gbo_muon_plan_set_timing(plan, True)
    gbo.gbo_muon_plan_phase_times(plan)  # reset
    adam_ev = [(ev(), ev()) for _ in range(args.steps)]
    p_start, p_end = ev(), ev()
    lp0 = gbo.gbo_launch_count()
    p_start.record(stream)
    for k in range(args.steps):
        step(adam_ev[k])
    p_end.record(stream)
    torch.cuda.synchronize()
    if graph is not None:  # the graph replays the kernels of one direct step
        launches = gbo.gbo_launch_count() - lp0
    phases = gbo.gbo_muon_plan_phase_times(plan)
    gbo.gbo_muon_plan_set_timing(plan, False)
    phase_run_ms = p_start.elapsed_time(p_end) / args.steps
    elapsed = start.elapsed_time(end) / 1e3
    step_ms = sorted((marks[k - 1] if k else start).elapsed_time(marks[k]) for k in range(args.steps))
    elapsed_max = max_over_ranks(elapsed, world)
    adam_ms = sum(a.elapsed_time(b) for a, b in adam_ev) / args.steps
    value = aggregate(args.steps, elapsed_max, world)
    if int(status.item()) != 0:
        raise RuntimeError("device status %d during the timed steps" % int(status.item()))

    # end to end: gradients from pinned host memory, norm read back
    e2e_value, h2d, up_gbs, e2e_wall, e2e_diag = None, 0, None, [], {}
    if args.e2e_steps > 0:
        bufs = [(g_flat, ag_flat)]
        plans = [plan]
        for _ in range(1, args.e2e_buffers):  # one more gradient buffer set, and its plan, each
            g_flat2, ag_flat2 = torch.empty_like(g_flat), torch.empty_like(ag_flat)
            entries2, off = [], 0
            for e in entries:
                n = e["w"].numel()
                entries2.append(dict(e, g=g_flat2[off:off + n].view(e["w"].shape)))
                off += n
            params2, off = [], 0
            for p, g, m, v in params:
                params2.append((p, ag_flat2[off:off + g.numel()].view(g.shape), m, v))
                off += g.numel()
            plan2 = gbo.gbo_muon_plan_create(entries2, precision=prec, normuon=wl.normuon, workspace_cap=cap)
            after_momentum.append(torch.cuda.Event())
            gbo.gbo_muon_plan_set_event(plan2, 0, after_momentum[len(bufs)])
            bound.append((plan2, params2, [p[1] for p in params2]))
            bufs.append((g_flat2, ag_flat2))
            plans.append(plan2)
        if args.e2e_copy == "kernel":  # the copy kernel's SMs stay free of the GEMMs
            for pl in plans:
                gbo.gbo_muon_plan_set_free_sms(pl, args.e2e_copy_sms)
        e2e_value, h2d, up_gbs, e2e_wall, e2e_diag = run_e2e(
            args.e2e_steps, world, bufs, step, total, after_momentum,
            copy_blocks=args.e2e_copy_sms if args.e2e_copy == "kernel" else 0)

    if rank != 0:
        return
    ms_step = elapsed_max * 1e3 / args.steps
    gram_ms, gram_n = phases["gram"]
    prod_ms, prod_n = phases["product"]
    sq_ms, sq_n = phases["square"]
    fin_ms, fin_n = phases["final"]
    gemm_ms = (gram_ms + prod_ms + sq_ms + fin_ms) / args.steps
    gemm_launches = (gram_n + prod_n + sq_n + fin_n) / args.steps
    # executed tensor FLOPs: the tile products, three TF32 passes each in the fp32 mode
    flops = info["ns_flops_executed"] * (3 if f32 else 1)
    achieved_tf = flops / (gemm_ms / 1e3) / 1e12
    counted_tf = info["ns_flops"] / (gemm_ms / 1e3) / 1e12
    peaks = load_peaks()
    # the Newton-Schulz launches are timed back to back inside 20 ms steps:
    # the burst bf16 rate is the denominator (the sustained, seconds-long
    # figure and the nominal datasheet peak are reported beside it)
    peak_tf = peaks["burst"]
    peak_src = peaks["source"] + ", burst"
    scale = 1.0
    if f32:  # TF32 runs at the nominal 1.1 / 2.25 of the bf16 dense rate
        scale = 1.1 / 2.25
        peak_tf *= scale
        peak_src += " x nominal TF32/bf16 ratio 1.1/2.25"
    tr = traffic_record(TC_KERNEL_SOURCES) if not f32 else None
    traffic = None
    if tr is not None:
        traffic = tr["bytes_per_unit"] * (flops / gemm_launches) / tr["unit_flops"]
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        t_cpu, desc = oracle_sample_time(wl, budget_elems=None)
        cpu = {"value": 1.0 / t_cpu, "unit": "steps/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": desc, "extrapolated": "the Muon part (one matrix per shape x count); AdamW + clip "
                                               "timed over every element"}
    hbm = peaks["hbm"]
    adam_bytes = 32.0 * n_adam
    # The step's floor: the executed tensor FLOPs at the tensor peak, or the
    # algorithmic bytes at HBM bandwidth, whichever is longer (perfect overlap
    # of the two).  Bytes: per Muon parameter G read, B read and written, W
    # read and written; per AdamW parameter 32 B.
    floor_bytes = floor_bytes_of(wl, torch)
    floor_tensor_ms, floor_hbm_ms = step_floor(flops / scale, floor_bytes, peaks)
    out = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if f32 else "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "description": wl.description, "muon_params": wl.muon_params,
                   "adamw_params": n_adam, "matrices": info["n_matrices"], "ns_steps": wl.ns_steps,
                   "ns_precision": ("fp32 operands as three TF32 products, fp32 accumulate" if f32
                                    else "bf16 operands, fp32 accumulate"),
                   "parallelism": "replicas" if world > 1 else "single",
                   "chain_gram": "separate launch" if args.separate_gram else "on chip (p <= 128)",
                   "tail_split": not args.no_tail_split,
                   "momentum_stream": not args.no_momentum_stream,
                   "cuda_graph": graph is not None,
                   "pdl": args.pdl,
                   "workspace_bytes": int(ws.numel()), "workspace_cap": cap or None,
                   "workspace_whole_table_bytes": int(ws_whole),
                   "chain_momentum": ("in the chain launch (wide p <= 128, bf16 G)"
                                      if args.fused_momentum and not args.separate_gram else "momentum kernel"),
                   "device": torch.cuda.get_device_name(),
                   "seed": "one seeded draw per tensor and role (workloads.seed: workload, tensor index, role)",
                   "l2": "working set ~20 GB per GPU, far above the 129 MB L2: no flush needed"},
        "roofline": {"bound": "tensor",
                     "kernel": ("ns_gemm_tf32_kernel" if f32 else "ns_gemm_tc_kernel")
                               + " (all Newton-Schulz launches), executed FLOPs",
                     "achieved": achieved_tf, "peak": peak_tf, "unit": "TFLOP/s", "frac": achieved_tf / peak_tf,
                     "peak_source": peak_src, "traffic": traffic,
                     "frac_of_sustained": achieved_tf / (peaks["sustained"] * scale),
                     "frac_of_nominal": achieved_tf / (NOMINAL_BF16_TFLOPS * scale),
                     "nominal_source": "NVIDIA GB300 datasheet: 2.25 PFLOP/s dense bf16 (TF32 1.1)",
                     "flops_per_launch": flops / gemm_launches, "ms_per_launch": gemm_ms / gemm_launches,
                     "basis": ("CUDA events on the launching stream around each phase of the plan, over a second "
                               "run of as many steps right after the timed one (the timed steps run without "
                               "phase events)")},
        "phases_ms_per_step": {k: v[0] / args.steps for k, v in phases.items()},
        "phase_run_ms_per_step": phase_run_ms,
        "step_ms": {"median": step_ms[len(step_ms) // 2], "min": step_ms[0], "max": step_ms[-1]},
        "step_floor": {"ms": max(floor_tensor_ms, floor_hbm_ms), "frac": max(floor_tensor_ms, floor_hbm_ms) / ms_step,
                       "tensor_ms": floor_tensor_ms, "hbm_ms": floor_hbm_ms, "bytes_per_step": floor_bytes,
                       "basis": "max(executed NS FLOPs / tensor peak, (G + B + W Muon traffic + 32 B per AdamW "
                                "parameter) / HBM copy bandwidth)"},
        "adamw_clip": {"ms": adam_ms, "GB/s": adam_bytes / (adam_ms / 1e3) / 1e9,
                       "frac_of_hbm": adam_bytes / (adam_ms / 1e3) / 1e9 / hbm,
                       "frac_of_nominal_hbm": adam_bytes / (adam_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                       "stream": "side stream, overlapped with the Muon GEMMs" if overlap else "main stream"},
        "ns_tflops": {"executed": achieved_tf, "counted_dense": counted_tf,
                      "executed_tflop_per_step": flops / 1e12, "counted_tflop_per_step": info["ns_flops"] / 1e12},
        "e2e": None if e2e_value is None else {"value": e2e_value, "unit": "steps/s",
                                               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 4,
                                               "overlap": ("gradient uploads run up to %d steps ahead of the "
                                                           "step that uses them (%d gradient buffer sets)"
                                                           % (args.e2e_buffers - 1, args.e2e_buffers)),
                                               "host_buffers": "page-locked, huge-page backed (hostmem)",
                                               "upload": ("copy kernel on %d SMs the plans leave free "
                                                          "(gbo_h2d_copy: SM loads over the C2C link)"
                                                          % args.e2e_copy_sms if args.e2e_copy == "kernel"
                                                          else "copy engine (cudaMemcpyAsync)"),
                                               "upload_GBps_alone": up_gbs,
                                               "upload_ms_alone": None if not up_gbs else h2d / up_gbs / 1e6,
                                               "steps": len(e2e_wall),
                                               "step_ms": {"median": statistics.median(e2e_wall),
                                                           "max": max(e2e_wall),
                                                           "over_2x_median": sum(
                                                               w > 2 * statistics.median(e2e_wall)
                                                               for w in e2e_wall),
                                                           "basis": "host wall time per step, up to its norm read; "
                                                                    "the first includes the first upload"},
                                               **e2e_diag},
        "gpu_launches": int(launches),
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    return out


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args)
    else:
        out = run_ours(args)
        if out is not None:
            extra = [] if args.extra in ("", "none") else [int(x) for x in args.extra.split(",")]
            extra = [x for x in extra if x != args.workload and not args.layers]
            if extra and world == 1:
                # the headline run's buffers are gone with run_ours; each set
                # is built, timed and freed in turn
                import gc
                import torch
                gc.collect()
                torch.cuda.empty_cache()
                peaks = load_peaks()
                out["extra_workloads"] = {}
                for index in extra:
                    out["extra_workloads"][str(index)] = run_extra_workload(index, peaks, dist_env()[2],
                                                                            use_graph=args.graph)
                    gc.collect()
            print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
