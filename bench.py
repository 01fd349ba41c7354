"""Benchmark of the LoRA delta operator: forward + backward per step.

Workload (the per-GEMM LoRA profile of page "Independent from-scratch
Qwen-14B step reimplementation ...", section "Finding 2"): M=8192 tokens,
K=N=4096, R=16, alpha=2, BF16 inputs with FP32 accumulation; X ~ N(0,1),
A ~ N(0,1/4096), B ~ N(0,1/16), dY ~ N(0,1e-2); seeded synthetic data.

One step = lora_delta_fwd + lora_delta_bwd through the C ABI (8 kernels),
called eagerly every step (no CUDA graph, no events inside the timed region).
Metric: algorithmic HBM bytes of the step / step time (GB/s); ms per step and
the fraction of the measured HBM copy peak are reported beside it. After the
timed region, untimed passes give the same steps replayed from a CUDA graph
(`graph_ms_per_step`) and the per-kernel CUDA-event breakdown (`kernels`).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --impl reference the CPU oracle is timed on the host cores instead (a
deliberately slow program: the parity reference, not a performance target).
For N > 1 (launched by torch.distributed.run) every rank runs its own replica
of the workload (the operator does not shard), and rank 0 prints one line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LoRA delta fwd+bwd ms & HBM GB/s (%roofline) at M=8192 K=N=4096 R=16"
# kernels of one step: the forward's three launches, the backward's five (R <= 16)
KERNELS_FWD = ["down U", "rows U", "up dY_lora"]
KERNELS_BWD = ["dy dU+dB", "rows dU+dB", "dX+dA", "combine dA"]   # rank <= 16: dX and dA in one launch
KERNELS = KERNELS_FWD + KERNELS_BWD
N_FWD = len(KERNELS_FWD)
FUSED_FWD = "fwd down+rows+up"   # lora_delta_fwd_fused: the same three steps in one launch
N_ROTATE = 3   # physical copies of the streamed inputs (X, dY), rotated step to step
HBM_NOMINAL_GBS = 7900.0   # GB300 HBM3e, nominal (context beside the measured copy peak)
GRAPH_STEPS = 48   # steps captured in the CUDA graph of the untimed graph pass
PROF_STEPS = 16    # steps of the untimed per-kernel event pass


def algorithmic_bytes(M, K, N, R):
    """Minimum bytes each step of the operator must move (each streamed operand
    read once per consuming kernel, each output written once, small operands
    counted once; dY is read once for both dU and dB), split by the kernel that
    moves them. The rows kernels write U and dU; the slice and chunk partial
    sums they and the final combine read are scratch (L2), not algorithmic
    bytes."""
    bf, f4 = 2, 4
    fwd = {
        "down U": M * K * bf + R * K * bf,                          # X, A -> U partials
        "rows U": M * R * bf,                                       # -> U
        "up dY_lora": M * R * bf + N * R * bf + M * N * f4,         # U, B -> dY_lora
    }
    return {
        "fwd down+rows+up": sum(fwd.values()),                      # the single-launch forward
        **fwd,
        "dy dU+dB": M * N * bf + N * R * bf + M * R * bf            # dY (read once), B, U -> dU, dB partials
                    + N * R * f4,                                   # (dB written by the combine)
        "rows dU+dB": M * R * bf,                                   # -> dU (and dB from its chunk partials)
        "dX+dA": M * K * bf + M * R * bf + R * K * bf               # X, dU, A (read once for both)
                 + M * K * f4 + R * K * f4,                         # -> dX, dA partials
        "combine dA": 0,
    }


def step_bytes(M, K, N, R):
    """Algorithmic bytes of one forward + backward step (the kernels of KERNELS)."""
    alg = algorithmic_bytes(M, K, N, R)
    return sum(alg[k] for k in KERNELS)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# DRAM traffic per launch from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by kernel, with the hash of the kernel sources
# the counters were taken on (every file under csrc/); after any change to the
# sources the line reports null until the counters are taken again.
NCU_TRAFFIC = {   # warm second step of `ncu --cache-control none` (profiles/train_step_M8192_K4096_N4096_R16.md)
    "down U": {"bytes": 72_347_904, "src_hash": "908bed44b4c14346"},
    "rows U": {"bytes": 109_056, "src_hash": "908bed44b4c14346"},
    "up dY_lora": {"bytes": 125_939_712, "src_hash": "908bed44b4c14346"},
    "dy dU+dB+rows dU (cluster)": {"bytes": 80_282_624, "src_hash": "908bed44b4c14346"},
    "dX+dA": {"bytes": 197_818_112, "src_hash": "908bed44b4c14346"},
    "combine dA+dB": {"bytes": 4_759_040, "src_hash": "908bed44b4c14346"},
}


def source_hash() -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "deterministic_arithmetic_gb300", "csrc")
    for name in sorted(os.listdir(d)):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={self.period}"], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        smax = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()) if rows else None}


def dist_setup():
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def kernel_event_pass(ld, names, n_fwd, steps, stream, fwd, bwd):
    """Average duration of each kernel of a forward + backward step (names: the forward's n_fwd
    kernels, then the backward's), from CUDA events the library records between its launches."""
    import torch

    n_bwd = len(names) - n_fwd
    fev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_fwd + 1)] for _ in range(steps)]
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_bwd + 1)] for _ in range(steps)]
    for evs in fev + bev:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(steps):
        ld.lora_delta_set_profile_events(fev[i])
        fwd(i)
        ld.lora_delta_set_profile_events(bev[i])
        bwd(i)
    ld.lora_delta_set_profile_events(None)
    torch.cuda.synchronize()
    out = {}
    for j, name in enumerate(names[:n_fwd]):
        out[name] = statistics.mean(f[j].elapsed_time(f[j + 1]) for f in fev)
    for j, name in enumerate(names[n_fwd:]):
        out[name] = statistics.mean(b[j].elapsed_time(b[j + 1]) for b in bev)
    return out


# ------------------------------------------------------------------ oracle
class OracleSample:
    """The CPU oracle's fwd+bwd (all 7 steps) on the first ``rows`` rows of the
    workload, all of K, N and R. Every step of the operator is linear in M, so
    the time scales to the full batch by M / rows."""

    def __init__(self, shape, rows: int, threads: int = 0):
        from deterministic_arithmetic_gb300 import synthetic as S
        from oracle import oracle as oracle_mod

        self.shape, self.rows = shape, rows
        self.o = oracle_mod.Oracle.load(threads=threads)
        w = S.Workload("sample", S.Shape(rows, shape.K, shape.N, shape.R, shape.alpha), S.train().std)
        self.d = w.generate(0)

    def seconds_full(self) -> float:
        d, a = self.d, self.shape.alpha
        t0 = time.perf_counter()
        f = self.o.fwd(d["x"], d["a"], d["b"], a)
        self.o.bwd(d["dy"], d["x"], d["a"], d["b"], f["u"], a)
        return (time.perf_counter() - t0) * self.shape.M / self.rows

    @property
    def threads(self) -> int:
        return self.o.n_threads

    def describe(self) -> str:
        sh = self.shape
        scale = "" if self.rows == sh.M else f"; time x{sh.M / self.rows:g} to the full batch"
        return (f"oracle fwd+bwd (all 7 steps) on {self.rows} of {sh.M} rows, full K={sh.K}, N={sh.N}, R={sh.R}, "
                f"{self.threads} threads{scale}")


def run_reference(args, world, rank):
    """The oracle as it stands, on the host cores, sized so that the whole
    --steps/--warmup run stays within about two minutes."""
    from deterministic_arithmetic_gb300 import synthetic as S

    if rank != 0:
        return
    shape = S.train().shape
    total_bytes = step_bytes(shape.M, shape.K, shape.N, shape.R)
    probe = OracleSample(shape, 64)
    per_row = probe.seconds_full() / shape.M
    rows = int(min(shape.M, max(16, args.reference_budget_s / max(1, args.steps + args.warmup) / per_row)))
    sample = OracleSample(shape, rows)
    for _ in range(args.warmup):
        sample.seconds_full()
    times = [sample.seconds_full() for _ in range(args.steps)]
    step_s = statistics.median(times)
    value = total_bytes / step_s / 1e9
    desc = sample.describe()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded splitmix64/Box-Muller)",
        "config": {"workload": "LoRA training step M=8192 K=N=4096 R=16 alpha=2", "sample": desc},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": sample.threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def fwd_variants(ld, Xs, A, B, alpha, M, K, N, R, dev, peak, steps=40, reps=25):
    """Forward only: FP32 dY_lora against the BF16 output variant, and the single-launch forward
    (lora_delta_fwd_fused) against the three launches of lora_delta_fwd; CUDA-graph timed like
    the main step (inputs rotated over the same copies of X). The single launch is also timed
    alone with CUDA events (its roofline fraction as one kernel)."""
    import torch

    out = {}
    bf, f4 = 2, 4
    for name, ydt, ysz in (("fwd_fp32_dy", torch.float32, f4), ("fwd_bf16_dy", torch.bfloat16, bf),
                           ("fwd_fused_fp32_dy", torch.float32, f4)):
        call = ld.lora_delta_fwd_fused if "fused" in name else ld.lora_delta_fwd
        Y = torch.empty((M, N), dtype=ydt, device=dev)
        U = torch.empty((M, R), dtype=torch.bfloat16, device=dev)
        wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), dev)
        for i in range(5):
            call(Xs[i % N_ROTATE], A, B, alpha, delta_y=Y, u=U, workspace=wf)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                gst = torch.cuda.current_stream(dev)
                for i in range(steps):
                    call(Xs[i % N_ROTATE], A, B, alpha, delta_y=Y, u=U, workspace=wf, stream=gst)
        torch.cuda.current_stream(dev).wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * steps)
        nbytes = M * K * bf + R * K * bf + 2 * M * R * bf + N * R * bf + M * N * ysz
        out[name] = {"ms": round(ms, 5), "algorithmic_bytes": nbytes, "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                     "launches_per_step": 1 if "fused" in name else 3}
        if "fused" in name:
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(8)]
            for i in range(8):
                ld.lora_delta_set_profile_events(ev[i])
                call(Xs[i % N_ROTATE], A, B, alpha, delta_y=Y, u=U, workspace=wf)
            ld.lora_delta_set_profile_events(None)
            torch.cuda.synchronize()
            k_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
            out[name]["kernel_event_ms"] = round(k_ms, 5)
            out[name]["kernel_frac"] = round(nbytes / (k_ms * 1e-3) / 1e9 / peak, 4)
        assert ld.lora_delta_device_status(wf) == 0
    return out


# Launch schedules of lora_delta_set_schedule measured beside the default (automatic) one:
# (name, schedule, cluster size, forward kernels, backward kernels)
SCHEDULES = [
    ("separate", 0, 0, KERNELS_FWD, KERNELS_BWD),
    ("cluster_reduce_cl4", 1, 4, ["down+rows U (cluster)", "up dY_lora"],
     ["dy dU+dB+rows dU (cluster)", "dX+dA", "combine dA+dB"]),
    ("cluster_single_cl2", 2, 2, ["fwd (cluster)"], ["bwd (cluster)", "combine dA+dB"]),
    ("cluster_single_cl4", 2, 4, ["fwd (cluster)"], ["bwd (cluster)", "combine dA+dB"]),
]
SCHEDULE_NAMES = {0: "separate launches", 1: "cluster reductions", 2: "single cluster launches", 3: "automatic"}


def schedule_kernels(fwd_schedule, bwd_schedule, M, K, N, R):
    """Kernel names of one step (forward's, then backward's) when the forward and the backward take
    the given schedules (as lora_delta_plan reports them), and the algorithmic bytes each moves."""
    alg = algorithmic_bytes(M, K, N, R)
    kb = dict(alg)
    kb.update({"down+rows U (cluster)": alg["down U"] + alg["rows U"],
               "dy dU+dB+rows dU (cluster)": alg["dy dU+dB"] + alg["rows dU+dB"], "combine dA+dB": 0,
               "fwd (cluster)": alg["down U"] + alg["rows U"] + alg["up dY_lora"],
               "bwd (cluster)": alg["dy dU+dB"] + alg["rows dU+dB"] + alg["dX+dA"]})
    by = {sched: (kf, kbw) for _, sched, _, kf, kbw in SCHEDULES}
    return by[fwd_schedule][0], by[bwd_schedule][1], kb


def schedule_variants(ld, Xs, DYs, A, B, alpha, M, K, N, R, dev, peak, steps=24, reps=10):
    """The training step under each cluster schedule (lora_delta_set_schedule): graph-replayed and
    eager step times like the main measurement, and the per-kernel CUDA-event pass with each
    kernel's fraction of the measured copy peak. Every schedule gives the same output bits (tested);
    the default stays the separate launches."""
    import torch

    _, _, kb = schedule_kernels(0, 0, M, K, N, R)   # bytes per kernel name (any schedule)
    total = step_bytes(M, K, N, R)
    Y = torch.empty((M, N), dtype=torch.float32, device=dev)
    U = torch.empty((M, R), dtype=torch.bfloat16, device=dev)
    DX = torch.empty((M, K), dtype=torch.float32, device=dev)
    DA = torch.empty((R, K), dtype=torch.float32, device=dev)
    DB = torch.empty((N, R), dtype=torch.float32, device=dev)
    DU = torch.empty((M, R), dtype=torch.bfloat16, device=dev)
    wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), dev)
    wb = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), dev)
    stream = torch.cuda.current_stream(dev)
    out = {}

    def fwd(i, st=None):
        ld.lora_delta_fwd(Xs[i % N_ROTATE], A, B, alpha, delta_y=Y, u=U, workspace=wf, stream=st or stream)

    def bwd(i, st=None):
        ld.lora_delta_bwd(DYs[i % N_ROTATE], Xs[i % N_ROTATE], A, B, U, alpha, dx=DX, da=DA, db=DB, du=DU,
                          workspace=wb, stream=st or stream)

    for name, sched, cl, kf, kbw in SCHEDULES:
        ld.lora_delta_set_schedule(sched, cl)
        try:
            for i in range(5):
                fwd(i)
                bwd(i)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(steps * reps // 4):
                fwd(i)
                bwd(i)
            e1.record(stream)
            torch.cuda.synchronize()
            eager_ms = e0.elapsed_time(e1) / (steps * reps // 4)
            graph = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                with torch.cuda.graph(graph, stream=cap):
                    gst = torch.cuda.current_stream(dev)
                    for i in range(steps):
                        fwd(i, gst)
                        bwd(i, gst)
            stream.wait_stream(cap)
            graph.replay()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            graph_ms = e0.elapsed_time(e1) / (reps * steps)
            del graph
            kavg = kernel_event_pass(ld, kf + kbw, len(kf), PROF_STEPS, stream, fwd, bwd)
            assert ld.lora_delta_device_status(wf) == 0 and ld.lora_delta_device_status(wb) == 0
        finally:
            ld.lora_delta_set_schedule(3, 0)
        out[f"schedule_{name}"] = {
            "launches_per_step": len(kf) + len(kbw),
            "ms_per_step": round(eager_ms, 5), "graph_ms_per_step": round(graph_ms, 5),
            "gbs": round(total / (eager_ms * 1e-3) / 1e9, 1),
            "kernels": {k: {"ms": round(kavg[k], 5), "algorithmic_bytes": kb[k],
                            "frac": round(kb[k] / (kavg[k] * 1e-3) / 1e9 / peak, 4) if kb[k] else None}
                        for k in kf + kbw},
        }
    return out


def bwd_variants(ld, Xs, DYs, A, B, alpha, M, K, N, R, dev, steps=40, reps=25):
    """Backward only, BF16 dY against the FP32-dY input variant (dV = bf16(fp32(dY * alpha))
    formed by a first launch), CUDA-graph timed, inputs rotated like the main step."""
    import torch

    out = {}
    bf, f4 = 2, 4
    U = torch.empty((M, R), dtype=torch.bfloat16, device=dev)
    wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), dev)
    ld.lora_delta_fwd(Xs[0], A, B, alpha, u=U, workspace=wf)
    DY32 = [d.float() for d in DYs]
    outs = dict(dx=torch.empty((M, K), dtype=torch.float32, device=dev),
                da=torch.empty((R, K), dtype=torch.float32, device=dev),
                db=torch.empty((N, R), dtype=torch.float32, device=dev),
                du=torch.empty((M, R), dtype=torch.bfloat16, device=dev))
    for name, dys, dsz, wsize in (("bwd_bf16_dy", DYs, bf, ld.lora_delta_bwd_workspace_size),
                                  ("bwd_f32_dy", DY32, f4, ld.lora_delta_bwd_f32dy_workspace_size)):
        wb = ld.new_workspace(wsize(M, K, N, R), dev)
        for i in range(5):
            ld.lora_delta_bwd(dys[i % N_ROTATE], Xs[i % N_ROTATE], A, B, U, alpha, workspace=wb, **outs)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                gst = torch.cuda.current_stream(dev)
                for i in range(steps):
                    ld.lora_delta_bwd(dys[i % N_ROTATE], Xs[i % N_ROTATE], A, B, U, alpha, workspace=wb, stream=gst,
                                      **outs)
        torch.cuda.current_stream(dev).wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * steps)
        nbytes = M * N * dsz + N * R * bf + M * R * bf + M * K * bf + R * K * bf + M * K * f4 + 2 * M * R * bf \
            + R * K * f4 + N * R * f4
        out[name] = {"ms": round(ms, 5), "algorithmic_bytes": nbytes, "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                     "launches_per_step": ld.lora_delta_plan(True, M, K, N, R)[1] + (0 if dsz == bf else 1)}
        assert ld.lora_delta_device_status(wb) == 0
    return out


def exact_variant(ld, Xs, DYs, A, B, alpha, M, K, N, R, dev, reps=5):
    """Exact mode of dA and dB (lora_delta_grads_exact: integer long-accumulator digits, one
    rounding) on the step's inputs, event-timed per launch pair (digits + reduce) through the
    library's profiling hook, inputs rotated like the main step."""
    import torch

    U = torch.empty((M, R), dtype=torch.bfloat16, device=dev)
    DU = torch.empty((M, R), dtype=torch.bfloat16, device=dev)
    wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), dev)
    wb = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), dev)
    ld.lora_delta_fwd(Xs[0], A, B, alpha, u=U, workspace=wf)
    ld.lora_delta_bwd(DYs[0], Xs[0], A, B, U, alpha, du=DU, workspace=wb)
    we = ld.new_workspace(ld.lora_delta_grads_exact_workspace_size(M, K, N, R), dev)
    da = torch.empty((R, K), dtype=torch.float32, device=dev)
    db = torch.empty((N, R), dtype=torch.float32, device=dev)
    for i in range(2):
        ld.lora_delta_grads_exact(DYs[i % N_ROTATE], Xs[i % N_ROTATE], U, DU, alpha, da=da, db=db, workspace=we)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    for i in range(reps):
        ld.lora_delta_set_profile_events(ev[i])
        ld.lora_delta_grads_exact(DYs[i % N_ROTATE], Xs[i % N_ROTATE], U, DU, alpha, da=da, db=db, workspace=we)
    ld.lora_delta_set_profile_events([])
    torch.cuda.synchronize()
    t_da = sorted(e[0].elapsed_time(e[1]) for e in ev)[reps // 2]
    t_db = sorted(e[1].elapsed_time(e[2]) for e in ev)[reps // 2]
    prod = M * R * (K + N)
    ms = t_da + t_db
    rate = prod / (ms * 1e-3) / 1e12
    # integer-issue roofline, measured: the library's probe of independent 32-bit wide
    # multiply-adds (the product step) in the digit kernel's launch shape, median of 5 launches
    sink = torch.empty(ld.library().lora_delta_exact_rate_probe_sink_bytes(), dtype=torch.uint8, device=dev)
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(5)]
    ld.lora_delta_exact_rate_probe(256, sink=sink)
    n_mad = 0
    for e in pev:
        e[0].record()
        n_mad = ld.lora_delta_exact_rate_probe(8192, sink=sink)
        e[1].record()
    torch.cuda.synchronize()
    p_ms = sorted(e[0].elapsed_time(e[1]) for e in pev)[2]
    peak = n_mad / (p_ms * 1e-3) / 1e12
    return {"grads_exact": {"ms": round(ms, 4), "ms_da": round(t_da, 4), "ms_db": round(t_db, 4),
                            "products": prod, "gproducts_per_s": round(rate * 1e3, 1),
                            "roofline": {"bound": "alu", "achieved": round(rate, 3), "peak": round(peak, 3),
                                         "unit": "Tproducts/s", "frac": round(rate / peak, 4),
                                         "peak_kind": "measured: independent 32-bit wide multiply-add chains in the "
                                                      "digit kernel's launch shape (lora_delta_exact_rate_probe)",
                                         "peak_probe_ms": round(p_ms, 4), "peak_probe_products": n_mad},
                            "launches_per_step": 4, "median_of": reps}}


def decode_variants(ld, dev, steps=50, reps=20, copies=8):
    """The decode batches of the pages' MLP width (M = 1, 8, 64; K5120 -> N17408; R64; alpha 1;
    random BF16 operands drawn on the device): the forward, and at M = 64 the backward too,
    CUDA-graph timed over `copies` rotated sets of every operand (weights included). The
    working set stays in L2 at these sizes, so the figures are latencies, not HBM rates."""
    import torch

    g = torch.Generator(device=dev)
    g.manual_seed(11)
    K, N, R, alpha = 5120, 17408, 64, 1.0
    bf, f4 = 2, 4

    def rnd(*shape, s=1.0):
        return (torch.randn(*shape, generator=g, device=dev) * s).to(torch.bfloat16)

    def graph_ms(call):
        for i in range(3):
            call(i, torch.cuda.current_stream(dev))
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                gst = torch.cuda.current_stream(dev)
                for i in range(steps):
                    call(i, gst)
        torch.cuda.current_stream(dev).wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * steps)

    out = {}
    for M in (1, 8, 64):
        As = [rnd(R, K, s=K ** -0.5) for _ in range(copies)]
        Bs = [rnd(N, R, s=R ** -0.5) for _ in range(copies)]
        Xs = [rnd(M, K) for _ in range(copies)]
        Ys = [torch.empty((M, N), dtype=torch.float32, device=dev) for _ in range(copies)]
        Us = [torch.empty((M, R), dtype=torch.bfloat16, device=dev) for _ in range(copies)]
        wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), dev)

        def fwd(i, st):
            j = i % copies
            ld.lora_delta_fwd(Xs[j], As[j], Bs[j], alpha, delta_y=Ys[j], u=Us[j], workspace=wf, stream=st)

        def fwd_fused(i, st):
            j = i % copies
            ld.lora_delta_fwd_fused(Xs[j], As[j], Bs[j], alpha, delta_y=Ys[j], u=Us[j], workspace=wf, stream=st)

        nbytes = M * K * bf + R * K * bf + 2 * M * R * bf + N * R * bf + M * N * f4
        for label, fn, launches in ((f"decode_fwd_M{M}", fwd, 3), (f"decode_fwd_fused_M{M}", fwd_fused, 1)):
            ms = graph_ms(fn)
            out[label] = {"ms": round(ms, 5), "algorithmic_bytes": nbytes, "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                          "launches_per_step": launches}
        assert ld.lora_delta_device_status(wf) == 0
        if M == 64:
            DYs = [rnd(M, N) for _ in range(copies)]
            wb = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), dev)
            dx = torch.empty((M, K), dtype=torch.float32, device=dev)
            da = torch.empty((R, K), dtype=torch.float32, device=dev)
            db = torch.empty((N, R), dtype=torch.float32, device=dev)
            du = torch.empty((M, R), dtype=torch.bfloat16, device=dev)

            def bwd(i, st):
                j = i % copies
                ld.lora_delta_bwd(DYs[j], Xs[j], As[j], Bs[j], Us[j], alpha, dx=dx, da=da, db=db, du=du,
                                  workspace=wb, stream=st)

            ms = graph_ms(bwd)
            nbytes = M * N * bf + N * R * bf + M * R * bf + M * K * bf + R * K * bf + M * K * f4 + 2 * M * R * bf \
                + R * K * f4 + N * R * f4
            out["decode_bwd_M64"] = {"ms": round(ms, 5), "algorithmic_bytes": nbytes,
                                     "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "launches_per_step": 6}
            assert ld.lora_delta_device_status(wb) == 0
    return out


def grouped_variants(ld, dev, peak, steps=10, reps=20):
    """The MLP insertion points of the pages (fc1 K5120 -> N17408, fc2 K17408 -> N5120,
    M4096, R16, alpha 1; random BF16 inputs drawn on the device), forward + backward of
    both sites: one grouped call per pass against two single-site calls per pass, each
    CUDA-graph timed; then an untimed per-kernel event pass of the single-site fc1 and fc2
    calls and of the grouped call, each kernel against its algorithmic bytes."""
    import torch

    g = torch.Generator(device=dev)
    g.manual_seed(7)
    M, R = 4096, 16

    def rnd(*shape, s=1.0):
        return (torch.randn(*shape, generator=g, device=dev) * s).to(torch.bfloat16)

    sites = []
    for K, N in ((5120, 17408), (17408, 5120)):
        sites.append(dict(x=rnd(M, K), a=rnd(R, K, s=K ** -0.5), b=rnd(N, R, s=R ** -0.5), dy=rnd(M, N, s=0.1),
                          alpha=1.0, delta_y=torch.empty((M, N), dtype=torch.float32, device=dev),
                          u=torch.empty((M, R), dtype=torch.bfloat16, device=dev),
                          dx=torch.empty((M, K), dtype=torch.float32, device=dev),
                          da=torch.empty((R, K), dtype=torch.float32, device=dev),
                          db=torch.empty((N, R), dtype=torch.float32, device=dev),
                          du=torch.empty((M, R), dtype=torch.bfloat16, device=dev),
                          wf=ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), dev),
                          wb=ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), dev)))
    fw_sites = [{k: s[k] for k in ("x", "a", "b", "alpha", "delta_y", "u")} for s in sites]
    bw_sites = [{k: s[k] for k in ("dy", "x", "a", "b", "u", "alpha", "dx", "da", "db", "du")} for s in sites]
    wfg = ld.new_workspace(sum(s["wf"].numel() for s in sites), dev)
    wbg = ld.new_workspace(sum(s["wb"].numel() for s in sites), dev)

    def separate(st):
        for s in sites:
            ld.lora_delta_fwd(s["x"], s["a"], s["b"], s["alpha"], delta_y=s["delta_y"], u=s["u"], workspace=s["wf"],
                              stream=st)
        for s in sites:
            ld.lora_delta_bwd(s["dy"], s["x"], s["a"], s["b"], s["u"], s["alpha"], dx=s["dx"], da=s["da"], db=s["db"],
                              du=s["du"], workspace=s["wb"], stream=st)

    def grouped(st):
        ld.lora_delta_fwd_grouped(fw_sites, workspace=wfg, stream=st)
        ld.lora_delta_bwd_grouped(bw_sites, workspace=wbg, stream=st)

    out = {}
    nbytes = sum(step_bytes(M, s["x"].shape[1], s["b"].shape[0], R) for s in sites)
    # single-site calls: each call's launch plan; a grouped call takes the separate launches once
    # for all sites (R <= 16: down, rows, up; dy, rows, dX + dA, combine)
    n_sep = sum(ld.lora_delta_plan(False, M, s["x"].shape[1], s["b"].shape[0], R)[1]
                + ld.lora_delta_plan(True, M, s["x"].shape[1], s["b"].shape[0], R)[1] for s in sites)
    for name, fn, launches in (("mlp_fc1_fc2_separate", separate, n_sep), ("mlp_fc1_fc2_grouped", grouped, 3 + 4)):
        for _ in range(3):
            fn(torch.cuda.current_stream(dev))
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                for _ in range(steps):
                    fn(torch.cuda.current_stream(dev))
        torch.cuda.current_stream(dev).wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * steps)
        out[name] = {"ms": round(ms, 5), "algorithmic_bytes": nbytes, "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                     "launches_per_step": launches}
    # per-kernel event pass (untimed): single-site fc1, single-site fc2, grouped fc1 + fc2
    stream = torch.cuda.current_stream(dev)

    def single(s):
        return (lambda i: ld.lora_delta_fwd(s["x"], s["a"], s["b"], s["alpha"], delta_y=s["delta_y"], u=s["u"],
                                            workspace=s["wf"], stream=stream),
                lambda i: ld.lora_delta_bwd(s["dy"], s["x"], s["a"], s["b"], s["u"], s["alpha"], dx=s["dx"],
                                            da=s["da"], db=s["db"], du=s["du"], workspace=s["wb"], stream=stream))

    passes = (("mlp_fc1", *single(sites[0]), sites[:1]), ("mlp_fc2", *single(sites[1]), sites[1:]),
              ("mlp_fc1_fc2_grouped", lambda i: ld.lora_delta_fwd_grouped(fw_sites, workspace=wfg, stream=stream),
               lambda i: ld.lora_delta_bwd_grouped(bw_sites, workspace=wbg, stream=stream), sites))
    for label, f, b, ss in passes:
        names = KERNELS
        kavg = kernel_event_pass(ld, names, N_FWD, 8, stream, f, b)
        alg = {k: sum(algorithmic_bytes(M, s["x"].shape[1], s["b"].shape[0], R)[k] for s in ss) for k in names}
        kern = {k: {"ms": round(kavg[k], 5), "algorithmic_bytes": alg[k],
                    "gbs": round(alg[k] / (kavg[k] * 1e-3) / 1e9, 1) if alg[k] else None,
                    "frac": round(alg[k] / (kavg[k] * 1e-3) / 1e9 / peak, 4) if alg[k] else None} for k in names}
        worst = min((k for k in names if alg[k]), key=lambda k: kern[k]["frac"])
        out.setdefault(label, {}).update({"kernels": kern, "worst_kernel": worst,
                                          "kernels_note": "untimed pass of 8 steps with a CUDA event between kernels"})
    for s in sites:
        assert ld.lora_delta_device_status(s["wf"]) == 0 and ld.lora_delta_device_status(s["wb"]) == 0
    assert ld.lora_delta_device_status(wfg) == 0 and ld.lora_delta_device_status(wbg) == 0
    return out


# ------------------------------------------------------------------ ours
def run_ours(args, world, rank, local):
    import torch

    from deterministic_arithmetic_gb300 import build_lib
    from deterministic_arithmetic_gb300 import lora_delta as ld
    from deterministic_arithmetic_gb300 import synthetic as S

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    if rank == 0 or not os.path.exists(build_lib.LIB):
        build_lib.build()
    barrier(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = S.train()
    sh = w.shape
    M, K, N, R, alpha = sh.M, sh.K, sh.N, sh.R, sh.alpha
    d = w.generate(0)

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    X0, A, B, DY0 = to_dev(d["x"]), to_dev(d["a"]), to_dev(d["b"]), to_dev(d["dy"])
    Xs = [X0] + [X0.clone() for _ in range(N_ROTATE - 1)]
    DYs = [DY0] + [DY0.clone() for _ in range(N_ROTATE - 1)]
    Y = torch.empty((M, N), dtype=torch.float32, device=dev)
    U = torch.empty((M, R), dtype=torch.bfloat16, device=dev)
    DX = torch.empty((M, K), dtype=torch.float32, device=dev)
    DA = torch.empty((R, K), dtype=torch.float32, device=dev)
    DB = torch.empty((N, R), dtype=torch.float32, device=dev)
    DU = torch.empty((M, R), dtype=torch.bfloat16, device=dev)
    wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), dev)
    wb = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), dev)
    stream = torch.cuda.current_stream(dev)
    ld.lora_delta_set_schedule(args.schedule, args.cluster)
    plan_f, plan_b = ld.lora_delta_plan(False, M, K, N, R), ld.lora_delta_plan(True, M, K, N, R)
    kf_names, kb_names, kbytes = schedule_kernels(plan_f[0], plan_b[0], M, K, N, R)
    assert (len(kf_names), len(kb_names)) == (plan_f[1], plan_b[1]), (plan_f, plan_b)
    knames = kf_names + kb_names

    def step(i):
        x, dy = Xs[i % N_ROTATE], DYs[i % N_ROTATE]
        ld.lora_delta_fwd(x, A, B, alpha, delta_y=Y, u=U, workspace=wf, stream=stream)
        ld.lora_delta_bwd(dy, x, A, B, U, alpha, dx=DX, da=DA, db=DB, du=DU, workspace=wb, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # Timed region: every step calls the two API entry points eagerly, as a training loop does.
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else int(
            os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local])) as clocks:
        start.record(stream)
        for i in range(args.steps):
            step(i)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = start.elapsed_time(stop)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    ms_step = elapsed_ms / args.steps
    status = (ld.lora_delta_device_status(wf), ld.lora_delta_device_status(wb))
    if status != (0, 0):
        raise SystemExit(f"device status block reports {status}")

    # Untimed: the same steps replayed from a CUDA graph (launch cost on the host and between
    # kernels as low as it gets), for comparison with the eager steps above.
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            gst = torch.cuda.current_stream(dev)
            for j in range(GRAPH_STEPS):
                x, dy = Xs[j % N_ROTATE], DYs[j % N_ROTATE]
                ld.lora_delta_fwd(x, A, B, alpha, delta_y=Y, u=U, workspace=wf, stream=gst)
                ld.lora_delta_bwd(dy, x, A, B, U, alpha, dx=DX, da=DA, db=DB, du=DU, workspace=wb, stream=gst)
    stream.wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_rep = max(1, min(20, args.steps // GRAPH_STEPS))
    g0.record(stream)
    for _ in range(n_rep):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = g0.elapsed_time(g1) / (n_rep * GRAPH_STEPS)
    del graph

    # Untimed: per-kernel CUDA events (a mark before the first kernel of each call and after each
    # kernel). The events sit between the kernels, so each figure includes its launch boundary.
    kavg = kernel_event_pass(ld, knames, len(kf_names), PROF_STEPS, stream,
                             lambda i: ld.lora_delta_fwd(Xs[i % N_ROTATE], A, B, alpha, delta_y=Y, u=U, workspace=wf,
                                                         stream=stream),
                             lambda i: ld.lora_delta_bwd(DYs[i % N_ROTATE], Xs[i % N_ROTATE], A, B, U, alpha, dx=DX,
                                                         da=DA, db=DB, du=DU, workspace=wb, stream=stream))
    alg = kbytes
    total_bytes = step_bytes(M, K, N, R)
    peak, peak_kind = measured_peaks()
    value = total_bytes * world / (ms_step * 1e-3) / 1e9
    dominant = max(kavg, key=lambda k: kavg[k])
    achieved = alg[dominant] / (kavg[dominant] * 1e-3) / 1e9
    src = source_hash()

    def ncu_traffic(k):
        tr = NCU_TRAFFIC.get(k)
        return tr["bytes"] if tr and tr.get("src_hash") == src else None

    traffic = ncu_traffic(dominant)

    # ---------------------------------------- forward variants (FP32 / BF16 dY_lora)
    variants = None
    if not args.no_variants:
        ld.lora_delta_set_schedule(3, 0)   # the variants choose their own schedules
        variants = fwd_variants(ld, Xs, A, B, alpha, M, K, N, R, dev, measured_peaks()[0])
        variants.update(bwd_variants(ld, Xs, DYs, A, B, alpha, M, K, N, R, dev))
        variants.update(schedule_variants(ld, Xs, DYs, A, B, alpha, M, K, N, R, dev, measured_peaks()[0]))
        variants.update(grouped_variants(ld, dev, measured_peaks()[0]))
        variants.update(exact_variant(ld, Xs, DYs, A, B, alpha, M, K, N, R, dev))
        variants.update(decode_variants(ld, dev))
        ld.lora_delta_set_schedule(args.schedule, args.cluster)

    # ----------------------------------------------------------- end to end
    e2e = None
    if not args.no_e2e:
        pin = dict(x=torch.from_numpy(d["x"].view(np.int16)).pin_memory(),
                   dy=torch.from_numpy(d["dy"].view(np.int16)).pin_memory(),
                   a=torch.from_numpy(d["a"].view(np.int16)).pin_memory(),
                   b=torch.from_numpy(d["b"].view(np.int16)).pin_memory())
        outs = dict(y=torch.empty((M, N), dtype=torch.float32).pin_memory(),
                    u=torch.empty((M, R), dtype=torch.int16).pin_memory(),
                    dx=torch.empty((M, K), dtype=torch.float32).pin_memory(),
                    da=torch.empty((R, K), dtype=torch.float32).pin_memory(),
                    db=torch.empty((N, R), dtype=torch.float32).pin_memory(),
                    du=torch.empty((M, R), dtype=torch.int16).pin_memory())
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in outs.values())
        # pipelined like a data loader: step i's inputs are copied in on one stream, its compute runs on
        # another and its outputs are copied out on a third, so copy-in of step i+1 and copy-out of step
        # i-1 overlap step i's kernels; device buffers are double-buffered (set i % 2)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        sets = []
        for k in range(2):
            sets.append(dict(x=Xs[k], dy=DYs[k], a=torch.empty_like(A), b=torch.empty_like(B),
                             y=torch.empty_like(Y), u=torch.empty_like(U), dx=torch.empty_like(DX),
                             da=torch.empty_like(DA), db=torch.empty_like(DB), du=torch.empty_like(DU),
                             wf=ld.new_workspace(wf.numel(), dev), wb=ld.new_workspace(wb.numel(), dev)))

        def ev():
            return torch.cuda.Event()

        def e2e_steps(n):
            done_in, done_compute, done_out = {}, {}, {}
            for i in range(n):
                b_ = sets[i % 2]
                with torch.cuda.stream(s_in):                      # copy-in (after step i-2 released the set)
                    if i - 2 in done_compute:
                        s_in.wait_event(done_compute[i - 2])
                    b_["x"].view(torch.int16).copy_(pin["x"], non_blocking=True)
                    b_["dy"].view(torch.int16).copy_(pin["dy"], non_blocking=True)
                    b_["a"].view(torch.int16).copy_(pin["a"], non_blocking=True)
                    b_["b"].view(torch.int16).copy_(pin["b"], non_blocking=True)
                    done_in[i] = ev(); done_in[i].record(s_in)
                stream.wait_event(done_in[i])                       # compute
                if i - 2 in done_out:
                    stream.wait_event(done_out[i - 2])
                ld.lora_delta_fwd(b_["x"], b_["a"], b_["b"], alpha, delta_y=b_["y"], u=b_["u"], workspace=b_["wf"],
                                  stream=stream)
                ld.lora_delta_bwd(b_["dy"], b_["x"], b_["a"], b_["b"], b_["u"], alpha, dx=b_["dx"], da=b_["da"],
                                  db=b_["db"], du=b_["du"], workspace=b_["wb"], stream=stream)
                done_compute[i] = ev(); done_compute[i].record(stream)
                with torch.cuda.stream(s_out):                     # copy-out
                    s_out.wait_event(done_compute[i])
                    outs["y"].copy_(b_["y"], non_blocking=True)
                    outs["u"].copy_(b_["u"].view(torch.int16), non_blocking=True)
                    outs["dx"].copy_(b_["dx"], non_blocking=True)
                    outs["da"].copy_(b_["da"], non_blocking=True)
                    outs["db"].copy_(b_["db"], non_blocking=True)
                    outs["du"].copy_(b_["du"].view(torch.int16), non_blocking=True)
                    done_out[i] = ev(); done_out[i].record(s_out)
            return done_out[n - 1]

        e2e_steps(3)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        last = e2e_steps(args.e2e_steps)
        s_out.wait_event(last)
        e1.record(s_out)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.e2e_steps
        e2e = {"value": round(total_bytes * world / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": args.e2e_steps,
               "pipeline": "copy-in, compute and copy-out of consecutive steps on three streams, 2 device buffer sets"}

    # ---------------------------------------------------------- CPU baseline
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = OracleSample(sh, min(M, args.oracle_rows))
        t_full = sample.seconds_full()
        cpu = {"value": round(total_bytes / t_full / 1e9, 4), "unit": "GB/s", "cores": sample.threads,
               "kind": "oracle", "sample": sample.describe(), "ms_per_step": round(t_full * 1e3, 1)}

    if rank == 0:
        clk = clocks.summary()
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded splitmix64/Box-Muller, BF16)",
            "config": {"workload": f"LoRA training step M=8192 K=N=4096 R=16 alpha=2 (fwd+bwd, {len(knames)} kernels)",
                       "schedule": SCHEDULE_NAMES[args.schedule]
                                   + f" (forward: {SCHEDULE_NAMES[plan_f[0]]}, backward: {SCHEDULE_NAMES[plan_b[0]]})"
                                   + (f", clusters of {args.cluster or 4}" if plan_f[0] or plan_b[0] else ""),
                       "M": M, "K": K, "N": N, "R": R, "alpha": alpha, "accumulate": "fp32",
                       "l2": f"inputs rotated over {N_ROTATE} physical copies of X and dY (384 MiB) and a 256 MiB "
                             "output stream per step, all larger than the 129 MB L2",
                       "parallelism": f"replicas x{world}",
                       "timing": "every timed step calls lora_delta_fwd and lora_delta_bwd eagerly (Python binding, "
                                 "C ABI); CUDA events only at the two ends of the timed region"},
            "graph_ms_per_step": round(graph_ms, 5),
            "graph_note": f"the same steps replayed from a CUDA graph of {GRAPH_STEPS} steps (untimed pass)",
            "steps_per_s": round(1e3 / ms_step, 1),
            "roofline_step": {"bound": "hbm", "achieved": round(total_bytes / (ms_step * 1e-3) / 1e9, 1),
                              "peak": peak, "unit": "GB/s", "frac": round(total_bytes / (ms_step * 1e-3) / 1e9 / peak, 4),
                              "peak_kind": peak_kind, "algorithmic_bytes": total_bytes,
                              "frac_of_nominal": round(total_bytes / (ms_step * 1e-3) / 1e9 / HBM_NOMINAL_GBS, 4),
                              "nominal_gbs": HBM_NOMINAL_GBS},
            "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "algorithmic_bytes": alg[dominant], "peak_kind": peak_kind},
            "kernels_note": f"untimed pass of {PROF_STEPS} steps with a CUDA event between kernels (each figure "
                            "includes its launch boundary; events stop the kernels' launch overlap)",
            "kernels": {k: {"ms": round(kavg[k], 5), "algorithmic_bytes": alg[k],
                            "gbs": round(alg[k] / (kavg[k] * 1e-3) / 1e9, 1) if alg[k] else None,
                            "frac": round(alg[k] / (kavg[k] * 1e-3) / 1e9 / peak, 4) if alg[k] else None,
                            "traffic": ncu_traffic(k)}
                        for k in knames},
            "gpu_launches": len(knames) * args.steps,
            "e2e": e2e,
            "variants": variants,
            "cpu_baseline": cpu,
            "clocks": clk,
            "provenance": json.loads(ld.lora_delta_describe()),
        }
        print(json.dumps(line), flush=True)


def profile_site(args):
    """A few forward + backward steps of one MLP insertion point (fc1: K5120 -> N17408, fc2:
    K17408 -> N5120; M4096, R16, alpha 1; device-drawn BF16 inputs), for an ncu capture of the
    kernels at that shape; prints nothing that is a measurement."""
    import torch
    from deterministic_arithmetic_gb300 import build_lib
    from deterministic_arithmetic_gb300 import lora_delta as ld

    build_lib.build()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    M, R = 4096, 16
    K, N = (5120, 17408) if args.profile_site == "fc1" else (17408, 5120)

    def rnd(*shape, s=1.0):
        return (torch.randn(*shape, generator=g, device=dev) * s).to(torch.bfloat16)

    x, a, b, dy = rnd(M, K), rnd(R, K, s=K ** -0.5), rnd(N, R, s=R ** -0.5), rnd(M, N, s=0.1)
    wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), dev)
    wb = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), dev)
    for _ in range(args.steps + args.warmup):
        y, u = ld.lora_delta_fwd(x, a, b, 1.0, workspace=wf)
        ld.lora_delta_bwd(dy, x, a, b, u, 1.0, workspace=wb)
    torch.cuda.synchronize()
    assert ld.lora_delta_device_status(wf) == 0 and ld.lora_delta_device_status(wb) == 0
    print(f"profile-site {args.profile_site}: M={M} K={K} N={N} R={R}, {args.steps + args.warmup} steps done")


def main():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--oracle-rows", type=int, default=8192, help="rows of the CPU-baseline oracle sample")
    p.add_argument("--reference-budget-s", type=float, default=120.0,
                   help="CPU seconds the --impl reference run may spend in total")
    p.add_argument("--schedule", type=int, choices=[0, 1, 2, 3], default=3,
                   help="launch schedule of the timed step (lora_delta_set_schedule): 0 separate launches, "
                        "1 cluster reductions, 2 single cluster launches, 3 automatic (the library's default)")
    p.add_argument("--cluster", type=int, choices=[0, 2, 4, 8], default=0, help="cluster size (0: default)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-variants", action="store_true", help="skip the forward-only FP32 / BF16 dY_lora timing")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile-site", choices=["fc1", "fc2"], default=None,
                   help="only run a few steps of one MLP site (for an ncu capture) and exit")
    args = p.parse_args()
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.profile_site:
        profile_site(args)
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
