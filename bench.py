#!/usr/bin/env python
"""Benchmark of the fused linear cross entropy forward+backward on GB300.

One step = one flce_fwd_bwd call over one batch of synthetic inputs (all stages: row
compaction, logits GEMM with online logsumexp, finalize, gradient formation, dX GEMM, dW
GEMM, reductions). Default workload: the Llama-3.1-8B-shaped head (BT=8192, H=4096,
V=128256, bf16, 16 sequences of 512 rows with the last row of each ignored, mean, z-loss
1e-4, dX and fp32 dW).

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--labelled-fraction F]
  python bench.py --impl reference ...   # the float64 CPU oracle on a bounded row sample
  python bench.py --op jsd ...           # the fused linear JSD distillation op (student
                                         # Llama-3.2-1B head vs Llama-3.1-8B teacher head)

Prints one JSON line (rank 0). Under torchrun each rank runs an independent replica on its
own GPU (the op has no exchange step); value = all ranks' tokens / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from linear_cross_entropy_logits_gb300 import inputs as I  # noqa: E402

METRIC = "FLCE fwd+bwd tokens/s and ms at 1 GB300; % of dense bf16 tensor peak"
UNIT = "tokens/s"
WORKLOAD_TITLES = {
    "tiny_fp32": "tiny fp32 FLCE",
    "llama1b": "Llama-3.2-1B-shaped head",
    "llama8b": "Llama-3.1-8B-shaped head",
    "large_vocab": "large-vocab long-context head",
    "frozen_head": "frozen-head (LoRA) variant",
    "llama2_7b": "32000-token head (H=4096)",
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--op", default="flce", choices=["flce", "jsd"])
    p.add_argument("--workload", default="llama8b", choices=list(I.WORKLOADS))
    p.add_argument("--dtype", default=None, choices=["bf16", "f16", "f32"],
                   help="override the workload's input dtype")
    p.add_argument("--dw-dtype", default="f32", choices=["f32", "same"],
                   help="dW / dbias accumulation dtype: fp32, or the input dtype")
    p.add_argument("--api", default="abi", choices=["abi", "torch"],
                   help="abi: the C ABI through the ctypes binding; torch: the autograd op "
                        "(loss = fused_linear_cross_entropy(X, W, targets); loss.backward())")
    p.add_argument("--labelled-fraction", type=float, default=None)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=20.0,
                   help="timed oracle seconds of the cpu_baseline leg")
    p.add_argument("--ref-seconds", type=float, default=100.0,
                   help="total oracle time budget of the --impl reference arm")
    p.add_argument("--bt", type=int, default=None,
                   help="override BT (smaller cases for profiler captures)")
    p.add_argument("--bounded-budget-gib", type=float, default=1.5,
                   help="also time the step at this workspace budget when the default one "
                        "holds the slab of every row (0: skip)")
    p.add_argument("--budget-gib", type=float, default=None,
                   help="workspace budget in GiB (default: the workload's cap, else the "
                        "library's default); sets the chunk rows R")
    return p.parse_args()


def workload_spec(args):
    ov = {}
    if args.labelled_fraction is not None:
        ov["labelled_fraction"] = args.labelled_fraction
    if args.bt is not None:
        ov["BT"] = args.bt
    if getattr(args, "dtype", None) is not None:
        ov["dtype"] = args.dtype
    if getattr(args, "budget_gib", None) is not None:
        ov["workspace_cap"] = int(args.budget_gib * 2 ** 30)
    return I.spec(args.workload, **ov)


def config_of(sp, n_lab, extra=None):
    c = {"workload": f"{WORKLOAD_TITLES[sp['name']]} ({sp['name']})", "BT": sp["BT"], "H": sp["H"],
         "V": sp["V"], "input_dtype": sp["dtype"], "n_labelled": int(n_lab),
         "reduction": sp["reduction"], "z_loss_scale": sp.get("z", 0.0),
         "bias": sp.get("bias_std") is not None, "dW": bool(sp["want_dW"]),
         "targets": sp.get("targets", "uniform"), "ignored_rows": sp.get("ignore", "none")}
    if sp.get("ignore") == "prompt_first":
        c["labelled_fraction"] = sp.get("labelled_fraction", 1.0)
    if extra:
        c.update(extra)
    return c


def flops_per_step(sp, n_lab):
    return (6 if sp["want_dW"] else 4) * n_lab * sp["H"] * sp["V"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def peak_for_region(peaks, src, region_ms):
    """The bf16 denominator for a timed region: the burst figure (cuBLAS timed alone) for a
    region under two seconds, which runs mostly before the power cap pulls the clocks
    down; the sustained figure (cuBLAS back to back for seconds) for a longer one."""
    if region_ms < 2000.0 or "bf16_tflops_sustained" not in peaks:
        return peaks["bf16_tflops"], f"bf16 burst ({src}; timed region {region_ms / 1000.0:.2f} s < 2 s)"
    return peaks["bf16_tflops_sustained"], f"bf16 sustained ({src}; timed region {region_ms / 1000.0:.1f} s)"


def fp32_fma_peak(peaks, dev):
    """FP32 FMA peak of the GPU from its unit counts and clock: 128 FP32 lanes per SM, two
    FLOPs per FMA, at the maximum SM clock."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = peaks.get("sm_max_mhz", 2070.0)
    return 2.0 * 128 * sms * mhz * 1e6 / 1e12, f"fp32 FMA: 2 x 128 lanes x {sms} SMs x {mhz:.0f} MHz"


def cpu_baseline_subprocess(args):
    """The oracle timed in a fresh process (this process's CUDA and threading state slowed
    the oracle's BLAS calls by 2x): the --impl reference arm of this script on the same
    workload, 2 steps of cpu_seconds/2 after a short warm-up. Returns its cpu_baseline."""
    argv = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--op", args.op,
            "--workload", args.workload, "--steps", "2", "--warmup", "1",
            "--ref-seconds", str(1.5 * args.cpu_seconds)]
    for flag, v in (("--labelled-fraction", args.labelled_fraction), ("--bt", args.bt),
                    ("--dtype", args.dtype), ("--budget-gib", args.budget_gib)):
        if v is not None:
            argv += [flag, str(v)]
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE")}
    r = subprocess.run(argv, capture_output=True, text=True, env=env, timeout=600)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    if r.returncode != 0 or not lines:
        return {"value": None, "error": (r.stderr or r.stdout)[-300:]}
    ref = json.loads(lines[-1])
    cb = dict(ref["cpu_baseline"])
    cb["process"] = "fresh subprocess (bench.py --impl reference, 2 steps)"
    return cb


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 50 ms, time-stamped on arrival by a reader thread; the
    summary keeps only the samples taken inside the timed region (mark_start / mark_end),
    so that idle clocks before or after it do not enter the median."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, dev):
        self.proc = None
        self.dev = dev
        self.rows = []
        self.t0 = self.t1 = None
        self.thread = None

    def _reader(self):
        for line in self.proc.stdout:
            if line.count(",") >= 8:
                self.rows.append((time.perf_counter(), line.strip().split(",")))

    def start(self):
        import threading
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", str(self.PERIOD_MS)]
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True, bufsize=1)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(2 * self.PERIOD_MS / 1000.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        # a sample reports the state of the preceding period: keep those that arrive
        # inside the region, plus the first one after it
        lo = self.t0 if self.t0 is not None else -float("inf")
        hi = (self.t1 if self.t1 is not None else float("inf")) + self.PERIOD_MS / 1000.0
        inside = [r for t, r in self.rows if lo <= t <= hi]
        rows = inside if inside else [r for _, r in self.rows]
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[1]) for r in rows) if v is not None]
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        pw = [v for v in (num(r[3]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "in_timed_region": bool(inside),
                "sm_mhz_min": min(sm) if sm else None, "power_w_max": max(pw) if pw else None,
                "period_ms": self.PERIOD_MS}


# ----------------------------------------------------------------------------- oracle timing
def oracle_prepare(sp, inp):
    """Untimed set-up of the oracle timing: the head weight (and bias) converted to float64
    once, the labelled rows listed. The timed calls then run the oracle on float64 arrays,
    on which its own per-block conversions are no-ops."""
    t = inp["targets"].numpy()
    return {"sp": sp, "t": t, "lab": np.nonzero(t != I.IGNORE_INDEX)[0],
            "W": I.to_numpy_exact(inp["W"]).astype(np.float64),
            "b": None if inp["bias"] is None else I.to_numpy_exact(inp["bias"]).astype(np.float64),
            "X": inp["X"],
            "go": inp["grad_out"].numpy() if inp["grad_out"] is not None else None}


def oracle_sample_rate(prep, seconds, rows_per_call=32, rng_seed=99, warmup_calls=1):
    """Time the float64 oracle (as it stands) on seeded samples of labelled rows of this
    workload until about `seconds` of CPU work, after `warmup_calls` untimed calls; returns
    (BT-tokens per second, rows, seconds). Ignored rows cost the oracle nothing, so labelled
    rows per second are scaled by BT / n_labelled to the metric's BT-token convention."""
    from oracle import flce_oracle as orc
    sp, t, lab, W, b, X, go = (prep[k] for k in ("sp", "t", "lab", "W", "b", "X", "go"))
    rng = np.random.default_rng(rng_seed)

    def call(rows):
        Xs = I.to_numpy_exact(X[torch.from_numpy(rows)]).astype(np.float64)
        gs = go[rows] if (go is not None and sp["reduction"] == "none") else None
        t0 = time.perf_counter()
        orc.flce_oracle(Xs, W, t[rows], bias=b, reduction=sp["reduction"],
                        z_loss_scale=sp.get("z", 0.0), grad_out=gs, want_dX=True,
                        want_dW=sp["want_dW"])
        return time.perf_counter() - t0

    for _ in range(warmup_calls):
        call(np.sort(rng.choice(lab, size=min(rows_per_call, lab.size), replace=False)))
    done, spent = 0, 0.0
    while spent < seconds:
        rows = np.sort(rng.choice(lab, size=min(rows_per_call, lab.size), replace=False))
        spent += call(rows)
        done += rows.size
    rate_lab = done / spent
    return rate_lab * sp["BT"] / max(lab.size, 1), done, spent


def jsd_oracle_sample_rate(sp, inp, seconds, rows_per_call=16, rng_seed=7):
    """Time the float64 JSD oracle (as it stands) on seeded samples of labelled rows of the
    distillation workload until about `seconds` of CPU work; returns (BT-tokens per second,
    rows, seconds), scaled by BT / n_labelled as for the cross-entropy op."""
    from oracle import jsd_oracle as jo
    lab_all = inp["labels"].numpy()
    lab = np.nonzero(lab_all != I.IGNORE_INDEX)[0]
    # the heads converted to float64 once, outside the timed calls
    Ws = I.to_numpy_exact(inp["Ws"]).astype(np.float64)
    Wt = I.to_numpy_exact(inp["Wt"]).astype(np.float64)
    rng = np.random.default_rng(rng_seed)
    done, spent = 0, 0.0
    while spent < seconds:
        rows = np.sort(rng.choice(lab, size=min(rows_per_call, lab.size), replace=False))
        idx = torch.from_numpy(rows)
        xs = I.to_numpy_exact(inp["Xs"][idx]).astype(np.float64)
        xt = I.to_numpy_exact(inp["Xt"][idx]).astype(np.float64)
        t0 = time.perf_counter()
        jo.jsd_oracle(xs, Ws, xt, Wt, lab_all[rows], beta=sp["beta"], temperature=sp["temperature"],
                      reduction=sp["reduction"], want_dX=True, want_dW=sp["want_dW"])
        spent += time.perf_counter() - t0
        done += rows.size
    return done / spent * sp["BT"] / max(lab.size, 1), done, spent


def step_percentiles(evs):
    """Median, p20 and p80 of the per-step device times between consecutive events."""
    t = sorted(a.elapsed_time(b) for a, b in zip(evs[:-1], evs[1:]))

    def pct(q):
        return float(np.percentile(np.asarray(t), q))
    return {"p20": pct(20), "median": pct(50), "p80": pct(80), "steps": len(t)}


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("internal_api") in ("openblas", "mkl", "blis")]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def traffic_record(run):
    """ncu DRAM bytes per GEMM launch, if taken with the current kernel sources on the
    configuration of this run (the record's "config": workload, BT, labelled rows, input and
    dW dtypes, chunk rows); None otherwise."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    if any(run.get(k) != v for k, v in rec.get("config", {"unmatched": True}).items()):
        return None
    return rec


# The sources the tensor-core GEMM kernel (the dominant kernel) is compiled from.
GEMM_SOURCES = ("flce_internal.cuh", "flce_tc.cu")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_cross_entropy_logits_gb300", "csrc")
    for name in GEMM_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(value, dist=None, device="cpu"):
    """Max of a per-rank scalar over all ranks (the bench reports the slowest replica)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- arms
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    sp = workload_spec(args)
    inp = I.generate(sp, seed=0)
    n_lab = int((inp["targets"] != I.IGNORE_INDEX).sum())
    prep = oracle_prepare(sp, inp)
    per_step_seconds = max(min(2.0, args.ref_seconds), args.ref_seconds / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        oracle_sample_rate(prep, per_step_seconds / 4, rng_seed=1)
    rows_total, secs_total = 0, 0.0
    for k in range(args.steps):
        _, rows, secs = oracle_sample_rate(prep, per_step_seconds, rng_seed=100 + k, warmup_calls=0)
        rows_total += rows
        secs_total += secs
    value = rows_total * sp["BT"] / max(n_lab, 1) / secs_total
    ms_per_step = sp["BT"] / value * 1000.0
    cores = cpu_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded torch.Generator)",
        "config": config_of(sp, n_lab, {"sample": "seeded samples of labelled rows"}),
        # the oracle never runs a whole step: ms_per_step is the time one step of all BT
        # rows would take at the measured rate
        "extrapolated": True, "timed_seconds": secs_total, "timed_rows": rows_total,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows_total} labelled rows in {args.steps} steps of "
                                   f"~{per_step_seconds:.0f} s, 32 rows per call (float64 oracle: "
                                   f"logits, lse, loss, dX and dW per row; W converted to float64 "
                                   f"once, untimed), scaled by BT/n_labelled; ms_per_step "
                                   f"extrapolated from {secs_total:.1f} s timed"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    from linear_cross_entropy_logits_gb300 import build as B
    B.build()
    from linear_cross_entropy_logits_gb300 import flce

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    sp = workload_spec(args)
    inp = I.generate(sp, seed=rank)
    n_lab = int((inp["targets"] != I.IGNORE_INDEX).sum())
    BT, H, V = sp["BT"], sp["H"], sp["V"]
    dt = I.TORCH_DTYPES[sp["dtype"]]
    X = inp["X"].to(dev)
    W = inp["W"].to(dev)
    tg = inp["targets"].to(dev)
    bias = inp["bias"].to(dev) if inp["bias"] is not None else None
    go = inp["grad_out"].to(dev) if inp["grad_out"] is not None else None
    ws_bytes = flce.workspace_size(BT, H, V, dt, sp.get("workspace_cap", 0))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    R = flce.chunk_rows(BT, H, V, dt, ws_bytes)
    nl = BT if sp["reduction"] == "none" else 1
    outs = {"loss": torch.empty(nl, dtype=torch.float32, device=dev),
            "z_loss": torch.empty(nl, dtype=torch.float32, device=dev),
            "acc": torch.empty(nl, dtype=torch.float32, device=dev),
            "lse": torch.empty(BT, dtype=torch.float32, device=dev),
            "pred": torch.empty(BT, dtype=torch.int64, device=dev),
            "n_labelled": torch.empty(1, dtype=torch.int32, device=dev),
            "status": torch.zeros(1, dtype=torch.int32, device=dev),
            "dX": torch.empty(BT, H, dtype=dt, device=dev)}
    acc_dt = torch.float32 if args.dw_dtype == "f32" else dt
    dW = torch.zeros(V, H, dtype=acc_dt, device=dev) if sp["want_dW"] else None
    dbias = torch.zeros(V, dtype=acc_dt, device=dev) if (sp["want_dW"] and bias is not None) else None
    prof = flce.Profiler()

    if args.api == "torch":
        from linear_cross_entropy_logits_gb300.torch_ops import fused_linear_cross_entropy
        Xp = X.detach().clone().requires_grad_(True)
        Wp = W.detach().clone().requires_grad_(sp["want_dW"])
        bp = bias.detach().clone().requires_grad_(sp["want_dW"]) if bias is not None else None

        def step(Xd=X, tgd=tg, god=go, profiler=None):
            # a training step's view: fresh .grad tensors each step
            Xp.grad = None
            Wp.grad = None
            if bp is not None:
                bp.grad = None
            loss = fused_linear_cross_entropy(Xp, Wp, tgd, bp, reduction=sp["reduction"],
                                              z_loss_scale=sp.get("z", 0.0),
                                              accum_dtype=acc_dt)
            if sp["reduction"] == "none":
                loss.backward(god)
            else:
                loss.backward()
            outs["loss"] = loss.detach().reshape(-1)
    else:
        def step(Xd=X, tgd=tg, god=go, profiler=None):
            flce.fwd_bwd(Xd, W, tgd, bias, reduction=sp["reduction"], z_loss_scale=sp.get("z", 0.0),
                         grad_out=god, want_dX=True, want_dW=sp["want_dW"], dW=dW, dbias=dbias,
                         workspace=ws, outputs=outs, check=False, profiler=profiler)

    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    st = flce.load().flce_get_status(outs["status"].data_ptr(), None, stream.cuda_stream)
    if st != flce.FLCE_OK:
        raise RuntimeError(f"warm-up status {flce.status_string(st)}")

    # ---- device-timed region
    clk = ClockSampler(dev)
    clk.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    prof.reset()
    torch.cuda.reset_peak_memory_stats(dev)
    mem0 = torch.cuda.memory_allocated(dev)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    clk.mark_start()
    evs[0].record(stream)
    for i in range(args.steps):
        step(profiler=prof)
        evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    clk.mark_end()
    if dist:
        dist.barrier()
    clocks = clk.stop()
    ms_total = evs[0].elapsed_time(evs[-1])
    per_step = step_percentiles(evs)
    transient = {"workspace_bytes": ws_bytes,
                 "allocated_in_timed_region_bytes": int(torch.cuda.max_memory_allocated(dev) - mem0)}
    stages = prof.read()
    ms_total = max_over_ranks(ms_total, dist, dev)
    ms_step = ms_total / args.steps
    value = BT * world / (ms_step / 1000.0)

    # ---- the same step with the workspace capped so that the exp slab holds fewer rows
    # than BT (R < BT): the memory / time trade of the budget argument
    bounded = None
    if (args.api == "abi" and world == 1 and args.budget_gib is None and R >= BT
            and args.bounded_budget_gib > 0):
        ws2_bytes = flce.workspace_size(BT, H, V, dt, int(args.bounded_budget_gib * 2 ** 30))
        R2 = flce.chunk_rows(BT, H, V, dt, ws2_bytes)
        if 0 < R2 < BT:
            ws2 = torch.empty(ws2_bytes, dtype=torch.uint8, device=dev)

            def step2():
                flce.fwd_bwd(X, W, tg, bias, reduction=sp["reduction"], z_loss_scale=sp.get("z", 0.0),
                             grad_out=go, want_dX=True, want_dW=sp["want_dW"], dW=dW, dbias=dbias,
                             workspace=ws2, outputs=outs, check=False)
            for _ in range(3):
                step2()
            torch.cuda.synchronize(dev)
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for _ in range(args.steps):
                step2()
            b1.record(stream)
            torch.cuda.synchronize(dev)
            ms2 = b0.elapsed_time(b1) / args.steps
            bounded = {"budget_bytes": int(args.bounded_budget_gib * 2 ** 30), "workspace_bytes": ws2_bytes,
                       "chunk_rows": R2, "chunks": -(-n_lab // R2), "ms_per_step": ms2,
                       "value": BT / (ms2 / 1000.0), "unit": UNIT,
                       "slab_bytes": R2 * -(-V // 256) * 256 * X.element_size()}
            del ws2

    # ---- end to end through the public API with pinned host inputs / outputs: every step
    # copies its token rows, targets (and per-token gradient) in from pinned host memory and
    # reads the loss back; the copy of step k+1 overlaps step k on a copy stream
    # (DoubleBufferedInputs), as a training loop feeding the op would run
    e2e = None
    if not args.no_e2e and args.api == "abi":
        from linear_cross_entropy_logits_gb300.feeder import DoubleBufferedInputs
        host = {"X": inp["X"].pin_memory(), "t": inp["targets"].pin_memory()}
        if inp["grad_out"] is not None:
            host["g"] = inp["grad_out"].pin_memory()
        lh = torch.empty(nl, dtype=torch.float32).pin_memory()
        feed = DoubleBufferedInputs(host, dev)

        def e2e_run(n, start=None):
            slot = feed.stage(host, after=start)
            for k in range(n):
                nxt = feed.stage(host) if k + 1 < n else None
                dv = feed.acquire(slot, stream)
                step(dv["X"], dv["t"], dv.get("g"))
                feed.release(slot, stream)
                lh.copy_(outs["loss"], non_blocking=True)
                slot = nxt

        e2e_run(2)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        e2e_run(args.steps, start=f0)
        f1.record(stream)
        torch.cuda.synchronize(dev)
        ms_e2e = f0.elapsed_time(f1) / args.steps
        ms_e2e = max_over_ranks(ms_e2e, dist, dev)
        e2e = {"value": BT * world / (ms_e2e / 1000.0), "unit": UNIT, "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": int(feed.h2d_bytes), "d2h_bytes_per_step": int(lh.numel() * 4),
               "copies": "H2D of step k+1 on a copy stream overlapping step k (double-buffered)"}

    # ---- roofline of the dominant kernel (per-stage CUDA events on the launching stream)
    peaks, peak_src = load_peaks()
    flops = flops_per_step(sp, n_lab)
    gemm_flops = 2.0 * n_lab * H * V
    dom = max(stages, key=lambda k: stages[k][0])
    dom_ms, dom_launches = stages[dom]
    per_step_dom_ms = dom_ms / args.steps
    stage_summary = {k: {"ms_per_step": v[0] / args.steps, "launches_per_step": v[1] / args.steps}
                     for k, v in stages.items() if v[1] > 0}
    rec = traffic_record({"workload": args.workload, "BT": BT, "n_labelled": n_lab, "dtype": sp["dtype"],
                          "dW_dtype": "f32" if args.dw_dtype == "f32" else sp["dtype"], "chunk_rows": R})
    if args.api == "torch":
        # the autograd op takes no profiler: whole-step numbers only
        roof = None
    elif dom in ("fwd", "dx", "dw", "bwd"):
        # "bwd": the dX and dW GEMMs in one launch (two GEMMs' FLOPs)
        achieved = gemm_flops * (2 if dom == "bwd" else 1) / (per_step_dom_ms / 1000.0) / 1e12
        if sp["dtype"] == "f32":
            # fp32 inputs run the SIMT FMA kernels: the bound is the FP32 FMA pipes
            peak, peak_kind = fp32_fma_peak(peaks, dev)
            bound = "alu"
        else:
            peak, peak_kind = peak_for_region(peaks, peak_src, evs[0].elapsed_time(evs[-1]))
            bound = "tensor"

        def gemm_entry(k):
            tf = gemm_flops * (2 if k == "bwd" else 1) / (stages[k][0] / args.steps / 1000.0) / 1e12
            return {"ms_per_step": stages[k][0] / args.steps, "tflops": tf, "frac": tf / peak,
                    "traffic": (rec["per_launch_bytes"].get(k) if rec else None)}
        roof = {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "peak_kind": peak_kind,
                "sm_mhz_median": (clocks or {}).get("sm_mhz"),
                "per_launch": (f"{4 if dom == 'bwd' else 2}*H*V FLOPs per labelled row x "
                               f"{n_lab * args.steps / max(stages[dom][1] / (2 if dom in ('dx', 'bwd') else 1), 1):.0f} "
                               f"rows per launch"),
                "traffic": (rec["per_launch_bytes"].get(dom) if rec else None),
                "traffic_source": "profiles/traffic.json (ncu, full size)" if rec else None,
                "gemms": {k: gemm_entry(k) for k in ("fwd", "dx", "dw", "bwd") if k in stages and stages[k][1] > 0}}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": None, "peak": peaks.get("hbm_gbs"),
                "unit": "GB/s", "frac": None, "traffic": None}
    tflops = flops / (ms_step / 1000.0) / 1e12

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if sp["dtype"] == "bf16" else sp["dtype"],
        "data": "synthetic (seeded torch.Generator; random-init head weights)",
        "config": config_of(sp, n_lab, {
            "parallelism": f"replicas x{world} (no exchange step)",
            "l2": f"no flush: W ({V * H * I.TORCH_DTYPES[sp['dtype']].itemsize / 1e9:.2f} GB) and the "
                  f"per-chunk slab exceed the 129 MB L2",
            "workspace_bytes": ws_bytes, "chunk_rows": R, "api": args.api,
            "dW_dtype": "f32" if args.dw_dtype == "f32" else sp["dtype"]}),
        "ms_per_step_percentiles": per_step,
        "transient": transient,
        "tokens_per_s_labelled": n_lab * world / (ms_step / 1000.0),
        "tflops": tflops, "flops_per_step": flops,
        "frac_of_bf16_peak": {"burst": tflops / peaks["bf16_tflops"],
                              "sustained": tflops / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]),
                              "source": peak_src},
        "roofline": roof,
        "stages": stage_summary,
        "gpu_launches": int(sum(v[1] for v in stages.values())) if args.api == "abi" else None,
        "clocks": clocks,
        "e2e": e2e,
        "slab_rows_below_bt": bounded,
        "context_vs_h200_public_default_ms": 53.039 if sp["name"] == "llama8b" else None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_subprocess(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_jsd(args):
    """The fused linear JSD distillation op on its synthetic workload (rank-local replicas
    under torchrun, like the cross-entropy op). FLOPs counted: the student and teacher
    logits GEMMs plus the student dX and dW GEMMs, 2 N V (3 Hs + Ht)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    sp = dict(I.DISTILL)
    if args.bt is not None:
        sp["BT"] = args.bt
    BT, Hs, Ht, V = sp["BT"], sp["Hs"], sp["Ht"], sp["V"]
    inp = I.generate_distill(sp, seed=rank)
    n_lab = int((inp["labels"] != I.IGNORE_INDEX).sum())
    flops = 2.0 * n_lab * V * (3 * Hs + Ht)
    cfg = {"workload": "distillation: Llama-3.2-1B-shaped student head vs Llama-3.1-8B-shaped "
                       "teacher head (distill)", "BT": BT, "Hs": Hs, "Ht": Ht, "V": V,
           "input_dtype": sp["dtype"], "beta": sp["beta"], "temperature": sp["temperature"],
           "reduction": sp["reduction"], "n_labelled": n_lab}
    metric = "fused linear JSD fwd+bwd tokens/s"
    if args.impl == "reference":
        if rank != 0:
            return
        per_step = max(min(2.0, args.ref_seconds), args.ref_seconds / max(args.steps + args.warmup, 1))
        jsd_oracle_sample_rate(sp, inp, per_step * args.warmup)
        value, done, spent = jsd_oracle_sample_rate(sp, inp, per_step * args.steps)
        print(json.dumps({"impl": "reference", "op": "fused_linear_jsd", "metric": metric, "value": value,
                          "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": BT / value * 1000.0, "higher_is_better": True, "scaling": "weak",
                          "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded torch.Generator)",
                          "config": cfg, "extrapolated": True, "timed_seconds": spent, "timed_rows": done,
                          "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(),
                                           "kind": "oracle",
                                           "sample": f"{done} seeded labelled rows, {spent:.1f} s of float64 "
                                                     f"oracle work (both heads' logits, loss, dX, dW)"},
                          "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return
    from linear_cross_entropy_logits_gb300 import build as B
    B.build()
    from linear_cross_entropy_logits_gb300 import flce
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    d = {k: v.to(dev) for k, v in inp.items()}
    dt = I.TORCH_DTYPES[sp["dtype"]]
    ws_bytes = flce.jsd_workspace_size(BT, Hs, Ht, V, dt, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    dW = torch.zeros(V, Hs, dtype=torch.float32, device=dev)
    outs = {"loss": torch.empty(1, device=dev), "n_labelled": torch.empty(1, dtype=torch.int32, device=dev),
            "status": torch.zeros(1, dtype=torch.int32, device=dev), "dX": torch.empty_like(d["Xs"])}
    prof = flce.Profiler()

    def step(profiler=None):
        flce.fused_linear_jsd(d["Xs"], d["Ws"], d["Xt"], d["Wt"], d["labels"], beta=sp["beta"],
                              temperature=sp["temperature"], dW=dW, workspace=ws, outputs=outs,
                              check=False, profiler=profiler)

    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    st = flce.load().flce_get_status(outs["status"].data_ptr(), None, stream.cuda_stream)
    if st != flce.FLCE_OK:
        raise RuntimeError(f"warm-up status {flce.status_string(st)}")
    clk = ClockSampler(dev)
    clk.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    prof.reset()
    torch.cuda.reset_peak_memory_stats(dev)
    mem0 = torch.cuda.memory_allocated(dev)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    clk.mark_start()
    evs[0].record(stream)
    for i in range(args.steps):
        step(prof)
        evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    clk.mark_end()
    if dist:
        dist.barrier()
    clocks = clk.stop()
    ms = max_over_ranks(evs[0].elapsed_time(evs[-1]), dist, dev) / args.steps
    per_step = step_percentiles(evs)
    transient = {"workspace_bytes": ws_bytes,
                 "allocated_in_timed_region_bytes": int(torch.cuda.max_memory_allocated(dev) - mem0)}
    stages = prof.read()

    # end to end through the public API: both heads' token rows and the labels copied in
    # from pinned host memory, the loss read back, every step (head weights stay resident)
    e2e = None
    if not args.no_e2e:
        from linear_cross_entropy_logits_gb300.feeder import DoubleBufferedInputs
        host = {k: inp[k].pin_memory() for k in ("Xs", "Xt", "labels")}
        lh = torch.empty(1, dtype=torch.float32).pin_memory()
        feed = DoubleBufferedInputs(host, dev)

        def e2e_run(n, start=None):
            slot = feed.stage(host, after=start)
            for k in range(n):
                nxt = feed.stage(host) if k + 1 < n else None
                dv = feed.acquire(slot, stream)
                flce.fused_linear_jsd(dv["Xs"], d["Ws"], dv["Xt"], d["Wt"], dv["labels"], beta=sp["beta"],
                                      temperature=sp["temperature"], dW=dW, workspace=ws, outputs=outs,
                                      check=False)
                feed.release(slot, stream)
                lh.copy_(outs["loss"], non_blocking=True)
                slot = nxt

        e2e_run(2)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        e2e_run(args.steps, start=f0)
        f1.record(stream)
        torch.cuda.synchronize(dev)
        ms_e2e = max_over_ranks(f0.elapsed_time(f1) / args.steps, dist, dev)
        e2e = {"value": BT * world / (ms_e2e / 1000.0), "unit": UNIT, "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": int(feed.h2d_bytes), "d2h_bytes_per_step": 4,
               "copies": "H2D of step k+1 on a copy stream overlapping step k (double-buffered)"}
    peaks, src = load_peaks()
    tflops = flops / (ms / 1000.0) / 1e12
    dom = max(("fwd", "dx", "dw", "bwd"), key=lambda k: stages[k][0])
    dom_flops = 2.0 * n_lab * V * {"fwd": Hs + Ht, "bwd": 2 * Hs}.get(dom, Hs)
    achieved = dom_flops / (stages[dom][0] / args.steps / 1000.0) / 1e12
    peak, peak_kind = peak_for_region(peaks, src, evs[0].elapsed_time(evs[-1]))
    line = {"op": "fused_linear_jsd", "metric": metric,
            "value": BT * world / (ms / 1000.0), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": sp["dtype"], "data": "synthetic (seeded torch.Generator)",
            "config": dict(cfg, workspace_bytes=ws_bytes, chunk_rows=None,
                           l2="no flush: the heads (0.5 + 1.05 GB) exceed the 129 MB L2"),
            "ms_per_step_percentiles": per_step, "transient": transient,
            "tflops": tflops, "frac_of_bf16_peak": {"burst": tflops / peaks["bf16_tflops"],
                                                     "sustained": tflops / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]),
                                                     "source": src},
            "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "peak_kind": peak_kind,
                         "sm_mhz_median": (clocks or {}).get("sm_mhz"), "traffic": None},
            "stages": {k: {"ms_per_step": v[0] / args.steps, "launches_per_step": v[1] / args.steps}
                       for k, v in stages.items() if v[1] > 0},
            "gpu_launches": int(sum(v[1] for v in stages.values())) if args.api == "abi" else None, "clocks": clocks, "e2e": e2e}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_subprocess(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.op == "jsd":
        run_jsd(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
