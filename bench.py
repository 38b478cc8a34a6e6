"""Benchmark of the KDA hot path on GB300.

One step = one pass of the whole path over one batch: the chunk table,
forward (saving for the backward) and backward of the 300M-shape layer call
(B=16, T=2048, H=8, dk=32, dv=64, bf16 inputs, fp32 state), i.e.
kda_fwd + kda_bwd through the C ABI.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launch stream; between steps a 512 MiB buffer is written so that the
L2 (129 MB on GB300) is flushed before every timed step.  Under torchrun each
rank runs its own batch (weak scaling, no collective on the data path); the
reported time is the max over ranks.  The line also carries the same step
with L2 left warm and the step captured once as a CUDA graph and replayed.

--impl reference times the plain CPU oracle (the only other implementation
of the method here) on the host cores, one full workload per step.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from kimi_delta_attention_bwd_gb300.inputs import BASE_SEED, WORKLOADS, custom, make_inputs, numpy_f64  # noqa: E402

METRIC = "KDA fwd and fwd+bwd tokens/s on 1 GB300 at 300M shape; % of roofline"
STEP_WORKLOAD = 3   # fwd+bwd training step at the 300M layer shape
FWD_WORKLOAD = 1    # forward only at the same shape
VARLEN_WORKLOAD = 2  # forward of one packed row of 32768 tokens (log-normal documents)
LARGE_WORKLOAD = 4   # fwd+bwd at dk = dv = 128, 16 heads, packed documents with states
PROFILES = os.path.join(ROOT, "profiles")


def algorithmic_bytes(w, kernel: str) -> float:
    """Algorithmic bytes one launch of `kernel` must move for workload w: each
    input it needs read once, each output it produces written once (bf16 io,
    fp32 parameters); per-chunk states and workspace are not counted."""
    e = 2 if w.dtype == "bf16" else 4
    th = w.B * w.T * w.H  # token-heads
    dk, dv = w.dk, w.dv
    inputs_fwd = e * (3 * dk + dv + 1)         # q, k, f, v, b
    grads = e * (3 * dk + dv + 1)               # dq, dk, df, dv, db
    per = {
        "fwd_chain": inputs_fwd + e * dv,       # reads q, k, f, v, b; writes o
        "fwd_chunk": inputs_fwd,                # reads q, k, f, v, b
        "fwd_state": e * dv,                    # writes o
        "fwd_intra": inputs_fwd,
        "fwd_scan": e * dv,                     # o
        "bwd_scan": e * dv,                     # dO (general path)
        "bwd_x": e * dv,                        # reads dO
        "bwd_grad": e * (dk + dv + 1) + e * dv + e * (dv + 1),  # reads k, f, v, b, dO; writes dv, db
        "bwd_gate": e * 3 * dk + e * 3 * dk,    # reads q, k, f; writes dq, dk, df
        "bwd_intra": inputs_fwd + e * dv + grads,
    }
    return float(per.get(kernel, 0)) * th


def step_bytes(w, backward=True, n_docs=None) -> float:
    """Algorithmic bytes of one step: every per-token input read once and
    every output written once (forward: q, k, f, v, b in, o out; backward:
    the same inputs and dO in, dq, dk, df, dv, db out), plus the fp32 states
    the workload carries (h0 in and h_final out; dh_final in and dh0 out)."""
    e = 2 if w.dtype == "bf16" else 4
    th = w.B * w.T * w.H
    fwd = e * (3 * w.dk + 2 * w.dv + 1)
    bwd = e * (3 * w.dk + 2 * w.dv + 1) + e * (3 * w.dk + w.dv + 1)
    states = 0
    if w.h0:
        states += 2 * (n_docs or w.B) * w.H * w.dk * w.dv * 4
    if backward and w.dh_final:
        states += 2 * (n_docs or w.B) * w.H * w.dk * w.dv * 4
    return float(th * (fwd + (bwd if backward else 0)) + states)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU baseline."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# Sources of the tensor-core kernels: their translation unit with its headers,
# and the host code that lays out their workspace and launches them.  A
# profile taken on these files stays valid while they are unchanged.
TC_SOURCES = ("kda_api.cu", "kda_fast.cu", "kda_internal.cuh", "kda_mma.cuh", "kda_tc.cuh")


def source_sha(files=None) -> str:
    """sha256 (16 hex digits) over the named kernel source files (default: all of csrc)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kimi_delta_attention_bwd_gb300", "csrc")
    for f in sorted(files or os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when absent or taken on different kernel sources (the entry names
    the source files its hash covers)."""
    p = os.path.join(PROFILES, "ncu_traffic.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    e = d.get(kernel)
    if not e or e.get("source_sha") != source_sha(e.get("source_files")):
        return None
    return e.get("bytes_per_launch")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            m = json.load(fh)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- oracle arm
def cpu_oracle_step(x, w):
    from oracle import oracle
    oracle.forward(x)
    if w.backward:
        oracle.backward(x, x["dO"], x.get("dh_final"))


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    w = WORKLOADS[STEP_WORKLOAD]
    x = numpy_f64(make_inputs(w))
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):
        cpu_oracle_step(x, w)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_oracle_step(x, w)
    el = time.perf_counter() - t0
    ms = 1e3 * el / max(1, args.steps)
    val = w.tokens / (ms / 1e3)
    line = {"metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, shapes of the 300M KDA layer)",
            "impl": "reference",
            "config": {"workload": w.name, "global_batch": w.B, "seq_len": w.T, "heads": w.H, "dk": w.dk,
                       "dv": w.dv, "parallelism": "single process, host cores"},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"each step = the full workload ({w.B}x{w.T} tokens x {w.H} heads, "
                                       "forward + backward) on the CPU oracle, threaded over (row, head)"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def cpu_baseline(min_seconds=10.0, max_reps=200):
    """The oracle as it stands on the host cores: full workload steps
    repeated until at least `min_seconds` have elapsed (a bounded sample of
    about 10 s of CPU work)."""
    w = WORKLOADS[STEP_WORKLOAD]
    x = numpy_f64(make_inputs(w))
    cpu_oracle_step(x, w)  # first touch of the output pages
    reps = 0
    t0 = time.perf_counter()
    while reps < max_reps:
        cpu_oracle_step(x, w)
        reps += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    el = time.perf_counter() - t0
    return {"value": reps * w.tokens / el, "unit": "tokens/s", "cores": os.cpu_count() or 1, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{reps} full workload steps ({w.B}x{w.T} tokens x {w.H} heads, fwd+bwd) in {el:.1f} s, "
                      "threaded over (row, head) units"}


# --------------------------------------------------------------- GPU arm
def make_step(w, inp, dev):
    from kimi_delta_attention_bwd_gb300 import _lib, kda_backward, kda_forward
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    prob = _lib.make_problem(w.B, w.T, w.H, w.dk, w.dv, w.torch_dtype, d["scale"], d.get("cu_seqlens"), None)
    ws = _lib.alloc_workspace(prob, w.backward, dev)
    o = torch.empty(w.B, w.T, w.H, w.dv, dtype=w.torch_dtype, device=dev)
    grads = None
    if w.backward:
        grads = {"dq": torch.empty_like(d["q"]), "dk": torch.empty_like(d["k"]), "dv": torch.empty_like(d["v"]),
                 "df": torch.empty_like(d["f"]), "db": torch.empty_like(d["b"]),
                 "dA_log": torch.empty(w.H, device=dev), "ddt_bias": torch.empty(w.H, w.dk, device=dev),
                 "dh0": None}

    n_docs = w.B if d.get("cu_seqlens") is None else int(d["cu_seqlens"].numel()) - 1
    if grads is not None and w.dh_final:
        grads["dh0"] = torch.empty(n_docs, w.H, w.dk, w.dv, device=dev)
    hf = torch.empty(n_docs, w.H, w.dk, w.dv, device=dev) if w.h0 else None

    def step():
        _, _, ctx = kda_forward(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"],
                                scale=d["scale"], h0=d.get("h0"), cu_seqlens=d.get("cu_seqlens"),
                                save_for_backward=w.backward, workspace=ws, out=o, want_final_state=w.h0,
                                final_state=hf)
        if w.backward:
            kda_backward(ctx, d["dO"], d.get("dh_final"), grads=grads)
    return step, d, grads


def workload_bench(wi, args, dev, flush, world, stream, hbm, rank, w=None):
    """One workload's step (forward, or forward + backward) timed as launched,
    then a second pass with per-kernel event brackets for the split and the
    dominant kernel's roofline.  w: a variant of workload wi (its inputs drawn
    with wi's seed)."""
    from kimi_delta_attention_bwd_gb300 import _lib
    w = WORKLOADS[wi] if w is None else w
    inp = make_inputs(w, seed=BASE_SEED + wi + 1000 * rank)
    n_docs = w.B if inp.get("cu_seqlens") is None else int(inp["cu_seqlens"].numel()) - 1
    step, _, _ = make_step(w, inp, dev)
    ms = max_over_ranks(time_steps(step, args.steps, args.warmup, flush, world, stream), world, dev)
    _lib.prof_start()
    time_steps(step, args.steps, 0, flush, world, stream)
    prof = _lib.prof_stop()
    del step
    torch.cuda.empty_cache()
    sb = step_bytes(w, w.backward, n_docs)
    dom = max(prof, key=lambda k: prof[k][0])
    dom_ms = prof[dom][0] / max(1, prof[dom][1])
    ab = algorithmic_bytes(w, dom)
    return {"value": world * w.tokens / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "workload": w.name,
            "roofline": {"bound": "hbm", "algorithmic_bytes": sb, "achieved": sb / (ms / 1e3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": sb / (ms / 1e3) / 1e9 / hbm},
            "dominant_kernel": {"kernel": dom, "launch_ms": dom_ms, "algorithmic_bytes_per_launch": ab,
                                "achieved": ab / (dom_ms / 1e3) / 1e9, "frac": ab / (dom_ms / 1e3) / 1e9 / hbm,
                                "traffic": ncu_traffic(dom)},
            "kernels_ms_per_step": {k: v[0] / args.steps for k, v in prof.items() if v[1]}}


DECODE_SEQS = 2048  # concurrent sequences of the decode step (fp32 state 134 MB, larger than L2)


def decode_bench(args, dev, flush, world, stream, hbm, rank):
    """Single-token step of DECODE_SEQS sequences at the 300M head shape."""
    from kimi_delta_attention_bwd_gb300 import kda_decode_step
    w = WORKLOADS[STEP_WORKLOAD]
    n, H, dk, dv = DECODE_SEQS, w.H, w.dk, w.dv
    inp = make_inputs(custom(n, 1, H, dk, dv, dtype="bf16", h0=True), seed=BASE_SEED + 77 + 1000 * rank,
                      with_grad_inputs=False)
    d = {k: (t.to(dev) if isinstance(t, torch.Tensor) else t) for k, t in inp.items()}
    q, k, v, f, b = (d[x][:, 0].contiguous() for x in ("q", "k", "v", "f", "b"))
    state = d["h0"].clone()
    o = torch.empty(n, H, dv, dtype=torch.bfloat16, device=dev)

    def step():
        kda_decode_step(q, k, v, f, b, d["A_log"], d["dt_bias"], state, scale=d["scale"], out=o)

    ms = max_over_ranks(time_steps(step, args.steps, args.warmup, flush, world, stream), world, dev)
    nbytes = n * H * (2 * dk * dv * 4 + 2 * (3 * dk + 2 * dv + 1))  # state in + out, q k f v o b
    achieved = nbytes / (ms / 1e3) / 1e9
    return {"value": world * n / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "workload": f"decode step, {n} sequences x {H} heads, {dk}/{dv}, bf16 io, fp32 state",
            "roofline": {"bound": "hbm", "kernel": "decode", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "algorithmic_bytes_per_launch": nbytes, "launch_ms": ms}}


def norm_gate_bench(args, dev, flush, world, stream, hbm, rank):
    """Gated RMSNorm epilogue forward and backward over the 300M layer's KDA
    output (16 x 2048 tokens x 8 heads rows of dv = 64, bf16)."""
    from kimi_delta_attention_bwd_gb300 import kda_norm_gate, kda_norm_gate_backward
    from kimi_delta_attention_bwd_gb300.inputs import norm_gate_inputs
    w = WORKLOADS[STEP_WORKLOAD]
    n, dv = w.B * w.T * w.H, w.dv
    d = {k: t.to(dev) for k, t in norm_gate_inputs(n, dv, "bf16", seed=BASE_SEED + 78 + 1000 * rank).items()}
    y = torch.empty_like(d["x"])
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    fwd_ms = max_over_ranks(time_steps(lambda: kda_norm_gate(d["x"], d["g"], d["w"], out=y), args.steps, args.warmup,
                                       flush, world, stream), world, dev)
    bwd_ms = max_over_ranks(time_steps(lambda: kda_norm_gate_backward(d["x"], d["g"], d["w"], d["dy"], workspace=ws),
                                       args.steps, args.warmup, flush, world, stream), world, dev)
    fb, bb = n * 3 * dv * 2, n * 5 * dv * 2  # x, g in, y out; x, g, dy in, dx, dg out
    return {"workload": f"gated RMSNorm epilogue, {n} rows x {dv}, bf16", "unit": "tokens/s",
            "fwd": {"value": world * w.tokens / (fwd_ms / 1e3), "ms_per_step": fwd_ms,
                    "roofline": {"bound": "hbm", "achieved": fb / (fwd_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                                 "frac": fb / (fwd_ms / 1e3) / 1e9 / hbm, "algorithmic_bytes_per_launch": fb}},
            "bwd": {"value": world * w.tokens / (bwd_ms / 1e3), "ms_per_step": bwd_ms,
                    "roofline": {"bound": "hbm", "achieved": bb / (bwd_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                                 "frac": bb / (bwd_ms / 1e3) / 1e9 / hbm, "algorithmic_bytes_per_launch": bb}}}


def short_conv_bench(args, dev, flush, world, stream, hbm, rank):
    """Short causal conv (width 4, silu) on the 300M layer's concatenated
    q | k | v (16 x 2048 tokens x C = H (2 dk + dv) = 1024 channels, bf16)."""
    from kimi_delta_attention_bwd_gb300 import _lib, kda_short_conv, kda_short_conv_backward
    from kimi_delta_attention_bwd_gb300.inputs import short_conv_inputs
    w = WORKLOADS[STEP_WORKLOAD]
    n, C = w.B * w.T, w.H * (2 * w.dk + w.dv)
    d = {k: t.to(dev) for k, t in short_conv_inputs(n, C, "bf16", seed=BASE_SEED + 79 + 1000 * rank).items()}
    y = torch.empty_like(d["x"])
    ws = torch.empty(_lib.kda_short_conv_workspace_size(n, C), dtype=torch.uint8, device=dev)
    fwd_ms = max_over_ranks(time_steps(lambda: kda_short_conv(d["x"], d["w"], out=y), args.steps, args.warmup,
                                       flush, world, stream), world, dev)
    bwd_ms = max_over_ranks(time_steps(lambda: kda_short_conv_backward(d["x"], d["w"], d["dy"], workspace=ws),
                                       args.steps, args.warmup, flush, world, stream), world, dev)
    fb, bb = n * C * 2 * 2, n * C * 3 * 2  # x in, y out; x, dy in, dx out
    return {"workload": f"short causal conv width 4 + silu, {n} tokens x {C} channels, bf16", "unit": "tokens/s",
            "fwd": {"value": world * n / (fwd_ms / 1e3), "ms_per_step": fwd_ms,
                    "roofline": {"bound": "hbm", "achieved": fb / (fwd_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                                 "frac": fb / (fwd_ms / 1e3) / 1e9 / hbm, "algorithmic_bytes_per_launch": fb}},
            "bwd": {"value": world * n / (bwd_ms / 1e3), "ms_per_step": bwd_ms,
                    "roofline": {"bound": "hbm", "achieved": bb / (bwd_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                                 "frac": bb / (bwd_ms / 1e3) / 1e9 / hbm, "algorithmic_bytes_per_launch": bb}}}


def fused_norm_bench(args, dev, flush, world, stream, hbm, rank):
    """KDA with the gated RMSNorm epilogue at the 300M layer shape: the fused
    entry points (kda_fwd_norm_gate + kda_bwd_norm_gate) against the same work
    composed of four calls (kda_fwd, kda_norm_gate_fwd, kda_norm_gate_bwd,
    kda_bwd), forward + backward, and the fused forward alone (inference: no
    save, o never written)."""
    from kimi_delta_attention_bwd_gb300 import (kda_backward, kda_backward_norm_gate, kda_forward,
                                                kda_forward_norm_gate, kda_norm_gate, kda_norm_gate_backward, _lib)
    from kimi_delta_attention_bwd_gb300.inputs import norm_gate_inputs
    w = WORKLOADS[STEP_WORKLOAD]
    inp = make_inputs(w, seed=BASE_SEED + STEP_WORKLOAD + 1000 * rank)
    d = {k: (t.to(dev) if isinstance(t, torch.Tensor) else t) for k, t in inp.items()}
    shape = (w.B, w.T, w.H, w.dv)
    ng = norm_gate_inputs(w.B * w.T * w.H, w.dv, "bf16", seed=BASE_SEED + 80 + 1000 * rank)
    g, wn, dy = ng["g"].reshape(shape).to(dev), ng["w"].to(dev), ng["dy"].reshape(shape).to(dev)
    prob = _lib.make_problem(w.B, w.T, w.H, w.dk, w.dv, w.torch_dtype, d["scale"])
    ws2 = _lib.alloc_workspace(prob, 2, dev)
    ws1 = _lib.alloc_workspace(prob, 1, dev)
    ws0 = _lib.alloc_workspace(prob, 0, dev)
    nws = torch.empty(_lib.kda_norm_gate_workspace_size(w.B * w.T * w.H, w.dv), dtype=torch.uint8, device=dev)
    x = (d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"])

    def fused():
        _, _, _, ctx = kda_forward_norm_gate(*x, g, wn, scale=d["scale"], workspace=ws2, want_final_state=False)
        kda_backward_norm_gate(ctx, dy, want_dh0=False)

    def composed():
        o, _, ctx = kda_forward(*x, scale=d["scale"], workspace=ws1, want_final_state=False)
        kda_norm_gate(o, g, wn)
        do, _, _ = kda_norm_gate_backward(o, g, wn, dy, workspace=nws)
        kda_backward(ctx, do, want_dh0=False)

    def fused_fwd():
        kda_forward_norm_gate(*x, g, wn, scale=d["scale"], workspace=ws0, save_for_backward=False,
                              want_final_state=False)

    def composed_fwd():
        o, _, _ = kda_forward(*x, scale=d["scale"], workspace=ws0, save_for_backward=False, want_final_state=False)
        kda_norm_gate(o, g, wn)

    res = {}
    for name, fn, back in (("fused_step", fused, True), ("composed_step", composed, True),
                           ("fused_fwd", fused_fwd, False), ("composed_fwd", composed_fwd, False)):
        ms = max_over_ranks(time_steps(fn, args.steps, args.warmup, flush, world, stream), world, dev)
        # algorithmic bytes: the KDA step's, plus g read and y written (and, backward, g and dy read, dg written)
        nb = step_bytes(w, back) + w.B * w.T * w.H * w.dv * 2 * (2 + (3 if back else 0))
        res[name] = {"value": world * w.tokens / (ms / 1e3), "ms_per_step": ms,
                     "roofline": {"bound": "hbm", "algorithmic_bytes": nb, "achieved": nb / (ms / 1e3) / 1e9,
                                  "peak": hbm, "unit": "GB/s", "frac": nb / (ms / 1e3) / 1e9 / hbm}}
    _lib.prof_start()
    time_steps(fused, args.steps, 0, flush, world, stream)
    prof = _lib.prof_stop()
    res["fused_kernels_ms_per_step"] = {k: v[0] / args.steps for k, v in prof.items() if v[1]}
    res["workload"] = f"{w.name} with the gated RMSNorm epilogue (g, dy ~ N(0,1) bf16, w ~ 1 + 0.1 N(0,1))"
    res["unit"] = "tokens/s"
    del ws0, ws1, ws2
    torch.cuda.empty_cache()
    return res


def fused_conv_bench(args, dev, flush, world, stream, hbm, rank):
    """The layer at the 300M shape: short conv (width 4, silu) on the q | k | v
    projection, KDA, gated RMSNorm, forward + backward.  Fused: kda_fwd_conv +
    kda_bwd_conv (the convolution applied to the rows the per-chunk kernels
    load, the norm inside the chains).  Composed: the standalone convolution
    on each of the q, k, v blocks, kda_fwd, kda_norm_gate_fwd; then
    kda_norm_gate_bwd, kda_bwd and the convolution's backward."""
    from kimi_delta_attention_bwd_gb300 import (kda_backward, kda_backward_conv, kda_forward, kda_forward_conv,
                                                kda_norm_gate, kda_norm_gate_backward, kda_short_conv,
                                                kda_short_conv_backward, _lib)
    from kimi_delta_attention_bwd_gb300.inputs import norm_gate_inputs, short_conv_inputs
    w = WORKLOADS[STEP_WORKLOAD]
    inp = make_inputs(w, seed=BASE_SEED + STEP_WORKLOAD + 1000 * rank)
    d = {k: (t.to(dev) if isinstance(t, torch.Tensor) else t) for k, t in inp.items()}
    N, H, dk, dv = w.B * w.T, w.H, w.dk, w.dv
    C = H * (2 * dk + dv)
    cv = short_conv_inputs(N, C, "bf16", seed=BASE_SEED + 81 + 1000 * rank)
    x, cw = cv["x"].reshape(w.B, w.T, C).to(dev), cv["w"].to(dev)
    xq, xk, xv = (x[..., a:b].contiguous() for a, b in ((0, H * dk), (H * dk, 2 * H * dk), (2 * H * dk, C)))
    cwq, cwk, cwv = cw[:H * dk].contiguous(), cw[H * dk:2 * H * dk].contiguous(), cw[2 * H * dk:].contiguous()
    shape = (w.B, w.T, H, dv)
    ng = norm_gate_inputs(N * H, dv, "bf16", seed=BASE_SEED + 82 + 1000 * rank)
    g, wn, dy = ng["g"].reshape(shape).to(dev), ng["w"].to(dev), ng["dy"].reshape(shape).to(dev)
    prob = _lib.make_problem(w.B, w.T, H, dk, dv, w.torch_dtype, d["scale"])
    ws3 = _lib.alloc_workspace(prob, 3, dev)
    ws1 = _lib.alloc_workspace(prob, 1, dev)
    cu_rows = torch.arange(0, (w.B + 1) * w.T, w.T, dtype=torch.int32, device=dev)  # the rows are the documents

    def fused():
        _, _, ctx = kda_forward_conv(x, cw, d["f"], d["b"], d["A_log"], d["dt_bias"], dk, dv, g=g, w=wn,
                                     scale=d["scale"], workspace=ws3, want_final_state=False)
        kda_backward_conv(ctx, dy, want_dh0=False)

    def composed():
        q = kda_short_conv(xq.view(N, -1), cwq, cu_rows).view(w.B, w.T, H, dk)
        k = kda_short_conv(xk.view(N, -1), cwk, cu_rows).view(w.B, w.T, H, dk)
        v = kda_short_conv(xv.view(N, -1), cwv, cu_rows).view(w.B, w.T, H, dv)
        o, _, ctx = kda_forward(q, k, v, d["f"], d["b"], d["A_log"], d["dt_bias"], scale=d["scale"], workspace=ws1,
                                want_final_state=False)
        kda_norm_gate(o, g, wn)
        do, _, _ = kda_norm_gate_backward(o, g, wn, dy)
        gr = kda_backward(ctx, do, want_dh0=False)
        kda_short_conv_backward(xq.view(N, -1), cwq, gr["dq"].view(N, -1), cu_rows)
        kda_short_conv_backward(xk.view(N, -1), cwk, gr["dk"].view(N, -1), cu_rows)
        kda_short_conv_backward(xv.view(N, -1), cwv, gr["dv"].view(N, -1), cu_rows)

    res = {}
    nb = step_bytes(w, True) + N * H * dv * 2 * 5  # the KDA step's bytes, x counted as q | k | v; g, y, dy, dg
    for name, fn in (("fused_step", fused), ("composed_step", composed)):
        ms = max_over_ranks(time_steps(fn, args.steps, args.warmup, flush, world, stream), world, dev)
        res[name] = {"value": world * w.tokens / (ms / 1e3), "ms_per_step": ms,
                     "roofline": {"bound": "hbm", "algorithmic_bytes": nb, "achieved": nb / (ms / 1e3) / 1e9,
                                  "peak": hbm, "unit": "GB/s", "frac": nb / (ms / 1e3) / 1e9 / hbm}}
    _lib.prof_start()
    time_steps(fused, args.steps, 0, flush, world, stream)
    prof = _lib.prof_stop()
    res["fused_kernels_ms_per_step"] = {k: v[0] / args.steps for k, v in prof.items() if v[1]}
    res["workload"] = f"{w.name}: short conv (x [{N}, {C}] bf16, taps ~ N(0, 0.25)) -> KDA -> gated RMSNorm"
    res["unit"] = "tokens/s"
    del ws1, ws3
    torch.cuda.empty_cache()
    return res


def time_steps(step, steps, warmup, flush, world, stream):
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return sum(a.elapsed_time(b) for a, b in evs) / steps


def graph_replay(step, stream):
    """Captures one step in a CUDA graph (after two eager warm-up steps on a
    side stream) and returns the callable that replays it on `stream`."""
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
        step()
    stream.wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    torch.cuda.synchronize()
    return g.replay


def e2e_pipelined(host, outs_host, d, ws, steps, warmup, world):
    """End to end through the public API, pipelined over three streams: every
    step copies its inputs from pinned host memory into one of two device
    input sets (copy-in stream), runs kda_forward + kda_backward into one of
    two gradient sets (compute stream) and reads every gradient back into
    pinned host memory (copy-out stream).  Events order each set's reuse, so
    step i+1's copy-in and step i-1's copy-out overlap step i's compute.
    Returns milliseconds per step over `steps` steps."""
    from kimi_delta_attention_bwd_gb300 import kda_backward, kda_forward
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    dev_in = [{k: torch.empty_like(d[k]) for k in host} for _ in range(2)]
    gd = [{k: torch.empty_like(d[k2]) for k, k2 in (("dq", "q"), ("dk", "k"), ("dv", "v"), ("df", "f"), ("db", "b"))}
          for _ in range(2)]
    for g in gd:
        g["dA_log"] = torch.empty_like(d["A_log"])
        g["ddt_bias"] = torch.empty_like(d["dt_bias"])
        g["dh0"] = None
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "cmp", "out")}

    def issue(i):
        p = i % 2
        if i >= 2:
            s_in.wait_event(ev["cmp"][p])  # step i - 2's compute has read this input set
            s_cmp.wait_event(ev["out"][p])  # and its copy-out has read this gradient set
        with torch.cuda.stream(s_in):
            for k in host:
                dev_in[p][k].copy_(host[k], non_blocking=True)
            ev["in"][p].record(s_in)
        s_cmp.wait_event(ev["in"][p])
        with torch.cuda.stream(s_cmp):
            x = dev_in[p]
            _, _, ctx = kda_forward(x["q"], x["k"], x["v"], x["f"], x["b"], x["A_log"], x["dt_bias"],
                                    scale=d["scale"], workspace=ws, want_final_state=False)
            kda_backward(ctx, x["dO"], None, want_dh0=False, grads=gd[p])
            ev["cmp"][p].record(s_cmp)
        s_out.wait_event(ev["cmp"][p])
        with torch.cuda.stream(s_out):
            for k in outs_host:
                outs_host[k].copy_(gd[p][k], non_blocking=True)
            ev["out"][p].record(s_out)

    cur = torch.cuda.current_stream()
    for i in range(warmup):
        issue(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(cur)
    for st in (s_in, s_cmp, s_out):
        st.wait_event(t0)
    for i in range(steps):
        issue(warmup + i)
    for st in (s_in, s_cmp, s_out):
        cur.wait_stream(st)
    t1.record(cur)
    torch.cuda.synchronize()
    barrier(world)
    return t0.elapsed_time(t1) / steps


def run_ours(args, rank, world, local):
    from kimi_delta_attention_bwd_gb300 import _lib
    from kimi_delta_attention_bwd_gb300.build import build
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    build()
    _lib.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    hbm, tflops, peak_kind = peaks()

    # forward-only at the same shape, the packed varlen forward and the large-head training step
    fwd = workload_bench(FWD_WORKLOAD, args, dev, flush, world, stream, hbm, rank)
    varlen = workload_bench(VARLEN_WORKLOAD, args, dev, flush, world, stream, hbm, rank)
    # the same packed row as a training step (with dO): both chains split on its long document
    vw = dataclasses.replace(WORKLOADS[VARLEN_WORKLOAD], backward=True,
                             name="varlen fwd+bwd, 1x32768 packed, H8, 32/64, bf16")
    varlen_step = workload_bench(VARLEN_WORKLOAD, args, dev, flush, world, stream, hbm, rank, w=vw)
    large = workload_bench(LARGE_WORKLOAD, args, dev, flush, world, stream, hbm, rank)
    dec = decode_bench(args, dev, flush, world, stream, hbm, rank)
    torch.cuda.empty_cache()
    ngate = norm_gate_bench(args, dev, flush, world, stream, hbm, rank)
    torch.cuda.empty_cache()
    sconv = short_conv_bench(args, dev, flush, world, stream, hbm, rank)
    torch.cuda.empty_cache()
    fnorm = fused_norm_bench(args, dev, flush, world, stream, hbm, rank)
    fconv = fused_conv_bench(args, dev, flush, world, stream, hbm, rank)

    # the training step (timed region with per-kernel event brackets and clock sampling)
    w = WORKLOADS[STEP_WORKLOAD]
    step, d, grads = make_step(w, make_inputs(w, seed=BASE_SEED + STEP_WORKLOAD + 1000 * rank), dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms = time_steps(step, args.steps, 0, flush, world, stream)  # as launched: dependent launches overlap
    clk = clocks.stop()
    # the per-kernel split from a second pass with CUDA-event brackets around every launch (the
    # brackets serialise the kernel boundaries, so their sum exceeds the step above)
    _lib.prof_start()
    time_steps(step, args.steps, 0, flush, world, stream)
    prof = _lib.prof_stop()
    ms = max_over_ranks(ms, world, dev)
    # secondary figures: the same step with L2 left warm, and replayed as one CUDA graph (flushed)
    warm_ms = max_over_ranks(time_steps(step, args.steps, 0, None, world, stream), world, dev)
    replay = graph_replay(step, stream)
    graph_ms = max_over_ranks(time_steps(replay, args.steps, args.warmup, flush, world, stream), world, dev)
    del replay
    value = world * w.tokens / (ms / 1e3)
    launches = int(sum(c for _, c in prof.values()))
    dom = max(prof, key=lambda k: prof[k][0])
    dom_ms = prof[dom][0] / max(1, prof[dom][1])
    ab = algorithmic_bytes(w, dom)
    achieved = ab / (dom_ms / 1e3) / 1e9
    traffic = ncu_traffic(dom)

    # end to end through the public API with host buffers
    from kimi_delta_attention_bwd_gb300 import kda_backward, kda_forward
    host = {k: d[k].cpu().pin_memory() for k in ("q", "k", "v", "f", "b", "dO", "A_log", "dt_bias")}
    dev_in = {k: torch.empty_like(d[k]) for k in host}
    outs_host = {k: torch.empty(grads[k].shape, dtype=grads[k].dtype).pin_memory()
                 for k in ("dq", "dk", "dv", "df", "db", "dA_log", "ddt_bias")}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs_host.values())
    from kimi_delta_attention_bwd_gb300 import _lib as L
    prob = L.make_problem(w.B, w.T, w.H, w.dk, w.dv, w.torch_dtype, d["scale"], None, None)
    ws = L.alloc_workspace(prob, True, dev)

    def e2e_step():
        for k in host:
            dev_in[k].copy_(host[k], non_blocking=True)
        _, _, ctx = kda_forward(dev_in["q"], dev_in["k"], dev_in["v"], dev_in["f"], dev_in["b"], dev_in["A_log"],
                                dev_in["dt_bias"], scale=d["scale"], workspace=ws, want_final_state=False)
        g = kda_backward(ctx, dev_in["dO"], None, want_dh0=False)
        for k in outs_host:
            outs_host[k].copy_(g[k], non_blocking=True)
    e2e_serial_ms = max_over_ranks(time_steps(e2e_step, args.steps, args.warmup, flush, world, stream), world, dev)
    e2e_ms = max_over_ranks(e2e_pipelined(host, outs_host, d, ws, args.steps, args.warmup, world), world, dev)

    cpu = cpu_baseline() if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, shapes of the 300M KDA layer)",
            "config": {"workload": w.name, "global_batch": w.B * world, "seq_len": w.T, "heads": w.H,
                       "dk": w.dk, "dv": w.dv, "parallelism": f"dp{world} (independent batches per GPU)",
                       "l2": "flushed between timed steps (512 MiB write)"},
            "fwd_value": fwd["value"], "fwd_roofline_frac": fwd["roofline"]["frac"],
            "fwd": fwd,
            "varlen_fwd": varlen,
            "varlen_step": varlen_step,
            "large_head_step": large,
            "decode": dec,
            "norm_gate": ngate,
            "norm_gate_fused": fnorm,
            "conv_norm_layer": fconv,
            "short_conv": sconv,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": traffic, "peak_kind": peak_kind,
                         "algorithmic_bytes_per_launch": ab, "launch_ms": dom_ms},
            "step_roofline": {"bound": "hbm", "algorithmic_bytes": step_bytes(w),
                              "achieved": step_bytes(w) / (ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                              "frac": step_bytes(w) / (ms / 1e3) / 1e9 / hbm},
            "secondary": {"warm_l2_ms_per_step": warm_ms, "cuda_graph_ms_per_step": graph_ms,
                          "note": "warm: no L2 flush between steps; cuda_graph: the step captured once and "
                                  "replayed, L2 flushed"},
            "kernels_ms_per_step": {k: v[0] / args.steps for k, v in prof.items() if v[1]},
            "gpu_launches": launches,
            "clocks": clk,
            "e2e": {"value": world * w.tokens / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "pipelined": "copy-in, compute and copy-out streams, two device input / gradient sets: step "
                                 "i+1's inputs and step i-1's gradients travel while step i computes",
                    "serial_ms_per_step": e2e_serial_ms},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    return 0


def ncu_pass(rows: int = 16):
    """One untimed pass for profiler captures (select launches with ncu's -k /
    -s / -c): a warm-up forward+backward of the bench step's workload, the same
    forward+backward again, then one decode step, the gated norm forward and
    backward, the short convolution forward and backward, one forward+backward
    with the gated norm fused into the chains (kda_fwd_norm_gate /
    kda_bwd_norm_gate), one of the fused layer (kda_fwd_conv / kda_bwd_conv
    with the norm) and one forward+backward of the packed varlen row (1 x 32768
    tokens, whose long document splits both chains: fwd_seg, bwd_seg), in that
    order.  rows < 16 runs the 300M step workloads on that many 2048-token rows
    (a smaller case for multi-pass captures); the varlen row stays whole."""
    from kimi_delta_attention_bwd_gb300 import (kda_backward, kda_backward_conv, kda_backward_norm_gate,
                                                kda_decode_step, kda_forward, kda_forward_conv,
                                                kda_forward_norm_gate, kda_norm_gate, kda_norm_gate_backward,
                                                kda_short_conv, kda_short_conv_backward)
    from kimi_delta_attention_bwd_gb300.inputs import norm_gate_inputs, short_conv_inputs
    dev = torch.device("cuda", 0)
    w = WORKLOADS[STEP_WORKLOAD]
    if rows != w.B:
        w = custom(rows, w.T, w.H, w.dk, w.dv, dtype=w.dtype, name=f"{rows}x{w.T} rows of the 300M layer")
    d = {k: (t.to(dev) if isinstance(t, torch.Tensor) else t) for k, t in make_inputs(w).items()}
    for _ in range(2):
        o, hf, ctx = kda_forward(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"], scale=d["scale"])
        kda_backward(ctx, d["dO"])
    di = {k: (t.to(dev) if isinstance(t, torch.Tensor) else t)
          for k, t in make_inputs(custom(DECODE_SEQS, 1, w.H, w.dk, w.dv, dtype="bf16", h0=True),
                                  with_grad_inputs=False).items()}
    state = di["h0"].clone()
    kda_decode_step(*(di[x][:, 0].contiguous() for x in ("q", "k", "v", "f", "b")), di["A_log"], di["dt_bias"], state,
                    scale=di["scale"])
    ng = {k: t.to(dev) for k, t in norm_gate_inputs(w.B * w.T * w.H, w.dv).items()}
    kda_norm_gate(ng["x"], ng["g"], ng["w"])
    kda_norm_gate_backward(ng["x"], ng["g"], ng["w"], ng["dy"])
    sc = {k: t.to(dev) for k, t in short_conv_inputs(w.B * w.T, 1024).items()}
    kda_short_conv(sc["x"], sc["w"])
    kda_short_conv_backward(sc["x"], sc["w"], sc["dy"])
    shape = (w.B, w.T, w.H, w.dv)
    _, _, _, nctx = kda_forward_norm_gate(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"],
                                          ng["g"].reshape(shape), ng["w"], scale=d["scale"])
    kda_backward_norm_gate(nctx, ng["dy"].reshape(shape))
    _, _, cctx = kda_forward_conv(sc["x"].reshape(w.B, w.T, -1), sc["w"], d["f"], d["b"], d["A_log"], d["dt_bias"],
                                  w.dk, w.dv, g=ng["g"].reshape(shape), w=ng["w"], scale=d["scale"])
    kda_backward_conv(cctx, ng["dy"].reshape(shape))
    vw = dataclasses.replace(WORKLOADS[VARLEN_WORKLOAD], backward=True)
    vi = make_inputs(vw, seed=BASE_SEED + VARLEN_WORKLOAD)
    dv_ = {k: (t.to(dev) if isinstance(t, torch.Tensor) else t) for k, t in vi.items()}
    _, _, vctx = kda_forward(dv_["q"], dv_["k"], dv_["v"], dv_["f"], dv_["b"], dv_["A_log"], dv_["dt_bias"],
                             scale=dv_["scale"], cu_seqlens=dv_["cu_seqlens"],
                             cu_seqlens_host=vi["cu_seqlens"].numpy())
    kda_backward(vctx, dv_["dO"])
    torch.cuda.synchronize()
    print("ncu pass done")
    return 0


def ncu_large_heads():
    """One untimed pass of the general (large-head) kernels for profiler
    captures: a warm-up forward+backward, then the same again, of one 8192-token
    row of the 128/128 packed workload (H 16, log-normal documents of median
    2048, h0 and dS_final, bf16) -- a quarter of that workload, so that a
    multi-pass capture stays small."""
    from kimi_delta_attention_bwd_gb300 import kda_backward, kda_forward
    from kimi_delta_attention_bwd_gb300.inputs import doc_lengths_rows
    dev = torch.device("cuda", 0)
    w = custom(1, 8192, 16, 128, 128, dtype="bf16", h0=True, dh_final=True)
    lens = doc_lengths_rows(1, 8192, 2048.0, np.random.RandomState(BASE_SEED + 4))
    inp = make_inputs(w, seed=BASE_SEED + 4, lengths=lens)
    d = {k: (t.to(dev) if isinstance(t, torch.Tensor) else t) for k, t in inp.items()}
    cu_host = inp["cu_seqlens"].numpy()
    for _ in range(2):
        o, hf, ctx = kda_forward(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"], scale=d["scale"],
                                 h0=d["h0"], cu_seqlens=d["cu_seqlens"], cu_seqlens_host=cu_host)
        kda_backward(ctx, d["dO"], d["dh_final"])
    torch.cuda.synchronize()
    print("ncu large-head pass done:", len(lens), "documents")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu-pass", action="store_true", help="one untimed pass of every kernel, for ncu captures")
    ap.add_argument("--ncu-rows", type=int, default=16, help="rows of the --ncu-pass step workloads (16: full size)")
    ap.add_argument("--ncu-large-heads", action="store_true",
                    help="one untimed pass of the large-head (128/128) kernels, for ncu captures")
    args = ap.parse_args()
    if args.ncu_pass:
        return ncu_pass(args.ncu_rows)
    if args.ncu_large_heads:
        return ncu_large_heads()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    if args.impl == "reference":
        # rank 0 alone times the oracle; the other ranks exit without work
        return run_reference(args, int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")))
    rank, world, local = dist_setup(args.gpus)
    rc = run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
