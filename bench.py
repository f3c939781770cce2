#!/usr/bin/env python3
"""Benchmark of the GB300 Mamba-2 SSD chunked forward.

One step = one SSD forward (all four chunk steps, or the fused kernel) over
one batch of the workload, inputs already resident in HBM.  Metric: tokens/s
(tokens = B*L) and ms per step at the large training shape
[B,L,H,P,N,chunk,G] = [8,4096,256,64,64,64,64] (fp32 public tensors, bf16
operands) unless --workload says otherwise.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle instead, on a bounded sample of the same workload.

Multi-GPU (torchrun, one process per GPU): each rank runs its own replica of
the workload on its own GPU (weak scaling; the path shards by batch and group
with no exchange), timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import signal
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import ssd_inputs  # noqa: E402

METRIC = "SSD fwd ms & tokens/s at [8,4096,256,64,64,64,64] on 1 GB300; % of roofline"
# The reference project's own number for this exact shape (AscendC on Ascend
# 910B3, 31.888 ms, README "Benchmark"): 8*4096 tokens / 31.888 ms.
PUBLISHED_TOKENS_PER_S = {"large_training": 8 * 4096 / 31.888e-3}
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2**20


# ---- helpers ---------------------------------------------------------------------

def rank_info():
    r = int(os.environ.get("RANK", "0"))
    w = int(os.environ.get("WORLD_SIZE", "1"))
    lr = int(os.environ.get("LOCAL_RANK", "0"))
    return r, w, lr


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(w) -> dict:
    """Public I/O of one forward, each tensor read or written once."""
    io = 4 if w.x_dtype == "f32" else 2
    nx = w.B * w.L * w.H * w.P
    nbc = w.B * w.L * w.G * w.N
    nst = w.B * w.H * w.P * w.N
    b = {
        "x": nx * io, "y": nx * io, "B": nbc * io, "C": nbc * io, "dt": w.B * w.L * w.H * 4,
        "params": w.H * 4 * (1 + (w.dt_bias_std is not None) + (w.D_std is not None)),
        "z": nx * io if w.z else 0,
        "h0": nst * 4 if w.h0_std is not None else 0,
        "final_state": nst * 4 if w.return_final_state else 0,
    }
    b["total"] = sum(b.values())
    return b


# fp32 FMA lanes: 152 SMs x 4 sub-partitions x 32 lanes, 2 flops per FMA, at
# the maximum SM clock (2070 MHz): the ceiling of CUDA-core fp32 arithmetic.
SM_COUNT = 152
FP32_LANES_PER_SM = 128
SM_MAX_MHZ = 2070.0


def fp32_alu_peak_tflops():
    try:
        mhz = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["sm_max_mhz"])
    except Exception:
        mhz = SM_MAX_MHZ
    return SM_COUNT * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def bwd_flops(w) -> int:
    """Algorithmic flops of one backward (2 per multiply-add), counting the
    contractions per (batch, head, chunk): the recomputed chunk state (Q P N),
    the adjoint's per-chunk sum (Q P N), C B^T once per group (Q^2 N), dyp x^T
    (Q^2 P), the intra-chunk parts of dx (Q^2 P), dB and dC (Q^2 N each), the
    inter-chunk parts of dx, dB and dC (Q P N each), and with z the recomputed
    pre-gate output (Q^2 N per group, Q^2 P, Q P N).  Elementwise work (decays,
    gate, reductions) is not counted."""
    Q, P, N = w.chunk, w.P, w.N
    hpg = w.H // w.G
    per = 5 * Q * P * N + 2 * Q * Q * P + 2 * Q * Q * N + Q * Q * N / hpg
    if w.z:
        per += Q * Q * N / hpg + Q * Q * P + Q * P * N
    chunks = -(-w.L // w.chunk)
    return int(2 * per * w.B * w.H * chunks)


def stage_bytes(w) -> dict:
    """Compulsory bytes of each chunked-plan kernel (its own inputs read once,
    its own outputs written once)."""
    io = 4 if w.x_dtype == "f32" else 2
    c = -(-w.L // w.chunk)
    nx = w.B * w.L * w.H * w.P
    nbc = w.B * w.L * w.G * w.N
    vec = w.B * w.H * c * w.chunk * 4
    st = w.B * c * w.H * w.P * w.N * 4
    nst = w.B * w.H * w.P * w.N * 4
    return {
        "chunk_cumsum": w.B * w.L * w.H * 4 + 2 * vec,
        "chunk_state": nx * io + nbc * io + 2 * vec + st,
        "state_passing": 2 * st + vec // w.chunk + (nst if w.return_final_state else 0)
        + (nst if w.h0_std is not None else 0),
        "chunk_scan": nx * io * (2 if w.z else 1) + 2 * nbc * io + 2 * vec + st + nx * io,
    }


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, enabled: bool = True):
        self.idx = device_index
        self.enabled = enabled
        self.proc = None
        self.path = None

    def __enter__(self):
        if not self.enabled:
            return self
        fd, self.path = tempfile.mkstemp(prefix="ssd_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.send_signal(signal.SIGTERM)
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def step_quantiles(per_step):
    """Median, 20th and 80th percentile of the per-step event times (ms)."""
    v = sorted(per_step)
    q = lambda f: v[min(len(v) - 1, int(round(f * (len(v) - 1))))]
    return {"median": round(q(0.5), 5), "p20": round(q(0.2), 5), "p80": round(q(0.8), 5)}


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, when the kernel's
    source is unchanged since the counters were taken (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        table = json.load(open(p))
    except Exception:
        return None
    ent = table.get(kernel, {}).get(workload)
    if not ent:
        return None
    src = os.path.join(ROOT, ent["source"])
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except Exception:
        return None
    if sha != ent["source_sha"]:
        return None
    return float(ent["dram_bytes_per_launch"])


# ---- the GPU arm ----------------------------------------------------------------------

def run_gpu(args):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    rank, world, lrank = rank_info()
    dist = None
    if world > 1:
        import torch.distributed as dist  # noqa: F811
        torch.cuda.set_device(lrank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", lrank if world > 1 else 0)
    torch.cuda.set_device(dev)
    w = ssd_inputs.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    inp = ssd_inputs.make(w, seed=w.seed + 1000 * rank)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    fin = torch.empty((w.B, w.H, w.P, w.N), device=dev) if w.return_final_state else None
    a = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk, y=y, final_state=fin,
                      D=d["D"], z=d["z"], dt_bias=d["dt_bias"], initial_states=d["initial_states"],
                      dt_softplus=w.dt_softplus, ops=args.ops or w.ops, plan=args.plan)
    plan = ssd.ssd_fwd_resolve_plan(a)
    fused_note = "taken"
    if plan != ssd.SSD_PLAN_FUSED:  # why the one-kernel plan is not running, in the library's words
        probe = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk, y=y, final_state=fin, D=d["D"],
                              z=d["z"], dt_bias=d["dt_bias"], initial_states=d["initial_states"],
                              dt_softplus=w.dt_softplus, ops=args.ops or w.ops, plan="fused")
        try:
            ssd.ssd_fwd_resolve_plan(probe)
            fused_note = "supported, not chosen" + (" (plan forced)" if args.plan != "auto" else "")
        except ssd.SsdError as exc:
            fused_note = "unavailable: " + exc.detail
    nws = ssd.ssd_fwd_workspace_size(a)
    ws = torch.zeros(max(nws, 256), dtype=torch.uint8, device=dev)
    a.workspace, a.workspace_bytes = ws.data_ptr(), nws
    stream = torch.cuda.current_stream(dev)
    sh = ssd._stream_handle(dev)
    ab = algorithmic_bytes(w)
    in_bytes = ab["x"] + ab["B"] + ab["C"] + ab["dt"] + ab["z"]
    flush = None
    if in_bytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        ssd.ssd_fwd(a, sh)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index, enabled=not args.no_clocks) as clk:
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(float(i))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        if not args.no_clocks:  # keep the sampler alive for a few samples
            extra_until = time.time() + 0.5
            while time.time() < extra_until:
                step()
            torch.cuda.synchronize(dev)
    clocks = clk.summary()
    per_step = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(per_step) / len(per_step)
    if dist:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    tokens = w.tokens * world
    value = tokens / (ms * 1e-3)

    # dominant kernel: time it alone with events on the launching stream
    hbm, peak_kind = peaks()
    kernels = ssd.ssd_fwd_describe(a)
    stages = None
    if plan == ssd.SSD_PLAN_FUSED:
        kname, kbytes, kms = "ssd_fused_kernel", ab["total"], ms
        launches_per_step = len(kernels)
        scope = ("one launch = the whole step" if launches_per_step == 1 else
                 f"whole step ({launches_per_step} launches: {', '.join(kernels)})")
    else:
        # several launches per step: the fraction is the path's algorithmic
        # bytes (public I/O only) over the whole step, the dominant stage named
        kname, _, _, stages = stage_timing(ssd, a, w, dev, sh, stream, args, kernels)
        kbytes, kms = ab["total"], ms
        launches_per_step = len(kernels)
        scope = f"whole step ({launches_per_step} launches; dominant stage {kname}, see stages)"
    achieved = kbytes / (kms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": hbm,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "traffic": traffic_for(kname, args.workload) if launches_per_step == 1 else None,
                "alg_bytes_per_launch": kbytes, "launch_ms": round(kms, 5), "scope": scope}
    path_roofline_ms = ab["total"] / (hbm * 1e9) * 1e3

    e2e = e2e_timing(ssd, inp, w, dev, args) if not args.no_e2e else None

    ops_name = {0: "f32", 1: "f16", 2: "bf16"}[a.ops]
    line = {
        "metric": METRIC if args.workload == "large_training" else f"SSD fwd tokens/s ({args.workload})",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (round(value / PUBLISHED_TOKENS_PER_S[args.workload], 3)
                        if args.workload in PUBLISHED_TOKENS_PER_S else None),
        "dtype": ops_name if any(k.endswith("_tc") or k == "ssd_fused_kernel" for k in kernels) else "f32",
        "data": "synthetic (seeded, pages' distributions)",
        "config": {"workload": f"{args.workload} {w.shape_tuple()} [B,L,H,P,N,chunk,G]"
                               + (" (batch overridden)" if args.batch else ""),
                   "plan": {1: "chunked", 2: "fused"}[plan], "fused_plan": fused_note, "ops_requested": ops_name,
                   "public_dtype": w.x_dtype, "tokens_per_step_per_gpu": w.tokens,
                   "l2": ("flushed between steps (256 MiB write)" if flush is not None
                          else f"inputs {in_bytes / 1e9:.2f} GB > 129 MB L2, no flush"),
                   "path_roofline_ms": round(path_roofline_ms, 4),
                   "path_frac_of_roofline": round(path_roofline_ms / ms, 4),
                   "step_ms_quantiles": step_quantiles(per_step),
                   "parallelism": f"replica x{world}" if world > 1 else "1 GPU"},
        "roofline": roofline,
        "kernels": kernels,
        "stages": stages,
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_seconds)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_decode(args):
    """Decode path: one ``ssd_decode_step`` per step for every sequence of the
    workload's batch (its final state is the carried state).  Each timed step
    follows a 256 MiB L2 flush, since the state of the large training shape
    (67 MB) would otherwise stay in the 129 MB L2; the flush buffer is written
    and then read back, so that the step does not pay for writing the flush's
    dirty lines back to HBM.  Prints its own JSON line."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = ssd_inputs.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    one = ssd_inputs.make(w.with_(L=1))
    cu = {k: (v[:, 0].to(dev).contiguous() if k in ("x", "dt", "B", "C", "z") and v is not None
              else (v.to(dev) if isinstance(v, torch.Tensor) else v)) for k, v in one.items()}
    gen = torch.Generator().manual_seed(w.seed + 77)
    state = (torch.randn((w.B, w.H, w.P, w.N), generator=gen) * 0.5).to(dev)
    y = torch.empty_like(cu["x"])
    a = ssd.make_decode_args(cu["x"], cu["dt"], cu["A"], cu["B"], cu["C"], state, y=y, D=cu["D"], z=cu["z"],
                             dt_bias=cu["dt_bias"], dt_softplus=w.dt_softplus)
    sh = ssd._stream_handle(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        ssd.ssd_decode_step(a, sh)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index, enabled=not args.no_clocks) as clk:
        torch.cuda.synchronize(dev)
        sink = torch.zeros((), device=dev)
        for i in range(args.steps):
            flush.fill_(float(i))
            sink += flush.sum()
            starts[i].record(stream)
            ssd.ssd_decode_step(a, sh)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        if not args.no_clocks:
            extra_until = time.time() + 0.5
            while time.time() < extra_until:
                ssd.ssd_decode_step(a, sh)
            torch.cuda.synchronize(dev)
    per_step = sorted(s.elapsed_time(e) for s, e in zip(starts, ends))
    ms = per_step[len(per_step) // 2]
    io = {"f32": 4, "f16": 2, "bf16": 2}[w.x_dtype]
    nbytes = (2 * w.B * w.H * w.P * w.N * 4                       # state read + written
              + w.B * w.H * w.P * io * (2 + (1 if w.z else 0))    # x, y (, z)
              + 2 * w.B * w.G * w.N * io + w.B * w.H * 4          # B, C, dt
              + w.H * 4 * (1 + (w.D_std is not None) + (w.dt_bias_std is not None)))
    hbm, peak_kind = peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    line = {
        "metric": f"SSD decode step tokens/s ({args.workload} state [{w.B},{w.H},{w.P},{w.N}])",
        "value": round(w.B / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded, pages' distributions)",
        "config": {"workload": f"decode, {args.workload} [B,H,P,N,G] = {[w.B, w.H, w.P, w.N, w.G]}",
                   "l2": "flushed before every timed step (256 MiB written, then read)",
                   "timing": "median of per-step events"},
        "roofline": {"bound": "hbm", "kernel": "decode_step_stream_kernel", "achieved": round(achieved, 1),
                     "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": traffic_for("decode_step_stream_kernel", args.workload),
                     "alg_bytes_per_launch": nbytes, "launch_ms": round(ms, 6)},
        "clocks": clk.summary(),
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def run_varlen(args):
    """Packed variable-length path: the workload's B*L tokens as B sequences
    of seeded random lengths (each 25-175 % of L, summing to B*L) packed along
    one batch row, one ``ssd_fwd_varlen`` per step.  Prints its own JSON line."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = ssd_inputs.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    T = w.B * w.L
    gen = torch.Generator().manual_seed(w.seed + 91)
    frac = torch.rand(w.B, generator=gen) * 1.5 + 0.25
    lengths = (frac / frac.sum() * T).long()
    lengths[-1] += T - int(lengths.sum())
    cu = torch.cat([torch.zeros(1, dtype=torch.long), torch.cumsum(lengths, 0)])
    packed = w.with_(B=1, L=T)
    inp = ssd_inputs.make(packed)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    fin = torch.empty((w.B, w.H, w.P, w.N), device=dev) if w.return_final_state else None
    a = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk, y=y, final_state=fin, D=d["D"], z=d["z"],
                      dt_bias=d["dt_bias"], dt_softplus=w.dt_softplus, ops=args.ops or w.ops, plan=args.plan)
    nws = ssd.ssd_fwd_varlen_workspace_size(a, cu)
    ws = torch.zeros(max(nws, 256), dtype=torch.uint8, device=dev)
    a.workspace, a.workspace_bytes = ws.data_ptr(), nws
    sh = ssd._stream_handle(dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        ssd.ssd_fwd_varlen(a, cu, sh)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index, enabled=not args.no_clocks) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            starts[i].record(stream)
            ssd.ssd_fwd_varlen(a, cu, sh)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        if not args.no_clocks:
            extra_until = time.time() + 0.5
            while time.time() < extra_until:
                ssd.ssd_fwd_varlen(a, cu, sh)
            torch.cuda.synchronize(dev)
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps
    ab = algorithmic_bytes(w)
    hbm, peak_kind = peaks()
    achieved = ab["total"] / (ms * 1e-3) / 1e9
    line = {
        "metric": f"SSD fwd tokens/s, packed variable-length sequences ({args.workload} tokens)",
        "value": round(T / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {0: "f32", 1: "f16", 2: "bf16"}[a.ops],
        "data": "synthetic (seeded, pages' distributions)",
        "config": {"workload": f"varlen: {w.B} sequences, lengths {lengths.tolist()}, total {T} tokens, "
                               f"[H,P,N,chunk,G] = {[w.H, w.P, w.N, w.chunk, w.G]}",
                   # the fused plan's workspace is the error word and the offsets; the chunked
                   # plan's holds one sequence's chunk states
                   "plan": "fused" if nws < 65536 else "chunked, per sequence"},
        "roofline": {"bound": "hbm", "kernel": "ssd_fused_kernel (varlen)", "achieved": round(achieved, 1),
                     "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": None, "alg_bytes_per_launch": ab["total"], "launch_ms": round(ms, 5)},
        "clocks": clk.summary(),
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def run_norm(args):
    """Forward + gated RMSNorm (a Mamba-2 block's SSD and the norm after it):
    the workload with a seeded z [B,L,H,P] and norm weight [H*P], groups of
    (H/G)*P channels.  Times the norm inside the fused kernel, and beside it
    the two-kernel route (the forward without its gate, then the norm kernel
    over y).  Prints its own JSON line."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = ssd_inputs.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    inp = ssd_inputs.make(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    gen = torch.Generator().manual_seed(w.seed + 77)
    z = torch.randn(inp["x"].shape, generator=gen).to(inp["x"].dtype).to(dev)
    nw = (torch.rand(w.H * w.P, generator=gen) + 0.5).to(dev)
    y = torch.empty_like(d["x"])
    fin = torch.empty((w.B, w.H, w.P, w.N), device=dev) if w.return_final_state else None
    ops = args.ops or w.ops
    fused = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk, y=y, final_state=fin, D=d["D"], z=z,
                          dt_bias=d["dt_bias"], initial_states=d["initial_states"], dt_softplus=w.dt_softplus,
                          ops=ops, plan=args.plan, norm_weight=nw, norm_eps=1e-5)
    plain = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk, y=y, final_state=fin, D=d["D"],
                          dt_bias=d["dt_bias"], initial_states=d["initial_states"], dt_softplus=w.dt_softplus,
                          ops=ops, plan=args.plan)
    kernels = ",".join(ssd.ssd_fwd_describe(fused))
    ws = torch.zeros(max(ssd.ssd_fwd_workspace_size(plain), ssd.ssd_fwd_workspace_size(fused), 256),
                     dtype=torch.uint8, device=dev)
    for a in (fused, plain):
        a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    sh = ssd._stream_handle(dev)
    stream = torch.cuda.current_stream(dev)
    Bb, L, H, P = y.shape
    y2, z2 = y.view(Bb * L, H * P), z.view(Bb * L, H * P)

    def two_kernels():
        ssd.ssd_fwd(plain, sh)
        ssd.ssd_gated_rmsnorm(y2, z2, nw, w.G, 1e-5, y2, sh)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            st[i].record(stream)
            fn()
            en[i].record(stream)
        torch.cuda.synchronize(dev)
        return sum(s_.elapsed_time(e_) for s_, e_ in zip(st, en)) / args.steps

    with ClockSampler(dev.index, enabled=not args.no_clocks) as clk:
        ms = timed(lambda: ssd.ssd_fwd(fused, sh))
        ms_two = timed(two_kernels)
    ab = algorithmic_bytes(w)
    nbytes = ab["total"] + y.numel() * y.element_size() + w.H * w.P * 4  # + z read, + the weight
    hbm, peak_kind = peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    line = {
        "metric": f"SSD fwd + gated RMSNorm tokens/s ({args.workload} {w.shape_tuple()})",
        "value": round(w.tokens / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {0: "f32", 1: "f16", 2: "bf16"}[fused.ops],
        "data": "synthetic (seeded, pages' distributions; z ~ N(0,1), weight ~ U(0.5, 1.5))",
        "config": {"workload": f"forward + gated RMSNorm, {args.workload} {w.shape_tuple()} [B,L,H,P,N,chunk,G], "
                               f"norm groups of {w.H // w.G * w.P} channels",
                   "kernels": kernels, "two_kernel_ms": round(ms_two, 5),
                   "l2": "inputs larger than L2, no flush"},
        "roofline": {"bound": "hbm", "kernel": kernels, "achieved": round(achieved, 1), "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": None,
                     "alg_bytes_per_launch": nbytes, "launch_ms": round(ms, 5)},
        "clocks": clk.summary(),
        "gpu_launches": args.steps * len(kernels.split(",")),
    }
    print(json.dumps(line), flush=True)


def measured_fp32_gemm_tflops(dev, n=8192, reps=3):
    """fp32 FMA throughput measured on this GPU: cuBLAS SGEMM with TF32 off
    (torch.matmul at 'highest' precision), n^3 multiply-adds, best of ``reps``
    CUDA-event timings after a warm-up."""
    prev = torch.get_float32_matmul_precision()
    torch.set_float32_matmul_precision("highest")
    try:
        a = torch.randn((n, n), device=dev)
        b = torch.randn((n, n), device=dev)
        torch.matmul(a, b)
        torch.cuda.synchronize(dev)
        best = math.inf
        for _ in range(reps):
            s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            torch.matmul(a, b)
            e0.record()
            torch.cuda.synchronize(dev)
            best = min(best, s0.elapsed_time(e0))
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.set_float32_matmul_precision(prev)


def measured_fp32_fma_tflops(dev, iters=32768, reps=5):
    """fp32 CUDA-core throughput measured on this GPU: the library's
    FMA-chain kernel (8 independent chains per thread, 8 CTAs of 256 threads
    per SM), best of ``reps`` CUDA-event timings after a warm-up launch."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    grid = 8 * torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.empty(grid * 256, device=dev)
    sh = ssd._stream_handle(dev)
    stream = torch.cuda.current_stream(dev)
    ssd.ssd_selftest_fma_rate(out, iters, grid, sh)
    torch.cuda.synchronize(dev)
    best = math.inf
    for _ in range(reps):
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        ssd.ssd_selftest_fma_rate(out, iters, grid, sh)
        e0.record(stream)
        torch.cuda.synchronize(dev)
        best = min(best, s0.elapsed_time(e0))
    return 2.0 * 8 * iters * 256 * grid / (best * 1e-3) / 1e12


def run_bwd(args):
    """Backward path: one ``ssd_bwd`` per step at the workload's shape (dy and
    dfinal seeded, all gradients written).  Prints its own JSON line; the
    roofline counts the backward's public I/O once (inputs x, dt, B, C, dy,
    dfinal, h0, z; outputs dx, ddt, dB, dC, dh0, dz)."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = ssd_inputs.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    inp = ssd_inputs.make(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    gen = torch.Generator().manual_seed(w.seed + 300)
    dy = torch.randn(inp["x"].shape, generator=gen).to(inp["x"].dtype).to(dev)
    dfinal = torch.randn((w.B, w.H, w.P, w.N), generator=gen).to(dev)
    f32 = dict(device=dev, dtype=torch.float32)
    g = {"dx": torch.empty_like(d["x"]), "ddt": torch.empty((w.B, w.L, w.H), **f32), "dA": torch.empty(w.H, **f32),
         "dB": torch.empty_like(d["B"]), "dC": torch.empty_like(d["C"]), "dh0": torch.empty((w.B, w.H, w.P, w.N), **f32),
         "dD": torch.empty(w.H, **f32) if d["D"] is not None else None,
         "dz": torch.empty_like(d["z"]) if d["z"] is not None else None,
         "ddt_bias": torch.empty(w.H, **f32) if d["dt_bias"] is not None else None}
    a = ssd.SsdBwdArgs()
    a.fwd = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                          initial_states=d["initial_states"], dt_softplus=w.dt_softplus)
    a.dy, a.dfinal = dy.data_ptr(), dfinal.data_ptr()
    for k in ("dx", "ddt", "dA", "dB", "dC", "dh0", "dD", "dz", "ddt_bias"):
        setattr(a, k, None if g[k] is None else g[k].data_ptr())
    nws = ssd.ssd_bwd_workspace_size(a)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    a.workspace, a.workspace_bytes = ws.data_ptr(), nws
    sh = ssd._stream_handle(dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        ssd.ssd_bwd(a, sh)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index, enabled=not args.no_clocks) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            starts[i].record(stream)
            ssd.ssd_bwd(a, sh)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps
    ab = algorithmic_bytes(w)
    nbytes = (2 * (ab["x"] + ab["B"] + ab["C"] + ab["dt"] + ab["z"]) + ab["x"]  # inputs and gradients, dy
              + 2 * w.B * w.H * w.P * w.N * 4 + ab["h0"])                           # dfinal, dh0, h0
    hbm, _ = peaks()
    flops = bwd_flops(w)
    tflops = flops / (ms * 1e-3) / 1e12
    derived = fp32_alu_peak_tflops()
    alu = measured_fp32_fma_tflops(dev)
    sgemm = measured_fp32_gemm_tflops(dev)
    has_z = d["z"] is not None
    # recompute 3 (+ chunk_scan with z); the gate (skipped for fp32 dy without z); adjoint, passing,
    # chunk, 2 group sums, head sum
    launches = 3 + has_z + (has_z or w.x_dtype != "f32") + 6
    line = {
        "metric": f"SSD backward tokens/s ({args.workload} {w.shape_tuple()})",
        "value": round(w.tokens / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded, pages' distributions)",
        "config": {"workload": f"backward, {args.workload} {w.shape_tuple()} [B,L,H,P,N,chunk,G]",
                   "workspace_gb": round(nws / 1e9, 2)},
        "roofline": {"bound": "alu", "kernel": f"whole backward ({launches} launches, fp32 CUDA cores)",
                     "achieved": round(tflops, 3), "peak": round(alu, 1),
                     "peak_kind": "measured: fp32 FMA-chain kernel (ssd_selftest_fma_rate), best of 5, this run",
                     "unit": "TFLOP/s", "frac": round(tflops / alu, 4), "traffic": None,
                     "derived_peak": {"tflops": round(derived, 1),
                                      "how": "152 SMs x 128 fp32 lanes x 2 flops x max SM clock"},
                     "alg_flops_per_step": flops, "launch_ms": round(ms, 4),
                     "measured_fp32": {"sgemm_tflops": round(sgemm, 2), "frac": round(tflops / sgemm, 4),
                                       "how": "cuBLAS SGEMM 8192^3, TF32 off, best of 3, this run"},
                     "hbm_view": {"alg_bytes_per_step": nbytes,
                                  "achieved_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "peak_gbs": hbm}},
        "clocks": clk.summary(),
        "gpu_launches": launches * args.steps,
    }
    print(json.dumps(line), flush=True)


def run_neighbor(args):
    """The SSD's neighbours, each timed alone (L2 flushed before every step):
    conv1d at the pages' test shape (B 1, D 10240, S 1024, W 4, fp32, bias,
    SiLU); gated RMSNorm at the y of the workload ([B, L, H*P], G groups, fp32).
    Prints its own JSON line."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator().manual_seed(17)
    w = ssd_inputs.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    if args.path == "conv1d":
        B, D, S, W = 1, 10240, 1024, 4
        x = torch.randn((B, D, S), generator=g).to(dev)
        wt = (torch.randn((D, W), generator=g) * 0.5).to(dev)
        bias = torch.randn(D, generator=g).to(dev)
        out = torch.empty_like(x)
        call = lambda sh: ssd.ssd_causal_conv1d(x, wt, bias, out, True, sh)
        nbytes = 2 * x.numel() * 4 + wt.numel() * 4 + D * 4
        name, cfg = "causal_conv1d_kernel", f"conv1d [B,D,S,W] = [{B},{D},{S},{W}] fp32, bias, SiLU"
        units = B * S
    else:
        B, L, D, G = w.B, w.L, w.H * w.P, w.G
        x = torch.randn((B, L, D), generator=g).to(dev)
        z = torch.randn((B, L, D), generator=g).to(dev)
        wn = (torch.rand(D, generator=g) + 0.5).to(dev)
        out = torch.empty_like(x)
        call = lambda sh: ssd.ssd_gated_rmsnorm(x, z, wn, G, 1e-5, out, sh)
        nbytes = 3 * x.numel() * 4 + D * 4
        name, cfg = "gated_rmsnorm_kernel", f"gated RMSNorm [B,L,D,G] = [{B},{L},{D},{G}] fp32"
        units = B * L
    sh = ssd._stream_handle(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.zeros((), device=dev)
    for _ in range(args.warmup):
        call(sh)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index, enabled=not args.no_clocks) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush.fill_(float(i))
            sink += flush.sum()
            starts[i].record(stream)
            call(sh)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    per = sorted(s.elapsed_time(e) for s, e in zip(starts, ends))
    ms = per[len(per) // 2]
    hbm, peak_kind = peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    line = {
        "metric": f"{args.path} tokens/s ({cfg})", "value": round(units / (ms * 1e-3), 1), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)",
        "config": {"workload": cfg, "l2": "flushed before every timed step (256 MiB written, then read)",
                   "timing": "median of per-step events"},
        "roofline": {"bound": "hbm", "kernel": name, "achieved": round(achieved, 1), "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": None,
                     "alg_bytes_per_launch": nbytes, "launch_ms": round(ms, 5)},
        "clocks": clk.summary(), "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def run_conv_ssd(args):
    """The causal conv1d + SiLU in front of the SSD (a Mamba-2 block's x, B, C
    before their convolution, width 4 with bias): the forward that convolves in
    its load stage, one ``ssd_fwd`` per step, against the two-kernel route
    (token-major conv kernels for x, B and C into separate buffers, then the
    forward on them) timed the same way on the same inputs.  Prints its own
    JSON line; its value is the one-call forward."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = ssd_inputs.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    inp = ssd_inputs.make(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    g = torch.Generator().manual_seed(23)
    W = 4
    cw = [(torch.randn((ch, W), generator=g) * 0.5).to(dev) for ch in (w.H * w.P, w.G * w.N, w.G * w.N)]
    cb = [(torch.randn(ch, generator=g) * 0.2).to(dev) for ch in (w.H * w.P, w.G * w.N, w.G * w.N)]
    conv = (cw[0], cb[0], cw[1], cb[1], cw[2], cb[2])
    y = torch.empty_like(d["x"])
    fin = torch.empty((w.B, w.H, w.P, w.N), device=dev) if w.return_final_state else None
    ops = args.ops or w.ops

    def make(x, Bm, Cm, conv_arg):
        a = ssd.make_args(x, d["dt"], d["A"], Bm, Cm, w.chunk, y=y, final_state=fin, D=d["D"], z=d["z"],
                          dt_bias=d["dt_bias"], initial_states=d["initial_states"], dt_softplus=w.dt_softplus,
                          ops=ops, plan=args.plan, conv=conv_arg)
        ws = torch.zeros(max(ssd.ssd_fwd_workspace_size(a), 256), dtype=torch.uint8, device=dev)
        a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
        return a, ws

    fused_args, ws1 = make(d["x"], d["B"], d["C"], conv)
    xc, Bc, Cc = torch.empty_like(d["x"]), torch.empty_like(d["B"]), torch.empty_like(d["C"])
    plain_args, ws2 = make(xc, Bc, Cc, None)
    sh = ssd._stream_handle(dev)
    stream = torch.cuda.current_stream(dev)

    def fused_step():
        ssd.ssd_fwd(fused_args, sh)

    def two_kernel_step():
        ssd.ssd_causal_conv1d_tokens(d["x"].view(w.B, w.L, -1), cw[0], cb[0], xc.view(w.B, w.L, -1), True, sh)
        ssd.ssd_causal_conv1d_tokens(d["B"].view(w.B, w.L, -1), cw[1], cb[1], Bc.view(w.B, w.L, -1), True, sh)
        ssd.ssd_causal_conv1d_tokens(d["C"].view(w.B, w.L, -1), cw[2], cb[2], Cc.view(w.B, w.L, -1), True, sh)
        ssd.ssd_fwd(plain_args, sh)

    def timed(step):
        for _ in range(args.warmup):
            step()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        return [st.elapsed_time(en) for st, en in zip(starts, ends)]

    with ClockSampler(dev.index, enabled=not args.no_clocks) as clk:
        per_two = timed(two_kernel_step)
        per_fused = timed(fused_step)
        if not args.no_clocks:
            extra_until = time.time() + 0.5
            while time.time() < extra_until:
                fused_step()
            torch.cuda.synchronize(dev)
    ms = sum(per_fused) / len(per_fused)
    ms_two = sum(per_two) / len(per_two)
    ab = algorithmic_bytes(w)
    nbytes = ab["total"] + sum(t.numel() * 4 for t in cw + cb)
    hbm, peak_kind = peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    kernels = ssd.ssd_fwd_describe(fused_args)
    line = {
        "metric": f"SSD fwd with the causal conv1d in front, tokens/s ({args.workload})",
        "value": round(w.tokens / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ops, "data": "synthetic (seeded, pages' distributions; conv width 4)",
        "config": {"workload": f"{args.workload} {w.shape_tuple()} [B,L,H,P,N,chunk,G] + conv1d W=4",
                   "step_ms_quantiles": step_quantiles(per_fused),
                   "two_kernel_ms": round(ms_two, 5), "two_kernel_quantiles": step_quantiles(per_two),
                   "speedup_over_two_kernels": round(ms_two / ms, 3),
                   "l2": f"inputs {(ab['x'] + ab['B'] + ab['C']) / 1e9:.2f} GB > 129 MB L2, no flush"},
        "roofline": {"bound": "hbm", "kernel": kernels[-1], "achieved": round(achieved, 1), "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": None,
                     "alg_bytes_per_launch": nbytes, "launch_ms": round(ms, 5)},
        "kernels": kernels,
        "clocks": clk.summary(),
        "gpu_launches": len(kernels) * args.steps,
    }
    print(json.dumps(line), flush=True)


def stage_timing(ssd, a, w, dev, sh, stream, args, kernels):
    """Time the four chunked-plan kernels one by one (events between launches)
    and return the dominant one with its algorithmic bytes, plus every stage's
    time."""
    c = -(-w.L // w.chunk)
    dtp = torch.empty((w.B, w.H, c, w.chunk), device=dev)
    cs = torch.empty_like(dtp)
    states = torch.empty((w.B, c, w.H, w.P, w.N), device=dev)
    names = ["chunk_cumsum", "chunk_state", "state_passing", "chunk_scan"]
    calls = [lambda: ssd.ssd_chunk_cumsum(a, dtp, cs, sh),
             lambda: ssd.ssd_chunk_state(a, dtp, cs, states, sh),
             lambda: ssd.ssd_state_passing(a, cs, states, sh),
             lambda: ssd.ssd_chunk_scan(a, dtp, cs, states, sh)]
    for _ in range(2):
        for f in calls:
            f()
    reps = max(3, min(args.steps, 10))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(reps)]
    torch.cuda.synchronize(dev)
    for r in range(reps):
        ev[r][0].record(stream)
        for i, f in enumerate(calls):
            f()
            ev[r][i + 1].record(stream)
    torch.cuda.synchronize(dev)
    t = [sum(ev[r][i].elapsed_time(ev[r][i + 1]) for r in range(reps)) / reps for i in range(4)]
    sb = stage_bytes(w)
    i = max(range(4), key=lambda j: t[j])
    stages = {kernels[j]: {"ms": round(t[j], 5), "alg_bytes": sb[names[j]],
                           "GB_per_s": round(sb[names[j]] / (t[j] * 1e-3) / 1e9, 1)} for j in range(4)}
    return kernels[i], sb[names[i]], t[i], stages


def e2e_timing(ssd, inp, w, dev, args):
    """Same metric through ssd_fwd_host: pinned host inputs copied in and y /
    final_state copied out inside the timed region."""
    h = {k: (v.contiguous().pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.empty_like(h["x"]).pin_memory()
    fin = torch.empty((w.B, w.H, w.P, w.N)).pin_memory() if w.return_final_state else None
    a = ssd.make_args(h["x"], h["dt"], h["A"], h["B"], h["C"], w.chunk, y=y, final_state=fin,
                      D=h["D"], z=h["z"], dt_bias=h["dt_bias"], initial_states=h["initial_states"],
                      dt_softplus=w.dt_softplus, ops=args.ops or w.ops, plan=args.plan)
    nws = ssd.ssd_fwd_host_workspace_size(a)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    a.workspace, a.workspace_bytes = ws.data_ptr(), nws
    sh = ssd._stream_handle(dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        ssd.ssd_fwd_host(a, sh)
    torch.cuda.synchronize(dev)
    steps = max(3, args.steps)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        starts[i].record(stream)
        ssd.ssd_fwd_host(a, sh)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    per_step = [st.elapsed_time(en) for st, en in zip(starts, ends)]
    ms = sum(per_step) / len(per_step)
    h2d = sum(v.numel() * v.element_size() for k, v in h.items()
              if isinstance(v, torch.Tensor))
    d2h = y.numel() * y.element_size() + (fin.numel() * 4 if fin is not None else 0)
    return {"value": round(w.tokens / (ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "steps": steps, "step_ms_quantiles": step_quantiles(per_step),
            "slowest_step": {"index": max(range(steps), key=per_step.__getitem__), "ms": round(max(per_step), 4)},
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# ---- the CPU oracle (cpu_baseline and --impl reference) --------------------------------

def _oracle_problem(inp):
    import oracle
    oracle.build()
    return oracle.Problem(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"], z=inp["z"],
                          dt_bias=inp["dt_bias"], initial_states=inp["initial_states"],
                          dt_softplus=inp["dt_softplus"])


def oracle_sample_size(w, prob, seconds, *, nthreads=0):
    """How many whole (batch, head) sequences of the workload the float64
    oracle finishes in about ``seconds`` (from one timed calibration run over
    one sequence per core)."""
    import oracle
    cores = nthreads or oracle.threads()
    total = w.B * w.H
    n = min(total, max(1, cores))
    t0 = time.perf_counter()
    oracle.recurrence(prob, [(i // w.H, i % w.H) for i in range(n)], nthreads=nthreads)
    per_pair = (time.perf_counter() - t0) / n
    return int(min(total, max(n, seconds / max(per_pair, 1e-9)))), cores


def oracle_timed(w, prob, n, *, nthreads=0, offset=0):
    """One timed oracle run over n whole sequences (starting at sequence
    ``offset``, wrapping around): (wall seconds, tokens processed, counted
    as the workload's tokens B*L times the share of its B*H sequences run)."""
    import oracle
    total = w.B * w.H
    pairs = [((offset + i) % total // w.H, (offset + i) % total % w.H) for i in range(n)]
    t0 = time.perf_counter()
    oracle.recurrence(prob, pairs, nthreads=nthreads)
    return time.perf_counter() - t0, w.tokens * n / total


def oracle_sample(w, inp, seconds, *, nthreads=0):
    """Time the float64 oracle on a bounded sample of the workload: whole
    (batch, head) sequences over the full L, as many as fit in ~``seconds``."""
    prob = _oracle_problem(inp)
    n, cores = oracle_sample_size(w, prob, seconds, nthreads=nthreads)
    dt, _ = oracle_timed(w, prob, n, nthreads=nthreads)
    total = w.B * w.H
    frac = n / total
    tok_s = w.tokens * frac / dt
    return {"value": round(tok_s, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {total} (batch, head) sequences over the full L={w.L} "
                      f"({frac * 100:.2f}% of one step), {dt:.2f} s wall",
            "seconds": round(dt, 3)}


def cpu_baseline(w, inp, seconds):
    return oracle_sample(w, inp, seconds)


def run_reference(args):
    """The float64 oracle as the reference arm.  Each step is one bounded
    sample of the workload (the same number of whole (batch, head) sequences
    every step, sized in the warm-up so that all steps take about
    --cpu-seconds); ms_per_step is a step's own measured wall time, and value
    is the tokens those steps processed over their total wall time."""
    rank, world, _ = rank_info()
    if rank != 0:
        return
    w = ssd_inputs.WORKLOADS[args.workload]
    inp = ssd_inputs.make(w)
    prob = _oracle_problem(inp)
    per_step = max(0.5, args.cpu_seconds / max(1, args.steps))
    n, cores = oracle_sample_size(w, prob, per_step)
    for i in range(args.warmup and 1 or 0):
        oracle_timed(w, prob, n, offset=i * n)
    walls, tokens = [], 0
    for i in range(args.steps):
        dt, tk = oracle_timed(w, prob, n, offset=i * n)
        walls.append(dt)
        tokens += tk
    value = tokens / sum(walls)
    ms = sum(walls) / len(walls) * 1e3
    total = w.B * w.H
    sample = (f"each step: {n} of {total} (batch, head) sequences over the full L={w.L} "
              f"({n / total * 100:.2f}% of the workload's tokens); {len(walls)} steps, "
              f"{sum(walls):.2f} s wall in total")
    line = {
        "impl": "reference",
        "metric": METRIC if args.workload == "large_training" else f"SSD fwd tokens/s ({args.workload})",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload} {w.shape_tuple()} [B,L,H,P,N,chunk,G]",
                   "what": "float64 CPU oracle (token-by-token recurrence), one bounded sample per step",
                   "tokens_per_step": round(w.tokens * n / total, 1),
                   "projected_full_workload_ms": round(w.tokens / value * 1e3, 1),
                   "step_ms_quantiles": step_quantiles([x * 1e3 for x in walls])},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(ssd_inputs.WORKLOADS), default="large_training")
    ap.add_argument("--plan", choices=["auto", "chunked", "fused"], default="auto")
    ap.add_argument("--ops", choices=["f32", "f16", "bf16"], default=None)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true", help="skip the nvidia-smi clock sampler")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (a smaller case of the same shape)")
    ap.add_argument("--path", choices=["forward", "decode", "varlen", "bwd", "conv1d", "rmsnorm", "norm",
                                       "conv_ssd"],
                    default="forward",
                    help="forward (default): the whole SSD forward; decode: one decode step per "
                         "sequence from a carried state; varlen: the forward over packed sequences "
                         "of random lengths; bwd: the backward; conv1d, rmsnorm: the neighbours alone; "
                         "norm: the forward with the gated RMSNorm of its output; conv_ssd: the forward "
                         "with the causal conv1d of x, B, C in front (in its load stage) against conv "
                         "kernels plus the forward")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the reference arm runs with --impl reference)")
    if args.path == "decode":
        run_decode(args)
        return
    if args.path == "varlen":
        run_varlen(args)
        return
    if args.path == "bwd":
        run_bwd(args)
        return
    if args.path == "norm":
        run_norm(args)
        return
    if args.path in ("conv1d", "rmsnorm"):
        run_neighbor(args)
        return
    if args.path == "conv_ssd":
        run_conv_ssd(args)
        return
    run_gpu(args)


if __name__ == "__main__":
    main()
