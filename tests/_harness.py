"""Helpers shared by the tests: run the library through its C ABI and the
oracle on the same seeded inputs, and compare them."""
from __future__ import annotations

import functools
import math

import numpy as np
import torch

import ssd_inputs

# Tolerances: fp32 operands ("exact" path) and fp16/bf16 operands with fp32
# accumulation, as rel-L2 over all compared elements and max|diff|/max|ref|.
TOL = {
    "f32": {"rel_l2": 1e-5, "max_abs_rel": 1e-4},
    "f16": {"rel_l2": 5e-3, "max_abs_rel": 2e-2},
    "bf16": {"rel_l2": 5e-3, "max_abs_rel": 2e-2},
}


def oracle_problem(oracle, inp, **over):
    kw = dict(D=inp["D"], z=inp["z"], dt_bias=inp["dt_bias"],
              initial_states=inp["initial_states"], dt_softplus=inp["dt_softplus"])
    kw.update(over)
    return oracle.Problem(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], **kw)


def to_device(inp, device="cuda"):
    out = {}
    for k, v in inp.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


def run_gpu(inp, *, chunk=None, ops=None, plan="auto", return_final=None, dt_limit=(0.0, math.inf)):
    """One ssd_fwd call through the C ABI on CUDA copies of ``inp``."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    d = to_device(inp)
    rf = inp["return_final_state"] if return_final is None else return_final
    res = ssd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], chunk or inp["chunk_size"],
                             dt_softplus=inp["dt_softplus"], return_final_state=rf, D=d["D"],
                             z=d["z"], dt_bias=d["dt_bias"], initial_states=d["initial_states"],
                             dt_limit=dt_limit, ops=ops, plan=plan)
    torch.cuda.synchronize()
    if rf:
        return res[0], res[1]
    return res, None


def pick_pairs(B, H, n, seed=0):
    """n distinct (b, h) pairs, always including the first and the last."""
    rng = np.random.default_rng(seed)
    total = B * H
    n = min(n, total)
    idx = set([0, total - 1])
    while len(idx) < n:
        idx.add(int(rng.integers(0, total)))
    return [(i // H, i % H) for i in sorted(idx)]


def gather_pairs(y, fin, pairs):
    """y [B,L,H,P] and fin [B,H,P,N] (torch, any device) -> float64 numpy
    [nbh,L,P] and [nbh,P,N] for the listed pairs."""
    ys = np.stack([y[b, :, h, :].double().cpu().numpy() for b, h in pairs])
    fs = None
    if fin is not None:
        fs = np.stack([fin[b, h].double().cpu().numpy() for b, h in pairs])
    return ys, fs


def assert_close(oracle, got, ref, mode, what=""):
    m = oracle.compare(got, ref)
    tol = TOL[mode]
    assert m["finite"], f"{what}: non-finite output"
    assert m["rel_l2"] <= tol["rel_l2"], f"{what}: rel_l2 {m['rel_l2']:.3e} > {tol['rel_l2']}"
    assert m["max_abs_rel"] <= tol["max_abs_rel"], \
        f"{what}: max_abs_rel {m['max_abs_rel']:.3e} > {tol['max_abs_rel']}"
    return m


@functools.lru_cache(maxsize=2)
def workload_inputs(name):
    """Inputs of a named workload (cached: the large ones take seconds to draw)."""
    w = ssd_inputs.WORKLOADS[name]
    return w, ssd_inputs.make(w)
