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


def stream_compare(oracle, prob, outs, B, H, *, block=64, want_final=True):
    """Compare GPU outputs with the oracle over EVERY (batch, head) sequence,
    recomputing the oracle block by block (``block`` sequences at a time, in
    float64) so that host memory stays bounded.

    ``outs`` maps a label to (y [B,L,H,P], final_state [B,H,P,N] or None),
    torch tensors on the GPU.  Returns {label: {"y": metrics, "final_state":
    metrics}} with the global rel-L2 and max|diff|/max|ref| over all elements,
    accumulated exactly as ``oracle.compare`` would over the whole tensors."""
    views = {}
    for k, (y, fin) in outs.items():
        Bq, L, Hq, P = y.shape
        yv = y.permute(0, 2, 1, 3).reshape(Bq * Hq, L, P)  # pair-major copy on the GPU
        fv = fin.reshape(Bq * Hq, fin.shape[2], fin.shape[3]) if (fin is not None and want_final) else None
        views[k] = (yv, fv)
    acc = {k: {w: [0.0, 0.0, 0.0, 0.0, True] for w in ("y", "final_state")} for k in outs}
    total = B * H
    for i0 in range(0, total, block):
        i1 = min(total, i0 + block)
        pairs = [(i // H, i % H) for i in range(i0, i1)]
        ref = oracle.recurrence(prob, pairs, want_final=want_final)
        for k, (yv, fv) in views.items():
            for what, got_t, r in (("y", yv, ref["y"]), ("final_state", fv, ref["final_state"])):
                if got_t is None or r is None:
                    continue
                g = got_t[i0:i1].double().cpu().numpy()
                d = g - r
                a = acc[k][what]
                a[0] += float(np.sum(d * d))
                a[1] += float(np.sum(r * r))
                a[2] = max(a[2], float(np.max(np.abs(d))) if d.size else 0.0)
                a[3] = max(a[3], float(np.max(np.abs(r))) if r.size else 0.0)
                a[4] = a[4] and bool(np.all(np.isfinite(g)))
    res = {}
    for k in outs:
        res[k] = {}
        for what, a in acc[k].items():
            if a[1] == 0.0 and a[3] == 0.0 and a[0] == 0.0:
                continue
            nd, nr = math.sqrt(a[0]), math.sqrt(a[1])
            res[k][what] = {"rel_l2": nd / nr if nr > 0 else nd,
                            "max_abs_rel": a[2] / a[3] if a[3] > 0 else a[2],
                            "max_abs": a[2], "finite": a[4]}
    return res


def assert_metrics(m, mode, what=""):
    tol = TOL[mode]
    assert m["finite"], f"{what}: non-finite output"
    assert m["rel_l2"] <= tol["rel_l2"], f"{what}: rel_l2 {m['rel_l2']:.3e} > {tol['rel_l2']}"
    assert m["max_abs_rel"] <= tol["max_abs_rel"], \
        f"{what}: max_abs_rel {m['max_abs_rel']:.3e} > {tol['max_abs_rel']}"
