"""GPU parity of the packed variable-length forward (``ssd_fwd_varlen``):
sequences of different lengths back to back along L of one batch row, each an
independent forward with its own initial and final state.  Reference: the
float64 oracle run on every sequence alone."""
import numpy as np
import pytest
import torch

import ssd_inputs
from _harness import assert_close

pytestmark = pytest.mark.gpu


def _packed(lengths, H, P, N, G, *, dtype, seed, feats):
    T = sum(lengths)
    f = dict(D=True, z=True, dt_bias=True) if feats else {}
    _, inp = ssd_inputs.custom(1, T, H, P, N, G, 64, seed=seed, x_dtype=dtype, ops=dtype, **f)
    h0 = None
    if feats:
        gen = torch.Generator().manual_seed(seed + 500)
        h0 = (torch.randn((len(lengths), H, P, N), generator=gen) * 0.1).float()
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return inp, h0, cu


def _oracle_per_sequence(oracle_mod, inp, h0, cu):
    ys, fins = [], []
    for s in range(len(cu) - 1):
        lo, hi = int(cu[s]), int(cu[s + 1])
        H, P = inp["x"].shape[2], inp["x"].shape[3]
        N = inp["B"].shape[3]
        if hi == lo:
            ys.append(np.zeros((0, H, P)))
            fins.append(h0[s].double().numpy() if h0 is not None else np.zeros((H, P, N)))
            continue
        cut = lambda t: None if t is None else t[:, lo:hi]
        prob = oracle_mod.Problem(cut(inp["x"]), cut(inp["dt"]), inp["A"], cut(inp["B"]), cut(inp["C"]),
                                  D=inp["D"], z=cut(inp["z"]), dt_bias=inp["dt_bias"],
                                  initial_states=None if h0 is None else h0[s:s + 1], dt_softplus=True)
        y, fin = oracle_mod.forward(prob)
        ys.append(y[0])
        fins.append(fin[0])
    return np.concatenate(ys, axis=0), np.stack(fins)


def _run(inp, h0, cu, *, ops, plan):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y, fin = ssd.mamba2_ssd_fwd_varlen(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, cu, dt_softplus=True,
                                       return_final_state=True, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                                       initial_states=None if h0 is None else h0.cuda(), ops=ops, plan=plan)
    torch.cuda.synchronize()
    return y, fin


LENGTHS = [64, 1, 130, 0, 77, 255, 128]


@pytest.mark.parametrize("io,ops", [("f32", "bf16"), ("bf16", "bf16"), ("f32", "f16")])
@pytest.mark.parametrize("feats", [False, True])
def test_varlen_fused_plan(oracle_mod, io, ops, feats):
    """P = N = 64 and an even number of heads per group: the fused kernel."""
    inp, h0, cu = _packed(LENGTHS, 8, 64, 64, 2, dtype=io, seed=41 + feats, feats=feats)
    y, fin = _run(inp, h0, cu, ops=ops, plan="fused")
    yr, fr = _oracle_per_sequence(oracle_mod, inp, h0, cu)
    assert_close(oracle_mod, y[0].double().cpu().numpy(), yr, ops, f"varlen fused {io}/{ops} y")
    assert_close(oracle_mod, fin.double().cpu().numpy(), fr, ops, f"varlen fused {io}/{ops} final")


@pytest.mark.parametrize("shape,ops,plan", [
    ((8, 64, 128, 2), "f32", "auto"),      # N = 128: the chunked plan, one sequence after another
    ((8, 64, 128, 2), "bf16", "auto"),
    ((8, 64, 64, 2), "bf16", "chunked"),   # a fused-capable shape, chunked on request
    ((6, 32, 48, 3), "f32", "auto"),       # odd heads per group
])
def test_varlen_chunked_plan(oracle_mod, shape, ops, plan):
    H, P, N, G = shape
    inp, h0, cu = _packed(LENGTHS, H, P, N, G, dtype="f32", seed=43, feats=True)
    y, fin = _run(inp, h0, cu, ops=ops, plan=plan)
    yr, fr = _oracle_per_sequence(oracle_mod, inp, h0, cu)
    assert_close(oracle_mod, y[0].double().cpu().numpy(), yr, ops, f"varlen chunked {shape} {ops} y")
    assert_close(oracle_mod, fin.double().cpu().numpy(), fr, ops, f"varlen chunked {shape} {ops} final")


def test_varlen_many_sequences_more_units_than_ctas(oracle_mod):
    """80 sequences of random length in 1..300 (fused plan, 80 x 32 units)."""
    rng = np.random.default_rng(7)
    lengths = rng.integers(1, 301, size=80).tolist()
    inp, h0, cu = _packed(lengths, 64, 64, 64, 16, dtype="bf16", seed=47, feats=True)
    y, fin = _run(inp, h0, cu, ops="bf16", plan="fused")
    pick = [0, 1, 17, 40, 79]
    sub_y, sub_f = [], []
    ref_y, ref_f = [], []
    for s in pick:
        lo, hi = int(cu[s]), int(cu[s + 1])
        part = {k: (v[:, lo:hi] if k in ("x", "dt", "B", "C", "z") else v) for k, v in inp.items()}
        prob = oracle_mod.Problem(part["x"], part["dt"], inp["A"], part["B"], part["C"], D=inp["D"],
                                  z=part["z"], dt_bias=inp["dt_bias"], initial_states=h0[s:s + 1],
                                  dt_softplus=True)
        yy, ff = oracle_mod.forward(prob)
        ref_y.append(yy[0]); ref_f.append(ff[0])
        sub_y.append(y[0, lo:hi].double().cpu().numpy()); sub_f.append(fin[s].double().cpu().numpy())
    assert_close(oracle_mod, np.concatenate(sub_y), np.concatenate(ref_y), "bf16", "varlen many y")
    assert_close(oracle_mod, np.stack(sub_f), np.stack(ref_f), "bf16", "varlen many final")


def test_varlen_equals_separate_calls():
    """The packed call gives the bits of one B = 1 call per sequence (fused plan both ways)."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    lengths = [128, 192, 64]
    inp, h0, cu = _packed(lengths, 8, 64, 64, 2, dtype="bf16", seed=49, feats=True)
    y, fin = _run(inp, h0, cu, ops="bf16", plan="fused")
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    for s in range(3):
        lo, hi = int(cu[s]), int(cu[s + 1])
        cut = lambda t: t[:, lo:hi].contiguous()
        ys, fs = ssd.mamba2_ssd_fwd(cut(d["x"]), cut(d["dt"]), d["A"], cut(d["B"]), cut(d["C"]), 64,
                                    dt_softplus=True, return_final_state=True, D=d["D"], z=cut(d["z"]),
                                    dt_bias=d["dt_bias"], initial_states=h0[s:s + 1].cuda(), ops="bf16",
                                    plan="fused")
        torch.cuda.synchronize()
        assert torch.equal(ys[0], y[0, lo:hi]) and torch.equal(fs[0], fin[s])
