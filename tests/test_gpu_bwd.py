"""GPU parity of the SSD backward (``ssd_bwd``) against the float64 oracle's
adjoint (itself pinned by central differences): every gradient, element by
element, over shapes with several chunks and ragged tails."""
import numpy as np
import pytest
import torch

import ssd_inputs
from _harness import assert_close, oracle_problem

pytestmark = pytest.mark.gpu

GRADS = ("dx", "ddt", "dA", "dB", "dC", "dD", "dz", "ddt_bias", "dh0")


def _case(shape, *, dtype="f32", feats=True, seed=0, **kw):
    B, L, H, P, N, G, Q = shape
    f = dict(D=True, z=True, dt_bias=True, h0=True) if feats else {}
    f.update(kw)
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=seed, x_dtype=dtype, ops=dtype, **f)
    gen = torch.Generator().manual_seed(seed + 300)
    dy = torch.randn(inp["x"].shape, generator=gen).to(inp["x"].dtype)
    dfinal = torch.randn((B, H, P, N), generator=gen).float() if feats else None
    return inp, dy, dfinal


def _gpu(inp, dy, dfinal, Q, dt_limit=(0.0, float("inf"))):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    g = ssd.mamba2_ssd_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], Q, dy.cuda(), dt_softplus=inp["dt_softplus"],
                           dfinal=None if dfinal is None else dfinal.cuda(), D=d["D"], z=d["z"],
                           dt_bias=d["dt_bias"], initial_states=d["initial_states"], dt_limit=dt_limit)
    torch.cuda.synchronize()
    return {k: v.double().cpu().numpy() for k, v in g.items()}


def _compare(oracle_mod, inp, dy, dfinal, got, mode, what, **over):
    ref = oracle_mod.backward(oracle_problem(oracle_mod, inp, **over), dy, dfinal)
    for k in GRADS:
        if k not in got:
            continue
        assert_close(oracle_mod, got[k], ref[k], mode, f"{what} {k}")


SHAPES = [
    # B, L, H, P, N, G, chunk
    (1, 64, 2, 64, 64, 1, 64),      # one chunk
    (2, 200, 4, 64, 64, 2, 64),     # several chunks, ragged tail, 2 heads per group
    (1, 130, 2, 32, 16, 1, 32),     # chunk 32
    (2, 96, 6, 48, 32, 3, 16),      # chunk 16, odd dims
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("feats", [False, True])
def test_bwd_matches_oracle(oracle_mod, shape, feats):
    inp, dy, dfinal = _case(shape, feats=feats, seed=sum(shape))
    got = _gpu(inp, dy, dfinal, shape[-1])
    _compare(oracle_mod, inp, dy, dfinal, got, "f32", f"bwd {shape} {feats}")


def test_bwd_with_an_active_dt_clamp_and_no_softplus(oracle_mod):
    shape = (2, 128, 4, 64, 64, 2, 64)
    inp, dy, dfinal = _case(shape, seed=5, dt_dist=("uniform", -0.5, 2.0))
    got = _gpu(inp, dy, dfinal, 64, dt_limit=(0.3, 1.2))
    _compare(oracle_mod, inp, dy, dfinal, got, "f32", "bwd clamp", dt_limit=(0.3, 1.2))
    inp2 = dict(inp, dt_softplus=False, dt=inp["dt"].abs() * 0.5)
    got2 = _gpu(inp2, dy, dfinal, 64)
    _compare(oracle_mod, inp2, dy, dfinal, got2, "f32", "bwd no softplus")


def test_bwd_bf16_inputs(oracle_mod):
    shape = (2, 192, 4, 64, 64, 2, 64)
    inp, dy, dfinal = _case(shape, dtype="bf16", seed=9)
    got = _gpu(inp, dy, dfinal, 64)
    # the gradients are computed in fp32 and rounded to bf16 where x is bf16
    _compare(oracle_mod, inp, dy, dfinal, got, "bf16", "bwd bf16")


def test_bwd_mid_size(oracle_mod):
    shape = (2, 1024, 16, 64, 64, 4, 64)
    inp, dy, dfinal = _case(shape, seed=11)
    got = _gpu(inp, dy, dfinal, 64)
    _compare(oracle_mod, inp, dy, dfinal, got, "f32", "bwd mid")


def test_bwd_at_the_large_training_shape_on_sampled_groups(oracle_mod):
    """The benched backward shape [1,4096,256,64,64,64,64] (the large training
    shape at batch 1, same seeds as the bench): the GPU runs the whole
    problem; the oracle runs three groups (first, one inside, last) with all
    of their heads, which fixes every gradient of those heads and groups
    exactly (heads interact only through the group sums of dB and dC)."""
    w = ssd_inputs.WORKLOADS["large_training"].with_(B=1)
    inp = ssd_inputs.make(w)
    gen = torch.Generator().manual_seed(w.seed + 300)
    dy = torch.randn(inp["x"].shape, generator=gen).to(inp["x"].dtype)
    dfinal = torch.randn((w.B, w.H, w.P, w.N), generator=gen).float()
    got = _gpu(inp, dy, dfinal, w.chunk)
    hpg = w.H // w.G
    groups = [0, 29, w.G - 1]
    heads = [g * hpg + j for g in groups for j in range(hpg)]
    sub = dict(inp, x=inp["x"][:, :, heads].contiguous(), dt=inp["dt"][:, :, heads].contiguous(),
               A=inp["A"][heads].contiguous(), B=inp["B"][:, :, groups].contiguous(),
               C=inp["C"][:, :, groups].contiguous())
    ref = oracle_mod.backward(oracle_problem(oracle_mod, sub), dy[:, :, heads].contiguous(),
                              dfinal[:, heads].contiguous())
    picks = {"dx": (slice(None), slice(None), heads), "ddt": (slice(None), slice(None), heads),
             "dA": (heads,), "dB": (slice(None), slice(None), groups), "dC": (slice(None), slice(None), groups),
             "dh0": (slice(None), heads)}
    for k, idx in picks.items():
        assert_close(oracle_mod, got[k][idx], ref[k], "f32", f"bwd large_training b1 {k}")


def test_bwd_is_deterministic():
    shape = (2, 256, 8, 64, 64, 2, 64)
    inp, dy, dfinal = _case(shape, seed=13)
    a = _gpu(inp, dy, dfinal, 64)
    b = _gpu(inp, dy, dfinal, 64)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_bwd_rejects_unsupported_shapes():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    inp, dy, dfinal = _case((1, 128, 2, 64, 128, 1, 64), feats=False, seed=1)
    with pytest.raises(ssd.SsdError) as ei:
        _gpu(inp, dy, dfinal, 64)
    assert ei.value.status == 2
