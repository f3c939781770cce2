"""GPU parity of the forward with the gated RMSNorm of its output (the step
after the SSD in a Mamba-2 block, ops-transformer MambaV2 article, section
4.6): y = rmsnorm over each group's (H/G)*P channels of (ssd * silu(z)), times
the weight.  Reference: the float64 oracle's forward without z, then the
oracle's gated RMSNorm, each pinned on its own.  Covers the norm inside the
fused kernel (head pairs of a group in one cluster of 1 or 2 CTAs) and the
second-kernel path (4 or 8 head pairs per group, the chunked plan, N = 128,
packed sequences, host buffers)."""
import numpy as np
import pytest
import torch

import ssd_inputs
from _harness import assert_close, oracle_problem, to_device

pytestmark = pytest.mark.gpu

EPS = 1e-5


def _case(B, L, H, P, N, G, chunk, *, dtype="f32", seed=0, D=True):
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, chunk, seed=seed, x_dtype=dtype, ops=dtype, D=D, z=True,
                               dt_bias=True, h0=True)
    w = (torch.rand(H * P, generator=torch.Generator().manual_seed(seed + 7)) + 0.5).float()
    return inp, w


def _reference(oracle_mod, inp, w, G):
    y, fin = oracle_mod.forward(oracle_problem(oracle_mod, inp, z=None))
    Bb, L, H, P = y.shape
    z = inp["z"].double().numpy()
    ref = oracle_mod.gated_rmsnorm(y.reshape(Bb, L, H * P), z.reshape(Bb, L, H * P), w.numpy(), G, EPS)
    return ref.reshape(Bb, L, H, P), fin


def _gpu(inp, w, chunk, *, ops, plan="auto"):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    d = to_device(inp)
    y, fin = ssd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], chunk, dt_softplus=True,
                                return_final_state=True, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                                initial_states=d["initial_states"], ops=ops, plan=plan, norm_weight=w.cuda(),
                                norm_eps=EPS)
    torch.cuda.synchronize()
    return y, fin


def _describe(inp, w, chunk, ops, plan="auto"):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    d = to_device(inp)
    a = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], chunk, y=torch.empty_like(d["x"]), D=d["D"],
                      z=d["z"], dt_bias=d["dt_bias"], initial_states=d["initial_states"], dt_softplus=True,
                      ops=ops, plan=plan, norm_weight=w.cuda(), norm_eps=EPS)
    return ssd.ssd_fwd_describe(a)


@pytest.mark.parametrize("H,G", [(4, 2), (8, 2)])   # 2, 4 heads per group: clusters of 1, 2
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_norm_in_the_fused_kernel(oracle_mod, H, G, dtype):
    inp, w = _case(2, 200, H, 64, 64, G, 64, dtype=dtype, seed=H + G)
    assert _describe(inp, w, 64, "bf16", "fused") == ["ssd_fused_kernel"]
    y, fin = _gpu(inp, w, 64, ops="bf16", plan="fused")
    ref, rfin = _reference(oracle_mod, inp, w, G)
    assert_close(oracle_mod, y.double().cpu().numpy(), ref, "bf16", f"fused norm H={H} G={G} {dtype}")
    assert_close(oracle_mod, fin.double().cpu().numpy(), rfin, "bf16", "final state")


def test_norm_in_the_fused_kernel_many_units_and_no_D(oracle_mod):
    """More units than CTAs (every cluster walks several groups), no D."""
    inp, w = _case(4, 256, 64, 64, 64, 16, 64, dtype="bf16", seed=3, D=False)
    assert _describe(inp, w, 64, "bf16", "fused") == ["ssd_fused_kernel"]
    y, _ = _gpu(inp, w, 64, ops="bf16", plan="fused")
    ref, _ = _reference(oracle_mod, inp, w, 16)
    assert_close(oracle_mod, y.double().cpu().numpy(), ref, "bf16", "fused norm, many units")


@pytest.mark.parametrize("shape,ops,plan,kernels", [
    ((2, 130, 32, 64, 64, 2, 64), "bf16", "fused", "ssd_fused_kernel,gated_rmsnorm"),  # 8 pairs per group
    ((2, 130, 16, 64, 64, 2, 64), "bf16", "fused", "ssd_fused_kernel,gated_rmsnorm"),  # 4 pairs per group
    ((2, 130, 8, 64, 64, 2, 64), "f32", "auto", None),                                 # chunked, fp32
    ((1, 300, 4, 64, 128, 1, 128), "bf16", "auto", None),                               # chunked, N = 128
    ((2, 96, 6, 32, 32, 3, 32), "f32", "auto", None),                                   # odd shapes
])
def test_norm_as_a_second_kernel(oracle_mod, shape, ops, plan, kernels):
    B, L, H, P, N, G, Q = shape
    inp, w = _case(B, L, H, P, N, G, Q, seed=sum(shape))
    desc = _describe(inp, w, Q, ops, plan)
    assert desc[-1] == "gated_rmsnorm", desc
    if kernels:
        assert ",".join(desc) == kernels
    y, fin = _gpu(inp, w, Q, ops=ops, plan=plan)
    ref, rfin = _reference(oracle_mod, inp, w, G)
    assert_close(oracle_mod, y.double().cpu().numpy(), ref, ops, f"norm second kernel {shape} {ops}")
    assert_close(oracle_mod, fin.double().cpu().numpy(), rfin, ops, "final state")


def test_fused_norm_is_deterministic_and_matches_the_two_kernel_path():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    inp, w = _case(2, 256, 8, 64, 64, 2, 64, dtype="bf16", seed=21)
    y1, _ = _gpu(inp, w, 64, ops="bf16", plan="fused")
    y2, _ = _gpu(inp, w, 64, ops="bf16", plan="fused")
    assert torch.equal(y1, y2)
    d = to_device(inp)
    ys = ssd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, dt_softplus=True, D=d["D"],
                            dt_bias=d["dt_bias"], initial_states=d["initial_states"], ops="bf16", plan="fused")
    Bb, L, H, P = ys.shape
    y3 = ssd.gated_rmsnorm(ys.reshape(Bb, L, H * P), d["z"].reshape(Bb, L, H * P), w.cuda(), 2, EPS)
    torch.cuda.synchronize()
    a, b = y1.reshape(Bb, L, H * P).double(), y3.double()
    rel = float((a - b).norm() / b.norm())
    assert rel < 1e-2, rel  # same operands; only the rounding of y (bf16) before the norm differs


def test_norm_with_packed_sequences(oracle_mod):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    lengths = [64, 1, 130, 77]
    T = sum(lengths)
    inp, w = _case(1, T, 8, 64, 64, 2, 64, seed=31)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    d = to_device(inp)
    h0 = inp["initial_states"].repeat(len(lengths), 1, 1, 1)
    y, fin = ssd.mamba2_ssd_fwd_varlen(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, cu, dt_softplus=True,
                                       return_final_state=True, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                                       initial_states=h0.cuda(), ops="bf16", plan="fused", norm_weight=w.cuda(),
                                       norm_eps=EPS)
    torch.cuda.synchronize()
    for s in range(len(lengths)):
        lo, hi = int(cu[s]), int(cu[s + 1])
        part = {k: (v[:, lo:hi] if k in ("x", "dt", "B", "C", "z") else v) for k, v in inp.items()}
        ref, _ = _reference(oracle_mod, part, w, 2)
        assert_close(oracle_mod, y[:, lo:hi].double().cpu().numpy(), ref, "bf16", f"varlen norm seq {s}")


def test_norm_through_host_buffers():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    inp, w = _case(4, 192, 8, 64, 64, 2, 64, seed=41)
    yd, fd = _gpu(inp, w, 64, ops="bf16")
    h = {k: (v.contiguous().pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.full_like(h["x"], float("nan")).pin_memory()
    fin = torch.full(fd.shape, float("nan")).pin_memory()
    wp = w.pin_memory()
    a = ssd.make_args(h["x"], h["dt"], h["A"], h["B"], h["C"], 64, y=y, final_state=fin, D=h["D"], z=h["z"],
                      dt_bias=h["dt_bias"], initial_states=h["initial_states"], dt_softplus=True, ops="bf16",
                      norm_weight=wp, norm_eps=EPS)
    ws = torch.empty(ssd.ssd_fwd_host_workspace_size(a), dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    ssd.ssd_fwd_host(a)
    torch.cuda.synchronize()
    assert torch.equal(y, yd.cpu()) and torch.equal(fin, fd.cpu())


def test_fused_norm_leaves_no_device_error():
    """No wait of the cluster exchange (or of the pipeline) gave up: the
    kernel's error word is clear after runs with clusters of 1 and 2 CTAs."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    for H in (4, 8):
        inp, w = _case(2, 256, H, 64, 64, 2, 64, dtype="bf16", seed=51 + H)
        d = to_device(inp)
        y = torch.empty_like(d["x"])
        a = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, y=y, D=d["D"], z=d["z"],
                          dt_bias=d["dt_bias"], initial_states=d["initial_states"], dt_softplus=True, ops="bf16",
                          plan="fused", norm_weight=w.cuda(), norm_eps=EPS)
        ws = torch.zeros(ssd.ssd_fwd_workspace_size(a), dtype=torch.uint8, device="cuda")
        a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
        for _ in range(3):
            ssd.ssd_fwd(a)
        ssd.ssd_check_device_error(a)  # raises on a set error word
        assert torch.isfinite(y).all()
