"""The causal conv1d + SiLU in front of the SSD (ops-transformer MambaV2
article, sections 1.4 and 4.1), as the forward's conv_* arguments: inside the
fused kernel at N = 64, else as token-major conv kernels into the workspace.
The reference is the oracle's conv1d followed by the oracle's forward; the
in-kernel conv must also equal the two-kernel route bit for bit (the same
arithmetic in the same order)."""
import numpy as np
import pytest
import torch

import ssd_inputs
from _harness import TOL, assert_close, oracle_problem, to_device

pytestmark = pytest.mark.gpu


def _conv_params(H, P, G, N, W, bias, seed):
    g = torch.Generator().manual_seed(seed)
    wx = torch.randn((H * P, W), generator=g) * 0.5
    wb = torch.randn((G * N, W), generator=g) * 0.5
    wc = torch.randn((G * N, W), generator=g) * 0.5
    bx = torch.randn(H * P, generator=g) * 0.2 if bias else None
    bb = torch.randn(G * N, generator=g) * 0.2 if bias else None
    bc = torch.randn(G * N, generator=g) * 0.2 if bias else None
    return wx, bx, wb, bb, wc, bc


def _oracle_conv(oracle_mod, t, w, b):
    """Token-major [B, L, C] through the oracle's conv1d (channels first)."""
    x = t.float().numpy().transpose(0, 2, 1)
    out = oracle_mod.causal_conv1d(x, w.numpy(), None if b is None else b.numpy(), silu=True)
    return out.transpose(0, 2, 1)


def _run(ssd, d, Q, ops, plan, conv=None, x=None, Bm=None, Cm=None):
    y = torch.empty_like(d["x"])
    fin = torch.empty((d["x"].shape[0], d["x"].shape[2], d["x"].shape[3], d["B"].shape[3]), device="cuda")
    a = ssd.make_args(d["x"] if x is None else x, d["dt"], d["A"], d["B"] if Bm is None else Bm,
                      d["C"] if Cm is None else Cm, Q, y=y, final_state=fin, D=d["D"], z=d["z"],
                      dt_bias=d["dt_bias"], initial_states=d["initial_states"], dt_softplus=True, ops=ops,
                      plan=plan, conv=conv)
    kernels = ssd.ssd_fwd_describe(a)
    ws = torch.empty(max(ssd.ssd_fwd_workspace_size(a), 256), dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    ssd.ssd_fwd(a)
    torch.cuda.synchronize()
    return y, fin, kernels


CASES = [
    # shape (B, L, H, P, N, G, chunk), io, ops, plan, W, bias, where the conv runs
    ((2, 256, 8, 64, 64, 2, 64), "f32", "bf16", "fused", 4, True, "kernel"),
    ((1, 200, 4, 64, 64, 1, 64), "bf16", "bf16", "fused", 4, False, "kernel"),   # ragged tail
    ((3, 448, 12, 64, 64, 3, 64), "f32", "f16", "fused", 2, True, "kernel"),     # 4 heads per group
    ((2, 384, 8, 64, 128, 2, 128), "f32", "bf16", "fused", 4, True, "tokens"),   # N = 128
    ((1, 200, 2, 64, 128, 1, 128), "f32", "f32", "chunked", 3, True, "tokens"),  # exact mode
]


@pytest.mark.parametrize("shape,io,ops,plan,W,bias,where", CASES)
@pytest.mark.parametrize("feat", ["plain", "all"])
def test_conv_then_ssd_matches_the_oracle(oracle_mod, shape, io, ops, plan, W, bias, where, feat):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, L, H, P, N, G, Q = shape
    f = dict(D=True, z=True, dt_bias=True, h0=True) if feat == "all" else {}
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=31 + L + W, x_dtype=io, ops=ops, **f)
    wx, bx, wb, bb, wc, bc = _conv_params(H, P, G, N, W, bias, seed=L)
    d = to_device(inp)
    conv = tuple(None if t is None else t.cuda() for t in (wx, bx, wb, bb, wc, bc))
    y, fin, kernels = _run(ssd, d, Q, ops, plan, conv=conv)
    assert (kernels[0] == "conv_tokens_kernel") == (where == "tokens"), kernels
    # oracle: conv1d of x, B, C, then the forward
    xc = _oracle_conv(oracle_mod, inp["x"].reshape(B, L, H * P), wx, bx).reshape(B, L, H, P)
    Bc = _oracle_conv(oracle_mod, inp["B"].reshape(B, L, G * N), wb, bb).reshape(B, L, G, N)
    Cc = _oracle_conv(oracle_mod, inp["C"].reshape(B, L, G * N), wc, bc).reshape(B, L, G, N)
    prob = oracle_problem(oracle_mod, dict(inp, x=xc, B=Bc, C=Cc))
    yr, fr = oracle_mod.forward(prob)
    assert_close(oracle_mod, y.double().cpu().numpy(), yr, ops, f"conv+ssd {shape} {io}/{ops} y")
    assert_close(oracle_mod, fin.double().cpu().numpy(), fr, ops, f"conv+ssd {shape} {io}/{ops} final")


@pytest.mark.parametrize("io,ops", [("f32", "bf16"), ("bf16", "bf16")])
def test_in_kernel_conv_equals_the_two_kernel_route(io, ops):
    """The fused kernel's conv warps and the token-major conv kernel compute the
    same values in the same order.  With bf16 tensors both round them to bf16,
    so the forward that convolves in its load stage equals the forward on the
    convolved tensors bit for bit; with fp32 tensors the in-kernel route rounds
    the convolved values to the operand dtype before the decay weight
    multiplies them, one rounding more, so the two agree to the operand
    tolerance."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, L, H, P, N, G, Q = 2, 640, 8, 64, 64, 2, 64
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=41, x_dtype=io, ops=ops, D=True, z=True, h0=True)
    wx, bx, wb, bb, wc, bc = (None if t is None else t.cuda() for t in _conv_params(H, P, G, N, 4, True, 5))
    d = to_device(inp)
    y1, f1, k1 = _run(ssd, d, Q, ops, "fused", conv=(wx, bx, wb, bb, wc, bc))
    assert k1 == ["ssd_fused_kernel"]
    xc, Bc, Cc = torch.empty_like(d["x"]), torch.empty_like(d["B"]), torch.empty_like(d["C"])
    ssd.ssd_causal_conv1d_tokens(d["x"].view(B, L, H * P), wx, bx, xc.view(B, L, H * P))
    ssd.ssd_causal_conv1d_tokens(d["B"].view(B, L, G * N), wb, bb, Bc.view(B, L, G * N))
    ssd.ssd_causal_conv1d_tokens(d["C"].view(B, L, G * N), wc, bc, Cc.view(B, L, G * N))
    y2, f2, _ = _run(ssd, d, Q, ops, "fused", x=xc, Bm=Bc, Cm=Cc)
    if io == "bf16":
        assert torch.equal(y1, y2) and torch.equal(f1, f2)
    else:
        for a, b in ((y1, y2), (f1, f2)):
            rel = float((a.double() - b.double()).norm() / b.double().norm())
            assert rel < TOL[ops]["rel_l2"], rel


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("W", [1, 2, 4])
def test_conv1d_tokens_matches_the_oracle(oracle_mod, dtype, W):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    g = torch.Generator().manual_seed(W)
    B, S, C = 2, 77, 136
    x = torch.randn((B, S, C), generator=g).to(dtype)
    w = torch.randn((C, W), generator=g) * 0.5
    b = torch.randn(C, generator=g) * 0.2
    out = torch.empty_like(x, device="cuda")
    ssd.ssd_causal_conv1d_tokens(x.cuda(), w.cuda(), b.cuda(), out)
    torch.cuda.synchronize()
    ref = _oracle_conv(oracle_mod, x, w, b)
    mode = "f32" if dtype == torch.float32 else "bf16"
    assert_close(oracle_mod, out.double().cpu().numpy(), ref, mode, f"conv1d tokens W={W}")
