"""GPU parity of the decode step (one token per sequence from a carried state,
``ssd_decode_step``) against the float64 oracle's step, which is the
recurrence for L = 1 (ops-transformer MambaV2 article, section 4.4: the final
state feeds the decode stage)."""
import numpy as np
import pytest
import torch

import ssd_inputs
from _harness import TOL, assert_close, oracle_problem

pytestmark = pytest.mark.gpu


def _step_inputs(B, H, P, N, G, *, dtype, seed, feats):
    """One token's inputs (drawn with the workloads' recipe, L = 1) and a state."""
    f = dict(D=True, z=True, dt_bias=True) if feats else {}
    _, inp = ssd_inputs.custom(B, 1, H, P, N, G, 16, seed=seed, x_dtype=dtype, ops=dtype, **f)
    gen = torch.Generator().manual_seed(seed + 1000)
    state = (torch.randn((B, H, P, N), generator=gen) * 0.5).float()
    one = {k: (v[:, 0] if k in ("x", "dt", "B", "C", "z") and v is not None else v) for k, v in inp.items()}
    return one, state


def _gpu_step(ssd, one, state):
    cu = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in one.items()}
    st = state.cuda().contiguous()
    y = ssd.mamba2_ssd_decode(cu["x"], cu["dt"], cu["A"], cu["B"], cu["C"], st, dt_softplus=True,
                              D=cu["D"], z=cu["z"], dt_bias=cu["dt_bias"])
    torch.cuda.synchronize()
    return y, st


def _oracle_step(oracle_mod, one, state):
    return oracle_mod.decode_step(one["x"], one["dt"], one["A"], one["B"], one["C"], state, D=one["D"],
                                  z=one["z"], dt_bias=one["dt_bias"], dt_softplus=True)


@pytest.mark.parametrize("shape", [
    # B, H, P, N, G
    (2, 4, 64, 64, 2),
    (3, 6, 48, 80, 3),    # P, N not multiples of 32
    (1, 2, 16, 128, 1),   # widest N
    (4, 8, 64, 64, 8),    # G = H
    (2, 4, 5, 7, 4),      # tiny odd dims
    (8, 64, 64, 128, 8),  # the streaming kernel, N = 128, more half-blocks than CTAs
    (2, 8, 64, 32, 4),    # the streaming kernel, N = 32
])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("feats", [False, True])
def test_decode_step_matches_oracle(oracle_mod, shape, dtype, feats):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, H, P, N, G = shape
    one, state = _step_inputs(B, H, P, N, G, dtype=dtype, seed=sum(shape) + (7 if feats else 0), feats=feats)
    y, st = _gpu_step(ssd, one, state)
    yr, sr = _oracle_step(oracle_mod, one, state)
    assert y.dtype == one["x"].dtype
    # the state is fp32 arithmetic throughout; y is rounded to the public dtype at the end
    assert_close(oracle_mod, st.double().cpu().numpy(), sr, "f32", f"decode {shape} {dtype} state")
    assert_close(oracle_mod, y.double().cpu().numpy(), yr, dtype if dtype != "f32" else "f32",
                 f"decode {shape} {dtype} y")


def test_decode_step_at_the_large_training_state_size(oracle_mod):
    """The state of the large training shape, [8,256,64,64] with G = 64."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    one, state = _step_inputs(8, 256, 64, 64, 64, dtype="f32", seed=33, feats=False)
    y, st = _gpu_step(ssd, one, state)
    yr, sr = _oracle_step(oracle_mod, one, state)
    assert_close(oracle_mod, st.double().cpu().numpy(), sr, "f32", "decode large state")
    assert_close(oracle_mod, y.double().cpu().numpy(), yr, "f32", "decode large y")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_continues_the_gpu_forward(oracle_mod, dtype):
    """Forward over the first L-k tokens (final state), then k decode steps:
    the outputs of the last k tokens and the final state match the oracle's
    forward over all L tokens."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, L, H, P, N, G, Q, k = 2, 200, 4, 64, 64, 2, 64, 5
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=91, x_dtype=dtype, ops=dtype, D=True, z=True,
                               dt_bias=True, h0=True)
    yr, fr = oracle_mod.forward(oracle_problem(oracle_mod, inp))
    cu = {kk: (v.cuda() if isinstance(v, torch.Tensor) else v) for kk, v in inp.items()}
    head = lambda t: t[:, :L - k].contiguous()
    _, st = ssd.mamba2_ssd_fwd(head(cu["x"]), head(cu["dt"]), cu["A"], head(cu["B"]), head(cu["C"]), Q,
                               dt_softplus=True, return_final_state=True, D=cu["D"], z=head(cu["z"]),
                               dt_bias=cu["dt_bias"], initial_states=cu["initial_states"], ops=dtype)
    ys = []
    for t in range(L - k, L):
        tok = lambda v: v[:, t].contiguous()
        ys.append(ssd.mamba2_ssd_decode(tok(cu["x"]), tok(cu["dt"]), cu["A"], tok(cu["B"]), tok(cu["C"]), st,
                                        dt_softplus=True, D=cu["D"], z=tok(cu["z"]), dt_bias=cu["dt_bias"]))
    torch.cuda.synchronize()
    yk = torch.stack(ys, dim=1).double().cpu().numpy()
    mode = "f32" if dtype == "f32" else dtype
    assert_close(oracle_mod, yk, yr[:, L - k:], mode, f"decode continuation {dtype} y")
    assert_close(oracle_mod, st.double().cpu().numpy(), fr, mode, f"decode continuation {dtype} final")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_streaming_kernel_with_many_units_per_cta(oracle_mod, dtype):
    """[64,512,32,32] with G = 8: 65536 half blocks over at most 912 CTAs, about
    72 units walked by each CTA with the next unit's loads in flight."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, H, P, N, G = 64, 512, 32, 32, 8
    one, state = _step_inputs(B, H, P, N, G, dtype=dtype, seed=61, feats=True)
    y, st = _gpu_step(ssd, one, state)
    yr, sr = _oracle_step(oracle_mod, one, state)
    assert_close(oracle_mod, st.double().cpu().numpy(), sr, "f32", f"decode many units {dtype} state")
    assert_close(oracle_mod, y.double().cpu().numpy(), yr, dtype, f"decode many units {dtype} y")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_step_with_an_unaligned_x_takes_the_streaming_kernel(oracle_mod, dtype):
    """x one element into its buffer (not 16-byte aligned): the streaming kernel
    reads x element by element; more half blocks (2048) than CTAs."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    one, state = _step_inputs(8, 128, 64, 64, 8, dtype=dtype, seed=12, feats=True)
    cu = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in one.items()}
    xb = torch.zeros(one["x"].numel() + 1, dtype=one["x"].dtype, device="cuda")
    x = xb[1:].view(one["x"].shape)
    x.copy_(cu["x"])
    assert x.data_ptr() % 16 != 0
    st = state.cuda().contiguous()
    y = ssd.mamba2_ssd_decode(x, cu["dt"], cu["A"], cu["B"], cu["C"], st, dt_softplus=True,
                              D=cu["D"], z=cu["z"], dt_bias=cu["dt_bias"])
    torch.cuda.synchronize()
    yr, sr = _oracle_step(oracle_mod, one, state)
    assert_close(oracle_mod, st.double().cpu().numpy(), sr, "f32", f"decode unaligned x {dtype} state")
    assert_close(oracle_mod, y.double().cpu().numpy(), yr, dtype, f"decode unaligned x {dtype} y")


def test_decode_step_with_an_unaligned_state_takes_the_scalar_kernel(oracle_mod):
    """A state that is not 16-byte aligned (a view 4 bytes into a buffer)."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    one, state = _step_inputs(2, 4, 32, 64, 2, dtype="f32", seed=8, feats=True)
    cu = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in one.items()}
    buf = torch.zeros(state.numel() + 1, device="cuda")
    st = buf[1:].view(state.shape)
    st.copy_(state.cuda())
    assert st.data_ptr() % 16 == 4
    y = ssd.mamba2_ssd_decode(cu["x"], cu["dt"], cu["A"], cu["B"], cu["C"], st, dt_softplus=True,
                              D=cu["D"], z=cu["z"], dt_bias=cu["dt_bias"])
    torch.cuda.synchronize()
    yr, sr = _oracle_step(oracle_mod, one, state)
    assert_close(oracle_mod, st.double().cpu().numpy(), sr, "f32", "decode unaligned state")
    assert_close(oracle_mod, y.double().cpu().numpy(), yr, "f32", "decode unaligned y")


def test_decode_step_is_deterministic():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    one, state = _step_inputs(4, 16, 64, 128, 4, dtype="bf16", seed=5, feats=True)
    y1, s1 = _gpu_step(ssd, one, state)
    y2, s2 = _gpu_step(ssd, one, state)
    assert torch.equal(y1, y2) and torch.equal(s1, s2)


def test_decode_rejects_bad_arguments_without_launching():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    one, state = _step_inputs(2, 4, 64, 64, 2, dtype="f32", seed=6, feats=False)
    cu = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in one.items()}
    wide = torch.zeros(2, 4, 64, 256, device="cuda")
    with pytest.raises(ssd.SsdError) as ei:
        ssd.mamba2_ssd_decode(cu["x"], cu["dt"], cu["A"], torch.zeros(2, 2, 256, device="cuda"),
                              torch.zeros(2, 2, 256, device="cuda"), wide)
    assert ei.value.status == 2
