"""GPU parity: the CUDA path, called through the C ABI, against the float64
oracle on the same seeded inputs.

Small shapes are compared element by element in full (several chunks and a
ragged tail); the five named workloads run at full size and are compared
element by element over every (batch, head) sequence, the oracle recomputing
them block by block.
"""
import math

import numpy as np
import pytest
import torch

import ssd_inputs
from _harness import (TOL, assert_close, assert_metrics, gather_pairs, oracle_problem, pick_pairs,
                      run_gpu, stream_compare, to_device, workload_inputs)

pytestmark = pytest.mark.gpu


def _mode(ops):
    return {"f32": "f32", "f16": "f16", "bf16": "bf16"}[ops]


def _full_compare(oracle_mod, inp, y, fin, mode, what):
    prob = oracle_problem(oracle_mod, inp)
    yr, fr = oracle_mod.forward(prob)
    assert_close(oracle_mod, y.double().cpu().numpy(), yr, mode, what + " y")
    if fin is not None:
        assert_close(oracle_mod, fin.double().cpu().numpy(), fr, mode, what + " final_state")


# ---- named workloads at full size ---------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "same_device", "large_training", "long_sequence",
                                  "gated_prefill"])
def test_named_workload(oracle_mod, name):
    """Each named workload at full size on both plans (auto, and the chunked
    plan forced), compared with the oracle over every (batch, head) sequence
    and every element of y and final_state."""
    w, inp = workload_inputs(name)
    outs = {}
    for plan in ("auto", "chunked"):
        y, fin = run_gpu(inp, ops=w.ops, plan=plan)
        assert y.dtype == inp["x"].dtype
        outs[plan] = (y, fin)
    if name == "tiny":
        for plan, (y, fin) in outs.items():
            _full_compare(oracle_mod, inp, y, fin, _mode(w.ops), f"{name} {plan}")
        return
    prob = oracle_problem(oracle_mod, inp)
    res = stream_compare(oracle_mod, prob, outs, w.B, w.H, want_final=w.return_final_state)
    for plan, r in res.items():
        assert "y" in r
        assert_metrics(r["y"], _mode(w.ops), f"{name} {plan} y (all {w.B * w.H} sequences)")
        if w.return_final_state:
            assert_metrics(r["final_state"], _mode(w.ops), f"{name} {plan} final_state")


# ---- small shapes, every feature, element by element ----------------------------

SHAPES = [
    # B, L, H, P, N, G, chunk
    (1, 128, 2, 64, 128, 1, 128),
    (2, 200, 4, 32, 64, 2, 64),      # ragged tail
    (1, 77, 3, 16, 16, 1, 16),       # tiny dims, ragged
    (2, 300, 8, 64, 64, 8, 64),      # G = H
    (1, 513, 4, 64, 128, 1, 256),    # one token past a chunk boundary
    (3, 96, 6, 48, 80, 3, 32),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("feat", ["plain", "all"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_shapes(oracle_mod, shape, feat, dtype):
    B, L, H, P, N, G, Q = shape
    f = dict(D=True, z=True, dt_bias=True, h0=True) if feat == "all" else {}
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=hash(shape) % 1000, x_dtype=dtype,
                               ops=dtype, **f)
    y, fin = run_gpu(inp, ops=dtype)
    _full_compare(oracle_mod, inp, y, fin, dtype, f"{shape} {feat} {dtype}")


@pytest.mark.parametrize("ops", ["f32", "f16", "bf16"])
def test_operand_modes(oracle_mod, ops):
    _, inp = ssd_inputs.custom(2, 256, 8, 64, 64, 2, 64, seed=21, ops=ops, h0=True, D=True)
    y, fin = run_gpu(inp, ops=ops)
    _full_compare(oracle_mod, inp, y, fin, ops, f"ops={ops}")


def test_dt_limit_and_no_softplus(oracle_mod):
    _, inp = ssd_inputs.custom(1, 160, 4, 32, 32, 2, 32, seed=22, dt_bias=True,
                               dt_dist=("uniform", -0.5, 1.5), dt_softplus=False)
    y, fin = run_gpu(inp, ops="f32", dt_limit=(0.05, 0.8))
    prob = oracle_problem(oracle_mod, inp, dt_limit=(0.05, 0.8))
    yr, fr = oracle_mod.forward(prob)
    assert_close(oracle_mod, y.double().cpu().numpy(), yr, "f32", "dt_limit y")
    assert_close(oracle_mod, fin.double().cpu().numpy(), fr, "f32", "dt_limit final")


# ---- the four steps, one at a time -------------------------------------------------

def _stage_setup(oracle_mod, shape=(2, 200, 4, 32, 64, 2, 64), dtype="f32", **feat):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, L, H, P, N, G, Q = shape
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=31, x_dtype=dtype, **feat)
    d = to_device(inp)
    c = -(-L // Q)
    y = torch.empty_like(d["x"])
    fin = torch.empty((B, H, P, N), device="cuda")
    args = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], Q, y=y, final_state=fin,
                         D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                         initial_states=d["initial_states"], dt_softplus=True)
    prob = oracle_problem(oracle_mod, inp)
    return ssd, inp, d, args, prob, (B, L, H, P, N, G, Q, c), y, fin


def test_stage_chunk_cumsum(oracle_mod):
    ssd, inp, d, args, prob, (B, L, H, P, N, G, Q, c), _, _ = _stage_setup(oracle_mod, dt_bias=True)
    dtp = torch.full((B, H, c, Q), float("nan"), device="cuda")
    cs = torch.full((B, H, c, Q), float("nan"), device="cuda")
    ssd.ssd_chunk_cumsum(args, dtp, cs)
    torch.cuda.synchronize()
    rd, rc = oracle_mod.chunk_cumsum(prob, Q)
    assert_close(oracle_mod, dtp.double().cpu().numpy(), rd, "f32", "dtp")
    assert_close(oracle_mod, cs.double().cpu().numpy(), rc, "f32", "cs")
    # past the ragged end: zero step, constant cumulative sum
    tail = L - (c - 1) * Q
    assert torch.all(dtp[:, :, -1, tail:] == 0)
    assert torch.all(cs[:, :, -1, tail:] == cs[:, :, -1, tail - 1:tail])


def test_stage_chunk_state(oracle_mod):
    ssd, inp, d, args, prob, (B, L, H, P, N, G, Q, c), _, _ = _stage_setup(oracle_mod, dt_bias=True)
    rd, rc = oracle_mod.chunk_cumsum(prob, Q)
    dtp = torch.from_numpy(rd).float().cuda()
    cs = torch.from_numpy(rc).float().cuda()
    states = torch.full((B, c, H, P, N), float("nan"), device="cuda")
    ssd.ssd_chunk_state(args, dtp, cs, states)
    torch.cuda.synchronize()
    ref = oracle_mod.chunk_local_states(prob, Q)              # [B*H, c, P, N]
    got = states.permute(0, 2, 1, 3, 4).reshape(B * H, c, P, N)
    assert_close(oracle_mod, got.double().cpu().numpy(), ref, "f32", "chunk states")


def test_stage_state_passing(oracle_mod):
    ssd, inp, d, args, prob, (B, L, H, P, N, G, Q, c), _, fin = _stage_setup(
        oracle_mod, h0=True, dt_bias=True)
    _, rc = oracle_mod.chunk_cumsum(prob, Q)
    local = oracle_mod.chunk_local_states(prob, Q).reshape(B, H, c, P, N)
    states = torch.from_numpy(local).float().permute(0, 2, 1, 3, 4).contiguous().cuda()
    cs = torch.from_numpy(rc).float().cuda()
    ssd.ssd_state_passing(args, cs, states)
    torch.cuda.synchronize()
    rec = oracle_mod.recurrence(prob, chunk=Q, want_y=False, want_chunk_states=True)
    got = states.permute(0, 2, 1, 3, 4).reshape(B * H, c, P, N)
    assert_close(oracle_mod, got.double().cpu().numpy(), rec["chunk_states"], "f32", "entering states")
    assert_close(oracle_mod, fin.double().cpu().numpy().reshape(B * H, P, N), rec["final_state"],
                 "f32", "final state")


def test_stage_chunk_scan(oracle_mod):
    ssd, inp, d, args, prob, (B, L, H, P, N, G, Q, c), y, _ = _stage_setup(
        oracle_mod, h0=True, D=True, z=True, dt_bias=True)
    rd, rc = oracle_mod.chunk_cumsum(prob, Q)
    rec = oracle_mod.recurrence(prob, chunk=Q, want_chunk_states=True)
    states = torch.from_numpy(rec["chunk_states"].reshape(B, H, c, P, N)).float()
    states = states.permute(0, 2, 1, 3, 4).contiguous().cuda()
    ssd.ssd_chunk_scan(args, torch.from_numpy(rd).float().cuda(), torch.from_numpy(rc).float().cuda(),
                       states)
    torch.cuda.synchronize()
    got = y.permute(0, 2, 1, 3).reshape(B * H, L, P)
    assert_close(oracle_mod, got.double().cpu().numpy(), rec["y"], "f32", "chunk scan y")


# ---- properties ------------------------------------------------------------------

def test_chunk_size_invariance(oracle_mod):
    _, inp = ssd_inputs.custom(1, 512, 4, 64, 128, 1, 64, seed=41, h0=True, D=True)
    outs = []
    for Q in (64, 128, 256):
        y, fin = run_gpu(inp, chunk=Q, ops="f32")
        outs.append((y.double().cpu().numpy(), fin.double().cpu().numpy()))
    yr, fr = oracle_mod.forward(oracle_problem(oracle_mod, inp))
    for y, f in outs:
        assert_close(oracle_mod, y, yr, "f32", "chunk invariance y")
        assert_close(oracle_mod, f, fr, "f32", "chunk invariance final")
    assert oracle_mod.compare(outs[0][0], outs[2][0])["rel_l2"] < 2e-6


@pytest.mark.parametrize("L1", [128, 150])
def test_split_consistency(oracle_mod, L1):
    _, inp = ssd_inputs.custom(2, 320, 4, 64, 64, 2, 64, seed=42, h0=True, D=True)
    y, fin = run_gpu(inp, ops="f32")
    head = {k: (v[:, :L1].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    _, fh = run_gpu(head, ops="f32")
    tail = {k: (v[:, L1:].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    tail["initial_states"] = fh.cpu()
    yt, ft = run_gpu(tail, ops="f32")
    m = oracle_mod.compare(yt.double().cpu().numpy(), y[:, L1:].double().cpu().numpy())
    assert m["rel_l2"] < 1e-5
    assert oracle_mod.compare(ft.double().cpu().numpy(), fin.double().cpu().numpy())["rel_l2"] < 1e-5


@pytest.mark.parametrize("name,plan", [("tiny", "auto"), ("same_device", "auto"),
                                       ("large_training", "auto"), ("gated_prefill", "auto")])
def test_bitwise_determinism(name, plan):
    w, inp = workload_inputs(name)
    y1, f1 = run_gpu(inp, ops=w.ops, plan=plan)
    y2, f2 = run_gpu(inp, ops=w.ops, plan=plan)
    assert torch.equal(y1, y2)
    if f1 is not None:
        assert torch.equal(f1, f2)


def test_outputs_stay_inside_their_buffers():
    """Canary guard bands around y and final_state, NaN-poisoned workspace."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    _, inp = ssd_inputs.custom(2, 200, 4, 64, 64, 2, 64, seed=43, h0=True, D=True, z=True)
    d = to_device(inp)
    B, L, H, P = inp["x"].shape
    N = inp["B"].shape[3]
    pad = 4096
    ybuf = torch.full((pad + B * L * H * P + pad,), 12345.0, device="cuda")
    fbuf = torch.full((pad + B * H * P * N + pad,), -777.0, device="cuda")
    y = ybuf[pad:pad + B * L * H * P].view(B, L, H, P)
    fin = fbuf[pad:pad + B * H * P * N].view(B, H, P, N)
    args = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, y=y, final_state=fin,
                         D=d["D"], z=d["z"], initial_states=d["initial_states"], dt_softplus=True)
    nws = ssd.ssd_fwd_workspace_size(args)
    ws = torch.full((nws // 4 + 1,), float("nan"), device="cuda")
    args.workspace, args.workspace_bytes = ws.data_ptr(), nws
    ssd.ssd_fwd(args)
    torch.cuda.synchronize()
    assert torch.all(ybuf[:pad] == 12345.0) and torch.all(ybuf[-pad:] == 12345.0)
    assert torch.all(fbuf[:pad] == -777.0) and torch.all(fbuf[-pad:] == -777.0)
    assert torch.isfinite(y).all() and torch.isfinite(fin).all()


def test_host_buffer_entry_matches_device_entry():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    _, inp = ssd_inputs.custom(2, 256, 4, 64, 64, 2, 64, seed=44, h0=True, D=True, z=True)
    yd, fd = run_gpu(inp, ops="f32")
    h = {k: (v.contiguous().pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.empty_like(h["x"]).pin_memory()
    B, L, H, P = h["x"].shape
    fin = torch.empty((B, H, P, h["B"].shape[3])).pin_memory()
    args = ssd.make_args(h["x"], h["dt"], h["A"], h["B"], h["C"], 64, y=y, final_state=fin,
                         D=h["D"], z=h["z"], initial_states=h["initial_states"], dt_softplus=True)
    nws = ssd.ssd_fwd_host_workspace_size(args)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    args.workspace, args.workspace_bytes = ws.data_ptr(), nws
    ssd.ssd_fwd_host(args)
    torch.cuda.synchronize()
    assert torch.equal(y, yd.cpu()) and torch.equal(fin, fd.cpu())


def _host_call(ssd, inp, chunk, ops, stream=None):
    h = {k: (v.contiguous().pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.full_like(h["x"], float("nan")).pin_memory()
    B, L, H, P = h["x"].shape
    fin = torch.full((B, H, P, h["B"].shape[3]), float("nan")).pin_memory()
    args = ssd.make_args(h["x"], h["dt"], h["A"], h["B"], h["C"], chunk, y=y, final_state=fin, D=h["D"], z=h["z"],
                         dt_bias=h["dt_bias"], initial_states=h["initial_states"], dt_softplus=True, ops=ops)
    nws = ssd.ssd_fwd_host_workspace_size(args)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    args.workspace, args.workspace_bytes = ws.data_ptr(), nws
    ssd.ssd_fwd_host(args, stream)
    return y, fin, (h, ws, args)


@pytest.mark.parametrize("B,L,H,P,G,ops", [
    (5, 192, 8, 64, 2, "bf16"),    # fused plan, 5 slices of one batch entry
    (11, 128, 4, 64, 1, "bf16"),   # 6 slices of 2, the last of 1
    (3, 33, 3, 16, 1, "f32"),      # per-batch strides not 256-byte multiples: one slice
])
def test_host_buffer_pipeline_matches_device_entry(B, L, H, P, G, ops):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    _, inp = ssd_inputs.custom(B, L, H, P, 64 if P == 64 else 32, G, 64 if P == 64 else 16, seed=B + L,
                               h0=True, D=True, z=True, dt_bias=True)
    chunk = 64 if P == 64 else 16
    d = to_device(inp)
    yd, fd = ssd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], chunk, dt_softplus=True,
                                return_final_state=True, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                                initial_states=d["initial_states"], ops=ops)
    y, fin, _ = _host_call(ssd, inp, chunk, ops)
    torch.cuda.synchronize()
    assert torch.equal(y, yd.cpu()) and torch.equal(fin, fd.cpu())


def _host_call_plan(ssd, inp, chunk, ops, plan, return_final=True):
    h = {k: (v.contiguous().pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.full_like(h["x"], float("nan")).pin_memory()
    B, L, H, P = h["x"].shape
    fin = torch.full((B, H, P, h["B"].shape[3]), float("nan")).pin_memory() if return_final else None
    args = ssd.make_args(h["x"], h["dt"], h["A"], h["B"], h["C"], chunk, y=y, final_state=fin, D=h["D"], z=h["z"],
                         dt_bias=h["dt_bias"], initial_states=h["initial_states"], dt_softplus=True, ops=ops,
                         plan=plan)
    nws = ssd.ssd_fwd_host_workspace_size(args)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    args.workspace, args.workspace_bytes = ws.data_ptr(), nws
    ssd.ssd_fwd_host(args)
    torch.cuda.synchronize()
    return y, fin


@pytest.mark.parametrize("B,L,H,G,ops,ret", [
    (2, 320, 8, 2, "bf16", True),    # fused plan, 5 sequence slices of 64 tokens
    (3, 300, 4, 1, "f16", True),     # a ragged last slice (44 tokens), f16 operands
    (2, 1024, 4, 2, "bf16", False),  # 16 slices; the carried state without a final_state output
])
def test_host_buffer_sequence_slices_on_the_fused_plan(B, L, H, G, ops, ret):
    """The fused plan at N = 64 sliced along the sequence (the fp32 state handed
    from slice to slice) equals one device call bit for bit."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    _, inp = ssd_inputs.custom(B, L, H, 64, 64, G, 64, seed=B * L + H, ops=ops, h0=True, D=True, z=True,
                               dt_bias=True)
    d = to_device(inp)
    args_probe = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, plan="fused", ops=ops)
    assert "ssd_fused_kernel" in ssd.ssd_fwd_describe(args_probe)
    res = ssd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, dt_softplus=True, return_final_state=ret,
                             D=d["D"], z=d["z"], dt_bias=d["dt_bias"], initial_states=d["initial_states"], ops=ops,
                             plan="fused")
    yd, fd = res if ret else (res, None)
    y, fin = _host_call_plan(ssd, inp, 64, ops, "fused", return_final=ret)
    assert torch.equal(y, yd.cpu())
    if ret:
        assert torch.equal(fin, fd.cpu())


def test_host_buffer_batch_slices_when_the_sequence_is_one_chunk():
    """A sequence of one chunk cannot be cut: the call goes in batch slices."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    _, inp = ssd_inputs.custom(6, 64, 4, 64, 64, 2, 64, seed=66, ops="bf16", h0=True, D=True)
    d = to_device(inp)
    yd, fd = ssd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, dt_softplus=True,
                                return_final_state=True, D=d["D"], initial_states=d["initial_states"], ops="bf16")
    y, fin = _host_call_plan(ssd, inp, 64, "bf16", "auto")
    assert torch.equal(y, yd.cpu()) and torch.equal(fin, fd.cpu())


def test_host_buffer_fused_n128_batch_slices(oracle_mod):
    """N = 128 on the fused plan goes in batch slices (its segments depend on the
    sequence length); each slice's segmentation differs from a whole-batch call,
    so it is held to the oracle."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    _, inp = ssd_inputs.custom(3, 1024, 4, 64, 128, 2, 128, seed=67, ops="bf16", h0=True, D=True)
    y, fin = _host_call_plan(ssd, inp, 128, "bf16", "fused")
    yr, fr = oracle_mod.forward(oracle_problem(oracle_mod, inp))
    assert_close(oracle_mod, y.double().numpy(), yr, "bf16", "host N=128 y")
    assert_close(oracle_mod, fin.double().numpy(), fr, "bf16", "host N=128 final_state")


def test_host_buffer_calls_back_to_back_stay_ordered():
    """Two calls on one stream with no synchronisation between them: the
    second call's copies in wait for the first call to finish."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    _, inp1 = ssd_inputs.custom(4, 256, 8, 64, 64, 2, 64, seed=61, h0=True)
    _, inp2 = ssd_inputs.custom(4, 256, 8, 64, 64, 2, 64, seed=62, h0=True)
    ref = []
    for inp in (inp1, inp2):
        d = to_device(inp)
        ref.append(ssd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, dt_softplus=True,
                                      return_final_state=True, initial_states=d["initial_states"], ops="bf16"))
    h = {k: (v.contiguous().pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp1.items()}
    h2 = {k: (v.contiguous().pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp2.items()}
    outs = []
    ws = None
    for hh in (h, h2):
        y = torch.full_like(hh["x"], float("nan")).pin_memory()
        fin = torch.full((4, 8, 64, 64), float("nan")).pin_memory()
        args = ssd.make_args(hh["x"], hh["dt"], hh["A"], hh["B"], hh["C"], 64, y=y, final_state=fin,
                             initial_states=hh["initial_states"], dt_softplus=True, ops="bf16")
        if ws is None:
            nws = ssd.ssd_fwd_host_workspace_size(args)
            ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
        args.workspace, args.workspace_bytes = ws.data_ptr(), ws.numel()  # one workspace for both calls
        ssd.ssd_fwd_host(args)
        outs.append((y, fin, args))
    torch.cuda.synchronize()
    for (y, fin, _), (yr, fr) in zip(outs, ref):
        assert torch.equal(y, yr.cpu()) and torch.equal(fin, fr.cpu())


def test_small_workspace_is_an_error_not_a_fault():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    _, inp = ssd_inputs.custom(1, 128, 2, 64, 64, 1, 64, seed=45)
    d = to_device(inp)
    y = torch.empty_like(d["x"])
    args = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, y=y, dt_softplus=True)
    nws = ssd.ssd_fwd_workspace_size(args)
    ws = torch.empty(nws - 256, dtype=torch.uint8, device="cuda")
    args.workspace, args.workspace_bytes = ws.data_ptr(), nws - 256
    with pytest.raises(ssd.SsdError) as ei:
        ssd.ssd_fwd(args)
    assert ei.value.status == 3
    ssd.ssd_check_device_error(ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, y=y,
                                             workspace=torch.zeros(256, dtype=torch.uint8, device="cuda")))


# ---- the fused tensor-core plan ---------------------------------------------------

FUSED_SHAPES = [
    # B, L, H, P, N, G, chunk  (P = N = chunk = 64, even heads per group)
    (1, 64, 2, 64, 64, 1, 64),       # one chunk, one unit
    (2, 256, 8, 64, 64, 2, 64),      # several chunks and units
    (1, 200, 4, 64, 64, 1, 64),      # ragged tail
    (3, 448, 12, 64, 64, 3, 64),     # 4 heads per group, 7 chunks
]


@pytest.mark.parametrize("shape", FUSED_SHAPES)
@pytest.mark.parametrize("feat", ["plain", "all"])
@pytest.mark.parametrize("io,ops", [("f32", "bf16"), ("f32", "f16"), ("bf16", "bf16")])
def test_fused_plan(oracle_mod, shape, feat, io, ops):
    B, L, H, P, N, G, Q = shape
    f = dict(D=True, z=True, dt_bias=True, h0=True) if feat == "all" else {}
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=7 + L + H, x_dtype=io, ops=ops, **f)
    y, fin = run_gpu(inp, ops=ops, plan="fused")
    _full_compare(oracle_mod, inp, y, fin, ops, f"fused {shape} {feat} {io}/{ops}")


@pytest.mark.parametrize("feat", ["plain", "all"])
def test_fused_plan_steep_decay(oracle_mod, feat):
    """Per-head decay rates from gentle to steep (|d A| up to ~24 per token):
    within-chunk decays far below fp32's range next to chunks that barely decay."""
    f = dict(D=True, z=True, dt_bias=True, h0=True) if feat == "all" else {}
    _, inp = ssd_inputs.custom(2, 448, 8, 64, 64, 2, 64, seed=81, ops="bf16",
                               dt_dist=("uniform", -3.0, 3.0), A_dist=("neg_uniform", 0.25, 8.0), **f)
    y, fin = run_gpu(inp, ops="bf16", plan="fused")
    _full_compare(oracle_mod, inp, y, fin, "bf16", f"fused steep decay {feat}")


def test_fused_plan_many_units(oracle_mod):
    """More units than CTAs, so each CTA walks several units in turn."""
    _, inp = ssd_inputs.custom(4, 128, 128, 64, 64, 32, 64, seed=77, ops="bf16", h0=True)
    y, fin = run_gpu(inp, ops="bf16", plan="fused")
    pairs = pick_pairs(4, 128, 12, seed=3)
    ref = oracle_mod.recurrence(oracle_problem(oracle_mod, inp), pairs)
    ys, fs = gather_pairs(y, fin, pairs)
    assert_close(oracle_mod, ys, ref["y"], "bf16", "fused many units y")
    assert_close(oracle_mod, fs, ref["final_state"], "bf16", "fused many units final")


def test_fused_plan_reports_no_device_error():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    _, inp = ssd_inputs.custom(2, 256, 8, 64, 64, 2, 64, seed=78, ops="bf16")
    d = to_device(inp)
    y = torch.empty_like(d["x"])
    args = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, y=y, dt_softplus=True,
                         ops="bf16", plan="fused")
    ws = torch.full((ssd.ssd_fwd_workspace_size(args),), 255, dtype=torch.uint8, device="cuda")
    args.workspace, args.workspace_bytes = ws.data_ptr(), ws.numel()
    ssd.ssd_fwd(args)
    ssd.ssd_check_device_error(args)


def test_fused_plan_rejects_unsupported_shape():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    _, inp = ssd_inputs.custom(1, 128, 2, 64, 96, 1, 64, seed=79, ops="bf16")  # N = 96
    with pytest.raises(ssd.SsdError) as ei:
        run_gpu(inp, ops="bf16", plan="fused")
    assert ei.value.status == 2


# ---- tensor-core chunk_state / chunk_scan (chunked plan, fp16/bf16 operands) ------------

def _stage_args(ssd, d, y, fin, Q, ops):
    return ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], Q, y=y, final_state=fin,
                         D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                         initial_states=d["initial_states"], dt_softplus=True, ops=ops)


@pytest.mark.parametrize("shape,ops", [((2, 300, 4, 64, 128, 2, 128), "bf16"),
                                       ((1, 512, 6, 64, 64, 3, 256), "f16"),
                                       ((2, 200, 2, 64, 128, 1, 64), "bf16")])
def test_stage_chunk_state_tensor_cores(oracle_mod, shape, ops):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, L, H, P, N, G, Q = shape
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=51, dt_bias=True)
    d = to_device(inp)
    c = -(-L // Q)
    args = _stage_args(ssd, d, torch.empty_like(d["x"]), None, Q, ops)
    prob = oracle_problem(oracle_mod, inp)
    rd, rc = oracle_mod.chunk_cumsum(prob, Q)
    states = torch.full((B, c, H, P, N), float("nan"), device="cuda")
    ssd.ssd_chunk_state(args, torch.from_numpy(rd).float().cuda(), torch.from_numpy(rc).float().cuda(), states)
    torch.cuda.synchronize()
    ref = oracle_mod.chunk_local_states(prob, Q)
    got = states.permute(0, 2, 1, 3, 4).reshape(B * H, c, P, N)
    assert_close(oracle_mod, got.double().cpu().numpy(), ref, ops, f"tc chunk states {shape}")


@pytest.mark.parametrize("shape,ops", [((2, 300, 4, 64, 128, 2, 128), "bf16"),
                                       ((1, 512, 6, 64, 64, 3, 256), "f16")])
def test_stage_chunk_scan_tensor_cores(oracle_mod, shape, ops):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, L, H, P, N, G, Q = shape
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=52, h0=True, D=True, z=True, dt_bias=True)
    d = to_device(inp)
    c = -(-L // Q)
    y = torch.full_like(d["x"], float("nan"))
    args = _stage_args(ssd, d, y, None, Q, ops)
    prob = oracle_problem(oracle_mod, inp)
    rd, rc = oracle_mod.chunk_cumsum(prob, Q)
    rec = oracle_mod.recurrence(prob, chunk=Q, want_chunk_states=True)
    states = torch.from_numpy(rec["chunk_states"].reshape(B, H, c, P, N)).float()
    states = states.permute(0, 2, 1, 3, 4).contiguous().cuda()
    ssd.ssd_chunk_scan(args, torch.from_numpy(rd).float().cuda(), torch.from_numpy(rc).float().cuda(), states)
    torch.cuda.synchronize()
    got = y.permute(0, 2, 1, 3).reshape(B * H, L, P)
    assert_close(oracle_mod, got.double().cpu().numpy(), rec["y"], ops, f"tc chunk scan {shape}")


@pytest.mark.parametrize("shape", [(1, 512, 4, 64, 64, 2, 256), (2, 384, 8, 64, 128, 2, 128),
                                   (1, 700, 4, 64, 128, 1, 256)])
@pytest.mark.parametrize("io,ops", [("f32", "bf16"), ("f32", "f16"), ("bf16", "bf16")])
def test_chunked_plan_tensor_cores(oracle_mod, shape, io, ops):
    B, L, H, P, N, G, Q = shape
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=53 + L, x_dtype=io, ops=ops, h0=True, D=True,
                               z=True, dt_bias=True)
    y, fin = run_gpu(inp, ops=ops, plan="chunked")
    _full_compare(oracle_mod, inp, y, fin, ops, f"tc chunked {shape} {io}/{ops}")
