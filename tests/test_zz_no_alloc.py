"""ssd_fwd_noalloc, the entry point for callers that cannot allocate device
memory (they run under an allocator they do not own, or in a plugin or a
latency-critical path where cudaMalloc is off limits).  It must give what
ssd_fwd gives with a caller-owned workspace, call after call, although every
call reuses the same scratch buffer inside the library.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import ssd_inputs
from _harness import TOL, oracle_problem, to_device

pytestmark = pytest.mark.gpu

CASES = [
    # (B, L, H, P, N, G, chunk), ops, public dtype, plan, a kernel the plan must launch
    ((1, 200, 2, 64, 128, 1, 128), "f32", "f32", "chunked", "chunk_scan"),    # CUDA-core kernels, ragged tail
    ((2, 384, 8, 64, 128, 2, 128), "bf16", "f32", "chunked", "chunk_scan_tc"),  # tensor-core kernels
    ((2, 256, 8, 64, 64, 2, 64), "bf16", "bf16", "fused", "ssd_fused_kernel"),       # fused plan
    ((1, 2048, 16, 64, 128, 1, 256), "bf16", "f32", "fused", "segment_state_kernel"),  # N = 128, segments
]


def _metrics(got, ref):
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    d = g - r
    return (float(np.linalg.norm(d) / max(np.linalg.norm(r), 1e-300)),
            float(np.max(np.abs(d)) / max(np.max(np.abs(r)), 1e-300)))


def _run(ssd, inp, Q, ops, plan, kernel, noalloc):
    d = to_device(inp)
    B, L, H, P = d["x"].shape
    y = torch.full_like(d["x"], float("nan"))
    fin = torch.full((B, H, P, d["B"].shape[3]), float("nan"), device="cuda")
    args = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], Q, y=y, final_state=fin, D=d["D"],
                         z=d["z"], dt_bias=d["dt_bias"], initial_states=d["initial_states"],
                         dt_softplus=True, ops=ops, plan=plan)
    assert kernel in ssd.ssd_fwd_describe(args), ssd.ssd_fwd_describe(args)
    if noalloc:
        ssd.ssd_fwd_noalloc(args)
    else:
        ws = torch.empty(max(ssd.ssd_fwd_workspace_size(args), 256), dtype=torch.uint8, device="cuda")
        args.workspace, args.workspace_bytes = ws.data_ptr(), ws.numel()
        ssd.ssd_fwd(args)
    torch.cuda.synchronize()
    return y, fin


@pytest.mark.parametrize("shape,ops,io,plan,kernel", CASES)
def test_noalloc_matches_ssd_fwd_on_consecutive_calls(oracle_mod, shape, ops, io, plan, kernel):
    """Two calls in a row with different inputs: each must equal ssd_fwd with a
    caller-owned workspace bit for bit (both run the same deterministic
    kernels, so any scratch left over from the previous call would show), and
    match the float64 oracle within the operand mode's tolerance."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, L, H, P, N, G, Q = shape
    for seed in (101, 202):  # two calls in a row, different inputs, same built-in scratch
        _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=seed, x_dtype=io, ops=ops, D=True, z=True,
                                   dt_bias=True, h0=True)
        y_ref, f_ref = _run(ssd, inp, Q, ops, plan, kernel, noalloc=False)
        y, f = _run(ssd, inp, Q, ops, plan, kernel, noalloc=True)
        for got, ref, what in ((y, y_ref, "y"), (f, f_ref, "final_state")):
            assert torch.isfinite(got.float()).all(), what
            if not torch.equal(got, ref):
                rel, mabs = _metrics(got, ref)
                raise AssertionError(f"{what} (seed {seed}) differs from ssd_fwd: rel_l2 {rel:.3e}, "
                                     f"max_abs_rel {mabs:.3e}")
        yr, fr = oracle_mod.forward(oracle_problem(oracle_mod, inp))
        tol = TOL[ops]
        for got, ref, what in ((y, yr, "y"), (f, fr, "final_state")):
            m = oracle_mod.compare(got.double().cpu().numpy(), ref)
            assert m["rel_l2"] <= tol["rel_l2"] and m["max_abs_rel"] <= tol["max_abs_rel"], (what, seed, m)


def test_noalloc_rejects_calls_larger_than_its_buffer():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    t = lambda *s: torch.empty(s, device="cuda")
    a = ssd.make_args(t(1, 64, 4, 64), t(1, 64, 4), t(4), t(1, 64, 2, 64), t(1, 64, 2, 64), 64,
                      y=t(1, 64, 4, 64), ops="f32", plan="chunked")
    a.B, a.L, a.H, a.G = 8, 4096, 256, 64  # chunk states alone would need 2 GiB
    with pytest.raises(ssd.SsdError) as ei:
        ssd.ssd_fwd_noalloc(a)
    assert ei.value.status == 3
    assert "built-in buffer" in str(ei.value)
