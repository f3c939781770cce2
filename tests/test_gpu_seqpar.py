"""GPU parity of the sequence-parallel exchange's kernels and of the whole
protocol with W ranks emulated in one process (phase 1 of every rank, the
gathered maps stacked, phase 3 of every rank; no collective).  Reference: the
float64 oracle's single-process forward."""
import numpy as np
import pytest
import torch

import ssd_inputs
from _harness import assert_close, oracle_problem

pytestmark = pytest.mark.gpu


def test_segment_log_decay_matches_the_oracle(oracle_mod):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    _, inp = ssd_inputs.custom(3, 300, 8, 16, 16, 2, 64, seed=71, dt_bias=True,
                               A_dist=("neg_uniform", 0.0, 4.0))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.empty(3, 8, device="cuda")
    a = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, dt_bias=d["dt_bias"], dt_softplus=True)
    ssd.ssd_segment_log_decay(a, out)
    torch.cuda.synchronize()
    _, cs = oracle_mod.chunk_cumsum(oracle_problem(oracle_mod, inp), 64)
    ref = cs[..., -1].sum(axis=-1)
    assert np.max(np.abs(out.double().cpu().numpy() - ref) / np.maximum(1.0, np.abs(ref))) < 1e-6


def test_state_fold_matches_the_definition():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    g = torch.Generator().manual_seed(3)
    nseg, B, H, P, N = 4, 2, 3, 16, 32
    la = -torch.rand((nseg, B, H), generator=g) * 3
    st = torch.randn((nseg, B, H, P, N), generator=g)
    out = torch.empty(B, H, P, N, device="cuda")
    ssd.ssd_state_fold(la.cuda(), st.cuda(), out)
    ref = torch.zeros(B, H, P, N, dtype=torch.float64)
    for q in range(nseg):
        ref = torch.exp(la[q].double())[..., None, None] * ref + st[q].double()
    assert torch.allclose(out.double().cpu(), ref, rtol=1e-5, atol=1e-6)
    zero = torch.full((B, H, P, N), 7.0, device="cuda")
    ssd.ssd_state_fold(la[:0].cuda(), st[:0].cuda(), zero)
    assert torch.count_nonzero(zero) == 0


@pytest.mark.parametrize("cuts,dtype", [
    ([0, 256, 512], "f32"),          # 2 ranks, on chunk boundaries
    ([0, 100, 333, 512], "f32"),     # 3 ranks, inside chunks
    ([0, 192, 320, 512], "bf16"),    # 3 ranks, tensor-core operands
])
def test_emulated_ranks_reproduce_the_forward(oracle_mod, cuts, dtype):
    from mamba_ssd_chunked_fwd_gb300 import seqpar
    B, L, H, P, N, G, Q = 2, 512, 8, 64, 64, 4, 64
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=73, x_dtype=dtype, ops=dtype, D=True, z=True,
                               dt_bias=True, h0=True)
    y_ref, fin_ref = oracle_mod.forward(oracle_problem(oracle_mod, inp))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    be = seqpar.LibraryBackend(Q, D=d["D"], dt_bias=d["dt_bias"], ops=dtype)
    W = len(cuts) - 1
    segs = []
    for r in range(W):
        lo, hi = cuts[r], cuts[r + 1]
        seg = {k: d[k][:, lo:hi].contiguous() for k in ("x", "dt", "B", "C", "z")}
        seg["A"] = d["A"]
        segs.append(seg)
    summ = [seqpar.segment_summary(be, segs[r], r, d["initial_states"]) for r in range(W)]
    log_decays = torch.stack([s[0] for s in summ])
    states = torch.stack([s[1] for s in summ])
    ys, fin = [summ[0][2]], summ[0][1]
    for r in range(1, W):
        y, fin = be.forward(segs[r], seqpar.entering_state(be, log_decays, states, r))
        ys.append(y)
    torch.cuda.synchronize()
    y = torch.cat(ys, dim=1).double().cpu().numpy()
    assert_close(oracle_mod, y, y_ref, dtype, f"seq-parallel {cuts} {dtype} y")
    assert_close(oracle_mod, fin.double().cpu().numpy(), fin_ref, dtype, f"seq-parallel {cuts} {dtype} final")
