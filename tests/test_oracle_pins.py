"""Pins for the float64 oracle: it is checked against things other than itself.

Each test fixes the oracle to a result the mathematics determines on its own:
the quadratic "attention form" of SSD duality computed by brute force, closed
forms (A = 0, dt' = 0, dt' -> 0, the memoryless limit, the scalar case),
linearity, group broadcast, split consistency, the chunked decomposition of
the ops-transformer MambaV2 article (sections 4.2-4.5), and softplus values
from an independent arbitrary-precision library.  Sources:
"Mamba-2 SSD for Ascend NPU" README ("Usage", "Implementation") and the
ops-transformer MambaV2 article (sections 1.1-1.3, 4.2-4.5).
"""
import math

import numpy as np
import pytest

import ssd_inputs


def _problem(oracle_mod, inp, **over):
    kw = dict(D=inp["D"], z=inp["z"], dt_bias=inp["dt_bias"],
              initial_states=inp["initial_states"], dt_softplus=inp["dt_softplus"])
    kw.update(over)
    return oracle_mod.Problem(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], **kw)


def _silu(v):
    return v / (1.0 + np.exp(-v))


def _np_softplus(u):
    return np.where(u > 0, u + np.log1p(np.exp(-np.abs(u))), np.log1p(np.exp(np.minimum(u, 0))))


def attention_form(x, dt, A, Bm, Cm, D=None, z=None, dt_bias=None, h0=None, softplus=True):
    """y = (Lmask o C B^T)(d o x) + diag(e^cs) C h0^T + D x, gated by silu(z).

    SSD duality (ops-transformer MambaV2 article, section 1.3): the recurrence
    equals a multiply by a semiseparable matrix, with Lmask[t,s] =
    exp(cs_t - cs_s) for s <= t (0 above the diagonal) and cs the inclusive
    cumulative sum of d*A over the whole sequence.  Written with no loop over
    time, in float64, for tiny sizes only.
    """
    x = np.asarray(x, np.float64); dt = np.asarray(dt, np.float64)
    Bm = np.asarray(Bm, np.float64); Cm = np.asarray(Cm, np.float64)
    Bb, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    r = H // G
    y = np.zeros((Bb, L, H, P))
    fin = np.zeros((Bb, H, P, N))
    tri = np.tril(np.ones((L, L), dtype=bool))
    for b in range(Bb):
        for h in range(H):
            g = h // r
            u = dt[b, :, h] + (0.0 if dt_bias is None else float(dt_bias[h]))
            d = _np_softplus(u) if softplus else u
            cs = np.cumsum(d * float(A[h]))
            diffm = cs[:, None] - cs[None, :]
            Lm = np.where(tri, np.exp(np.where(tri, diffm, 0.0)), 0.0)
            CB = Cm[b, :, g, :] @ Bm[b, :, g, :].T            # [L, L]
            xs = d[:, None] * x[b, :, h, :]                   # [L, P]
            yy = (Lm * CB) @ xs
            if h0 is not None:
                hh = np.asarray(h0[b, h], np.float64)         # [P, N]
                yy += np.exp(cs)[:, None] * (Cm[b, :, g, :] @ hh.T)
            if D is not None:
                yy += float(D[h]) * x[b, :, h, :]
            if z is not None:
                yy *= _silu(np.asarray(z[b, :, h, :], np.float64))
            y[b, :, h, :] = yy
            w = np.exp(cs[-1] - cs) * d                        # [L]
            f = (x[b, :, h, :] * w[:, None]).T @ Bm[b, :, g, :]
            if h0 is not None:
                f += np.exp(cs[-1]) * np.asarray(h0[b, h], np.float64)
            fin[b, h] = f
    return y, fin


def _rel(a, b):
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-300))


@pytest.mark.parametrize("feat", [
    dict(),
    dict(D=True, z=True, dt_bias=True, h0=True),
    dict(h0=True, dt_bias=True),
])
@pytest.mark.parametrize("dims", [(2, 33, 4, 8, 5, 2), (1, 48, 3, 4, 16, 1), (1, 17, 6, 3, 7, 3)])
def test_attention_form_equals_recurrence(oracle_mod, feat, dims):
    B, L, H, P, N, G = dims
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, 16, seed=11 + L, **feat)
    prob = _problem(oracle_mod, inp)
    y, fin = oracle_mod.forward(prob)
    ya, fa = attention_form(inp["x"].float().numpy(), inp["dt"].numpy(), inp["A"].numpy(),
                            inp["B"].float().numpy(), inp["C"].float().numpy(),
                            D=None if inp["D"] is None else inp["D"].numpy(),
                            z=None if inp["z"] is None else inp["z"].float().numpy(),
                            dt_bias=None if inp["dt_bias"] is None else inp["dt_bias"].numpy(),
                            h0=None if inp["initial_states"] is None else inp["initial_states"].numpy())
    assert _rel(y, ya) < 1e-12
    assert _rel(fin, fa) < 1e-12


def test_zero_decay_is_cumulative_sum(oracle_mod):
    """A = 0: h_t = h0 + sum_{s<=t} d_s x_s B_s^T, a pure running sum."""
    B, L, H, P, N, G = 2, 40, 2, 5, 6, 1
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, 16, seed=3, h0=True)
    inp["A"] = inp["A"] * 0.0
    prob = _problem(oracle_mod, inp)
    y, fin = oracle_mod.forward(prob)
    x = inp["x"].double().numpy(); Bm = inp["B"].double().numpy(); Cm = inp["C"].double().numpy()
    d = _np_softplus(inp["dt"].double().numpy())
    h0 = inp["initial_states"].double().numpy()
    outer = np.einsum("blh,blhp,bln->blhpn", d, x, Bm[:, :, 0, :])
    hs = np.cumsum(outer, axis=1) + h0[:, None]
    yref = np.einsum("blhpn,bln->blhp", hs, Cm[:, :, 0, :])
    assert _rel(y, yref) < 1e-12
    assert _rel(fin, hs[:, -1]) < 1e-12


def test_zero_step_keeps_initial_state(oracle_mod):
    """dt' = 0 (no softplus, dt = 0): y_t = C_t h0^T + D x_t, final = h0 exactly."""
    B, L, H, P, N, G = 1, 20, 4, 3, 5, 2
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, 8, seed=4, h0=True, D=True)
    inp["dt"] = inp["dt"] * 0.0
    prob = _problem(oracle_mod, inp, dt_softplus=False)
    y, fin = oracle_mod.forward(prob)
    h0 = inp["initial_states"].double().numpy()
    Cm = inp["C"].double().numpy(); x = inp["x"].double().numpy(); D = inp["D"].double().numpy()
    g = np.arange(H) // (H // G)
    yref = np.einsum("blhn,bhpn->blhp", Cm[:, :, g, :], h0) + D[None, None, :, None] * x
    assert np.array_equal(fin, h0)
    assert _rel(y, yref) < 1e-13


def test_small_step_limit(oracle_mod):
    """dt' = eps: y/eps -> sum_{s<=t} (C_t . B_s) x_s with an O(eps) error."""
    B, L, H, P, N, G = 1, 24, 2, 4, 6, 1
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, 8, seed=5)
    eps = 1e-7
    inp["dt"] = inp["dt"] * 0.0 + eps
    prob = _problem(oracle_mod, inp, dt_softplus=False)
    y, _ = oracle_mod.forward(prob)
    x = inp["x"].double().numpy(); Bm = inp["B"].double().numpy(); Cm = inp["C"].double().numpy()
    CB = np.einsum("btn,bsn->bts", Cm[:, :, 0], Bm[:, :, 0])
    CB = CB * np.tril(np.ones((L, L)))[None]
    yref = np.einsum("bts,bshp->bthp", CB, x)
    rel = _rel(y / eps, yref)
    assert rel < 50 * eps * L
    assert rel > 0.0  # the decay is really applied


def test_memoryless_limit(oracle_mod):
    """A = -1e4 and dt' >= ln 2: exp(dt' A) underflows to 0, so
    y_t = dt'_t (C_t . B_t) x_t."""
    B, L, H, P, N, G = 2, 30, 4, 3, 5, 2
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, 8, seed=6, h0=True)
    inp["A"] = inp["A"] * 0.0 - 1e4
    prob = _problem(oracle_mod, inp)
    y, _ = oracle_mod.forward(prob)
    x = inp["x"].double().numpy(); Bm = inp["B"].double().numpy(); Cm = inp["C"].double().numpy()
    d = _np_softplus(inp["dt"].double().numpy())
    g = np.arange(H) // (H // G)
    cb = np.einsum("blhn,blhn->blh", Cm[:, :, g], Bm[:, :, g])
    yref = (d * cb)[..., None] * x
    assert _rel(y, yref) < 1e-13


def test_scalar_textbook_case(oracle_mod):
    """B=H=G=P=N=1: y_t = C_t sum_s (prod_{s<r<=t} a_r) d_s B_s x_s, with the
    products formed explicitly in plain Python."""
    L = 25
    _, inp = ssd_inputs.custom(1, L, 1, 1, 1, 1, 8, seed=7, dt_bias=True)
    prob = _problem(oracle_mod, inp)
    y, _ = oracle_mod.forward(prob)
    x = [float(v) for v in inp["x"].flatten()]
    dt = [float(v) for v in inp["dt"].flatten()]
    Bv = [float(v) for v in inp["B"].flatten()]
    Cv = [float(v) for v in inp["C"].flatten()]
    A = float(inp["A"][0]); bias = float(inp["dt_bias"][0])
    d = [math.log1p(math.exp(u + bias)) for u in dt]
    a = [math.exp(dd * A) for dd in d]
    for t in range(L):
        acc = 0.0
        for s in range(t + 1):
            prod = 1.0
            for r in range(s + 1, t + 1):
                prod *= a[r]
            acc += prod * d[s] * Bv[s] * x[s]
        assert abs(y.flatten()[t] - Cv[t] * acc) <= 1e-13 * max(1.0, abs(Cv[t] * acc))


def test_linearity_in_x_and_h0(oracle_mod):
    B, L, H, P, N, G = 1, 30, 2, 4, 5, 1
    _, i1 = ssd_inputs.custom(B, L, H, P, N, G, 8, seed=8, h0=True, D=True)
    _, i2 = ssd_inputs.custom(B, L, H, P, N, G, 8, seed=9, h0=True, D=True)
    i3 = dict(i1)
    i3["x"] = (i1["x"].double() + i2["x"].double()).float()
    i3["initial_states"] = (i1["initial_states"].double() + i2["initial_states"].double()).float()
    i2 = dict(i2, dt=i1["dt"], B=i1["B"], C=i1["C"], A=i1["A"], D=i1["D"])
    y1, f1 = oracle_mod.forward(_problem(oracle_mod, i1))
    y2, f2 = oracle_mod.forward(_problem(oracle_mod, i2))
    y3, f3 = oracle_mod.forward(_problem(oracle_mod, i3))
    # i3's x and h0 were rounded to float32 after the sum
    assert _rel(y3, y1 + y2) < 1e-6
    assert _rel(f3, f1 + f2) < 1e-6


def test_group_broadcast(oracle_mod):
    """G < H gives the same result as G = H with B and C repeated per head."""
    B, L, H, P, N, G = 2, 20, 6, 3, 4, 2
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, 8, seed=10, h0=True, D=True, z=True)
    y, fin = oracle_mod.forward(_problem(oracle_mod, inp))
    rep = dict(inp)
    idx = np.arange(H) // (H // G)
    rep["B"] = inp["B"][:, :, idx]
    rep["C"] = inp["C"][:, :, idx]
    y2, fin2 = oracle_mod.forward(_problem(oracle_mod, rep))
    assert np.array_equal(y, y2) and np.array_equal(fin, fin2)
    # and a different group really changes the result
    swap = dict(inp)
    swap["B"] = inp["B"].flip(2)
    y3, _ = oracle_mod.forward(_problem(oracle_mod, swap))
    assert _rel(y3, y) > 1e-2


@pytest.mark.parametrize("L1", [16, 21])
def test_split_consistency(oracle_mod, L1):
    """run[0,L1) -> h; run[L1,L) from h0 = h reproduces the tail and the final
    state (the state carry of the ops-transformer article, section 4.4)."""
    B, L, H, P, N, G = 2, 48, 2, 4, 6, 1
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, 16, seed=12, h0=True, D=True)
    y, fin = oracle_mod.forward(_problem(oracle_mod, inp))
    head = {k: (v[:, :L1] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    _, fh = oracle_mod.forward(_problem(oracle_mod, head))
    tail = {k: (v[:, L1:] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    tail["initial_states"] = fh.astype(np.float32)
    yt, ft = oracle_mod.forward(_problem(oracle_mod, tail))
    assert _rel(yt, y[:, L1:]) < 1e-6
    assert _rel(ft, fin) < 1e-6


def test_softplus_against_arbitrary_precision(oracle_mod):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    for u in [-30.0, -5.0, -1.0, 0.0, 0.5, 1.0, 20.0, 30.0, 60.0]:
        want = float(mp.log(1 + mp.exp(mp.mpf(u))))
        got = oracle_mod.softplus(u)
        assert abs(got - want) <= 2e-16 * abs(want), (u, got, want)
    assert oracle_mod.softplus(0.0) == math.log(2.0)


def test_dt_pipeline_order(oracle_mod):
    """Bias is added first, then softplus, then the clamp ("softplus / clamp /
    decay").  The values are chosen so that any other order differs."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    x = np.zeros((1, 4, 1, 1), np.float32)
    dt = np.array([-1.0, 0.3, 3.0, -4.0], np.float32).reshape(1, 4, 1)
    A = np.array([-1.0], np.float32)
    Bm = np.zeros((1, 4, 1, 1), np.float32)
    bias = np.array([0.5], np.float32)
    lo, hi = 0.1, 0.9
    prob = oracle_mod.Problem(x, dt, A, Bm, Bm, dt_bias=bias, dt_softplus=True, dt_limit=(lo, hi))
    dtp, cs = oracle_mod.chunk_cumsum(prob, 4)
    for i, raw in enumerate([-1.0, 0.3, 3.0, -4.0]):
        sp = float(mp.log(1 + mp.exp(mp.mpf(raw) + mp.mpf(0.5))))
        want = min(max(sp, lo), hi)
        assert abs(dtp[0, 0, 0, i] - want) < 1e-15
    # no clamp by default
    prob2 = oracle_mod.Problem(x, dt, A, Bm, Bm, dt_bias=bias, dt_softplus=True)
    dtp2, _ = oracle_mod.chunk_cumsum(prob2, 4)
    assert abs(dtp2[0, 0, 0, 2] - float(mp.log(1 + mp.exp(mp.mpf(3.5))))) < 1e-15


def test_chunk_cumsum_and_tail(oracle_mod):
    """cs steps by d*A inside each chunk, restarts at each chunk, and past the
    end of a ragged sequence the step is 0 so cs holds its last value."""
    B, L, H, P, N, G, Q = 2, 37, 3, 2, 2, 1, 16
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=13, dt_bias=True)
    prob = _problem(oracle_mod, inp)
    dtp, cs = oracle_mod.chunk_cumsum(prob, Q)
    c = -(-L // Q)
    assert dtp.shape == (B, H, c, Q)
    A = inp["A"].double().numpy()
    u = inp["dt"].double().numpy() + inp["dt_bias"].double().numpy()[None, None, :]
    d = np.log1p(np.exp(u))  # u is small here, the plain form is exact enough
    dpad = np.zeros((B, c * Q, H)); dpad[:, :L] = d
    dref = dpad.reshape(B, c, Q, H).transpose(0, 3, 1, 2)
    assert np.max(np.abs(dtp - dref)) < 1e-14
    steps = np.diff(np.concatenate([np.zeros((B, H, c, 1)), cs], axis=-1), axis=-1)
    assert np.max(np.abs(steps - dtp * A[None, :, None, None])) < 1e-13
    assert np.all(cs[:, :, -1, L - (c - 1) * Q:] == cs[:, :, -1, L - (c - 1) * Q - 1:L - (c - 1) * Q])


@pytest.mark.parametrize("Q", [8, 16, 32])
def test_chunked_decomposition(oracle_mod, Q):
    """The chunked SSD of the ops-transformer article, sections 4.3-4.5,
    rebuilt from oracle pieces, equals the recurrence for every chunk size:
      local state   dS_k = sum_j exp(cs_last - cs_j) d_j x_j B_j^T
      passing       S_{k+1} = exp(cs_last_k) S_k + dS_k
      scan          y_i = exp(cs_i) C_i S_k^T + sum_{j<=i} (C_i.B_j) exp(cs_i - cs_j) d_j x_j
    """
    B, L, H, P, N, G = 1, 45, 4, 3, 5, 2
    _, inp = ssd_inputs.custom(B, L, H, P, N, G, Q, seed=14, h0=True, D=True, z=True)
    prob = _problem(oracle_mod, inp)
    rec = oracle_mod.recurrence(prob, chunk=Q, want_chunk_states=True)
    dtp, cs = oracle_mod.chunk_cumsum(prob, Q)
    local = oracle_mod.chunk_local_states(prob, Q)
    c = -(-L // Q)
    x = inp["x"].double().numpy(); Bm = inp["B"].double().numpy(); Cm = inp["C"].double().numpy()
    D = inp["D"].double().numpy(); z = inp["z"].double().numpy()
    pad = c * Q - L
    xp = np.pad(x, ((0, 0), (0, pad), (0, 0), (0, 0)))
    Bp = np.pad(Bm, ((0, 0), (0, pad), (0, 0), (0, 0)))
    Cp = np.pad(Cm, ((0, 0), (0, pad), (0, 0), (0, 0)))
    zp = np.pad(z, ((0, 0), (0, pad), (0, 0), (0, 0)))
    r = H // G
    for i_bh, (b, h) in enumerate(rec["bh"]):
        g = h // r
        S = rec["chunk_states"][i_bh]
        for k in range(c):
            sl = slice(k * Q, (k + 1) * Q)
            csk, dk = cs[b, h, k], dtp[b, h, k]
            xs, Bs, Cs = xp[b, sl, h], Bp[b, sl, g], Cp[b, sl, g]
            w = np.exp(csk[-1] - csk) * dk
            dS = (xs * w[:, None]).T @ Bs
            assert _rel(local[i_bh, k], dS) < 1e-12
            if k + 1 < c:
                assert _rel(S[k + 1], np.exp(csk[-1]) * S[k] + dS) < 1e-12
            mask = np.tril(np.ones((Q, Q), dtype=bool))
            dec = np.where(mask, np.exp(np.where(mask, csk[:, None] - csk[None, :], 0.0)), 0.0)
            yk = np.exp(csk)[:, None] * (Cs @ S[k].T) + ((Cs @ Bs.T) * dec) @ (dk[:, None] * xs)
            yk = (yk + D[h] * xs) * _silu(zp[b, sl, h])
            n = min(Q, L - k * Q)
            assert _rel(yk[:n], rec["y"][i_bh, k * Q:k * Q + n]) < 1e-12
    fin = rec["final_state"]
    last = c - 1
    S_last = rec["chunk_states"][:, last]
    dS_last = local[:, last]
    a_last = np.exp(np.array([cs[b, h, last, -1] for b, h in rec["bh"]]))
    assert _rel(fin, a_last[:, None, None] * S_last + dS_last) < 1e-12


def test_oracle_rejects_bad_arguments(oracle_mod):
    _, inp = ssd_inputs.custom(1, 8, 2, 2, 2, 1, 4, seed=1)
    prob = _problem(oracle_mod, inp)
    with pytest.raises(ValueError):
        oracle_mod.recurrence(prob, [(0, 5)])
    with pytest.raises(ValueError):
        oracle_mod.recurrence(prob, [(3, 0)])


# ---- decode step (one token from a carried state) -------------------------------

def test_decode_step_scalar_closed_form(oracle_mod):
    """B = H = G = P = N = 1: one step by hand, s' = a s + d x b, y = (c s' + D x) silu(z)."""
    s0, x, dt, A, b, c, D, z, bias = 0.3, -1.2, 0.4, -0.7, 0.9, -1.1, 0.25, 0.6, -0.2
    f = lambda v, shp: np.full(shp, v, np.float32)
    yo, so = oracle_mod.decode_step(f(x, (1, 1, 1)), f(dt, (1, 1)), f(A, (1,)), f(b, (1, 1, 1)),
                                    f(c, (1, 1, 1)), f(s0, (1, 1, 1, 1)), D=f(D, (1,)),
                                    z=f(z, (1, 1, 1)), dt_bias=f(bias, (1,)))
    # the inputs were rounded to float32 on the way in: recompute from those values
    r = lambda v: float(np.float32(v))
    d = math.log1p(math.exp(r(dt) + r(bias)))
    s1 = math.exp(d * r(A)) * r(s0) + d * r(x) * r(b)
    y = (r(c) * s1 + r(D) * r(x)) * (r(z) / (1.0 + math.exp(-r(z))))
    assert abs(so[0, 0, 0, 0] - s1) <= 1e-12 * abs(s1)
    assert abs(yo[0, 0, 0] - y) <= 1e-12 * abs(y)


def test_decode_continues_the_forward(oracle_mod):
    """Stepping the last token from the state after L-1 tokens gives the
    forward's last output and final state (group broadcast G < H, D, z, bias)."""
    _, inp = ssd_inputs.custom(2, 33, 4, 8, 16, 2, 16, seed=21, D=True, z=True, dt_bias=True, h0=True)
    prob = _problem(oracle_mod, inp)
    y_full, fin_full = oracle_mod.forward(prob)
    head = {k: (v[:, :-1] if k in ("x", "dt", "B", "C", "z") else v) for k, v in inp.items()}
    _, fin_head = oracle_mod.forward(_problem(oracle_mod, head))
    t = -1
    yd, sd = oracle_mod.decode_step(inp["x"][:, t], inp["dt"][:, t], inp["A"], inp["B"][:, t],
                                    inp["C"][:, t], fin_head.astype(np.float32), D=inp["D"],
                                    z=inp["z"][:, t], dt_bias=inp["dt_bias"])
    # the carried state passes through float32 once: agreement to float32 rounding
    assert oracle_mod.compare(yd, y_full[:, t])["rel_l2"] < 1e-6
    assert oracle_mod.compare(sd, fin_full)["rel_l2"] < 1e-6


# ---- backward (adjoint) against finite differences of the forward ------------------

def _loss(oracle_mod, tensors, flags, dy, dfinal):
    prob = oracle_mod.Problem(tensors["x"], tensors["dt"], tensors["A"], tensors["B"], tensors["C"],
                              D=tensors.get("D"), z=tensors.get("z"), dt_bias=tensors.get("dt_bias"),
                              initial_states=tensors.get("h0"), **flags)
    y, fin = oracle_mod.forward(prob)
    return float(np.sum(y * dy) + np.sum(fin * dfinal))


@pytest.mark.parametrize("case", ["all_features", "grouped", "clamped"])
def test_backward_matches_central_differences(oracle_mod, case):
    """Every gradient of the adjoint recurrence, coordinate by coordinate,
    against (L(t + e) - L(t - e)) / (t+ - t-) of the forward oracle, with t+-
    the float32 values actually fed to it.  Linear inputs (x, B, C, D, h0) are
    exact up to rounding; dt, A, bias and z carry an O(e^2) truncation."""
    if case == "grouped":
        _, inp = ssd_inputs.custom(2, 5, 4, 3, 2, 2, 16, seed=31, D=True, dt_bias=True, h0=True)
        flags = dict(dt_softplus=True)
    elif case == "clamped":
        _, inp = ssd_inputs.custom(1, 6, 2, 2, 3, 1, 16, seed=32, D=True, h0=True,
                                   dt_dist=("uniform", -0.5, 2.0))
        flags = dict(dt_softplus=True, dt_limit=(0.3, 1.2))
    else:
        _, inp = ssd_inputs.custom(1, 6, 2, 3, 4, 1, 16, seed=33, D=True, z=True, dt_bias=True, h0=True)
        flags = dict(dt_softplus=True)
    rng = np.random.default_rng(7)
    Bb, L, H, P = inp["x"].shape
    N = inp["B"].shape[3]
    dy = rng.standard_normal((Bb, L, H, P)).astype(np.float32)
    dfinal = rng.standard_normal((Bb, H, P, N)).astype(np.float32)
    t = {"x": inp["x"].numpy(), "dt": inp["dt"].numpy(), "A": inp["A"].numpy(), "B": inp["B"].numpy(),
         "C": inp["C"].numpy(), "D": inp["D"].numpy(), "h0": inp["initial_states"].numpy()}
    if inp["z"] is not None:
        t["z"] = inp["z"].numpy()
    if inp["dt_bias"] is not None:
        t["dt_bias"] = inp["dt_bias"].numpy()
    prob = oracle_mod.Problem(t["x"], t["dt"], t["A"], t["B"], t["C"], D=t["D"], z=t.get("z"),
                              dt_bias=t.get("dt_bias"), initial_states=t["h0"], **flags)
    g = oracle_mod.backward(prob, dy, dfinal)
    names = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "h0": "dh0", "z": "dz",
             "dt_bias": "ddt_bias"}
    for name, gname in names.items():
        if name not in t:
            continue
        base = t[name]
        fd = np.zeros(base.shape)
        for idx in np.ndindex(base.shape):
            eps = 1e-3 * max(1.0, abs(float(base[idx])))
            plus, minus = base.copy(), base.copy()
            plus[idx] = np.float32(base[idx] + eps)
            minus[idx] = np.float32(base[idx] - eps)
            lp = _loss(oracle_mod, {**t, name: plus}, flags, dy, dfinal)
            lm = _loss(oracle_mod, {**t, name: minus}, flags, dy, dfinal)
            fd[idx] = (lp - lm) / (float(plus[idx]) - float(minus[idx]))
        got = np.asarray(g[gname], dtype=np.float64).reshape(fd.shape)
        scale = max(1.0, float(np.max(np.abs(fd))))
        assert np.max(np.abs(got - fd)) <= 2e-5 * scale, (case, name, np.max(np.abs(got - fd)), scale)
    if case == "clamped":
        # some steps sit outside the clamp: their raw-dt gradient is exactly zero
        d = np.logaddexp(0.0, t["dt"].astype(np.float64))
        outside = (d < 0.3) | (d > 1.2)
        assert outside.any() and np.all(g["ddt"][outside] == 0.0)


# ---- the SSD's neighbours: causal conv1d + SiLU, gated RMSNorm -------------------

def test_causal_conv1d_matches_numpy_convolve(oracle_mod):
    """Each channel is numpy's full convolution with the reversed taps, first S
    outputs (the causal part), plus bias, through SiLU."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 5, 17))
    w = rng.standard_normal((5, 4))
    bias = rng.standard_normal(5)
    out = oracle_mod.causal_conv1d(x, w, bias)
    for b in range(2):
        for d in range(5):
            full = np.convolve(x[b, d], w[d][::-1])[:17] + bias[d]
            ref = full / (1.0 + np.exp(-full))
            assert np.allclose(out[b, d], ref, rtol=1e-13, atol=1e-13)


def test_causal_conv1d_impulse_and_causality(oracle_mod):
    """A unit impulse at step 3 reproduces the taps (in order) from step 3 on
    and nothing before it; no bias, no SiLU."""
    x = np.zeros((1, 2, 12))
    x[0, :, 3] = 1.0
    w = np.array([[1.0, 2.0, 3.0, 4.0], [0.5, -1.0, 0.0, 2.0]])
    out = oracle_mod.causal_conv1d(x, w, silu=False)
    assert np.all(out[0, :, :3] == 0.0)
    assert np.allclose(out[0, 0, 3:7], [4.0, 3.0, 2.0, 1.0]) and np.allclose(out[0, 1, 3:7], [2.0, 0.0, -1.0, 0.5])
    assert np.all(out[0, :, 7:] == 0.0)


def test_gated_rmsnorm_closed_forms(oracle_mod):
    """With the gate at z -> +inf (silu(z) ~ z, here z large so silu(z)/z = 1 to
    1e-15) a group of equal values v normalises to sign(v) * w; scaling x
    leaves the output unchanged when eps = 0; one group of D equals the plain
    RMSNorm of the whole row."""
    D, G = 12, 3
    x = np.full((2, D), -2.5)
    z = np.full((2, D), 40.0)
    w = np.linspace(0.5, 2.0, D)
    out = oracle_mod.gated_rmsnorm(x, z, w, G, 0.0)
    assert np.allclose(out, -w[None, :], rtol=1e-12)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, D))
    z = rng.standard_normal((3, D))
    a = oracle_mod.gated_rmsnorm(x, z, w, G, 0.0)
    b = oracle_mod.gated_rmsnorm(7.0 * x, z, w, G, 0.0)
    assert np.allclose(a, b, rtol=1e-12)
    v = x * z / (1.0 + np.exp(-z))
    one = v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + 1e-5) * w
    assert np.allclose(oracle_mod.gated_rmsnorm(x, z, w, 1, 1e-5), one, rtol=1e-12)


def test_gated_rmsnorm_groups_are_runs_of_consecutive_channels(oracle_mod):
    """The article's grouped norm (ops-transformer MambaV2 article, section 4.6)
    normalises each of G runs of D/G consecutive channels on its own.  A row
    whose k-th run holds one constant c_k (distinct magnitudes) must come out as
    sign(c_k) * w channel by channel when eps = 0: a strided grouping (channel d
    in group d mod G) mixes the constants and fails, and so does a transposed
    reshape."""
    D, G = 12, 3
    c = np.array([0.5, -3.0, 7.0])
    x = np.repeat(c, D // G)[None, :]            # [c0 c0 c0 c0 c1 c1 ... c2]
    z = np.full((1, D), 40.0)                    # silu(40) = 40 to 4e-18
    w = np.linspace(0.25, 3.0, D)
    out = oracle_mod.gated_rmsnorm(x, z, w, G, 0.0)
    assert np.allclose(out[0], np.repeat(np.sign(c), D // G) * w, rtol=1e-12, atol=0)
    # the strided reading would give c_k / rms(c) * w, which differs for every run here
    strided_rms = np.sqrt(np.mean(c ** 2))
    assert not np.allclose(out[0], np.repeat(c / strided_rms, D // G) * w, rtol=1e-3)


def test_gated_rmsnorm_eps_inside_the_root_and_the_gate(oracle_mod):
    """eps sits inside the root: a run of equal gated values v gives
    v / sqrt(v^2 + eps) * w (with eps outside it would be v / (|v| + eps) * w,
    which differs at the values chosen).  With runs of one channel the gate is
    visible on its own: z = 1 gives silu(1) = 1 / (1 + e^-1) =
    0.7310585786300049 (the logistic function at 1), z = 0 gives 0, so the
    output is 0 there whatever x is."""
    D, G = 8, 2
    x = np.full((1, D), 0.01)
    z = np.full((1, D), 40.0)
    w = np.linspace(0.5, 2.0, D)
    eps = 0.1
    v = 0.4                                       # 0.01 * silu(40)
    out = oracle_mod.gated_rmsnorm(x, z, w, G, eps)
    assert np.allclose(out[0], v / np.sqrt(v * v + eps) * w, rtol=1e-12)
    assert not np.allclose(out[0], v / (v + eps) * w, rtol=1e-3)
    # groups of one channel: out = v / sqrt(v^2 + eps) * w with v = x silu(z)
    x1 = np.array([[2.0, -1.5, 3.0, 0.7]])
    z1 = np.array([[1.0, 1.0, 0.0, 1.0]])
    w1 = np.array([1.0, 2.0, 3.0, 4.0])
    s1 = 0.7310585786300049
    v1 = x1[0] * np.array([s1, s1, 0.0, s1])
    out1 = oracle_mod.gated_rmsnorm(x1, z1, w1, 4, 1e-3)
    assert np.allclose(out1[0], v1 / np.sqrt(v1 * v1 + 1e-3) * w1, rtol=1e-12, atol=1e-300)
    assert out1[0, 2] == 0.0
