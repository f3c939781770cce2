"""float64 CPU oracle for the Mamba-2 SSD forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product path (``mamba_ssd_chunked_fwd_gb300``)
never imports it, and this package never imports the product.

The arithmetic lives in ``ssd_oracle.c`` (the token-by-token recurrence, the
definition stated in the "Mamba-2 SSD for Ascend NPU" README, sections "Usage"
and "Implementation", and in the ops-transformer MambaV2 article, section 1.1).
This module only builds that file with gcc and marshals numpy arrays into it.

Inputs may be given as numpy arrays or CPU torch tensors of any float dtype;
they are widened to float32 (exact for fp32, bf16 and fp16) before the C code
widens them again, exactly, to float64.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("L", ctypes.c_int64), ("H", ctypes.c_int64),
        ("P", ctypes.c_int64), ("N", ctypes.c_int64), ("G", ctypes.c_int64),
        ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p), ("A", ctypes.c_void_p),
        ("Bm", ctypes.c_void_p), ("Cm", ctypes.c_void_p), ("D", ctypes.c_void_p),
        ("z", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p), ("h0", ctypes.c_void_p),
        ("dt_softplus", ctypes.c_int), ("has_dt_limit", ctypes.c_int),
        ("dt_min", ctypes.c_double), ("dt_max", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile ssd_oracle.c with gcc (-O2, OpenMP, no fast-math)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fno-fast-math", "-std=c99", "-shared", "-fPIC",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.oracle_softplus.restype = ctypes.c_double
        lib.oracle_softplus.argtypes = [ctypes.c_double]
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_recurrence.restype = ctypes.c_int
        lib.oracle_recurrence.argtypes = [
            ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_chunk_cumsum.restype = ctypes.c_int
        lib.oracle_chunk_cumsum.argtypes = [
            ctypes.POINTER(_Problem), ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_chunk_local_states.restype = ctypes.c_int
        lib.oracle_chunk_local_states.argtypes = [
            ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int]
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [
            ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        _lib = lib
    return _lib


def _f32(a):
    """Widen to a contiguous float32 numpy array (exact for fp32/bf16/fp16)."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        import torch
        a = a.detach().to("cpu")
        if a.dtype != torch.float32:
            a = a.to(torch.float32)
        a = a.contiguous().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


class Problem:
    """The inputs of one SSD forward, held as float32 numpy arrays.

    Shapes follow the README's public tensors: x [B,L,H,P], dt [B,L,H], A [H],
    B/C [B,L,G,N], D [H], z [B,L,H,P], dt_bias [H], initial_states [B,H,P,N].
    ``dt_limit`` is a (lo, hi) pair; the clamp is applied only when it differs
    from the no-op default (0, +inf).
    """

    def __init__(self, x, dt, A, B, C, *, D=None, z=None, dt_bias=None,
                 initial_states=None, dt_softplus=True, dt_limit=(0.0, math.inf)):
        self.x, self.dt, self.A = _f32(x), _f32(dt), _f32(A)
        self.B, self.C = _f32(B), _f32(C)
        self.D, self.z, self.dt_bias = _f32(D), _f32(z), _f32(dt_bias)
        self.h0 = _f32(initial_states)
        self.dt_softplus = bool(dt_softplus)
        lo, hi = float(dt_limit[0]), float(dt_limit[1])
        self.has_dt_limit = not (lo == 0.0 and hi == math.inf)
        self.dt_min, self.dt_max = lo, hi
        Bb, L, H, P = self.x.shape
        G, N = self.B.shape[2], self.B.shape[3]
        self.dims = (Bb, L, H, P, N, G)
        assert self.dt.shape == (Bb, L, H)
        assert self.A.shape == (H,)
        assert self.B.shape == (Bb, L, G, N) and self.C.shape == (Bb, L, G, N)
        assert H % G == 0
        if self.D is not None:
            assert self.D.shape == (H,)
        if self.z is not None:
            assert self.z.shape == self.x.shape
        if self.dt_bias is not None:
            assert self.dt_bias.shape == (H,)
        if self.h0 is not None:
            assert self.h0.shape == (Bb, H, P, N)

    def _struct(self):
        Bb, L, H, P, N, G = self.dims

        def ptr(a):
            return None if a is None else a.ctypes.data

        return _Problem(Bb, L, H, P, N, G, ptr(self.x), ptr(self.dt), ptr(self.A),
                        ptr(self.B), ptr(self.C), ptr(self.D), ptr(self.z),
                        ptr(self.dt_bias), ptr(self.h0), int(self.dt_softplus),
                        int(self.has_dt_limit), self.dt_min, self.dt_max)


def _bh_array(prob: Problem, bh):
    Bb, _, H = prob.dims[0], prob.dims[1], prob.dims[2]
    if bh is None:
        bh = [(b, h) for b in range(Bb) for h in range(H)]
    arr = np.ascontiguousarray(np.asarray(bh, dtype=np.int64).reshape(-1, 2))
    return arr


def threads() -> int:
    """Number of OpenMP threads the oracle uses by default."""
    return int(_load().oracle_threads())


def softplus(u: float) -> float:
    return float(_load().oracle_softplus(float(u)))


def recurrence(prob: Problem, bh=None, *, chunk=None, want_y=True, want_final=True,
               want_chunk_states=False, nthreads=0):
    """Token-by-token recurrence for the listed (b, h) pairs (default: all).

    Returns a dict with float64 arrays:
      y            [nbh, L, P]
      final_state  [nbh, P, N]
      chunk_states [nbh, c, P, N]  state entering each chunk (needs ``chunk``)
    and ``bh`` (the [nbh, 2] pair list).
    """
    lib = _load()
    Bb, L, H, P, N, G = prob.dims
    bha = _bh_array(prob, bh)
    nbh = bha.shape[0]
    y = np.empty((nbh, L, P), np.float64) if want_y else None
    fin = np.empty((nbh, P, N), np.float64) if want_final else None
    cs = None
    if want_chunk_states:
        assert chunk and chunk > 0
        c = -(-L // chunk)
        cs = np.empty((nbh, c, P, N), np.float64)
    st = prob._struct()
    rc = lib.oracle_recurrence(ctypes.byref(st), bha.ctypes.data, nbh,
                               None if y is None else y.ctypes.data,
                               None if fin is None else fin.ctypes.data,
                               int(chunk or 0), None if cs is None else cs.ctypes.data,
                               int(nthreads))
    if rc != 0:
        raise ValueError("oracle_recurrence rejected its arguments")
    return {"y": y, "final_state": fin, "chunk_states": cs, "bh": bha}


def forward(prob: Problem, *, chunk=None, nthreads=0):
    """Full forward in the public layout: y [B,L,H,P], final_state [B,H,P,N]."""
    Bb, L, H, P, N, G = prob.dims
    r = recurrence(prob, None, chunk=chunk, nthreads=nthreads)
    y = r["y"].reshape(Bb, H, L, P).transpose(0, 2, 1, 3)
    fin = r["final_state"].reshape(Bb, H, P, N)
    return np.ascontiguousarray(y), fin


def chunk_cumsum(prob: Problem, chunk: int):
    """dt' and the within-chunk inclusive cumsum of dt'*A, both [B,H,c,chunk]."""
    lib = _load()
    Bb, L, H, P, N, G = prob.dims
    c = -(-L // chunk)
    dtp = np.empty((Bb, H, c, chunk), np.float64)
    cs = np.empty((Bb, H, c, chunk), np.float64)
    st = prob._struct()
    if lib.oracle_chunk_cumsum(ctypes.byref(st), int(chunk), dtp.ctypes.data, cs.ctypes.data):
        raise ValueError("oracle_chunk_cumsum rejected its arguments")
    return dtp, cs


def chunk_local_states(prob: Problem, chunk: int, bh=None, nthreads=0):
    """State each chunk produces from a zero start, [nbh, c, P, N]."""
    lib = _load()
    Bb, L, H, P, N, G = prob.dims
    bha = _bh_array(prob, bh)
    c = -(-L // chunk)
    out = np.empty((bha.shape[0], c, P, N), np.float64)
    st = prob._struct()
    if lib.oracle_chunk_local_states(ctypes.byref(st), bha.ctypes.data, bha.shape[0],
                                     int(chunk), out.ctypes.data, int(nthreads)):
        raise ValueError("oracle_chunk_local_states rejected its arguments")
    return out


def backward(prob: Problem, dy, dfinal=None, *, nthreads=0):
    """Gradients of L = sum(dy * y) + sum(dfinal * final_state) with respect
    to every input of the forward, by the adjoint of the token recurrence (the
    SSD backward named in the "Mamba-2 SSD for Ascend NPU" README, "Limitations
    and roadmap"; the recurrence of the README's "Implementation").

    dy [B,L,H,P], dfinal [B,H,P,N] or None.  Returns float64 arrays in the
    public layouts: dx [B,L,H,P], dB, dC [B,L,G,N] (heads of a group summed),
    ddt [B,L,H] (with respect to the raw dt), dA, dD, ddt_bias [H] (batch
    summed), dz [B,L,H,P] (zeros without z), dh0 [B,H,P,N].
    """
    lib = _load()
    Bb, L, H, P, N, G = prob.dims
    bha = _bh_array(prob, None)
    nbh = bha.shape[0]
    dy32 = _f32(dy)
    assert dy32.shape == (Bb, L, H, P)
    dy_pairs = np.ascontiguousarray(dy32.transpose(0, 2, 1, 3).reshape(nbh, L, P))
    df = None
    if dfinal is not None:
        df = _f32(dfinal)
        assert df.shape == (Bb, H, P, N)
        df = np.ascontiguousarray(df.reshape(nbh, P, N))
    dx = np.empty((nbh, L, P)); dBh = np.empty((nbh, L, N)); dCh = np.empty((nbh, L, N))
    ddt = np.empty((nbh, L)); dA = np.empty(nbh); dD = np.empty(nbh); dbias = np.empty(nbh)
    dz = np.empty((nbh, L, P)); dh0 = np.empty((nbh, P, N))
    st = prob._struct()
    ptr = lambda a: None if a is None else a.ctypes.data
    rc = lib.oracle_backward(ctypes.byref(st), bha.ctypes.data, nbh, dy_pairs.ctypes.data, ptr(df),
                             dx.ctypes.data, dBh.ctypes.data, dCh.ctypes.data, ddt.ctypes.data,
                             dA.ctypes.data, dD.ctypes.data, dbias.ctypes.data, dz.ctypes.data,
                             dh0.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_backward rejected its arguments")
    hpg = H // G
    per_head = lambda a, w: a.reshape(Bb, H, L, w).transpose(0, 2, 1, 3)  # [B,L,H,w]
    out = {
        "dx": np.ascontiguousarray(per_head(dx, P)),
        "dB": per_head(dBh, N).reshape(Bb, L, G, hpg, N).sum(axis=3),
        "dC": per_head(dCh, N).reshape(Bb, L, G, hpg, N).sum(axis=3),
        "ddt": np.ascontiguousarray(ddt.reshape(Bb, H, L).transpose(0, 2, 1)),
        "dA": dA.reshape(Bb, H).sum(axis=0),
        "dD": dD.reshape(Bb, H).sum(axis=0),
        "ddt_bias": dbias.reshape(Bb, H).sum(axis=0),
        "dz": np.ascontiguousarray(per_head(dz, P)),
        "dh0": dh0.reshape(Bb, H, P, N),
    }
    return out


def decode_step(x, dt, A, B, C, state, *, D=None, z=None, dt_bias=None, dt_softplus=True,
                dt_limit=(0.0, math.inf)):
    """One recurrent step for a single new token, continuing from ``state``:
    the recurrence above for L = 1 with initial state ``state``
    (ops-transformer MambaV2 article, section 4.4: the final state feeds the
    decode stage).  x/z [B,H,P], dt [B,H], B/C [B,G,N], state [B,H,P,N]
    (widened to float32, exact for fp32 input).  Returns (y [B,H,P],
    new_state [B,H,P,N]) in float64.  Parity of this step rests on the pins of
    the recurrence; the continuation test pins the slicing done here."""
    def one(t):
        if t is None:
            return None
        t = _f32(t)
        return t.reshape((t.shape[0], 1) + t.shape[1:])

    prob = Problem(one(x), one(dt), A, one(B), one(C), D=D, z=one(z), dt_bias=dt_bias,
                   initial_states=state, dt_softplus=dt_softplus, dt_limit=dt_limit)
    y, fin = forward(prob)
    return y[:, 0], fin


def causal_conv1d(x, w, bias=None, *, silu=True):
    """Depthwise causal convolution along the sequence, then SiLU
    (ops-transformer MambaV2 article, sections 1.4 and 4.1: kernel width 4,
    bias, SiLU; the reference there is a grouped convolution with W-1 zeros of
    left padding, truncated to the first S steps).  x [B,D,S], w [D,W],
    bias [D]:  out[b,d,t] = silu(bias[d] + sum_k w[d,k] x[b,d,t-(W-1)+k]),
    x = 0 before the first step.  float64; written out term by term."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    Bb, D, S = x.shape
    W = w.shape[1]
    out = np.zeros((Bb, D, S))
    for k in range(W):
        shift = W - 1 - k  # tap k reads the input `shift` steps back
        out[:, :, shift:] += w[None, :, k, None] * x[:, :, :S - shift]
    if bias is not None:
        out += np.asarray(bias, dtype=np.float64)[None, :, None]
    if silu:
        out = out / (1.0 + np.exp(-out))
    return out


def gated_rmsnorm(x, z, w, groups, eps):
    """Gated, grouped RMSNorm (ops-transformer MambaV2 article, section 4.6):
    v = x * silu(z), normalised by the root mean square of v over each of the
    `groups` runs of D/groups consecutive channels (plus eps inside the root),
    times w.  x, z [..., D], w [D].  float64."""
    x = np.asarray(x, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    D = x.shape[-1]
    v = x * (z / (1.0 + np.exp(-z)))
    vg = v.reshape(v.shape[:-1] + (groups, D // groups))
    r = np.sqrt(np.mean(vg * vg, axis=-1, keepdims=True) + eps)
    return (vg / r).reshape(v.shape) * w


def compare(got, ref):
    """Global error metrics in float64: rel-L2, max|diff|/max|ref|, max|diff|."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    diff = g - r
    nref = float(np.linalg.norm(r.ravel()))
    ndiff = float(np.linalg.norm(diff.ravel()))
    mref = float(np.max(np.abs(r))) if r.size else 0.0
    mdiff = float(np.max(np.abs(diff))) if r.size else 0.0
    return {
        "rel_l2": ndiff / nref if nref > 0 else ndiff,
        "max_abs_rel": mdiff / mref if mref > 0 else mdiff,
        "max_abs": mdiff,
        "finite": bool(np.all(np.isfinite(g))),
    }
