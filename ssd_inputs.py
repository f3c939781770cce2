"""Seeded synthetic inputs for the Mamba-2 SSD forward.

This module only draws random tensors; it holds none of the method's
arithmetic.  Both the float64 oracle (through the tests) and the CUDA library
(through the tests, the smoke check and the benchmark) are fed from here, so
they always see the same bits.

The workloads are the five shapes quoted for the SSD forward, written
[B, L, H, P, N, chunk, G] as in the "Mamba-2 SSD for Ascend NPU" README
("Benchmark" table and its notes; "Usage" for the tiny demo):

* ``tiny``            [1,128,2,64,128,128,1]    fp32, exact operands, final state
* ``same_device``     [4,2048,16,64,128,128,4]  fp32 public, fp16 operands, y only
* ``large_training``  [8,4096,256,64,64,64,64]  fp32 public, bf16 operands, final state
* ``long_sequence``   [1,16384,32,64,128,256,1] fp32 public, bf16 operands, dt_bias, final
* ``gated_prefill``   [2,8192,128,64,128,256,8] bf16 x/B/C/z, D, z gate, h0, final

Draw order is fixed: x, dt, A, B, C, dt_bias, D, z, initial_states (absent
tensors are skipped), all from one ``torch.Generator`` on the CPU seeded with
the workload's seed.  Low-precision tensors are drawn in float32 and rounded
to nearest-even by the cast.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int
    H: int
    P: int
    N: int
    G: int
    chunk: int
    seed: int
    x_dtype: str = "f32"          # dtype of x, B, C (and z, y)
    bc_dtype: str = "f32"
    ops: str = "f32"              # operand precision of the contractions
    dt_dist: tuple = ("uniform", 0.0, 1.0)
    A_dist: tuple = ("neg_uniform", 0.0, 1.0)
    dt_bias_std: float | None = None
    D_std: float | None = None
    z: bool = False
    h0_std: float | None = None
    return_final_state: bool = True
    dt_softplus: bool = True
    notes: dict = field(default_factory=dict, compare=False)

    @property
    def tokens(self) -> int:
        return self.B * self.L

    def shape_tuple(self):
        """[B, L, H, P, N, chunk, G], the order the README uses."""
        return [self.B, self.L, self.H, self.P, self.N, self.chunk, self.G]

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 128, 2, 64, 128, 1, 128, seed=1),
    "same_device": Workload("same_device", 4, 2048, 16, 64, 128, 4, 128, seed=2,
                            ops="f16", return_final_state=False),
    "large_training": Workload("large_training", 8, 4096, 256, 64, 64, 64, 64, seed=3,
                               ops="bf16"),
    "long_sequence": Workload("long_sequence", 1, 16384, 32, 64, 128, 1, 256, seed=4,
                              ops="bf16", dt_dist=("uniform", 0.001, 0.1),
                              A_dist=("neg_exp_uniform", 0.0, math.log(16.0)),
                              dt_bias_std=0.1),
    "gated_prefill": Workload("gated_prefill", 2, 8192, 128, 64, 128, 8, 256, seed=5,
                              x_dtype="bf16", bc_dtype="bf16", ops="bf16",
                              A_dist=("neg_uniform", 0.5, 8.0), D_std=1.0, z=True,
                              h0_std=0.1),
}


def _draw(dist, shape, gen):
    kind = dist[0]
    if kind == "uniform":
        lo, hi = dist[1], dist[2]
        return torch.rand(shape, generator=gen) * (hi - lo) + lo
    if kind == "neg_uniform":          # A = -U(lo, hi)
        lo, hi = dist[1], dist[2]
        return -(torch.rand(shape, generator=gen) * (hi - lo) + lo)
    if kind == "neg_exp_uniform":      # A = -exp(U(lo, hi))
        lo, hi = dist[1], dist[2]
        return -torch.exp(torch.rand(shape, generator=gen) * (hi - lo) + lo)
    if kind == "const":
        return torch.full(shape, float(dist[1]))
    raise ValueError(f"unknown distribution {dist}")


def make(w: Workload, seed: int | None = None) -> dict:
    """Draw the inputs of workload ``w`` on the CPU.

    Returns a dict with keys x, dt, A, B, C, dt_bias, D, z, initial_states
    (None where the workload has no such tensor) plus the flags
    dt_softplus / return_final_state / chunk_size.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed if seed is None else seed)
    xd, bd = _DT[w.x_dtype], _DT[w.bc_dtype]
    x = torch.randn((w.B, w.L, w.H, w.P), generator=gen).to(xd)
    dt = _draw(w.dt_dist, (w.B, w.L, w.H), gen).float()
    A = _draw(w.A_dist, (w.H,), gen).float()
    Bm = torch.randn((w.B, w.L, w.G, w.N), generator=gen).to(bd)
    Cm = torch.randn((w.B, w.L, w.G, w.N), generator=gen).to(bd)
    dt_bias = None
    if w.dt_bias_std is not None:
        dt_bias = (torch.randn((w.H,), generator=gen) * w.dt_bias_std).float()
    D = None
    if w.D_std is not None:
        D = (torch.randn((w.H,), generator=gen) * w.D_std).float()
    z = None
    if w.z:
        z = torch.randn((w.B, w.L, w.H, w.P), generator=gen).to(xd)
    h0 = None
    if w.h0_std is not None:
        h0 = (torch.randn((w.B, w.H, w.P, w.N), generator=gen) * w.h0_std).float()
    return {"x": x, "dt": dt, "A": A, "B": Bm, "C": Cm, "dt_bias": dt_bias, "D": D,
            "z": z, "initial_states": h0, "dt_softplus": w.dt_softplus,
            "return_final_state": w.return_final_state, "chunk_size": w.chunk}


def custom(B, L, H, P, N, G, chunk, *, seed=0, ops="f32", x_dtype="f32", D=False, z=False,
           dt_bias=False, h0=False, dt_dist=("uniform", 0.0, 1.0),
           A_dist=("neg_uniform", 0.0, 1.0), return_final_state=True, dt_softplus=True):
    """A small workload of any shape, drawn with the same recipe."""
    w = Workload("custom", B, L, H, P, N, G, chunk, seed=seed, x_dtype=x_dtype,
                 bc_dtype=x_dtype, ops=ops, dt_dist=dt_dist, A_dist=A_dist,
                 dt_bias_std=0.1 if dt_bias else None, D_std=1.0 if D else None, z=z,
                 h0_std=0.1 if h0 else None, return_final_state=return_final_state,
                 dt_softplus=dt_softplus)
    return w, make(w)
