"""The sequence-parallel exchange on CPU ranks: two gloo processes split the
tokens of every sequence, exchange their segments' (log-decay, state) maps and
must reproduce the float64 oracle's single-process forward.  The local
computations use the oracle (no GPU here); what is tested is the protocol of
``mamba_ssd_chunked_fwd_gb300.seqpar``: segment order, rank 0's initial
state, the exclusive fold, the final state on the last rank."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import ssd_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class OracleBackend:
    """The three local computations of the protocol, done by the float64
    oracle on CPU (results handed over as float32 tensors, as on GPUs)."""

    def __init__(self, oracle_mod, chunk, *, D=None, dt_bias=None):
        self.o, self.chunk, self.D, self.dt_bias = oracle_mod, chunk, D, dt_bias

    def _prob(self, seg, h0):
        return self.o.Problem(seg["x"], seg["dt"], seg["A"], seg["B"], seg["C"], D=self.D, z=seg.get("z"),
                              dt_bias=self.dt_bias, initial_states=h0, dt_softplus=True)

    def forward(self, seg, initial_states):
        y, fin = self.o.forward(self._prob(seg, initial_states))
        return torch.from_numpy(y).float(), torch.from_numpy(fin).float()

    def log_decay(self, seg):
        # total of d_t A[h] over the segment: each chunk's last cumulative value, summed
        _, cs = self.o.chunk_cumsum(self._prob(seg, None), self.chunk)
        return torch.from_numpy(cs[..., -1].sum(axis=-1)).float()

    def fold(self, log_decays, states):
        S = torch.zeros(states.shape[1:], dtype=torch.float64)
        for q in range(states.shape[0]):
            S = torch.exp(log_decays[q].double())[..., None, None] * S + states[q].double()
        return S.float()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, cut, feats, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    from mamba_ssd_chunked_fwd_gb300 import seqpar
    os.environ["MASTER_ADDR"], os.environ["MASTER_PORT"] = "127.0.0.1", str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _, inp = ssd_inputs.custom(2, 150, 4, 16, 8, 2, 32, seed=61, **feats)
        lo, hi = cut[rank], cut[rank + 1]
        seg = {k: inp[k][:, lo:hi].contiguous() for k in ("x", "dt", "B", "C")}
        seg["A"] = inp["A"]
        if inp["z"] is not None:
            seg["z"] = inp["z"][:, lo:hi].contiguous()
        be = OracleBackend(oracle, 32, D=inp["D"], dt_bias=inp["dt_bias"])
        y, fin = seqpar.ssd_fwd_seq_parallel(seg, backend=be, initial_states=inp["initial_states"])
        torch.save({"y": y, "final": fin}, os.path.join(out_dir, f"rank{rank}.pt"))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("cut,feats", [
    ([0, 64, 150], {}),                                                    # split on a chunk boundary
    ([0, 77, 150], dict(D=True, z=True, dt_bias=True, h0=True)),           # split inside a chunk
])
def test_two_gloo_ranks_reproduce_the_forward(oracle_mod, tmp_path, cut, feats):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), cut, feats, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    _, inp = ssd_inputs.custom(2, 150, 4, 16, 8, 2, 32, seed=61, **feats)
    prob = oracle_mod.Problem(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"], z=inp["z"],
                              dt_bias=inp["dt_bias"], initial_states=inp["initial_states"], dt_softplus=True)
    y_ref, fin_ref = oracle_mod.forward(prob)
    parts = [torch.load(os.path.join(tmp_path, f"rank{r}.pt")) for r in range(world)]
    y = torch.cat([p["y"] for p in parts], dim=1).double().numpy()
    # the exchanged maps pass through float32 once: agreement to float32 rounding
    assert oracle_mod.compare(y, y_ref)["rel_l2"] < 2e-6
    assert oracle_mod.compare(parts[-1]["final"].double().numpy(), fin_ref)["rel_l2"] < 2e-6
