"""Sequence-parallel SSD forward: the token dimension of every sequence split
across the ranks of a process group.

Rank r of W holds tokens [L_r, L_{r+1}) of all B sequences (all heads).  Per
(b, h) a segment acts on the state entering it as an affine map,
S_out = exp(a) S_in + S_seg, with a = the segment's total d_t A[h] and S_seg its
final state from a zero start: the rule the chunk_state_passing step applies
between chunks (ops-transformer MambaV2 article, section 4.4), applied here
between segments held by different ranks.  Three phases:

1. local   -- the forward over the rank's segment from a zero state (rank 0:
              from the sequence's initial state) gives S_seg; the segment's
              total log-decay a comes from ``ssd_segment_log_decay``.  Rank 0's
              outputs are already final.
2. exchange -- all-gather of (a, S_seg): P*N*4 + 4 bytes per (b, h) per rank.
3. local   -- the state entering the segment is the fold of the maps of ranks
              0..r-1 (``ssd_state_fold``); the forward over the segment from
              that state gives the rank's y and, on the last rank, the final
              state of the whole sequence.

Every arithmetic step runs in the library's kernels (through ``backend``);
this module moves tensors between ranks and calls the entry points.  The
backend is pluggable so that the protocol can be exercised on CPU ranks.
"""
from __future__ import annotations

import math

import torch


class LibraryBackend:
    """The three local computations on the GPU through libssd_gb300.so."""

    def __init__(self, chunk_size, *, dt_softplus=True, D=None, dt_bias=None, dt_limit=(0.0, math.inf),
                 ops=None, plan="auto"):
        self.chunk = chunk_size
        self.kw = dict(dt_softplus=dt_softplus, D=D, dt_bias=dt_bias, dt_limit=dt_limit, ops=ops, plan=plan)

    def forward(self, seg, initial_states):
        """(y, final_state) of the segment from ``initial_states`` (None: zero)."""
        from . import mamba2_ssd_fwd
        return mamba2_ssd_fwd(seg["x"], seg["dt"], seg["A"], seg["B"], seg["C"], self.chunk,
                              return_final_state=True, z=seg.get("z"), initial_states=initial_states,
                              **self.kw)

    def log_decay(self, seg):
        from . import make_args, ssd_segment_log_decay, _stream_handle
        Bb, _, H, _ = seg["x"].shape
        out = torch.empty((Bb, H), device=seg["x"].device, dtype=torch.float32)
        a = make_args(seg["x"], seg["dt"], seg["A"], seg["B"], seg["C"], self.chunk,
                      dt_bias=self.kw["dt_bias"], dt_softplus=self.kw["dt_softplus"],
                      dt_limit=self.kw["dt_limit"])
        ssd_segment_log_decay(a, out, _stream_handle(seg["x"].device))
        return out

    def fold(self, log_decays, states):
        """State entering the segment after ``len(states)`` segments."""
        from . import ssd_state_fold, _stream_handle
        out = torch.empty(states.shape[1:], device=states.device, dtype=torch.float32)
        ssd_state_fold(log_decays.contiguous(), states.contiguous(), out, _stream_handle(states.device))
        return out


def segment_summary(backend, seg, rank, initial_states=None):
    """Phase 1: (log_decay [B,H], S_seg [B,H,P,N], y or None).  Rank 0 runs
    from the sequence's initial state, so its y is already the final output."""
    h0 = initial_states if rank == 0 else None
    y, S = backend.forward(seg, h0)
    return backend.log_decay(seg), S, (y if rank == 0 else None)


def entering_state(backend, log_decays, states, rank):
    """Phase 3a: the state entering rank ``rank``'s segment, from the gathered
    maps of all ranks ([W,B,H] and [W,B,H,P,N]); only ranks < rank are used."""
    return backend.fold(log_decays[:rank], states[:rank])


def ssd_fwd_seq_parallel(seg, *, backend, group=None, initial_states=None):
    """Sequence-parallel forward of this rank's segment ``seg`` (a dict with
    x [B,L_r,H,P], dt [B,L_r,H], A [H], B/C [B,L_r,G,N] and optionally z) over
    the ranks of ``group`` (torch.distributed, initialised by the caller; rank
    order = segment order).  ``initial_states`` is read on rank 0 only.

    Returns (y [B,L_r,H,P], final_state [B,H,P,N]); final_state is that of the
    whole sequence on the last rank and the state after this rank's segment on
    the others.
    """
    import torch.distributed as dist
    rank, world = dist.get_rank(group), dist.get_world_size(group)

    def all_gather(t):
        parts = [torch.empty_like(t) for _ in range(world)]
        dist.all_gather(parts, t.contiguous(), group=group)
        return torch.stack(parts)

    a, S, y0 = segment_summary(backend, seg, rank, initial_states)
    log_decays = all_gather(a)   # [W, B, H]
    states = all_gather(S)       # [W, B, H, P, N]
    if rank == 0:
        return y0, S
    S_in = entering_state(backend, log_decays, states, rank)
    return backend.forward(seg, S_in)
