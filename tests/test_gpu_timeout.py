"""The bounded device-side waits give up instead of hanging, and the host
learns of it: a wait that runs out sets the workspace error word, the kernel
returns, ssd_check_device_error reports SSD_ERR_TIMEOUT (status 5), and the
context stays usable for the next call.  No GPU fault is involved: the wait
that runs out is on an mbarrier that nothing arrives on, with a 1 ms limit."""
import time

import numpy as np
import pytest
import torch

import ssd_inputs
from _harness import to_device

pytestmark = pytest.mark.gpu

SSD_ERR_TIMEOUT = 5


def _fused_args(ssd):
    _, inp = ssd_inputs.custom(1, 128, 4, 64, 64, 2, 64, seed=11, ops="bf16")
    d = to_device(inp)
    y = torch.empty_like(d["x"])
    a = ssd.make_args(d["x"], d["dt"], d["A"], d["B"], d["C"], 64, y=y, dt_softplus=True, ops="bf16",
                      plan="fused")
    ws = torch.zeros(max(ssd.ssd_fwd_workspace_size(a), 256), dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    return a, ws, (d, y)


def test_error_word_maps_to_the_timeout_status():
    """A nonzero error word left in a fused-plan workspace (written from the
    host) reads back as SSD_ERR_TIMEOUT; a clean run reads back as OK."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    a, ws, keep = _fused_args(ssd)
    assert "ssd_fused_kernel" in ssd.ssd_fwd_describe(a)
    ssd.ssd_fwd(a)
    ssd.ssd_check_device_error(a)  # clean run: no error
    ws[:4].copy_(torch.tensor([1, 0, 0, 0], dtype=torch.uint8))
    with pytest.raises(ssd.SsdError) as ei:
        ssd.ssd_check_device_error(a)
    assert ei.value.status == SSD_ERR_TIMEOUT
    ssd.ssd_fwd(a)  # the next call clears the word again
    ssd.ssd_check_device_error(a)


def test_a_bounded_wait_that_nothing_releases_gives_up():
    """The library's mbarrier wait on a barrier nobody arrives on returns after
    its limit; the kernel records it and exits.  The control case (the thread
    arrives first) leaves the word clear.  A forward afterwards still runs
    cleanly on the same context."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    a, _, keep = _fused_args(ssd)
    probe = ssd.make_args(*[keep[0][k] for k in ("x", "dt", "A", "B", "C")], 64, y=keep[1], ops="bf16")
    probe.workspace, probe.workspace_bytes = ws.data_ptr(), ws.numel()

    t0 = time.perf_counter()
    ssd.ssd_selftest_wait_timeout(ws, 1000, arrive=False)
    with pytest.raises(ssd.SsdError) as ei:
        ssd.ssd_check_device_error(probe)
    elapsed = time.perf_counter() - t0
    assert ei.value.status == SSD_ERR_TIMEOUT
    assert elapsed < 5.0, elapsed  # gave up after ~1 ms, not after a hang

    ssd.ssd_selftest_wait_timeout(ws, 1000, arrive=True)
    ssd.ssd_check_device_error(probe)  # released wait: no error

    ssd.ssd_fwd(a)  # the context is intact
    ssd.ssd_check_device_error(a)
    assert torch.isfinite(keep[1].float()).all()
