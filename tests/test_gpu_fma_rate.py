"""The fp32 FMA-chain kernel behind the backward's measured CUDA-core peak
does the work it is credited with: each thread's stored sum equals the closed
form of its 8 chains a <- a*m + c after `iters` steps (a geometric series),
and the timed rate lies between a third of and just above the GPU's nominal
fp32 rate (SMs x 128 lanes x 2 flops x clock)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

M, C = 0.9999, 1e-4  # the kernel's multiplier and addend


def _closed_form(iters, threads):
    m, c = np.float64(np.float32(M)), np.float64(np.float32(C))
    t = np.arange(threads, dtype=np.float64)
    total = np.zeros(threads)
    for k in range(8):
        a0 = (np.float32(1e-3) * t.astype(np.float32)).astype(np.float64) + k  # fp32 start, exact + k
        total += m ** iters * a0 + c * (1.0 - m ** iters) / (1.0 - m)
    return total


@pytest.mark.parametrize("iters", [8, 1024])
def test_fma_chain_values_match_the_closed_form(iters):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    grid = 3
    out = torch.full((grid * 256,), float("nan"), device="cuda")
    ssd.ssd_selftest_fma_rate(out, iters, grid)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64).reshape(grid, 256)
    want = _closed_form(iters, 256)
    # fp32 rounding per step: at most iters * 2^-24 relative on each chain of size <= 8
    bound = 8 * 8.0 * iters * 2.0 ** -24 + 1e-6
    for b in range(grid):
        np.testing.assert_allclose(got[b], want, rtol=0, atol=bound)


def test_fma_rate_is_plausible():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    props = torch.cuda.get_device_properties(0)
    grid = 8 * props.multi_processor_count
    iters = 16384
    out = torch.empty(grid * 256, device="cuda")
    ssd.ssd_selftest_fma_rate(out, iters, grid)
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(3):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        ssd.ssd_selftest_fma_rate(out, iters, grid)
        e.record()
        torch.cuda.synchronize()
        best = min(best, s.elapsed_time(e))
    tflops = 2.0 * 8 * iters * 256 * grid / (best * 1e-3) / 1e12
    nominal = props.multi_processor_count * 128 * 2 * 2.07e9 / 1e12  # max SM clock 2070 MHz
    assert nominal / 3 < tflops < nominal * 1.05, (tflops, nominal)
