"""GPU parity of the SSD's neighbours against the float64 oracle: the causal
conv1d + SiLU and the gated grouped RMSNorm (ops-transformer MambaV2 article,
sections 1.4, 4.1 and 4.6)."""
import numpy as np
import pytest
import torch

from _harness import assert_close

pytestmark = pytest.mark.gpu

_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.mark.parametrize("shape", [(1, 10240, 1024, 4), (2, 96, 1500, 4), (3, 5, 7, 2), (1, 64, 2049, 8), (2, 33, 300, 1),
                                   (2, 7, 3072, 8)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("feats", [(True, True), (False, False)])
def test_causal_conv1d(oracle_mod, shape, dtype, feats):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, D, S, W = shape
    use_bias, silu = feats
    g = torch.Generator().manual_seed(sum(shape))
    x = torch.randn((B, D, S), generator=g).to(_DT[dtype])
    w = torch.randn((D, W), generator=g) * 0.5
    bias = torch.randn(D, generator=g) if use_bias else None
    out = ssd.causal_conv1d(x.cuda(), w.cuda(), None if bias is None else bias.cuda(), silu=silu)
    torch.cuda.synchronize()
    ref = oracle_mod.causal_conv1d(x.double().numpy(), w.numpy(), None if bias is None else bias.numpy(), silu=silu)
    assert out.dtype == x.dtype
    assert_close(oracle_mod, out.double().cpu().numpy(), ref, dtype, f"conv1d {shape} {dtype}")


# group sizes 256, 32, 4096 (two passes), 25, 512, 500, 128, 60; then 32, 64, 128 with the groups
# a multiple of 8, 4, 2 (several groups per warp)
@pytest.mark.parametrize("shape", [(2, 512, 16384, 64), (3, 7, 96, 3), (1, 5, 4096, 1), (4, 33, 200, 8),
                                   (2, 9, 1024, 2), (1, 3, 1000, 2), (1, 17, 384, 3), (2, 11, 300, 5),
                                   (2, 9, 512, 16), (1, 13, 512, 8), (3, 5, 512, 4)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gated_rmsnorm(oracle_mod, shape, dtype):
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, S, D, G = shape
    g = torch.Generator().manual_seed(sum(shape) + 1)
    x = torch.randn((B, S, D), generator=g).to(_DT[dtype])
    z = torch.randn((B, S, D), generator=g).to(_DT[dtype])
    w = torch.rand(D, generator=g) + 0.5
    out = ssd.gated_rmsnorm(x.cuda(), z.cuda(), w.cuda(), G, 1e-5)
    torch.cuda.synchronize()
    ref = oracle_mod.gated_rmsnorm(x.double().numpy(), z.double().numpy(), w.numpy(), G, 1e-5)
    assert_close(oracle_mod, out.double().cpu().numpy(), ref, dtype, f"rmsnorm {shape} {dtype}")


def test_causal_conv1d_unaligned_rows(oracle_mod):
    """fp32 rows that start off a 16-byte boundary take the scalar loads."""
    import mamba_ssd_chunked_fwd_gb300 as ssd
    B, D, S, W = 2, 6, 1028, 4
    g = torch.Generator().manual_seed(17)
    flat = torch.randn(B * D * S + 1, generator=g)
    w = torch.randn((D, W), generator=g) * 0.5
    x = flat.cuda()[1:].view(B, D, S)
    out = ssd.causal_conv1d(x, w.cuda(), None, silu=True)
    torch.cuda.synchronize()
    ref = oracle_mod.causal_conv1d(flat[1:].view(B, D, S).double().numpy(), w.numpy(), None, silu=True)
    assert_close(oracle_mod, out.double().cpu().numpy(), ref, "f32", "conv1d unaligned")


def test_neighbours_are_deterministic():
    import mamba_ssd_chunked_fwd_gb300 as ssd
    g = torch.Generator().manual_seed(3)
    x = torch.randn((2, 64, 999), generator=g).cuda()
    w = torch.randn((64, 4), generator=g).cuda()
    assert torch.equal(ssd.causal_conv1d(x, w), ssd.causal_conv1d(x, w))
    y = torch.randn((4, 100, 512), generator=g).cuda()
    z = torch.randn((4, 100, 512), generator=g).cuda()
    wn = torch.rand(512, generator=g).cuda()
    assert torch.equal(ssd.gated_rmsnorm(y, z, wn, 4), ssd.gated_rmsnorm(y, z, wn, 4))
