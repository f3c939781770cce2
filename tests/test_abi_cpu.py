"""The C-ABI library builds, loads and exports every symbol include/ssd.h
declares; host-side validation answers without a GPU (no compute calls)."""
import ctypes
import os
import re

import pytest
import torch

import mamba_ssd_chunked_fwd_gb300 as ssd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "ssd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = ssd.load_library()
    names = _declared_functions()
    assert "ssd_fwd" in names and "ssd_chunk_scan" in names
    for name in names:
        assert hasattr(lib, name), f"missing export {name}"
    assert lib.ssd_abi_version() == 4


def test_status_strings():
    lib = ssd.load_library()
    for code in range(6):
        assert lib.ssd_status_string(code)
    assert lib.ssd_status_string(0) == b"ok"


def _args(**over):
    kw = dict(B=1, L=128, H=4, P=64, N=64, G=2)
    kw.update({k: over.pop(k) for k in list(over) if k in kw})
    x = torch.empty((kw["B"], kw["L"], kw["H"], kw["P"]))
    dt = torch.empty((kw["B"], kw["L"], kw["H"]))
    A = torch.empty((kw["H"],))
    Bm = torch.empty((kw["B"], kw["L"], kw["G"], kw["N"]))
    chunk = over.pop("chunk", 64)
    a = ssd.make_args(x, dt, A, Bm, Bm, chunk, y=x, **over)
    return a


def _status(fn, a):
    out = ctypes.c_size_t(0)
    return fn(ctypes.byref(a), ctypes.byref(out)), out.value


def test_workspace_size_for_valid_shape():
    lib = ssd.load_library()
    a = _args()
    st, n = _status(lib.ssd_fwd_workspace_size, a)
    assert st == 0
    # chunked plan: error word + dtp + cs + states
    c = 2
    assert n >= 256 + 2 * 1 * 4 * c * 64 * 4 + 1 * c * 4 * 64 * 64 * 4


@pytest.mark.parametrize("field,value,code", [
    ("B", 0, 1), ("L", -3, 1), ("H", 0, 1), ("P", 0, 1), ("G", 3, 1),
    ("chunk", 24, 2), ("chunk", 512, 2), ("P", 72, 2), ("N", 256, 2),
    ("ops", 7, 1), ("plan", 9, 1), ("x_dtype", 5, 1), ("bc_dtype", 2, 2),
])
def test_validation_rejects(field, value, code):
    lib = ssd.load_library()
    a = _args()
    setattr(a, field, value)
    st, _ = _status(lib.ssd_fwd_workspace_size, a)
    assert st == code, (field, value, st, lib.ssd_last_error_detail())
    assert lib.ssd_last_error_detail()


def test_dt_limit_must_be_ordered():
    lib = ssd.load_library()
    a = _args(dt_limit=(0.5, 0.1))
    st, _ = _status(lib.ssd_fwd_workspace_size, a)
    assert st == 1


def test_missing_pointers_rejected_before_any_launch():
    lib = ssd.load_library()
    a = _args()
    a.x = None
    assert lib.ssd_fwd(ctypes.byref(a), None) == 1
    a = _args()
    a.y = None
    assert lib.ssd_fwd(ctypes.byref(a), None) == 1
    a = _args()
    assert lib.ssd_chunk_cumsum(ctypes.byref(a), None, None, None) == 1


def test_missing_workspace_rejected():
    lib = ssd.load_library()
    a = _args()
    a.workspace = None
    assert lib.ssd_fwd(ctypes.byref(a), None) == 3
    assert b"workspace" in lib.ssd_last_error_detail()


def test_misaligned_state_rejected():
    lib = ssd.load_library()
    a = _args()
    a.final_state = 8  # not 16-byte aligned
    assert lib.ssd_fwd(ctypes.byref(a), None) == 1


def test_norm_needs_z_and_a_finite_eps():
    lib = ssd.load_library()
    a = _args()
    a.norm_weight, a.norm_eps, a.z = 4096, 1e-5, None
    assert lib.ssd_fwd(ctypes.byref(a), None) == 1
    assert b"needs z" in lib.ssd_last_error_detail()
    a = _args()
    a.norm_weight, a.norm_eps, a.z = 4096, float("nan"), 4096
    assert lib.ssd_fwd(ctypes.byref(a), None) == 1


def test_backward_rejects_the_norm():
    lib = ssd.load_library()
    b = ssd.SsdBwdArgs()
    b.fwd = _args()
    b.fwd.norm_weight, b.fwd.z = 4096, 4096
    assert lib.ssd_bwd(ctypes.byref(b), None) == 2


def test_python_binding_raises_with_detail():
    a = _args()
    a.G = 3
    with pytest.raises(ssd.SsdError) as ei:
        ssd.ssd_fwd_workspace_size(a)
    assert "G" in str(ei.value)


def test_fused_plan_request_is_checked():
    a = _args(plan="fused")
    lib = ssd.load_library()
    plan = ctypes.c_int32(-1)
    st = lib.ssd_fwd_resolve_plan(ctypes.byref(a), ctypes.byref(plan))
    assert st in (0, 2)
    if st == 0:
        assert plan.value == ssd.SSD_PLAN_FUSED


def test_describe_names_the_kernels_each_workload_runs():
    """The named workloads run on the tensor cores (the fused kernel, at N = 128
    after the segment passes when it cuts the walk into segments); only the
    fp32 tiny workload uses the CUDA-core chunk steps.  Without a GPU the SM
    count reads as 1, so no walk is cut into segments here."""
    import ssd_inputs
    expect = {
        "tiny": ["chunk_cumsum", "chunk_state", "state_passing", "chunk_scan"],
        "same_device": ["ssd_fused_kernel"],
        "large_training": ["ssd_fused_kernel"],
        "long_sequence": ["ssd_fused_kernel"],
        "gated_prefill": ["ssd_fused_kernel"],
    }
    dt_of = {"f32": torch.float32, "bf16": torch.bfloat16}
    for name, w in ssd_inputs.WORKLOADS.items():
        xd = dt_of[w.x_dtype]
        a = ssd.make_args(torch.empty((1, 1, w.H, w.P), dtype=xd), torch.empty((1, 1, w.H)), torch.empty(w.H),
                          torch.empty((1, 1, w.G, w.N), dtype=xd), torch.empty((1, 1, w.G, w.N), dtype=xd),
                          w.chunk, ops=w.ops)
        a.B, a.L = w.B, w.L
        a.x = a.Bm = a.Cm = 4096  # any 16-byte aligned address: describe only inspects alignment
        assert ssd.ssd_fwd_describe(a) == expect[name], name


def _decode_args(**over):
    a = ssd.SsdDecodeArgs()
    a.B, a.H, a.P, a.N, a.G = 2, 4, 64, 64, 2
    fake = 1 << 20  # never dereferenced: every case below fails validation first
    a.x = a.dt = a.A = a.Bm = a.Cm = a.state = a.y = fake
    a.x_dtype, a.dt_softplus, a.dt_min, a.dt_max = 0, 1, 0.0, float("inf")
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,code", [
    ("B", 0, 1), ("H", -1, 1), ("P", 0, 1), ("G", 3, 1), ("N", 256, 2), ("x_dtype", 7, 1),
    ("state", None, 1), ("y", None, 1), ("Bm", None, 1), ("dt_min", 1.0, 1),
])
def test_decode_validation_rejects(field, value, code):
    lib = ssd.load_library()
    a = _decode_args(**{field: value})
    if field == "dt_min":
        a.dt_max = 0.5
    assert lib.ssd_decode_step(ctypes.byref(a), None) == code
    assert lib.ssd_last_error_detail().decode()


@pytest.mark.parametrize("cu,code", [
    ([0, 10, 5, 64], 1),     # decreasing
    ([1, 10, 64], 1),        # does not start at 0
    ([0, 10, 63], 1),        # does not end at L
    ([0], 1),                # no sequence
])
def test_varlen_offsets_are_validated(cu, code):
    lib = ssd.load_library()
    a = _args(B=1, L=64)
    arr = (ctypes.c_int64 * len(cu))(*cu)
    out = ctypes.c_size_t(0)
    assert lib.ssd_fwd_varlen_workspace_size(ctypes.byref(a), arr, len(cu) - 1, ctypes.byref(out)) == code
    assert lib.ssd_fwd_varlen(ctypes.byref(a), arr, len(cu) - 1, None) == code
    assert lib.ssd_last_error_detail().decode()


def test_varlen_needs_a_single_batch_row():
    lib = ssd.load_library()
    a = _args(B=2, L=64)
    arr = (ctypes.c_int64 * 3)(0, 30, 64)
    out = ctypes.c_size_t(0)
    assert lib.ssd_fwd_varlen_workspace_size(ctypes.byref(a), arr, 2, ctypes.byref(out)) == 1
    a = _args(B=1, L=64)
    assert lib.ssd_fwd_varlen_workspace_size(ctypes.byref(a), arr, 2, ctypes.byref(out)) == 0
    assert out.value >= 256


def test_neighbour_validation_without_a_gpu():
    lib = ssd.load_library()
    fake = ctypes.c_void_p(1 << 20)
    # conv1d: W too wide, zero dims, missing pointer, unknown dtype
    assert lib.ssd_causal_conv1d(1, 8, 16, 9, 0, fake, fake, None, 1, fake, None) == 2
    assert lib.ssd_causal_conv1d(1, 0, 16, 4, 0, fake, fake, None, 1, fake, None) == 1
    assert lib.ssd_causal_conv1d(1, 8, 16, 4, 0, None, fake, None, 1, fake, None) == 1
    assert lib.ssd_causal_conv1d(1, 8, 16, 4, 5, fake, fake, None, 1, fake, None) == 1
    # RMSNorm: groups not dividing D, negative eps, missing z
    assert lib.ssd_gated_rmsnorm(4, 10, 3, 1e-5, 0, fake, fake, fake, fake, None) == 1
    assert lib.ssd_gated_rmsnorm(4, 12, 3, -1.0, 0, fake, fake, fake, fake, None) == 1
    assert lib.ssd_gated_rmsnorm(4, 12, 3, 1e-5, 0, fake, None, fake, fake, None) == 1


def test_selftest_validation_without_a_gpu():
    """The bounded-wait self-test rejects a missing or misaligned workspace and
    an out-of-range limit before anything is enqueued."""
    import ctypes
    lib = ssd.load_library()
    assert lib.ssd_selftest_wait_timeout(None, 1000, 0, None) == 1
    buf = ctypes.create_string_buffer(512)
    base = ctypes.addressof(buf)
    aligned = (base + 255) // 256 * 256
    assert lib.ssd_selftest_wait_timeout(ctypes.c_void_p(aligned + 4), 1000, 0, None) == 1
    assert lib.ssd_selftest_wait_timeout(ctypes.c_void_p(aligned), 0, 0, None) == 1
    assert lib.ssd_selftest_wait_timeout(ctypes.c_void_p(aligned), 2000000, 0, None) == 1
    # the FMA-rate kernel: null out, iters not a multiple of 8, grid out of range, out too small
    assert lib.ssd_selftest_fma_rate(None, 256, 64, 1, None) == 1
    assert lib.ssd_selftest_fma_rate(ctypes.c_void_p(aligned), 256, 60, 1, None) == 1
    assert lib.ssd_selftest_fma_rate(ctypes.c_void_p(aligned), 256, 64, 0, None) == 1
    assert lib.ssd_selftest_fma_rate(ctypes.c_void_p(aligned), 255, 64, 1, None) == 1


def test_conv_arguments_are_validated_without_a_gpu():
    """The conv1d in front of the SSD: width 0..4, the three weights required,
    16-byte aligned x, B, C; the host-buffer, packed and backward entries do
    not take it."""
    import ctypes
    lib = ssd.load_library()
    a = _args()
    a.conv_width = 5
    assert lib.ssd_fwd(ctypes.byref(a), None) == 2
    a.conv_width = 4
    assert lib.ssd_fwd(ctypes.byref(a), None) == 1   # no weights
    a.conv_x_weight = a.conv_b_weight = a.conv_c_weight = 1 << 20
    size = ctypes.c_size_t(0)
    assert lib.ssd_fwd_host_workspace_size(ctypes.byref(a), ctypes.byref(size)) == 2
    assert lib.ssd_fwd_host(ctypes.byref(a), None) == 2
    cu = (ctypes.c_int64 * 2)(0, a.L)
    assert lib.ssd_fwd_varlen(ctypes.byref(a), cu, 1, None) == 2
    assert lib.ssd_causal_conv1d_tokens(1, 8, 6, 4, 0, 1 << 20, 1 << 20, None, 1, 1 << 21, None) == 2  # C % 4
    assert lib.ssd_causal_conv1d_tokens(1, 8, 8, 5, 0, 1 << 20, 1 << 20, None, 1, 1 << 21, None) == 2  # W > 4
