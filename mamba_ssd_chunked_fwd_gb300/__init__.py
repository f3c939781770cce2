"""GB300 (sm_103a) Mamba-2 SSD chunked forward: thin Python binding.

Every step of the computation runs in the CUDA kernels of
``libssd_gb300.so``; this module only marshals torch tensors (device memory
and the current stream) into the C ABI of ``include/ssd.h``.  The binding
functions carry the C names (``ssd_fwd``, ``ssd_chunk_cumsum``,
``ssd_chunk_state``, ``ssd_state_passing``, ``ssd_chunk_scan``,
``ssd_fwd_host`` ...).  ``mamba2_ssd_fwd`` mirrors the public call of the
"Mamba-2 SSD for Ascend NPU" README ("Usage": mamba2_ssd_fwd(x, dt, A, B, C,
chunk_size, dt_softplus, return_final_state) plus D, z, dt_bias, dt_limit and
initial_states).

There is no fallback: if the library cannot be built or loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import math
import threading

import torch

from . import _build

__all__ = [
    "SSD_F32", "SSD_F16", "SSD_BF16", "SSD_OPS_F32", "SSD_OPS_F16", "SSD_OPS_BF16",
    "SSD_PLAN_AUTO", "SSD_PLAN_CHUNKED", "SSD_PLAN_FUSED", "SsdError", "SsdFwdArgs",
    "load_library", "library_path", "make_args", "ssd_fwd", "ssd_fwd_workspace_size",
    "ssd_fwd_resolve_plan", "ssd_fwd_describe", "ssd_fwd_noalloc", "ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing",
    "ssd_chunk_scan", "ssd_fwd_host", "ssd_fwd_host_workspace_size", "ssd_check_device_error",
    "mamba2_ssd_fwd", "SsdDecodeArgs", "make_decode_args", "ssd_decode_step", "mamba2_ssd_decode",
    "ssd_segment_log_decay", "ssd_state_fold", "ssd_fwd_varlen", "ssd_fwd_varlen_workspace_size",
    "mamba2_ssd_fwd_varlen", "SsdBwdArgs", "ssd_bwd", "ssd_bwd_workspace_size", "mamba2_ssd_bwd",
    "ssd_causal_conv1d", "ssd_gated_rmsnorm", "causal_conv1d", "gated_rmsnorm",
]

SSD_F32, SSD_F16, SSD_BF16 = 0, 1, 2
SSD_OPS_F32, SSD_OPS_F16, SSD_OPS_BF16 = 0, 1, 2
SSD_PLAN_AUTO, SSD_PLAN_CHUNKED, SSD_PLAN_FUSED = 0, 1, 2
_PLAN_NAMES = {"auto": SSD_PLAN_AUTO, "chunked": SSD_PLAN_CHUNKED, "fused": SSD_PLAN_FUSED}
_OPS_NAMES = {"f32": SSD_OPS_F32, "fp32": SSD_OPS_F32, "f16": SSD_OPS_F16, "fp16": SSD_OPS_F16,
              "bf16": SSD_OPS_BF16}
_DTYPE_CODES = {torch.float32: SSD_F32, torch.float16: SSD_F16, torch.bfloat16: SSD_BF16}
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
           3: "workspace missing or too small", 4: "CUDA error", 5: "device-side wait timed out"}


class SsdError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {_STATUS.get(status, status)} ({detail})")
        self.status = status
        self.detail = detail


class SsdFwdArgs(ctypes.Structure):
    """Mirror of ``ssd_fwd_args`` in include/ssd.h."""
    _fields_ = [
        ("B", ctypes.c_int64), ("L", ctypes.c_int64), ("H", ctypes.c_int64),
        ("P", ctypes.c_int64), ("N", ctypes.c_int64), ("G", ctypes.c_int64),
        ("chunk", ctypes.c_int64),
        ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p), ("A", ctypes.c_void_p),
        ("Bm", ctypes.c_void_p), ("Cm", ctypes.c_void_p), ("D", ctypes.c_void_p),
        ("z", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p), ("initial_state", ctypes.c_void_p),
        ("y", ctypes.c_void_p), ("final_state", ctypes.c_void_p),
        ("x_dtype", ctypes.c_int32), ("bc_dtype", ctypes.c_int32), ("z_dtype", ctypes.c_int32),
        ("y_dtype", ctypes.c_int32), ("ops", ctypes.c_int32), ("plan", ctypes.c_int32),
        ("dt_softplus", ctypes.c_int32), ("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("norm_weight", ctypes.c_void_p), ("norm_eps", ctypes.c_float),
        ("conv_x_weight", ctypes.c_void_p), ("conv_x_bias", ctypes.c_void_p),
        ("conv_b_weight", ctypes.c_void_p), ("conv_b_bias", ctypes.c_void_p),
        ("conv_c_weight", ctypes.c_void_p), ("conv_c_bias", ctypes.c_void_p),
        ("conv_width", ctypes.c_int32),
    ]


class SsdDecodeArgs(ctypes.Structure):
    """Mirror of ``ssd_decode_args`` in include/ssd.h."""
    _fields_ = [
        ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("P", ctypes.c_int64),
        ("N", ctypes.c_int64), ("G", ctypes.c_int64),
        ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p), ("A", ctypes.c_void_p),
        ("Bm", ctypes.c_void_p), ("Cm", ctypes.c_void_p), ("D", ctypes.c_void_p),
        ("z", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p), ("state", ctypes.c_void_p),
        ("y", ctypes.c_void_p), ("x_dtype", ctypes.c_int32), ("dt_softplus", ctypes.c_int32),
        ("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float),
    ]


class SsdBwdArgs(ctypes.Structure):
    """Mirror of ``ssd_bwd_args`` in include/ssd.h."""
    _fields_ = [
        ("fwd", SsdFwdArgs), ("dy", ctypes.c_void_p), ("dfinal", ctypes.c_void_p), ("dx", ctypes.c_void_p),
        ("ddt", ctypes.c_void_p), ("dA", ctypes.c_void_p), ("dB", ctypes.c_void_p), ("dC", ctypes.c_void_p),
        ("dD", ctypes.c_void_p), ("dz", ctypes.c_void_p), ("ddt_bias", ctypes.c_void_p), ("dh0", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


_lock = threading.Lock()
_lib = None

# C entry points: name -> argument types (all return ssd_status / int32)
_P = ctypes.POINTER(SsdFwdArgs)
_SIGS = {
    "ssd_fwd_workspace_size": [_P, ctypes.POINTER(ctypes.c_size_t)],
    "ssd_fwd_resolve_plan": [_P, ctypes.POINTER(ctypes.c_int32)],
    "ssd_fwd": [_P, ctypes.c_void_p],
    "ssd_chunk_cumsum": [_P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
    "ssd_chunk_state": [_P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
    "ssd_state_passing": [_P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
    "ssd_chunk_scan": [_P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
    "ssd_fwd_host_workspace_size": [_P, ctypes.POINTER(ctypes.c_size_t)],
    "ssd_fwd_host": [_P, ctypes.c_void_p],
    "ssd_check_device_error": [_P, ctypes.c_void_p],
    "ssd_selftest_wait_timeout": [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int32, ctypes.c_void_p],
    "ssd_selftest_fma_rate": [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p],
    "ssd_fwd_describe": [_P, ctypes.c_char_p, ctypes.c_size_t],
    "ssd_fwd_noalloc": [_P, ctypes.c_void_p],
    "ssd_decode_step": [ctypes.POINTER(SsdDecodeArgs), ctypes.c_void_p],
    "ssd_segment_log_decay": [_P, ctypes.c_void_p, ctypes.c_void_p],
    "ssd_fwd_varlen_workspace_size": [_P, ctypes.c_void_p, ctypes.c_int64, ctypes.POINTER(ctypes.c_size_t)],
    "ssd_bwd_workspace_size": [ctypes.POINTER(SsdBwdArgs), ctypes.POINTER(ctypes.c_size_t)],
    "ssd_bwd": [ctypes.POINTER(SsdBwdArgs), ctypes.c_void_p],
    "ssd_causal_conv1d": [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                          ctypes.c_void_p],
    "ssd_causal_conv1d_tokens": [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                 ctypes.c_void_p],
    "ssd_gated_rmsnorm": [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, ctypes.c_int32,
                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
    "ssd_fwd_varlen": [_P, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p],
    "ssd_state_fold": [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
}


def library_path() -> str:
    return _build.LIB


def load_library(build: bool = True):
    """Build (if stale) and load libssd_gb300.so.  Raises if that fails."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build else _build.LIB
            lib = ctypes.CDLL(path)
            for name, argtypes in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = argtypes
                fn.restype = ctypes.c_int32
            lib.ssd_abi_version.restype = ctypes.c_int32
            lib.ssd_abi_version.argtypes = []
            lib.ssd_status_string.restype = ctypes.c_char_p
            lib.ssd_status_string.argtypes = [ctypes.c_int32]
            lib.ssd_last_error_detail.restype = ctypes.c_char_p
            lib.ssd_last_error_detail.argtypes = []
            _lib = lib
    return _lib


def _check(status: int, where: str):
    if status != 0:
        detail = load_library().ssd_last_error_detail().decode(errors="replace")
        raise SsdError(status, where, detail)


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("every tensor passed to the SSD library must be contiguous")
    return t.data_ptr()


def _stream_handle(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def make_args(x, dt, A, B, C, chunk_size, *, y=None, final_state=None, D=None, z=None,
              dt_bias=None, initial_states=None, dt_softplus=False,
              dt_limit=(0.0, math.inf), ops=None, plan="auto", workspace=None, norm_weight=None,
              norm_eps=1e-5, conv=None) -> SsdFwdArgs:
    """Fill an ``ssd_fwd_args`` from tensors (device or host; no copies).

    ``conv``: optional (x_weight, x_bias, B_weight, B_bias, C_weight, C_bias)
    of the causal conv1d + SiLU in front of the SSD (weights [channels, W]
    fp32, biases [channels] fp32 or None); x, B and C are then the
    activations before the convolution."""
    Bb, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    io = _DTYPE_CODES.get(x.dtype)
    if io is None:
        raise ValueError(f"unsupported dtype {x.dtype}")
    if ops is None:
        ops = {SSD_F32: "f32", SSD_F16: "f16", SSD_BF16: "bf16"}[io]
    a = SsdFwdArgs()
    a.B, a.L, a.H, a.P, a.N, a.G, a.chunk = Bb, L, H, P, N, G, int(chunk_size)
    a.x, a.dt, a.A, a.Bm, a.Cm = _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C)
    a.D, a.z, a.dt_bias, a.initial_state = _ptr(D), _ptr(z), _ptr(dt_bias), _ptr(initial_states)
    a.y, a.final_state = _ptr(y), _ptr(final_state)
    a.x_dtype = io
    a.bc_dtype = _DTYPE_CODES.get(B.dtype, -1)
    a.z_dtype = _DTYPE_CODES.get(z.dtype, -1) if z is not None else io
    a.y_dtype = _DTYPE_CODES.get(y.dtype, -1) if y is not None else io
    a.ops = _OPS_NAMES[ops] if isinstance(ops, str) else int(ops)
    a.plan = _PLAN_NAMES[plan] if isinstance(plan, str) else int(plan)
    a.dt_softplus = 1 if dt_softplus else 0
    a.dt_min, a.dt_max = float(dt_limit[0]), float(dt_limit[1])
    if workspace is not None:
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    a.norm_weight, a.norm_eps = _ptr(norm_weight), float(norm_eps)
    if conv is not None:
        wx, bx, wb, bb, wc, bc = conv
        a.conv_x_weight, a.conv_x_bias = _ptr(wx), _ptr(bx)
        a.conv_b_weight, a.conv_b_bias = _ptr(wb), _ptr(bb)
        a.conv_c_weight, a.conv_c_bias = _ptr(wc), _ptr(bc)
        a.conv_width = int(wx.shape[-1])
    return a


# ---- the C entry points, one Python function each ----------------------------

def ssd_fwd_workspace_size(args: SsdFwdArgs) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().ssd_fwd_workspace_size(ctypes.byref(args), ctypes.byref(out)),
           "ssd_fwd_workspace_size")
    return int(out.value)


def ssd_fwd_resolve_plan(args: SsdFwdArgs) -> int:
    out = ctypes.c_int32(0)
    _check(load_library().ssd_fwd_resolve_plan(ctypes.byref(args), ctypes.byref(out)),
           "ssd_fwd_resolve_plan")
    return int(out.value)


def ssd_fwd_describe(args: SsdFwdArgs) -> list:
    """Kernels ssd_fwd would launch for these arguments, in order."""
    buf = ctypes.create_string_buffer(256)
    _check(load_library().ssd_fwd_describe(ctypes.byref(args), buf, 256), "ssd_fwd_describe")
    return buf.value.decode().split(",")


def ssd_fwd(args: SsdFwdArgs, stream=None):
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_fwd(ctypes.byref(args), s), "ssd_fwd")


def ssd_fwd_noalloc(args: SsdFwdArgs, stream=None):
    """ssd_fwd with the scratch taken from the library's built-in 64 MiB
    buffer instead of args.workspace (for callers that cannot allocate)."""
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_fwd_noalloc(ctypes.byref(args), s), "ssd_fwd_noalloc")


def ssd_chunk_cumsum(args: SsdFwdArgs, dtp, cs, stream=None):
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_chunk_cumsum(ctypes.byref(args), _ptr(dtp), _ptr(cs), s),
           "ssd_chunk_cumsum")


def ssd_chunk_state(args: SsdFwdArgs, dtp, cs, states, stream=None):
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_chunk_state(ctypes.byref(args), _ptr(dtp), _ptr(cs), _ptr(states), s),
           "ssd_chunk_state")


def ssd_state_passing(args: SsdFwdArgs, cs, states, stream=None):
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_state_passing(ctypes.byref(args), _ptr(cs), _ptr(states), s),
           "ssd_state_passing")


def ssd_chunk_scan(args: SsdFwdArgs, dtp, cs, states, stream=None):
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_chunk_scan(ctypes.byref(args), _ptr(dtp), _ptr(cs), _ptr(states), s),
           "ssd_chunk_scan")


def ssd_fwd_host_workspace_size(args: SsdFwdArgs) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().ssd_fwd_host_workspace_size(ctypes.byref(args), ctypes.byref(out)),
           "ssd_fwd_host_workspace_size")
    return int(out.value)


def ssd_fwd_host(args: SsdFwdArgs, stream=None):
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_fwd_host(ctypes.byref(args), s), "ssd_fwd_host")


def ssd_check_device_error(args: SsdFwdArgs, stream=None):
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_check_device_error(ctypes.byref(args), s), "ssd_check_device_error")


def ssd_selftest_wait_timeout(workspace, timeout_us: int, arrive: bool = False, stream=None):
    """Run the bounded-wait self-test into ``workspace`` (a CUDA uint8 tensor
    of at least 256 bytes): one bounded mbarrier wait that nothing releases
    (or, with ``arrive``, one that completes at once)."""
    s = stream if stream is not None else _stream_handle()
    if workspace.numel() * workspace.element_size() < 256:
        raise ValueError("the self-test needs a workspace of at least 256 bytes")
    _check(load_library().ssd_selftest_wait_timeout(_ptr(workspace), int(timeout_us), int(bool(arrive)), s),
           "ssd_selftest_wait_timeout")


def ssd_selftest_fma_rate(out, iters: int, grid: int, stream=None):
    """Launch the fp32 FMA-chain measurement kernel into ``out`` (a CUDA
    float32 tensor of at least grid * 256 elements); 4096 * iters * grid
    flops."""
    s = stream if stream is not None else _stream_handle()
    if out.dtype != torch.float32:
        raise ValueError("out must be float32")
    _check(load_library().ssd_selftest_fma_rate(_ptr(out), out.numel(), int(iters), int(grid), s),
           "ssd_selftest_fma_rate")


def _cu_host(cu_seqlens):
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int64).cpu().contiguous()
    return cu, cu.numel() - 1


def ssd_fwd_varlen_workspace_size(args: SsdFwdArgs, cu_seqlens) -> int:
    cu, nseq = _cu_host(cu_seqlens)
    out = ctypes.c_size_t(0)
    _check(load_library().ssd_fwd_varlen_workspace_size(ctypes.byref(args), cu.data_ptr(), nseq,
                                                        ctypes.byref(out)), "ssd_fwd_varlen_workspace_size")
    return int(out.value)


def ssd_fwd_varlen(args: SsdFwdArgs, cu_seqlens, stream=None):
    """Packed variable-length forward; cu_seqlens (nseq + 1 offsets) stays on
    the host (any int sequence or CPU tensor)."""
    cu, nseq = _cu_host(cu_seqlens)
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_fwd_varlen(ctypes.byref(args), cu.data_ptr(), nseq, s), "ssd_fwd_varlen")


def ssd_segment_log_decay(args: SsdFwdArgs, log_decay, stream=None):
    """log_decay [B,H] fp32 <- sum over the segment's tokens of d_t * A[h]."""
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_segment_log_decay(ctypes.byref(args), _ptr(log_decay), s),
           "ssd_segment_log_decay")


def ssd_state_fold(log_decay, states, out, stream=None):
    """out [B,H,P,N] <- fold of the segment maps (log_decay [nseg,B,H],
    states [nseg,B,H,P,N], fp32): S = 0; S = exp(a_q) S + S_q for each q."""
    nseg, Bb, H, P, N = states.shape
    if tuple(log_decay.shape) != (nseg, Bb, H) or tuple(out.shape) != (Bb, H, P, N):
        raise ValueError("ssd_state_fold: log_decay [nseg,B,H], states [nseg,B,H,P,N], out [B,H,P,N]")
    if any(t.dtype != torch.float32 for t in (log_decay, states, out)):
        raise ValueError("ssd_state_fold takes fp32 tensors")
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_state_fold(nseg, Bb, H, P, N, _ptr(log_decay), _ptr(states), _ptr(out), s),
           "ssd_state_fold")


# ---- the README-style call ---------------------------------------------------

def mamba2_ssd_fwd(x, dt, A, B, C, chunk_size, dt_softplus=False, return_final_state=False, *,
                   D=None, z=None, dt_bias=None, dt_limit=(0.0, math.inf), initial_states=None,
                   ops=None, plan="auto", workspace=None, out=None, norm_weight=None, norm_eps=1e-5,
                   conv=None):
    """SSD forward on the GPU.  Returns ``out`` or ``(out, final_state)``.

    x [B,L,H,P], dt [B,L,H] fp32, A [H] fp32, B/C [B,L,G,N], D [H] fp32,
    z [B,L,H,P], dt_bias [H] fp32, initial_states [B,H,P,N] fp32; x, B, C, z
    share a dtype (fp32, fp16 or bf16) and the output takes it.  ``ops``
    ("f32" | "f16" | "bf16") is the operand precision of the contractions
    (default: that of x).  With ``norm_weight`` (fp32 [H*P], z required) the
    output is the gated RMSNorm of the SSD, groups of (H/G)*P channels.
    With ``conv`` = (x_weight, x_bias, B_weight, B_bias, C_weight, C_bias)
    (weights [channels, W] fp32, W <= 4; biases or None), x, B and C are the
    activations before the causal conv1d + SiLU of a Mamba-2 block, which runs
    in front of the SSD.
    Allocation of out, final_state and the workspace is done here with torch;
    all compute runs in libssd_gb300.so on the current stream.
    """
    if not x.is_cuda:
        raise ValueError("mamba2_ssd_fwd takes CUDA tensors; use ssd_fwd_host for host buffers")
    y = out if out is not None else torch.empty_like(x)
    fin = None
    if return_final_state:
        Bb, L, H, P = x.shape
        fin = torch.empty((Bb, H, P, B.shape[3]), device=x.device, dtype=torch.float32)
    args = make_args(x, dt, A, B, C, chunk_size, y=y, final_state=fin, D=D, z=z, dt_bias=dt_bias,
                     initial_states=initial_states, dt_softplus=dt_softplus, dt_limit=dt_limit,
                     ops=ops, plan=plan, norm_weight=norm_weight, norm_eps=norm_eps, conv=conv)
    if workspace is None:
        nbytes = ssd_fwd_workspace_size(args)
        workspace = torch.empty(max(nbytes, 256), device=x.device, dtype=torch.uint8)
    args.workspace, args.workspace_bytes = workspace.data_ptr(), workspace.numel()
    ssd_fwd(args, _stream_handle(x.device))
    return (y, fin) if return_final_state else y


# ---- decode: one recurrent step from a carried state ---------------------------

def make_decode_args(x, dt, A, B, C, state, *, y=None, D=None, z=None, dt_bias=None,
                     dt_softplus=False, dt_limit=(0.0, math.inf)) -> SsdDecodeArgs:
    """Fill an ``ssd_decode_args`` from tensors: x/z/y [B,H,P], dt [B,H],
    B/C [B,G,N], state [B,H,P,N] fp32 (updated in place)."""
    Bb, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    io = _DTYPE_CODES.get(x.dtype)
    if io is None:
        raise ValueError(f"unsupported dtype {x.dtype}")
    for t in (B, C) + ((z,) if z is not None else ()) + ((y,) if y is not None else ()):
        if t.dtype != x.dtype:
            raise ValueError("x, B, C, z and y must share one dtype")
    if state.dtype != torch.float32:
        raise ValueError("state must be fp32")
    a = SsdDecodeArgs()
    a.B, a.H, a.P, a.N, a.G = Bb, H, P, N, G
    a.x, a.dt, a.A, a.Bm, a.Cm = _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C)
    a.D, a.z, a.dt_bias, a.state, a.y = _ptr(D), _ptr(z), _ptr(dt_bias), _ptr(state), _ptr(y)
    a.x_dtype = io
    a.dt_softplus = 1 if dt_softplus else 0
    a.dt_min, a.dt_max = float(dt_limit[0]), float(dt_limit[1])
    return a


def ssd_decode_step(args: SsdDecodeArgs, stream=None):
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_decode_step(ctypes.byref(args), s), "ssd_decode_step")


def mamba2_ssd_decode(x, dt, A, B, C, state, dt_softplus=False, *, D=None, z=None, dt_bias=None,
                      dt_limit=(0.0, math.inf), out=None):
    """One decode step on the GPU: advances ``state`` [B,H,P,N] (fp32, in
    place) by one token and returns y [B,H,P] in x's dtype.  x/z [B,H,P],
    dt [B,H] fp32, B/C [B,G,N].  All compute runs in libssd_gb300.so on the
    current stream."""
    if not x.is_cuda:
        raise ValueError("mamba2_ssd_decode takes CUDA tensors")
    y = out if out is not None else torch.empty_like(x)
    args = make_decode_args(x, dt, A, B, C, state, y=y, D=D, z=z, dt_bias=dt_bias,
                            dt_softplus=dt_softplus, dt_limit=dt_limit)
    ssd_decode_step(args, _stream_handle(x.device))
    return y


def mamba2_ssd_fwd_varlen(x, dt, A, B, C, chunk_size, cu_seqlens, dt_softplus=False, return_final_state=False,
                          *, D=None, z=None, dt_bias=None, dt_limit=(0.0, math.inf), initial_states=None,
                          ops=None, plan="auto", out=None, norm_weight=None, norm_eps=1e-5):
    """Packed variable-length SSD forward on the GPU: x [1,T,H,P], dt [1,T,H],
    B/C [1,T,G,N], z like x; sequence s holds tokens [cu_seqlens[s],
    cu_seqlens[s+1]) and starts from initial_states[s] (or 0).  Returns y, or
    (y, final_state [nseq,H,P,N]); ``norm_weight`` as in ``mamba2_ssd_fwd``.
    All compute runs in libssd_gb300.so."""
    if not x.is_cuda:
        raise ValueError("mamba2_ssd_fwd_varlen takes CUDA tensors")
    cu, nseq = _cu_host(cu_seqlens)
    y = out if out is not None else torch.empty_like(x)
    fin = None
    if return_final_state:
        fin = torch.empty((nseq, x.shape[2], x.shape[3], B.shape[3]), device=x.device, dtype=torch.float32)
    args = make_args(x, dt, A, B, C, chunk_size, y=y, final_state=fin, D=D, z=z, dt_bias=dt_bias,
                     initial_states=initial_states, dt_softplus=dt_softplus, dt_limit=dt_limit, ops=ops,
                     plan=plan, norm_weight=norm_weight, norm_eps=norm_eps)
    nbytes = ssd_fwd_varlen_workspace_size(args, cu)
    ws = torch.empty(max(nbytes, 256), device=x.device, dtype=torch.uint8)
    args.workspace, args.workspace_bytes = ws.data_ptr(), ws.numel()
    ssd_fwd_varlen(args, cu, _stream_handle(x.device))
    return (y, fin) if return_final_state else y


# ---- backward ------------------------------------------------------------------

def ssd_bwd_workspace_size(args: SsdBwdArgs) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().ssd_bwd_workspace_size(ctypes.byref(args), ctypes.byref(out)), "ssd_bwd_workspace_size")
    return int(out.value)


def ssd_bwd(args: SsdBwdArgs, stream=None):
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_bwd(ctypes.byref(args), s), "ssd_bwd")


def mamba2_ssd_bwd(x, dt, A, B, C, chunk_size, dy, dt_softplus=False, *, dfinal=None, D=None, z=None,
                   dt_bias=None, dt_limit=(0.0, math.inf), initial_states=None, want_dh0=True):
    """Gradients of sum(dy * y) + sum(dfinal * final_state) of the forward with
    these inputs, on the GPU.  Returns a dict: dx, ddt, dA, dB, dC and, when
    the matching input is given, dD, dz, ddt_bias, plus dh0 (if want_dh0).
    Tensors as for mamba2_ssd_fwd; dy like x, dfinal [B,H,P,N] fp32.  All
    compute runs in libssd_gb300.so on the current stream."""
    if not x.is_cuda:
        raise ValueError("mamba2_ssd_bwd takes CUDA tensors")
    Bb, L, H, P = x.shape
    N = B.shape[3]
    f32 = dict(device=x.device, dtype=torch.float32)
    g = {"dx": torch.empty_like(x), "ddt": torch.empty((Bb, L, H), **f32), "dA": torch.empty((H,), **f32),
         "dB": torch.empty_like(B), "dC": torch.empty_like(C)}
    if D is not None:
        g["dD"] = torch.empty((H,), **f32)
    if z is not None:
        g["dz"] = torch.empty_like(z)
    if dt_bias is not None:
        g["ddt_bias"] = torch.empty((H,), **f32)
    if want_dh0:
        g["dh0"] = torch.empty((Bb, H, P, N), **f32)
    a = SsdBwdArgs()
    a.fwd = make_args(x, dt, A, B, C, chunk_size, D=D, z=z, dt_bias=dt_bias, initial_states=initial_states,
                      dt_softplus=dt_softplus, dt_limit=dt_limit)
    a.dy, a.dfinal = _ptr(dy), _ptr(dfinal)
    a.dx, a.ddt, a.dA, a.dB, a.dC = (_ptr(g[k]) for k in ("dx", "ddt", "dA", "dB", "dC"))
    a.dD, a.dz, a.ddt_bias, a.dh0 = (_ptr(g.get(k)) for k in ("dD", "dz", "ddt_bias", "dh0"))
    nbytes = ssd_bwd_workspace_size(a)
    ws = torch.empty(max(nbytes, 256), device=x.device, dtype=torch.uint8)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    ssd_bwd(a, _stream_handle(x.device))
    return g


# ---- the SSD's neighbours ----------------------------------------------------------

def ssd_causal_conv1d(x, w, bias, out, silu=True, stream=None):
    """C entry: x, out [B,D,S]; w [D,W] fp32; bias [D] fp32 or None."""
    Bb, D, S = x.shape
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_causal_conv1d(Bb, D, S, w.shape[1], _DTYPE_CODES[x.dtype], _ptr(x), _ptr(w),
                                            _ptr(bias), 1 if silu else 0, _ptr(out), s), "ssd_causal_conv1d")


def ssd_causal_conv1d_tokens(x, w, bias, out, silu=True, stream=None):
    """C entry: token-major x, out [B,S,C]; w [C,W] fp32; bias [C] fp32 or None."""
    Bb, S, C = x.shape
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_causal_conv1d_tokens(Bb, S, C, w.shape[1], _DTYPE_CODES[x.dtype], _ptr(x), _ptr(w),
                                                   _ptr(bias), 1 if silu else 0, _ptr(out), s),
           "ssd_causal_conv1d_tokens")


def ssd_gated_rmsnorm(x, z, w, groups, eps, out, stream=None):
    """C entry: x, z, out [..., D] (rows = the leading dims); w [D] fp32."""
    D = x.shape[-1]
    rows = x.numel() // D
    s = stream if stream is not None else _stream_handle()
    _check(load_library().ssd_gated_rmsnorm(rows, D, groups, float(eps), _DTYPE_CODES[x.dtype], _ptr(x), _ptr(z),
                                            _ptr(w), _ptr(out), s), "ssd_gated_rmsnorm")


def causal_conv1d(x, w, bias=None, silu=True):
    """Depthwise causal conv1d (+ bias) then SiLU on the GPU; x [B,D,S]."""
    out = torch.empty_like(x)
    ssd_causal_conv1d(x, w, bias, out, silu, _stream_handle(x.device))
    return out


def gated_rmsnorm(x, z, w, groups, eps=1e-5):
    """(x * silu(z)) normalised per group of D/groups channels, times w, on the GPU."""
    out = torch.empty_like(x)
    ssd_gated_rmsnorm(x, z, w, groups, eps, out, _stream_handle(x.device))
    return out
