"""Python binding of the C ABI in include/jfa.h (argument marshalling only).

Every step of the attention runs in the library's CUDA kernels; this module only
checks tensors, allocates outputs and workspace through PyTorch's allocator, and
passes raw device pointers plus the current CUDA stream.  There is no CPU path:
without the built library, or with CPU tensors, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

from . import build as _build

JFA_OK = 0
STATUS_NAMES = {0: "JFA_OK", 1: "JFA_ERR_INVALID_ARG", 2: "JFA_ERR_UNSUPPORTED", 3: "JFA_ERR_WORKSPACE",
                4: "JFA_ERR_CUDA", 5: "JFA_ERR_BAD_OFFSETS", 6: "JFA_ERR_TIMEOUT"}

# Every symbol include/jfa.h declares.
EXPORTED_SYMBOLS = ("jfa_workspace_size", "jfa_forward", "jfa_forward_noalloc", "jfa_backward", "jfa_check_status",
                    "jfa_status_string", "jfa_last_launch_count", "jfa_last_error", "jfa_timing_enable",
                    "jfa_timing_read", "jfa_trace_configure", "jfa_selftest_wait_timeout", "jfa_wait_limit_ns",
                    "jfa_set_nsp_max_tiles")
KERNEL_KINDS = ("plan", "forward", "bwd_preprocess", "bwd_dkdv", "bwd_dq", "bwd_fused", "bwd_nsp")


class JfaError(RuntimeError):
    def __init__(self, status: int, what: str):
        detail = ""
        if status == 4:
            try:
                detail = " -- " + load_library(build_if_missing=False).jfa_last_error().decode()
            except Exception:
                pass
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status_string(status)}){detail}")
        self.status = status


class _Bias(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("table", ctypes.c_void_p), ("num_buckets", ctypes.c_int),
                ("center", ctypes.c_int), ("grad", ctypes.c_void_p), ("values", ctypes.c_void_p),
                ("block_offsets", ctypes.c_void_p), ("plane", ctypes.c_int64), ("values_grad", ctypes.c_void_p)]


_LIB = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load the in-tree shared library (building it first if asked and needed)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB_PATH
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"jagged attention library not built ({path} missing); run build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.jfa_workspace_size.argtypes = [i32, i32, i32, i64, i64, i32]
    lib.jfa_workspace_size.restype = sz
    lib.jfa_forward.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i64, i64, ctypes.POINTER(_Bias), f32, i32,
                                vp, vp, vp, sz, vp]
    lib.jfa_forward.restype = i32
    lib.jfa_forward_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i64, i64, ctypes.POINTER(_Bias), f32,
                                        i32, vp, vp, vp]
    lib.jfa_forward_noalloc.restype = i32
    lib.jfa_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i64, i64,
                                 ctypes.POINTER(_Bias), f32, i32, vp, vp, vp, vp, sz, vp]
    lib.jfa_backward.restype = i32
    lib.jfa_check_status.argtypes = [vp, vp]
    lib.jfa_check_status.restype = i32
    lib.jfa_status_string.argtypes = [i32]
    lib.jfa_status_string.restype = ctypes.c_char_p
    lib.jfa_last_launch_count.argtypes = []
    lib.jfa_last_launch_count.restype = i32
    lib.jfa_last_error.argtypes = []
    lib.jfa_last_error.restype = ctypes.c_char_p
    lib.jfa_timing_enable.argtypes = [i32]
    lib.jfa_timing_enable.restype = i32
    lib.jfa_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int), i32]
    lib.jfa_timing_read.restype = i32
    lib.jfa_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint64, vp]
    lib.jfa_selftest_wait_timeout.restype = i32
    lib.jfa_set_nsp_max_tiles.argtypes = [i32]
    lib.jfa_set_nsp_max_tiles.restype = i32
    lib.jfa_wait_limit_ns.argtypes = [i64, i32, i64]
    lib.jfa_wait_limit_ns.restype = ctypes.c_uint64
    lib.jfa_trace_configure.argtypes = [vp, sz, i32]
    lib.jfa_trace_configure.restype = i32
    _LIB = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library(build_if_missing=False).jfa_status_string(int(status)).decode()
    except Exception:  # library not loadable: fall back to the enum name
        return STATUS_NAMES.get(status, "unknown")


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check_values(name, t, rows=None, H=None, d=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 3 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [T, H, d] tensor")
    if H is not None and (t.shape[1] != H or t.shape[2] != d):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected [*, {H}, {d}]")
    if rows is not None and t.shape[0] != rows:
        raise ValueError(f"{name} has {t.shape[0]} rows, expected {rows}")


def _check_lse(t, H, Tq):
    if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 or tuple(t.shape) != (H, Tq)
            or not t.is_contiguous()):
        raise ValueError(f"lse must be a contiguous float32 CUDA tensor [{H}, {Tq}]")


def _check_workspace(ws, nbytes, device):
    """A caller-given workspace: contiguous bytes on the inputs' device, at least `nbytes`
    long (its size is passed to the library in bytes, whatever its dtype)."""
    if not isinstance(ws, torch.Tensor) or not ws.is_cuda or ws.device != device or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor on the inputs' device")
    have = ws.numel() * ws.element_size()
    if have < nbytes:
        raise ValueError(f"workspace holds {have} bytes, the call needs {nbytes}")
    if ws.data_ptr() % 256:
        raise ValueError("workspace must start on a 256-byte boundary")
    return have


def _check_offsets(name, off):
    if not isinstance(off, torch.Tensor) or not off.is_cuda or off.dtype != torch.int64 or off.dim() != 1 \
            or not off.is_contiguous() or off.numel() < 2:
        raise ValueError(f"{name} must be a contiguous int64 CUDA tensor [B+1] with B >= 1")


def _bias_struct(bias, center, H, grad=None, jagged_bias=None, jagged_bias_grad=None):
    if jagged_bias is not None:
        if bias is not None or grad is not None:
            raise ValueError("a general jagged bias excludes the relative-position table and its gradient")
        values, boff = jagged_bias
        if (not values.is_cuda or values.dtype != torch.bfloat16 or values.dim() != 2 or values.shape[0] != H
                or not values.is_contiguous()):
            raise ValueError("jagged bias values must be a contiguous bf16 CUDA tensor [H, plane]")
        _check_offsets("jagged bias block offsets", boff)
        gptr = None
        if jagged_bias_grad is not None:
            if (jagged_bias_grad.dtype != torch.bfloat16 or tuple(jagged_bias_grad.shape) != tuple(values.shape)
                    or not jagged_bias_grad.is_contiguous() or jagged_bias_grad.device != values.device):
                raise ValueError("jagged_bias_grad must be a contiguous bf16 tensor shaped like the bias values")
            gptr = jagged_bias_grad.data_ptr()
        return (_Bias(2, None, 0, 0, None, values.data_ptr(), boff.data_ptr(), values.shape[1], gptr),
                (values, boff))
    if jagged_bias_grad is not None:
        raise ValueError("jagged_bias_grad needs a general jagged bias")
    if bias is None:
        if grad is not None:
            raise ValueError("bias_grad needs a bias table")
        return None, None
    if not bias.is_cuda or bias.dtype != torch.float32 or bias.dim() != 2 or bias.shape[0] != H:
        raise ValueError("bias must be a float32 CUDA tensor [H, num_buckets]")
    bias = bias.contiguous()
    gptr = None
    if grad is not None:
        if (grad.device != bias.device or grad.dtype != torch.float32 or tuple(grad.shape) != tuple(bias.shape)
                or not grad.is_contiguous()):
            raise ValueError("bias_grad must be a contiguous float32 tensor shaped like the bias table, on its device")
        gptr = grad.data_ptr()
    return _Bias(1, bias.data_ptr(), bias.shape[1], int(center), gptr), bias


def workspace_size(B, H, d, total_q, total_kv, backward) -> int:
    return int(load_library().jfa_workspace_size(B, H, d, total_q, total_kv, 1 if backward else 0))


def new_workspace(B, H, d, total_q, total_kv, backward, device) -> torch.Tensor:
    """A zero-initialised workspace for jfa_forward (backward=False) or jfa_backward."""
    return _workspace(workspace_size(B, H, d, total_q, total_kv, backward), device)


def _workspace(nbytes, device):
    # 256-byte alignment is guaranteed by the caching allocator; the status header must
    # start zeroed
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


def jfa_forward(q, k, v, q_offsets, kv_offsets, bias=None, bias_center=0, scale=None, causal=False,
                out=None, lse=None, workspace=None, stream=None, jagged_bias=None):
    """out, lse = jfa_forward(...): the C-ABI forward on PyTorch-allocated device memory.

    q: bf16 [Tq, H, d]; k, v: bf16 [Tk, H, d]; offsets: int64 [B+1] on the device.
    bias: optional fp32 [H, num_buckets] relative-position table (bucket j - i + bias_center).
    jagged_bias: optional (values bf16 [H, plane], block offsets int64 [B+1]): a general
    bias, one Lq x Lk block per sequence with rows padded to 8 elements (see jfa.h).
    Returns out bf16 [Tq, H, d] and lse fp32 [H, Tq].  The call is asynchronous on
    the current stream; device-side errors are reported by jfa_check_status(workspace).
    """
    lib = load_library()
    _check_values("q", q)
    Tq, H, d = q.shape
    _check_values("k", k, H=H, d=d)
    _check_values("v", v, rows=k.shape[0], H=H, d=d)
    _check_offsets("q_offsets", q_offsets)
    _check_offsets("kv_offsets", kv_offsets)
    B = q_offsets.numel() - 1
    if kv_offsets.numel() != B + 1:
        raise ValueError("q_offsets and kv_offsets must have the same length")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    bstruct, bias_keep = _bias_struct(bias, bias_center, H, jagged_bias=jagged_bias)
    for name, t in (("k", k), ("v", v), ("q_offsets", q_offsets), ("kv_offsets", kv_offsets)):
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_values("out", out, rows=Tq, H=H, d=d)
    if lse is None:
        lse = torch.empty((H, Tq), dtype=torch.float32, device=q.device)
    else:
        _check_lse(lse, H, Tq)
    nbytes = int(lib.jfa_workspace_size(B, H, d, Tq, k.shape[0], 0))
    if workspace is None:
        workspace = _workspace(nbytes, q.device)
    ws_bytes = _check_workspace(workspace, nbytes, q.device)
    st = lib.jfa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), q_offsets.data_ptr(), kv_offsets.data_ptr(),
                         B, H, d, Tq, k.shape[0], ctypes.byref(bstruct) if bstruct is not None else None,
                         scale, 1 if causal else 0, out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
                         ws_bytes, _stream_handle(stream))
    if st != JFA_OK:
        raise JfaError(st, "jfa_forward")
    del bias_keep
    return out, lse, workspace


def jfa_backward(dout, q, k, v, out, lse, q_offsets, kv_offsets, bias=None, bias_center=0, scale=None,
                 causal=False, dq=None, dk=None, dv=None, workspace=None, stream=None, bias_grad=None,
                 jagged_bias=None, jagged_bias_grad=None):
    """dq, dk, dv, workspace = jfa_backward(...): gradients of sum(dout * out).  With
    `bias_grad` (a float32 tensor shaped like `bias`) the bias table's gradient is written
    into it as well; with `jagged_bias_grad` (a bf16 tensor shaped like a general bias's
    values) that bias's gradient (dS at every block element)."""
    lib = load_library()
    _check_values("q", q)
    Tq, H, d = q.shape
    for name, t, rows in (("dout", dout, Tq), ("out", out, Tq), ("k", k, None), ("v", v, k.shape[0])):
        _check_values(name, t, rows=rows, H=H, d=d)
    _check_lse(lse, H, Tq)
    _check_offsets("q_offsets", q_offsets)
    _check_offsets("kv_offsets", kv_offsets)
    B = q_offsets.numel() - 1
    if kv_offsets.numel() != B + 1:
        raise ValueError("q_offsets and kv_offsets must have the same length")
    for name, t in (("dout", dout), ("k", k), ("v", v), ("out", out), ("lse", lse), ("q_offsets", q_offsets),
                    ("kv_offsets", kv_offsets)):
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    bstruct, bias_keep = _bias_struct(bias, bias_center, H, bias_grad, jagged_bias, jagged_bias_grad)
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t is not None:
            _check_values(name, t, rows=ref.shape[0], H=H, d=d)
            if t.device != q.device:
                raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nbytes = int(lib.jfa_workspace_size(B, H, d, Tq, k.shape[0], 1))
    if workspace is None:
        workspace = _workspace(nbytes, q.device)
    ws_bytes = _check_workspace(workspace, nbytes, q.device)
    st = lib.jfa_backward(dout.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr(), q_offsets.data_ptr(), kv_offsets.data_ptr(), B, H, d, Tq, k.shape[0],
                          ctypes.byref(bstruct) if bstruct is not None else None, scale, 1 if causal else 0,
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(), ws_bytes,
                          _stream_handle(stream))
    if st != JFA_OK:
        raise JfaError(st, "jfa_backward")
    del bias_keep
    return dq, dk, dv, workspace


def jfa_check_status(workspace, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status of the last call."""
    return int(load_library().jfa_check_status(workspace.data_ptr(), _stream_handle(stream)))


def jfa_set_nsp_max_tiles(max_tiles: int) -> int:
    """Sequences of 2 .. max_tiles query tiles take the non-sequence-parallel backward pass
    (0 or 1: none, the default); returns the previous setting.  Process-wide."""
    prev = int(load_library().jfa_set_nsp_max_tiles(int(max_tiles)))
    if prev < 0:
        raise ValueError(f"max_tiles must be in 0 .. 16, got {max_tiles}")
    return prev


def jfa_nsp_max_tiles() -> int:
    return int(load_library().jfa_set_nsp_max_tiles(-1))


def jfa_last_launch_count() -> int:
    return int(load_library().jfa_last_launch_count())


def jfa_timing_enable(on: bool) -> None:
    load_library().jfa_timing_enable(1 if on else 0)


def jfa_timing_read() -> dict:
    """{kind: (total_ms, launches)} for the launches recorded since the last read."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    st = load_library().jfa_timing_read(ms, cnt, n)
    if st != JFA_OK:
        raise JfaError(st, "jfa_timing_read")
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}


def jfa_trace_configure(buffer: Optional[torch.Tensor], kernel_kind: str = "forward") -> None:
    """Developer tracing: record pipeline events of the first CTA of every later launch of
    `kernel_kind` into `buffer` (a CUDA int64/uint8 tensor); None turns tracing off."""
    lib = load_library()
    if buffer is None:
        st = lib.jfa_trace_configure(None, 0, -1)
    else:
        st = lib.jfa_trace_configure(buffer.data_ptr(), buffer.numel() * buffer.element_size(),
                                     KERNEL_KINDS.index(kernel_kind))
    if st != JFA_OK:
        raise JfaError(st, "jfa_trace_configure")


def decode_trace(buffer: torch.Tensor):
    """Split a trace buffer into per-role lists of (sm_clock, event_id), dropping unused
    entries (the buffer should be zeroed before tracing)."""
    flat = buffer.detach().cpu().view(torch.int64).numpy()
    cap = flat.size // 5
    raw = flat[:5 * cap].reshape(5, cap)
    roles = []
    for r in range(5):
        ent = [int(x) & 0xFFFFFFFFFFFFFFFF for x in raw[r] if int(x) != 0]
        roles.append([(e >> 16, e & 0xFF) for e in ent])
    return roles


class JaggedAttention(torch.autograd.Function):
    """Differentiable jagged attention: out = JaggedAttention.apply(q, k, v, q_offsets,
    kv_offsets, bias, bias_center, scale, causal, jagged_bias_values, jagged_bias_offsets).
    lse is saved for the backward; the relative-position table and a general jagged bias's
    values get their gradients when they require them."""

    @staticmethod
    def forward(ctx, q, k, v, q_offsets, kv_offsets, bias=None, bias_center=0, scale=None, causal=False,
                jb_values=None, jb_offsets=None):
        jb = (jb_values, jb_offsets) if jb_values is not None else None
        out, lse, _ = jfa_forward(q, k, v, q_offsets, kv_offsets, bias, bias_center, scale, causal, jagged_bias=jb)
        ctx.save_for_backward(q, k, v, out, lse, q_offsets, kv_offsets, bias, jb_values, jb_offsets)
        ctx.cfg = (bias_center, scale, causal)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse, q_offsets, kv_offsets, bias, jb_values, jb_offsets = ctx.saved_tensors
        bias_center, scale, causal = ctx.cfg
        jb = (jb_values, jb_offsets) if jb_values is not None else None
        dbias = torch.empty_like(bias) if bias is not None and ctx.needs_input_grad[5] else None
        djb = torch.empty_like(jb_values) if jb_values is not None and ctx.needs_input_grad[9] else None
        dq, dk, dv, _ = jfa_backward(dout.contiguous(), q, k, v, out, lse, q_offsets, kv_offsets, bias,
                                     bias_center, scale, causal, bias_grad=dbias, jagged_bias=jb,
                                     jagged_bias_grad=djb)
        return dq, dk, dv, None, None, dbias, None, None, None, djb, None


def jagged_attention(q, k, v, q_offsets, kv_offsets, bias=None, bias_center=0, scale=None, causal=False,
                     jagged_bias=None):
    jb_values, jb_offsets = jagged_bias if jagged_bias is not None else (None, None)
    return JaggedAttention.apply(q, k, v, q_offsets, kv_offsets, bias, bias_center, scale, causal, jb_values,
                                 jb_offsets)
