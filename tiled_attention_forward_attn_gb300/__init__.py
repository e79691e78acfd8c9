"""Fused attention forward for GB300 (sm_103a) — Python binding.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libfa.so`` behind the C ABI of ``include/fa.h``.  There is no
CPU or PyTorch fallback; if the library is missing, every call raises.

Names follow the C ABI: :func:`fa_fwd` takes preallocated device tensors;
:func:`attention_forward` allocates the outputs and calls :func:`fa_fwd`.
Also: :func:`fa_fwd_host` (the forward for tensors in host memory, copies
included), :func:`fa_fwd_splitkv` / :func:`attention_forward_splitkv` (few
queries against many keys) and :func:`fa_fwd_splitkv_static`,
:func:`fa_bwd` / :func:`attention_backward` (gradients, bf16 or fp16),
:func:`attention` (forward and backward as one torch.autograd function),
:func:`fa_fwd_splitkv_host` and :func:`fa_bwd_host` (host tensors, copies included),
:func:`attention_forward_order_ablation` (the two loop orders), and the
device status / test-hook functions.  :func:`reload_library` switches to
another build of the library, e.g. ``GUARDED_LIB_PATH`` (every tile origin,
TMEM range and store bounds-checked; FA_DEVICE_STATUS_BOUNDS on a failure).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import _build

__all__ = [
    "FAError", "fa_fwd", "attention_forward", "fa_strerror", "fa_version", "fa_fwd_strided",
    "fa_bwd_strided",
    "fa_fwd_host", "fa_fwd_host_workspace_bytes",
    "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_bytes", "fa_fwd_splitkv_num_splits",
    "attention_forward_splitkv", "fa_fwd_splitkv_static", "fa_fwd_splitkv_static_scratch_bytes",
    "fa_fwd_splitkv_host", "fa_fwd_splitkv_host_workspace_bytes",
    "fa_bwd", "fa_bwd_workspace_bytes", "fa_bwd_host", "fa_bwd_host_workspace_bytes",
    "attention_backward", "attention", "attention_forward_order_ablation",
    "fa_get_device_status", "fa_clear_device_status", "fa_set_wait_limit_ns",
    "fa_set_fault_injection", "load_library", "reload_library", "LIB_PATH", "GUARDED_LIB_PATH",
    "FA_DEVICE_STATUS_TIMEOUT", "FA_DEVICE_STATUS_BOUNDS", "FA_INJECT_SKIP_FIRST_V_LOAD",
]

LIB_PATH = _build.LIB_PATH
GUARDED_LIB_PATH = _build.GUARDED_LIB_PATH
FA_DEVICE_STATUS_TIMEOUT = 1
FA_DEVICE_STATUS_BOUNDS = 2
FA_INJECT_SKIP_FIRST_V_LOAD = 1

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    """A non-zero return code from the C ABI."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: error {code}: {fa_strerror(code)}")


def load_library(path: str | None = None):
    """Load libfa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library not built: {path} is missing "
                "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        lib = ctypes.CDLL(path)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.fa_fwd.restype = i
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.fa_fwd_strided.restype = i
        lib.fa_fwd_strided.argtypes = [vp, i64p, vp, i64p, vp, i64p, vp, i64p, vp, i, i, i, i, i,
                                       i, f, vp]
        lib.fa_fwd_host.restype = i
        lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, ctypes.c_size_t,
                                    vp]
        lib.fa_fwd_host_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_fwd_host_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_strerror.restype = ctypes.c_char_p
        lib.fa_strerror.argtypes = [i]
        lib.fa_get_device_status.restype = i
        lib.fa_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.fa_clear_device_status.restype = i
        lib.fa_clear_device_status.argtypes = []
        lib.fa_set_wait_limit_ns.restype = i
        lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        lib.fa_set_fault_injection.restype = i
        lib.fa_set_fault_injection.argtypes = [ctypes.c_uint]
        lib.fa_version.restype = i
        lib.fa_version.argtypes = []
        lib.fa_fwd_splitkv.restype = i
        lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp,
                                       ctypes.c_size_t, vp]
        lib.fa_fwd_splitkv_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_fwd_splitkv_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.fa_fwd_splitkv_num_splits.restype = i
        lib.fa_fwd_splitkv_num_splits.argtypes = [i, i, i, i, i, i]
        lib.fa_bwd.restype = i
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp,
                               ctypes.c_size_t, vp]
        lib.fa_bwd_ex.restype = i
        lib.fa_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp,
                                  ctypes.c_size_t, vp]
        lib.fa_bwd_strided.restype = i
        lib.fa_bwd_strided.argtypes = [vp, i64p, vp, i64p, vp, i64p, vp, i64p, vp, vp, i64p, vp,
                                       i64p, vp, i64p, vp, i64p, i, i, i, i, i, i, f, vp,
                                       ctypes.c_size_t, vp]
        lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_fwd_order_ablation.restype = i
        lib.fa_fwd_order_ablation.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp,
                                              ctypes.c_size_t, vp]
        lib.fa_fwd_order_ablation_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_fwd_order_ablation_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.fa_fwd_splitkv_static.restype = i
        lib.fa_fwd_splitkv_static.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_splitkv_static_scratch_bytes.restype = ctypes.c_size_t
        lib.fa_fwd_splitkv_static_scratch_bytes.argtypes = []
        lib.fa_fwd_splitkv_host.restype = i
        lib.fa_fwd_splitkv_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp,
                                            ctypes.c_size_t, vp]
        lib.fa_fwd_splitkv_host_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_fwd_splitkv_host_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.fa_bwd_host.restype = i
        lib.fa_bwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp,
                                    ctypes.c_size_t, vp]
        lib.fa_bwd_host_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_bwd_host_workspace_bytes.argtypes = [i, i, i, i]
        _lib = lib
        return lib


def reload_library(path: str | None = None):
    """Make later calls use the library at `path` (default: LIB_PATH), e.g.
    GUARDED_LIB_PATH; returns it.  Each build keeps its own device status
    word."""
    global _lib
    with _lock:
        _lib = None
    return load_library(path)


def fa_strerror(code: int) -> str:
    return load_library().fa_strerror(int(code)).decode()


def fa_version() -> int:
    return int(load_library().fa_version())


def _check(code: int, where: str):
    if code != 0:
        raise FAError(code, where)


def fa_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int,
               N: int, d: int, causal: bool, scale: float, stream: int = 0) -> int:
    """Direct call with integer device addresses; returns the C return code."""
    return int(load_library().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(N),
                                     int(d), int(bool(causal)), float(scale), stream or None))


def _dims(t):
    if t.dim() != 4:
        raise ValueError("expected a [B, H, N, d] tensor")
    return tuple(int(x) for x in t.shape)


FA_DTYPE_BF16 = 0
FA_DTYPE_FP16 = 1


def fa_fwd_strided(q_ptr: int, q_strides, k_ptr: int, k_strides, v_ptr: int, v_strides,
                   o_ptr: int, o_strides, lse_ptr: int, dtype: int, B: int, H: int, N: int,
                   d: int, causal: bool, scale: float, stream: int = 0) -> int:
    """Direct call of the strided entry point; strides are 3-tuples of
    element strides (batch, head, row) or None; returns the C return code."""
    def arr(st):
        if st is None:
            return None
        return (ctypes.c_int64 * 3)(*[int(x) for x in st])

    return int(load_library().fa_fwd_strided(
        q_ptr, arr(q_strides), k_ptr, arr(k_strides), v_ptr, arr(v_strides), o_ptr,
        arr(o_strides), lse_ptr, int(dtype), int(B), int(H), int(N), int(d), int(bool(causal)),
        float(scale), stream or None))


def fa_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """Attention forward into preallocated CUDA tensors.

    q, k, v, o: ``[B, H, N, d]`` tensors of one dtype, ``torch.bfloat16`` or
    ``torch.float16``, on one CUDA device, any strides with the last
    dimension contiguous (strides multiples of 8 elements); lse:
    ``torch.float32`` ``[B, H, N]`` contiguous.  Enqueued on ``stream``
    (default: the current torch stream of q's device); asynchronous.
    """
    import torch

    B, H, N, d = _dims(q)
    for name, t in (("k", k), ("v", v), ("o", o)):
        if tuple(t.shape) != (B, H, N, d):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {(B, H, N, d)}")
    if tuple(lse.shape) != (B, H, N):
        raise ValueError(f"lse has shape {tuple(lse.shape)}, expected {(B, H, N)}")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"q must be bfloat16 or float16, got {q.dtype}")
    for name, t, dt in (("q", q, q.dtype), ("k", k, q.dtype), ("v", v, q.dtype),
                        ("o", o, q.dtype), ("lse", lse, torch.float32)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.device != q.device:
            raise ValueError("all tensors must be on one device")
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if t.stride(3) != 1 and d > 1:
            raise ValueError(f"{name} must have a contiguous last dimension")
    if not lse.is_contiguous():
        raise ValueError("lse must be contiguous")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    dtype = FA_DTYPE_FP16 if q.dtype == torch.float16 else FA_DTYPE_BF16

    def st(t):  # a dimension of extent 1 is never stepped: its stride is irrelevant
        return tuple(0 if t.shape[i] == 1 else t.stride(i) for i in range(3))

    with torch.cuda.device(q.device):
        _check(fa_fwd_strided(q.data_ptr(), st(q), k.data_ptr(), st(k), v.data_ptr(), st(v),
                              o.data_ptr(), st(o), lse.data_ptr(), dtype, B, H, N, d, causal,
                              scale, handle), "fa_fwd")


def fa_fwd_host_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    """Device workspace bytes fa_fwd_host needs (0 on invalid arguments)."""
    return int(load_library().fa_fwd_host_workspace_bytes(B, H, N, d))


def fa_fwd_host(q, k, v, o, lse, causal: bool, scale: float, workspace, stream=None) -> None:
    """Forward with host tensors (C ABI ``fa_fwd_host``): copies Q, K, V into
    ``workspace`` on the device, runs the forward and copies O and LSE back,
    all queued on ``stream``; synchronise it before reading ``o``, ``lse``.

    q, k, v, o: contiguous CPU tensors ``[B, H, N, d]`` of one type
    (``torch.bfloat16`` or ``torch.float16``; page-locked for asynchronous
    copies); lse: contiguous CPU ``torch.float32`` ``[B, H, N]``; workspace: a
    CUDA byte tensor of at least :func:`fa_fwd_host_workspace_bytes` bytes
    (its device is the one used).
    """
    import torch

    B, H, N, d = _dims(q)
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q must be torch.bfloat16 or torch.float16")
    for name, t, dt, shape in (("k", k, q.dtype, (B, H, N, d)), ("v", v, q.dtype, (B, H, N, d)),
                               ("o", o, q.dtype, (B, H, N, d)), ("lse", lse, torch.float32, (B, H, N)),
                               ("q", q, q.dtype, (B, H, N, d))):
        if tuple(t.shape) != shape or t.dtype != dt or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU {dt} tensor of shape {shape}")
    if not workspace.is_cuda or workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a CUDA uint8 tensor")
    with torch.cuda.device(workspace.device):
        if stream is None:
            stream = torch.cuda.current_stream(workspace.device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        dtype = FA_DTYPE_FP16 if q.dtype == torch.float16 else FA_DTYPE_BF16
        rc = load_library().fa_fwd_host(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dtype,
            B, H, N, d, int(bool(causal)), float(scale), workspace.data_ptr(),
            workspace.numel(), handle or None)
        _check(rc, "fa_fwd_host")


def _host_stream(workspace, stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_host(name, t, dt, shape):
    if tuple(t.shape) != tuple(shape) or t.dtype != dt or t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CPU {dt} tensor of shape {tuple(shape)}")


def fa_fwd_splitkv_host_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int,
                                        num_splits: int = 0) -> int:
    """Device workspace bytes fa_fwd_splitkv_host needs on the current device."""
    return int(load_library().fa_fwd_splitkv_host_workspace_bytes(B, H, Nq, Nk, d, num_splits))


def fa_fwd_splitkv_host(q, k, v, o, lse, causal: bool, scale: float, num_splits: int, workspace,
                        stream=None) -> None:
    """Split-KV forward with host tensors (C ABI ``fa_fwd_splitkv_host``):
    copies Q, K, V into ``workspace``, runs the split-KV path and copies O
    and LSE back, all queued on ``stream``; synchronise before reading.

    q, o: contiguous CPU bf16 ``[B, H, Nq, d]``; k, v: ``[B, H, Nk, d]``;
    lse: CPU float32 ``[B, H, Nq]``; workspace: a CUDA uint8 tensor of at
    least :func:`fa_fwd_splitkv_host_workspace_bytes` bytes."""
    import torch

    B, H, Nq, d = _dims(q)
    Nk = int(k.shape[2])
    for name, t, dt, shape in (("q", q, torch.bfloat16, (B, H, Nq, d)),
                               ("k", k, torch.bfloat16, (B, H, Nk, d)),
                               ("v", v, torch.bfloat16, (B, H, Nk, d)),
                               ("o", o, torch.bfloat16, (B, H, Nq, d)),
                               ("lse", lse, torch.float32, (B, H, Nq))):
        _check_host(name, t, dt, shape)
    if not workspace.is_cuda or workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a CUDA uint8 tensor")
    with torch.cuda.device(workspace.device):
        rc = load_library().fa_fwd_splitkv_host(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk,
            d, int(bool(causal)), float(scale), int(num_splits), workspace.data_ptr(),
            workspace.numel(), _host_stream(workspace, stream) or None)
        _check(rc, "fa_fwd_splitkv_host")


def fa_bwd_host_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    """Device workspace bytes fa_bwd_host needs (0 on invalid arguments)."""
    return int(load_library().fa_bwd_host_workspace_bytes(B, H, N, d))


def fa_bwd_host(q, k, v, o, lse, dout, dq, dk, dv, causal: bool, scale: float, workspace,
                stream=None) -> None:
    """Backward with host tensors (C ABI ``fa_bwd_host``): copies Q, K, V, O,
    LSE, dO into ``workspace``, runs the backward and copies dQ, dK, dV
    back, all queued on ``stream``; synchronise before reading.

    q, k, v, o, dout, dq, dk, dv: contiguous CPU tensors ``[B, H, N, d]`` of
    one type (bf16 or fp16); lse: CPU float32 ``[B, H, N]``; workspace: a CUDA
    uint8 tensor of at least :func:`fa_bwd_host_workspace_bytes` bytes."""
    import torch

    B, H, N, d = _dims(q)
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q must be torch.bfloat16 or torch.float16")
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq), ("dk", dk),
                    ("dv", dv), ("q", q)):
        _check_host(name, t, q.dtype, (B, H, N, d))
    _check_host("lse", lse, torch.float32, (B, H, N))
    if not workspace.is_cuda or workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a CUDA uint8 tensor")
    with torch.cuda.device(workspace.device):
        dtype = FA_DTYPE_FP16 if q.dtype == torch.float16 else FA_DTYPE_BF16
        rc = load_library().fa_bwd_host(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dtype, B, H, N, d,
            int(bool(causal)), float(scale), workspace.data_ptr(), workspace.numel(),
            _host_stream(workspace, stream) or None)
        _check(rc, "fa_bwd_host")


def attention_forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Allocate ``O`` (bf16) and ``LSE`` (fp32) and run :func:`fa_fwd`.

    ``scale`` defaults to ``1/sqrt(d)``.  O has q's dtype and is contiguous.
    Returns ``(O, LSE)``.
    """
    import torch

    B, H, N, d = _dims(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty((B, H, N, d), dtype=q.dtype, device=q.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def fa_fwd_splitkv_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int,
                                   num_splits: int = 0) -> int:
    """Workspace bytes fa_fwd_splitkv needs (0 on invalid arguments)."""
    return int(load_library().fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits))


def fa_fwd_splitkv_num_splits(B: int, H: int, Nq: int, Nk: int, d: int,
                              num_splits: int = 0) -> int:
    """Key ranges fa_fwd_splitkv uses (0 on invalid arguments)."""
    return int(load_library().fa_fwd_splitkv_num_splits(B, H, Nq, Nk, d, num_splits))


def fa_fwd_splitkv(q, k, v, o, lse, causal: bool, scale: float, num_splits: int = 0,
                   workspace=None, stream=None) -> None:
    """Split-KV attention forward into preallocated CUDA tensors.

    q, o: ``torch.bfloat16`` ``[B, H, Nq, d]`` (Nq <= 16); k, v: ``[B, H, Nk, d]``;
    lse: ``torch.float32`` ``[B, H, Nq]``.  ``workspace``: a CUDA byte tensor of
    at least :func:`fa_fwd_splitkv_workspace_bytes`; allocated here when None.
    """
    import torch

    B, H, Nq, d = _dims(q)
    Bk, Hk, Nk, dk = _dims(k)
    if (Bk, Hk, dk) != (B, H, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, H, Nk, d] matching q's B, H, d")
    if tuple(o.shape) != (B, H, Nq, d) or tuple(lse.shape) != (B, H, Nq):
        raise ValueError("o must be [B, H, Nq, d] and lse [B, H, Nq]")
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("o", o, torch.bfloat16),
                        ("lse", lse, torch.float32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous {dt} CUDA tensor on q's device")
    with torch.cuda.device(q.device):
        if workspace is None:
            nbytes = fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits)
            if nbytes == 0:
                raise FAError(2, "fa_fwd_splitkv_workspace_bytes")
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        rc = load_library().fa_fwd_splitkv(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk,
            d, int(bool(causal)), float(scale), int(num_splits), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), handle or None)
        _check(rc, "fa_fwd_splitkv")


def attention_forward_splitkv(q, k, v, causal: bool = False, scale: float | None = None,
                              num_splits: int = 0, stream=None):
    """Allocate O and LSE (and a workspace) and run :func:`fa_fwd_splitkv`."""
    import torch

    B, H, Nq, d = _dims(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    fa_fwd_splitkv(q, k, v, o, lse, causal, scale, num_splits, None, stream)
    return o, lse


def fa_fwd_splitkv_static_scratch_bytes() -> int:
    """Size of the scratch array built into the library for
    :func:`fa_fwd_splitkv_static`."""
    return int(load_library().fa_fwd_splitkv_static_scratch_bytes())


def fa_fwd_splitkv_static(q, k, v, o, lse, causal: bool, scale: float, num_splits: int = 0,
                          stream=None) -> None:
    """:func:`fa_fwd_splitkv` without a workspace and without any device
    allocation, for callers that cannot allocate: the scratch is the
    library's built-in array (shared by every call on a device; order calls
    on one stream).  Tensors as for :func:`fa_fwd_splitkv`."""
    import torch

    B, H, Nq, d = _dims(q)
    Bk, Hk, Nk, dk = _dims(k)
    if (Bk, Hk, dk) != (B, H, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, H, Nk, d] matching q's B, H, d")
    if tuple(o.shape) != (B, H, Nq, d) or tuple(lse.shape) != (B, H, Nq):
        raise ValueError("o must be [B, H, Nq, d] and lse [B, H, Nq]")
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("o", o, torch.bfloat16),
                        ("lse", lse, torch.float32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous {dt} CUDA tensor on q's device")
    with torch.cuda.device(q.device):
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        rc = load_library().fa_fwd_splitkv_static(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk,
            d, int(bool(causal)), float(scale), int(num_splits), handle or None)
        _check(rc, "fa_fwd_splitkv_static")


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    """Workspace bytes fa_bwd needs (0 on invalid arguments)."""
    return int(load_library().fa_bwd_workspace_bytes(B, H, N, d))


def _arr3(st):
    return None if st is None else (ctypes.c_int64 * 3)(*[int(x) for x in st])


def fa_bwd_strided(ptrs, strides, lse_ptr: int, dtype: int, B: int, H: int, N: int, d: int,
                   causal: bool, scale: float, workspace_ptr: int, workspace_bytes: int,
                   stream: int = 0) -> int:
    """Direct call of the strided backward entry point.

    ``ptrs``: device addresses of (q, k, v, o, dout, dq, dk, dv); ``strides``:
    eight 3-tuples of element strides (batch, head, row) or None, in the same
    order.  Returns the C return code."""
    q, k, v, o, do, dq, dk, dv = (int(x) for x in ptrs)
    sq, sk, sv, so, sdo, sdq, sdk, sdv = (_arr3(x) for x in strides)
    return int(load_library().fa_bwd_strided(
        q, sq, k, sk, v, sv, o, so, lse_ptr, do, sdo, dq, sdq, dk, sdk, dv, sdv, int(dtype),
        int(B), int(H), int(N), int(d), int(bool(causal)), float(scale), workspace_ptr,
        int(workspace_bytes), stream or None))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, causal: bool, scale: float, workspace=None,
           stream=None) -> None:
    """Attention backward into preallocated CUDA tensors (C ABI ``fa_bwd_strided``).

    q, k, v, o, dout, dq, dk, dv: ``[B, H, N, d]`` CUDA tensors of one element
    type, ``torch.bfloat16`` or ``torch.float16``, on one device, any strides
    with the last dimension contiguous (strides multiples of 8 elements), d a
    multiple of 16 from 16 to 128; lse: contiguous ``torch.float32``
    ``[B, H, N]`` (o and lse from :func:`fa_fwd`).
    ``workspace``: a CUDA byte tensor of at least :func:`fa_bwd_workspace_bytes`;
    allocated here when None.
    """
    import torch

    B, H, N, d = _dims(q)
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q must be torch.bfloat16 or torch.float16")
    elem = q.dtype
    tensors = (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq), ("dk", dk),
               ("dv", dv))
    for name, t in tensors[1:]:
        if tuple(t.shape) != (B, H, N, d):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {(B, H, N, d)}")
    if tuple(lse.shape) != (B, H, N):
        raise ValueError(f"lse has shape {tuple(lse.shape)}, expected {(B, H, N)}")
    for name, t in tensors:
        if t.dtype != elem or not t.is_cuda or t.device != q.device:
            raise ValueError(f"{name} must be a {elem} CUDA tensor on q's device")
        if t.stride(3) != 1:
            raise ValueError(f"{name} must have a contiguous last dimension")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or \
            lse.device != q.device:
        raise ValueError("lse must be a contiguous torch.float32 CUDA tensor on q's device")

    def st(t):  # a dimension of extent 1 is never stepped: its stride is irrelevant
        return tuple(0 if t.shape[i] == 1 else t.stride(i) for i in range(3))

    with torch.cuda.device(q.device):
        if workspace is None:
            nbytes = fa_bwd_workspace_bytes(B, H, N, d)
            if nbytes == 0:
                raise FAError(3, "fa_bwd_workspace_bytes")
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        dtype = FA_DTYPE_FP16 if elem == torch.float16 else FA_DTYPE_BF16
        rc = fa_bwd_strided([t.data_ptr() for _, t in tensors], [st(t) for _, t in tensors],
                            lse.data_ptr(), dtype, B, H, N, d, causal, scale,
                            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                            handle)
        _check(rc, "fa_bwd_strided")


def attention_backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
                       stream=None):
    """Allocate dQ, dK, dV and run :func:`fa_bwd`; returns ``(dQ, dK, dV)``."""
    import torch

    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, causal, scale, None, stream)
    return dq, dk, dv


_autograd_fn = None


def _attention_function():
    """The torch.autograd.Function behind :func:`attention`, made on first use."""
    global _autograd_fn
    if _autograd_fn is None:
        import torch

        class AttentionFunction(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, causal, scale):
                o, lse = attention_forward(q, k, v, causal=causal, scale=scale)
                ctx.save_for_backward(q, k, v, o, lse)
                ctx.causal, ctx.scale = causal, scale
                return o

            @staticmethod
            def backward(ctx, grad_o):
                q, k, v, o, lse = ctx.saved_tensors
                # Autograd may hand over an expanded or otherwise strided
                # gradient; the backward wants unit column stride and strides
                # that are multiples of 8 elements.
                ok = grad_o.dtype == q.dtype and grad_o.stride(3) == 1 and all(
                    grad_o.shape[i] == 1 or grad_o.stride(i) % 8 == 0 for i in range(3))
                dout = grad_o if ok else grad_o.to(q.dtype).contiguous()
                dq, dk, dv = attention_backward(q, k, v, o, lse, dout, causal=ctx.causal,
                                                scale=ctx.scale)
                return dq, dk, dv, None, None

        _autograd_fn = AttentionFunction
    return _autograd_fn


def attention(q, k, v, causal: bool = False, scale: float | None = None):
    """Differentiable attention for PyTorch training code: the forward runs
    :func:`fa_fwd` and keeps O and LSE; ``.backward()`` runs :func:`fa_bwd`
    (head dimensions that are multiples of 16 up to 128 for the backward).
    q, k, v: ``[B, H, N, d]`` CUDA tensors, bf16 or fp16.  Returns O."""
    if scale is None:
        scale = 1.0 / math.sqrt(_dims(q)[3])
    return _attention_function().apply(q, k, v, bool(causal), float(scale))


def attention_forward_order_ablation(q, k, v, causal: bool, scale: float, order: int,
                                     workspace=None, out=None, stream=None):
    """The forward in loop order 1 (K/V outer, O/m/l through HBM) or 2 (Q
    outer, state on chip) via ``fa_fwd_order_ablation``; contiguous bf16
    ``[B, H, N, d]`` CUDA tensors, d 64 or 128.  Returns ``(O, LSE)``
    (``out`` = preallocated ``(O, LSE)`` to reuse)."""
    import torch

    B, H, N, d = _dims(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or \
                tuple(t.shape) != (B, H, N, d):
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor [B, H, N, d]")
    with torch.cuda.device(q.device):
        if out is None:
            out = (torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32,
                                                    device=q.device))
        o, lse = out
        if workspace is None:
            nbytes = load_library().fa_fwd_order_ablation_workspace_bytes(B, H, N, d, order)
            workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        rc = load_library().fa_fwd_order_ablation(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
            int(bool(causal)), float(scale), int(order), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), handle or None)
        _check(rc, "fa_fwd_order_ablation")
    return o, lse


def fa_get_device_status() -> int:
    """Sticky device status bits of the current device (synchronises it)."""
    st = ctypes.c_uint(0)
    _check(load_library().fa_get_device_status(ctypes.byref(st)), "fa_get_device_status")
    return int(st.value)


def fa_clear_device_status() -> None:
    _check(load_library().fa_clear_device_status(), "fa_clear_device_status")


def fa_set_wait_limit_ns(ns: int) -> None:
    _check(load_library().fa_set_wait_limit_ns(int(ns)), "fa_set_wait_limit_ns")


def fa_set_fault_injection(flags: int) -> None:
    _check(load_library().fa_set_fault_injection(int(flags)), "fa_set_fault_injection")


def nominal_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """4·B·H·N²·d, halved when causal (the metric's nominal count)."""
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f
