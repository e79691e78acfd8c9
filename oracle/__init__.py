"""Oracle for exact attention — TEST INFRASTRUCTURE, not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA path never calls it, and it
imports nothing from the CUDA path.

Two independent fp64 restatements live here:

* ``attention`` / ``scores`` / ``safe_softmax`` — the plain definition (C,
  fp64, OpenMP over rows) from "Parsing FlashAttention (2): FlashAttention-v1
  forward pass" §1.1 and §2.1 eqs (1)-(5): materialise a score row, mask,
  take the max, exponentiate, sum, normalise, multiply by V.
* ``oracle.online`` — the tiled online-softmax algorithm in the pages' own
  step order (numpy, fp64), used to show the method reaches the definition.

The C source is compiled with the host gcc by :func:`build`; nothing here
links CUDA.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile ``attention_oracle.c`` into ``oracle/_build/liboracle.so``."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_safe_softmax.restype = None
            lib.oracle_safe_softmax.argtypes = [_f64p, ctypes.c_int64, _f64p, _f64p, _f64p, _f64p]
            lib.oracle_scores.restype = None
            lib.oracle_scores.argtypes = [_u16p, _u16p, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                          ctypes.c_int64, _f64p]
            lib.oracle_attention_rect.restype = ctypes.c_int
            lib.oracle_attention_rect.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64,
                                                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.c_int, ctypes.c_double, _i64p,
                                                  ctypes.c_int64, _f64p, _f64p, _f64p,
                                                  ctypes.c_int]
            lib.oracle_attention_rect_fmt.restype = ctypes.c_int
            lib.oracle_attention_rect_fmt.argtypes = lib.oracle_attention_rect.argtypes + [
                ctypes.c_int]
            lib.oracle_attention_bwd.restype = ctypes.c_int
            lib.oracle_attention_bwd.argtypes = [_u16p, _u16p, _u16p, _u16p, ctypes.c_int64,
                                                 ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                                 ctypes.c_double, _f64p, _f64p, _f64p,
                                                 ctypes.c_int, ctypes.c_int]
            lib.oracle_f16_to_double.restype = ctypes.c_double
            lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                             _i64p, ctypes.c_int64, _f64p, _f64p, _f64p,
                                             ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _ptr(a, t):
    return a.ctypes.data_as(t)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return np.ascontiguousarray(a)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64 (elementwise)."""
    lib = _load()
    flat = _u16(bits).ravel()
    return np.array([lib.oracle_bf16_to_double(int(b)) for b in flat],
                    dtype=np.float64).reshape(np.shape(bits))


def f16_to_f64(bits) -> np.ndarray:
    """Exact widening of IEEE binary16 bit patterns to fp64 (elementwise)."""
    lib = _load()
    flat = _u16(bits).ravel()
    return np.array([lib.oracle_f16_to_double(int(b)) for b in flat],
                    dtype=np.float64).reshape(np.shape(bits))


_FORMATS = {"bf16": 0, "f16": 1}


def safe_softmax(x):
    """Safe softmax of one fp64 vector (page 1 §2.1 eqs (1)-(5)).

    Returns ``(m, shifted, l, p)``: the max, ``x - m``, ``sum exp(x - m)``
    and the probabilities.
    """
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    n = x.size
    shifted = np.empty(n)
    p = np.empty(n)
    m = ctypes.c_double()
    l = ctypes.c_double()
    lib.oracle_safe_softmax(_ptr(x, _f64p), n, _ptr(shifted, _f64p), _ptr(p, _f64p),
                            ctypes.byref(m), ctypes.byref(l))
    return m.value, shifted, l.value, p


def scores(q, k, scale: float = 1.0, causal: bool = False, row_offset: int = 0):
    """Score block ``scale * q @ k.T`` in fp64 (rows of q are queries
    ``row_offset ..``; causal masks ``j > i`` with -inf)."""
    lib = _load()
    q = _u16(q)
    k = _u16(k)
    nq, d = q.shape
    nk, d2 = k.shape
    if d != d2:
        raise ValueError("q and k disagree on d")
    out = np.empty((nq, nk))
    lib.oracle_scores(_ptr(q, _u16p), _ptr(k, _u16p), nq, nk, d, float(scale),
                      int(bool(causal)), int(row_offset), _ptr(out, _f64p))
    return out


def attention(q, k, v, causal: bool, scale: float, rows=None,
              return_probs: bool = False, threads: int = 0, dtype: str = "bf16"):
    """Exact attention forward on bf16 (or fp16) inputs, in fp64.

    q: uint16 bit patterns (``dtype`` "bf16" or "f16") shaped ``[..., Nq, d]``;
    k, v: ``[..., Nk, d]``
    (leading dims equal and flattened into independent slices).  Causal
    masking is aligned to the end of the keys: query i sees keys
    ``0 .. Nk - Nq + i`` (``0 .. i`` when Nq == Nk).  ``rows``: optional 1-D
    array of query indices evaluated in every slice (default: all).  Returns
    ``(O, LSE)`` (and ``P`` if ``return_probs``) as fp64 arrays shaped
    ``[..., n_rows, d]`` / ``[..., n_rows]`` / ``[..., n_rows, Nk]``.
    """
    lib = _load()
    q, k, v = _u16(q), _u16(k), _u16(v)
    if k.shape != v.shape or q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1]:
        raise ValueError("q [..., Nq, d] and k, v [..., Nk, d] disagree")
    lead = q.shape[:-2]
    Nq, d = q.shape[-2:]
    Nk = k.shape[-2]
    BH = int(np.prod(lead)) if lead else 1
    if rows is None:
        rows_arr = None
        n_rows = Nq
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = rows_arr.size
    o = np.empty((BH, n_rows, d))
    lse = np.empty((BH, n_rows))
    p = np.empty((BH, n_rows, Nk)) if return_probs else None
    if dtype not in _FORMATS:
        raise ValueError(f"dtype must be one of {sorted(_FORMATS)}")
    rc = lib.oracle_attention_rect_fmt(
        _ptr(q, _u16p), _ptr(k, _u16p), _ptr(v, _u16p), BH, Nq, Nk, d, int(bool(causal)),
        float(scale), None if rows_arr is None else _ptr(rows_arr, _i64p), n_rows,
        _ptr(o, _f64p), _ptr(lse, _f64p), None if p is None else _ptr(p, _f64p), int(threads),
        _FORMATS[dtype])
    if rc != 0:
        raise ValueError(f"oracle_attention_rect failed with code {rc}")
    o = o.reshape(lead + (n_rows, d))
    lse = lse.reshape(lead + (n_rows,))
    if return_probs:
        return o, lse, p.reshape(lead + (n_rows, Nk))
    return o, lse


def attention_bwd(q, k, v, dout, causal: bool, scale: float, threads: int = 0,
                  dtype: str = "bf16"):
    """Exact gradients of the attention forward, in fp64.

    q, k, v, dout: uint16 bit patterns (``dtype`` "bf16" or "f16") shaped
    ``[..., N, d]`` (square attention; causal: query i sees keys 0..i).
    Returns ``(dQ, dK, dV)`` as fp64 arrays of the same shape: the gradients
    of ``sum(dout * O)`` with respect to Q, K and V, from the softmax
    Jacobian written out (no tiling).
    """
    lib = _load()
    q, k, v, dout = _u16(q), _u16(k), _u16(v), _u16(dout)
    if not (q.shape == k.shape == v.shape == dout.shape):
        raise ValueError("q, k, v and dout must share the shape [..., N, d]")
    if dtype not in _FORMATS:
        raise ValueError(f"dtype must be one of {sorted(_FORMATS)}")
    N, d = q.shape[-2:]
    BH = int(np.prod(q.shape[:-2])) if q.ndim > 2 else 1
    dq, dk, dv = (np.empty(q.shape, dtype=np.float64) for _ in range(3))
    rc = lib.oracle_attention_bwd(_ptr(q, _u16p), _ptr(k, _u16p), _ptr(v, _u16p),
                                  _ptr(dout, _u16p), BH, N, d, int(bool(causal)), float(scale),
                                  _ptr(dq, _f64p), _ptr(dk, _f64p), _ptr(dv, _f64p),
                                  int(threads), _FORMATS[dtype])
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd failed with code {rc}")
    return dq, dk, dv
