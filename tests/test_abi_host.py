"""Host-side checks of the C ABI (no GPU needed, no kernel launched):
the library builds and loads, exports every function include/fa.h declares,
and rejects bad arguments with the documented codes before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

# Codes from include/fa.h
FA_OK, FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_HEAD_DIM, FA_ERR_ALIGN = 0, 1, 2, 3, 4
FA_ERR_SCALE, FA_ERR_ALIAS, FA_ERR_DEVICE, FA_ERR_LAUNCH = 5, 6, 7, 8


@pytest.fixture(scope="module")
def lib():
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    return fa.load_library()


def _declared_functions():
    names = []
    for fname in sorted(os.listdir(HEADER_DIR)):
        if not fname.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fname)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("fa_fwd", "fa_strerror", "fa_get_device_status", "fa_clear_device_status",
                     "fa_set_wait_limit_ns", "fa_set_fault_injection", "fa_version"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared in include/*.h but not exported: {missing}"


def test_guarded_build_exports_every_declared_symbol(lib):
    """The bounds-checked twin (FA_GUARDED=1) is built beside the library and
    exports the same C ABI."""
    from tiled_attention_forward_attn_gb300 import _build

    glib = ctypes.CDLL(_build.GUARDED_LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(glib, n)]
    assert not missing, f"not exported by the guarded build: {missing}"


def test_strerror_and_version(lib):
    for code in range(0, 10):
        assert isinstance(lib.fa_strerror(code), bytes) and lib.fa_strerror(code)
    assert lib.fa_strerror(12345) == b"unknown error code"
    assert lib.fa_version() >= 100


A16 = 0x10000  # fake, 16-byte aligned addresses (never dereferenced)


def _call(lib, q=A16, k=2 * A16, v=3 * A16, o=4 * A16, lse=5 * A16, B=1, H=1, N=128, d=64,
          causal=0, scale=0.125):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, None)


@pytest.mark.parametrize("which", ["q", "k", "v", "o", "lse"])
def test_null_pointers_rejected(lib, which):
    assert _call(lib, **{which: 0}) == FA_ERR_NULL


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(N=0), dict(B=-1), dict(N=-5),
                                dict(causal=2), dict(B=65536, H=65536),
                                dict(B=2, N=2 ** 30)])
def test_bad_shapes_rejected(lib, kw):
    assert _call(lib, **kw) == FA_ERR_SHAPE


@pytest.mark.parametrize("d", [0, 8, 24, 127, 144, 192, 240, 272])
def test_unsupported_head_dim_rejected(lib, d):
    assert _call(lib, d=d) == FA_ERR_HEAD_DIM


@pytest.mark.parametrize("d", [16, 32, 48, 80, 96, 112, 256])
def test_multiple_of_16_head_dims_accepted(lib, d):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a device is present; covered by the GPU tests")
    # Validation passes; only the missing device stops the call.
    assert _call(lib, d=d) in (FA_ERR_LAUNCH, FA_ERR_DEVICE)


FA_ERR_DTYPE, FA_ERR_STRIDE = 12, 13


def _strided(lib, qs=None, ks=None, vs=None, os_=None, dtype=0, B=2, H=3, N=100, d=64, o=None,
             lse=None):
    def arr(st):
        return None if st is None else (ctypes.c_int64 * 3)(*st)

    big = 1 << 24  # buffers far apart: no aliasing unless intended
    o = 4 * big if o is None else o
    lse = 5 * big if lse is None else lse
    return lib.fa_fwd_strided(big, arr(qs), 2 * big, arr(ks), 3 * big, arr(vs), o, arr(os_), lse,
                              dtype, B, H, N, d, 0, 0.1, None)


def test_strided_validation(lib):
    import torch

    no_dev = not torch.cuda.is_available()
    assert _strided(lib, dtype=2) == FA_ERR_DTYPE
    assert _strided(lib, qs=(-64, 64, 64)) == FA_ERR_STRIDE  # negative
    assert _strided(lib, ks=(19200, 6400, 68)) == FA_ERR_STRIDE  # not a multiple of 8
    assert _strided(lib, vs=(1 << 38, 64, 64)) == FA_ERR_STRIDE  # too large
    # o rows overlapping (row stride below d), o heads overlapping
    assert _strided(lib, os_=(19200, 6400, 32)) == FA_ERR_STRIDE
    assert _strided(lib, os_=(19200, 64, 64)) == FA_ERR_STRIDE
    # [B, N, H, d] memory viewed as [B, H, N, d] is disjoint; so are padded rows
    # and inputs shared across heads (stride 0).
    if no_dev:
        for kw in (dict(os_=(19200, 64, 192)), dict(os_=(20000, 6400, 64)),
                   dict(ks=(6400, 0, 64), vs=(6400, 0, 64)), dict(dtype=1)):
            assert _strided(lib, **kw) in (FA_ERR_LAUNCH, FA_ERR_DEVICE), kw
    # the output's strided span overlapping an input is aliasing
    assert _strided(lib, o=3 * (1 << 24) + 4096, os_=(19200, 64, 192)) == FA_ERR_ALIAS


@pytest.mark.parametrize("kw", [dict(q=A16 + 2), dict(k=2 * A16 + 8), dict(v=3 * A16 + 1),
                                dict(o=4 * A16 + 4), dict(lse=5 * A16 + 2)])
def test_misaligned_pointers_rejected(lib, kw):
    assert _call(lib, **kw) == FA_ERR_ALIGN


@pytest.mark.parametrize("scale", [float("nan"), float("inf"), float("-inf")])
def test_non_finite_scale_rejected(lib, scale):
    assert _call(lib, scale=scale) == FA_ERR_SCALE


def test_aliasing_outputs_rejected(lib):
    # o == q
    assert _call(lib, o=A16) == FA_ERR_ALIAS
    # lse inside v (v spans 128*64*2 bytes)
    assert _call(lib, lse=3 * A16 + 1024) == FA_ERR_ALIAS
    # lse inside o
    assert _call(lib, lse=4 * A16 + 64) == FA_ERR_ALIAS


def test_valid_arguments_without_a_device_report_an_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a device is present; covered by the GPU tests")
    assert _call(lib) in (FA_ERR_LAUNCH, FA_ERR_DEVICE)


def test_python_binding_validates_before_calling(lib):
    torch = pytest.importorskip("torch")
    import tiled_attention_forward_attn_gb300 as fa

    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises((ValueError, TypeError)):
        fa.fa_fwd(q, q, q, q.clone(), torch.zeros(1, 1, 8), False, 0.1)  # CPU tensors
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q[:, :, :4], q, q.clone(), torch.zeros(1, 1, 8), False, 0.1)


def test_status_hooks_accept_arguments(lib):
    assert lib.fa_set_wait_limit_ns(ctypes.c_ulonglong(0)) == FA_OK
    assert lib.fa_set_fault_injection(0) == FA_OK
    assert lib.fa_get_device_status(None) == FA_ERR_NULL


# ---------------------------------------------------------------- split-KV

FA_ERR_WORKSPACE = 10


def _split(lib, q=A16, k=2 * A16, v=3 * A16, o=4 * A16, lse=5 * A16, B=1, H=1, Nq=1, Nk=128,
           d=64, causal=0, scale=0.125, splits=0, ws=6 * A16, ws_bytes=1 << 20):
    return lib.fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, splits, ws,
                              ws_bytes, None)


@pytest.mark.parametrize("which", ["q", "k", "v", "o", "lse"])
def test_splitkv_null_pointers_rejected(lib, which):
    assert _split(lib, **{which: 0}) == FA_ERR_NULL


@pytest.mark.parametrize("kw", [dict(Nq=0), dict(Nq=17), dict(Nk=0), dict(B=0),
                                dict(causal=1, Nq=5, Nk=4), dict(splits=-1), dict(splits=257),
                                dict(B=256, H=256)])
def test_splitkv_bad_shapes_rejected(lib, kw):
    assert _split(lib, **kw) == FA_ERR_SHAPE


def test_splitkv_head_dim_alignment_scale(lib):
    assert _split(lib, d=96) == FA_ERR_HEAD_DIM
    assert _split(lib, ws=6 * A16 + 8) == FA_ERR_ALIGN
    assert _split(lib, scale=float("nan")) == FA_ERR_SCALE
    assert _split(lib, o=A16) == FA_ERR_ALIAS


def test_splitkv_workspace_size_formula(lib):
    # Nk=1000 -> 16 tiles of 64 keys; 4 requested splits -> 4 tiles each.
    assert lib.fa_fwd_splitkv_num_splits(1, 2, 3, 1000, 64, 4) == 4
    # 7 requested -> 3 tiles per split -> 6 ranges cover the 16 tiles
    assert lib.fa_fwd_splitkv_num_splits(1, 2, 3, 1000, 64, 7) == 6
    # partial outputs 4*2*3*64 fp32 = 6144 B, log-sum-exps 24 fp32 -> 256 B (256-byte rounding)
    assert lib.fa_fwd_splitkv_workspace_bytes(1, 2, 3, 1000, 64, 4) == 6144 + 256
    # more splits than tiles: capped at one tile per split
    assert lib.fa_fwd_splitkv_num_splits(1, 1, 1, 300, 128, 50) == 5
    assert lib.fa_fwd_splitkv_workspace_bytes(1, 1, 17, 300, 128, 2) == 0  # Nq > 16


def test_splitkv_without_device_reports_an_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a device is present; covered by the GPU tests")
    assert _split(lib) in (FA_ERR_LAUNCH, FA_ERR_DEVICE)
    assert lib.fa_fwd_splitkv_num_splits(1, 1, 1, 1000, 64, 0) == 0  # needs the device


def test_bwd_validation(lib):
    import torch

    big = 1 << 24
    args = dict(q=big, k=2 * big, v=3 * big, o=4 * big, lse=5 * big, do=6 * big, dq=7 * big,
                dk=8 * big, dv=9 * big, B=1, H=2, N=300, d=64, causal=1, scale=0.1,
                ws=10 * big, ws_bytes=1 << 20)

    def call(**kw):
        a = dict(args, **kw)
        return lib.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"],
                          a["dv"], a["B"], a["H"], a["N"], a["d"], a["causal"], a["scale"],
                          a["ws"], a["ws_bytes"], None)

    # 2 rows of D and LSE*log2(e) per head, padded to 384 rows: 2 * 2 * 384 * 4 bytes
    assert lib.fa_bwd_workspace_bytes(1, 2, 300, 64) == 6144
    # head dimensions: multiples of 16 from 16 to 128
    assert lib.fa_bwd_workspace_bytes(1, 2, 300, 96) == 6144
    assert lib.fa_bwd_workspace_bytes(1, 2, 300, 16) == 6144
    for bad in (0, 8, 72, 144, 256):
        assert lib.fa_bwd_workspace_bytes(1, 2, 300, bad) == 0
        assert call(d=bad) == FA_ERR_HEAD_DIM
    assert call(q=0) == FA_ERR_NULL
    assert call(N=0) == FA_ERR_SHAPE
    assert call(dk=8 * big + 8) == FA_ERR_ALIGN
    assert call(scale=float("nan")) == FA_ERR_SCALE
    assert call(ws_bytes=6000) == FA_ERR_WORKSPACE
    assert call(dq=big) == FA_ERR_ALIAS            # dq over q
    assert call(dv=8 * big + 64) == FA_ERR_ALIAS   # dv inside dk
    assert call(ws=9 * big) == FA_ERR_ALIAS        # workspace over dv
    if not torch.cuda.is_available():
        assert call() in (FA_ERR_LAUNCH, FA_ERR_DEVICE)


def test_bwd_ex_validation(lib):
    """fa_bwd_ex: the element type is checked first; an fp16 call is
    validated like a bf16 one."""
    import torch

    big = 1 << 24
    base = [big, 2 * big, 3 * big, 4 * big, 5 * big, 6 * big, 7 * big, 8 * big, 9 * big]

    def call(dtype, d=64, ws_bytes=1 << 20, q=big):
        ptrs = [q] + base[1:]
        return lib.fa_bwd_ex(*ptrs, dtype, 1, 2, 300, d, 1, 0.1, 10 * big, ws_bytes, None)

    assert call(7) == FA_ERR_DTYPE
    assert call(-1) == FA_ERR_DTYPE
    assert call(1, q=0) == FA_ERR_NULL
    assert call(1, d=72) == FA_ERR_HEAD_DIM
    assert call(1, d=256) == FA_ERR_HEAD_DIM
    assert call(1, ws_bytes=6000) == FA_ERR_WORKSPACE
    if not torch.cuda.is_available():
        assert call(1) in (FA_ERR_LAUNCH, FA_ERR_DEVICE)
        assert call(0) in (FA_ERR_LAUNCH, FA_ERR_DEVICE)


def test_bwd_strided_validation(lib):
    """fa_bwd_strided: strides are checked like fa_fwd_strided's (non-negative
    multiples of 8 below 2^38), the gradients' elements must not overlap, and
    the aliasing check uses each tensor's strided span."""
    import torch

    big = 1 << 24
    B, H, N, d = 2, 3, 100, 64

    def call(strides=None, ptrs=None, dtype=0):
        st = list(strides or [None] * 8)
        arr = [None if x is None else (ctypes.c_int64 * 3)(*x) for x in st]
        p = list(ptrs or [big * (i + 1) for i in range(8)])
        return lib.fa_bwd_strided(p[0], arr[0], p[1], arr[1], p[2], arr[2], p[3], arr[3],
                                  9 * big, p[4], arr[4], p[5], arr[5], p[6], arr[6], p[7], arr[7],
                                  dtype, B, H, N, d, 1, 0.1, 10 * big, 1 << 20, None)

    def one(i, st):
        s = [None] * 8
        s[i] = st
        return s

    bnhd = (N * H * d, d, H * d)  # [B, N, H, d] memory viewed as [B, H, N, d]
    assert call(dtype=2) == FA_ERR_DTYPE
    for i in range(8):
        assert call(one(i, (-64, 64, 64))) == FA_ERR_STRIDE, i
        assert call(one(i, (19200, 6400, 68))) == FA_ERR_STRIDE, i
        assert call(one(i, (1 << 38, 64, 64))) == FA_ERR_STRIDE, i
    # overlapping gradient rows or heads; the same strides on an input are allowed
    for i in (5, 6, 7):
        assert call(one(i, (19200, 6400, 32))) == FA_ERR_STRIDE, i
        assert call(one(i, (19200, 64, 64))) == FA_ERR_STRIDE, i
    # dq starting 4 KiB below k: its strided span reaches into k
    ptrs = [big * (i + 1) for i in range(8)]
    ptrs[5] = 2 * big - 4096
    assert call(one(5, bnhd), ptrs) == FA_ERR_ALIAS
    # dk, dv interleaved within one [B, N, 2, H, d] buffer: distinct
    # elements but overlapping spans, rejected as aliasing
    ptrs = [big * (i + 1) for i in range(8)]
    ptrs[7] = ptrs[6] + H * d * 2
    s = [None] * 8
    s[6] = s[7] = (N * 2 * H * d, d, 2 * H * d)
    assert call(s, ptrs) == FA_ERR_ALIAS
    if not torch.cuda.is_available():
        for st in ([bnhd] * 8, one(1, (6400, 0, 64)), [None] * 8):
            assert call(st) in (FA_ERR_LAUNCH, FA_ERR_DEVICE)


def test_strides_whose_span_overflows_are_rejected(lib):
    """A stride times its extent is checked before it is formed: a batch
    stride of 2^37 elements over 2^20 batches (a 2^57-element span) is
    rejected with FA_ERR_STRIDE by the forward and the backward, instead of
    wrapping around in 64-bit arithmetic; the same stride over 2 batches is
    valid."""
    import torch

    big = 1 << 40
    huge = (1 << 37, 64, 64)

    def fwd(B, qs):
        st = (ctypes.c_int64 * 3)(*qs)
        return lib.fa_fwd_strided(big, st, 2 * big, None, 3 * big, None, 4 * big, None,
                                  5 * big, 0, B, 1, 8, 64, 0, 0.1, None)

    def bwd(B, qs):
        st = (ctypes.c_int64 * 3)(*qs)
        ptrs = [big * (i + 1) for i in range(8)]
        return lib.fa_bwd_strided(ptrs[0], st, ptrs[1], None, ptrs[2], None, ptrs[3], None,
                                  9 * big, ptrs[4], None, ptrs[5], None, ptrs[6], None,
                                  ptrs[7], None, 0, B, 1, 8, 64, 0, 0.1, 10 * big, 1 << 30, None)

    assert fwd(1 << 20, huge) == FA_ERR_STRIDE
    assert bwd(1 << 20, huge) == FA_ERR_STRIDE
    if not torch.cuda.is_available():
        assert fwd(2, huge) in (FA_ERR_LAUNCH, FA_ERR_DEVICE)
        assert bwd(2, huge) in (FA_ERR_LAUNCH, FA_ERR_DEVICE)


def test_workspace_queries_return_zero_for_rejected_shapes(lib):
    """Every size query answers 0, without overflowing, for a shape its entry
    point rejects as too large."""
    n = 1 << 30
    assert lib.fa_bwd_workspace_bytes(n, n, n, 64) == 0
    assert lib.fa_bwd_host_workspace_bytes(n, n, n, 64) == 0
    assert lib.fa_fwd_host_workspace_bytes(n, n, n, 64) == 0
    assert lib.fa_fwd_order_ablation_workspace_bytes(n, n, n, 64, 1) == 0
    assert lib.fa_fwd_splitkv_workspace_bytes(n, n, 16, n, 64, 0) == 0
    # and a shape just inside the limits still has a size
    assert lib.fa_bwd_workspace_bytes(1, 1, 1 << 20, 64) == 2 * (1 << 20) * 4
    assert lib.fa_fwd_order_ablation_workspace_bytes(1, 1, 1000, 64, 1) > 0


def test_fwd_host_validation(lib):
    """fa_fwd_host rejects bad arguments before queueing any copy (no GPU
    needed for these checks)."""
    import torch

    big = 1 << 24
    need = lib.fa_fwd_host_workspace_bytes(1, 2, 300, 64)
    # Q, K, V, O: 2 heads x 300 rows x 64 x 2 bytes, rounded to 256; LSE 2400 -> 2560
    assert need == 4 * 76800 + 2560
    assert lib.fa_fwd_host_workspace_bytes(1, 2, 300, 72) == 0

    def call(q=big, o=4 * big, lse=5 * big, dtype=0, d=64, causal=1, ws=1 << 30,
             ws_bytes=1 << 22):
        return lib.fa_fwd_host(q, 2 * big, 3 * big, o, lse, dtype, 1, 2, 300, d, causal, 0.1, ws,
                               ws_bytes, None)

    assert call(q=0) == FA_ERR_NULL
    assert call(dtype=5) == FA_ERR_DTYPE
    assert call(d=72) == FA_ERR_HEAD_DIM
    assert call(causal=2) == FA_ERR_SHAPE
    assert call(ws_bytes=need - 1) == FA_ERR_WORKSPACE
    assert call(ws=(1 << 30) + 16) == FA_ERR_ALIGN
    assert call(o=big + 64) == FA_ERR_ALIAS          # O over Q
    assert call(lse=4 * big + 256) == FA_ERR_ALIAS   # LSE inside O
    if not torch.cuda.is_available():
        assert call() in (FA_ERR_LAUNCH, FA_ERR_DEVICE)


def _r256(x):
    return (x + 255) // 256 * 256


def test_splitkv_host_validation(lib):
    """fa_fwd_splitkv_host rejects bad arguments before queueing any copy."""
    import torch

    big = 1 << 24
    # With num_splits > 0 the sizes need no device.
    part = lib.fa_fwd_splitkv_workspace_bytes(1, 2, 5, 1000, 64, 4)
    need = lib.fa_fwd_splitkv_host_workspace_bytes(1, 2, 5, 1000, 64, 4)
    assert part > 0
    assert need == (2 * _r256(2 * 5 * 64 * 2) + 2 * _r256(2 * 1000 * 64 * 2) + _r256(2 * 5 * 4)
                    + _r256(part))
    assert lib.fa_fwd_splitkv_host_workspace_bytes(1, 2, 5, 1000, 96, 4) == 0

    def call(q=big, Nq=5, d=64, causal=1, scale=0.1):
        return lib.fa_fwd_splitkv_host(q, 2 * big, 3 * big, 4 * big, 5 * big, 1, 2, Nq, 1000, d,
                                       causal, scale, 4, 1 << 30, 1 << 26, None)

    assert call(q=0) == FA_ERR_NULL
    assert call(Nq=17) == FA_ERR_SHAPE
    assert call(d=96) == FA_ERR_HEAD_DIM
    assert call(causal=2) == FA_ERR_SHAPE
    assert call(scale=float("inf")) == FA_ERR_SCALE
    if not torch.cuda.is_available():
        assert call() in (FA_ERR_LAUNCH, FA_ERR_DEVICE)


def test_bwd_host_validation(lib):
    """fa_bwd_host rejects bad arguments before queueing any copy."""
    import torch

    big = 1 << 24
    need = lib.fa_bwd_host_workspace_bytes(1, 2, 300, 64)
    ws_bwd = lib.fa_bwd_workspace_bytes(1, 2, 300, 64)
    assert ws_bwd == 2 * 2 * 384 * 4
    assert need == 8 * _r256(2 * 300 * 64 * 2) + _r256(2 * 300 * 4) + _r256(ws_bwd)
    assert lib.fa_bwd_host_workspace_bytes(1, 2, 300, 72) == 0

    def call(q=big, dq=7 * big, dtype=0, d=64, causal=1, ws=1 << 30, ws_bytes=1 << 24):
        return lib.fa_bwd_host(q, 2 * big, 3 * big, 4 * big, 5 * big, 6 * big, dq, 8 * big,
                               9 * big, dtype, 1, 2, 300, d, causal, 0.1, ws, ws_bytes, None)

    assert call(q=0) == FA_ERR_NULL
    assert call(dtype=4) == 12  # FA_ERR_DTYPE
    assert call(d=72) == FA_ERR_HEAD_DIM
    assert call(causal=2) == FA_ERR_SHAPE
    assert call(ws_bytes=need - 1) == 10  # FA_ERR_WORKSPACE
    assert call(ws=(1 << 30) + 16) == FA_ERR_ALIGN
    assert call(dq=big + 128) == FA_ERR_ALIAS  # dQ over Q
    if not torch.cuda.is_available():
        assert call() in (FA_ERR_LAUNCH, FA_ERR_DEVICE)

