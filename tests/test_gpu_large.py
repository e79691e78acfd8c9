"""GPU parity at sizes past 32-bit offsets.

Every large tensor in these cases holds more than 2^31 elements (over 4 GiB),
so an element or byte offset formed in 32 bits would put a head's rows in the
wrong place.  The inputs are a few seeded heads repeated along the head axis
on the device (a copy, no arithmetic); the heads compared with the oracle are
the first, the ones on both sides of the 2^31-element boundary (which falls
inside a head: the row count is ragged) and the last.
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import compare

pytestmark = pytest.mark.gpu

SRC = 8  # distinct seeded heads, repeated along H


@pytest.fixture(scope="module")
def fa(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.load_library()
    return fa


@pytest.fixture(autouse=True)
def _release(cuda_device):
    yield
    import torch

    torch.cuda.synchronize(cuda_device)
    torch.cuda.empty_cache()


def _repeat(bits, B, H, dev, dtype="bf16"):
    """[1, SRC, N, d] seeded heads -> [B, H, N, d] on the device, head h of
    every batch being source head h % SRC."""
    t = workloads.as_torch(bits, dtype).to(dev)
    return t.repeat(B, H // SRC, 1, 1)


def _checked_heads(B, H, per_head):
    """Flat (b * H + h) indices: first, around element 2^31, last."""
    boundary = (1 << 31) // per_head
    assert B * H * per_head > (1 << 31) + per_head
    assert (1 << 31) % per_head != 0  # the boundary falls inside a head
    return sorted({0, boundary - 1, boundary, boundary + 1, B * H - 1})


def _head(a, flat, H):
    return a[flat // H, flat % H]


@pytest.mark.parametrize("d,B,H", [(128, 2, 20480), (256, 1, 16384)])
def test_forward_past_2_31_elements(fa, cuda_device, d, B, H):
    import torch

    N = 600
    scale = 1.0 / math.sqrt(d)
    q, k, v = workloads.generate_shape(1, SRC, N, d, seed=2200 + d, qk_std=1.5)
    qd, kd, vd = (_repeat(a, B, H, cuda_device) for a in (q, k, v))
    o, lse = fa.attention_forward(qd, kd, vd, causal=True, scale=scale)
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    refs = {}
    for flat in _checked_heads(B, H, N * d):
        s = (flat % H) % SRC
        if s not in refs:
            refs[s] = oracle.attention(q[:, s:s + 1], k[:, s:s + 1], v[:, s:s + 1], True, scale)
        o_ref, lse_ref = refs[s]
        compare(_head(o, flat, H).float().cpu().numpy()[None, None],
                _head(lse, flat, H).cpu().numpy()[None, None], o_ref, lse_ref,
                f"d{d} head {flat}")
    del qd, kd, vd, o, lse


def test_backward_past_2_31_elements(fa, cuda_device):
    import torch

    from test_gpu_bwd import check_grads

    B, H, N, d = 2, 20480, 600, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = workloads.generate_shape(1, SRC, N, d, seed=2300, qk_std=1.5)
    do = workloads.generate_shape(1, SRC, N, d, seed=2301)[0]
    qd, kd, vd, dod = (_repeat(a, B, H, cuda_device) for a in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=True, scale=scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=True, scale=scale)
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    refs = {}
    for flat in _checked_heads(B, H, N * d):
        s = (flat % H) % SRC
        if s not in refs:
            sl = slice(s, s + 1)
            refs[s] = oracle.attention_bwd(q[:, sl], k[:, sl], v[:, sl], do[:, sl], True, scale)
        got = [_head(t, flat, H).float().cpu().numpy().astype(np.float64)[None, None]
               for t in (dq, dk, dv)]
        check_grads(got, refs[s], f"head {flat}")
    del qd, kd, vd, dod, o, lse, dq, dk, dv


def test_splitkv_past_2_31_elements(fa, cuda_device):
    import torch

    B, H, Nq, Nk, d = 1, 1024, 16, 20000, 128
    scale = 1.0 / math.sqrt(d)
    q = workloads.generate_shape(1, SRC, Nq, d, seed=2400, qk_std=1.5)[0]
    _, k, v = workloads.generate_shape(1, SRC, Nk, d, seed=2401, qk_std=1.5)
    qd, kd, vd = (_repeat(a, B, H, cuda_device) for a in (q, k, v))
    o, lse = fa.attention_forward_splitkv(qd, kd, vd, causal=True, scale=scale)
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    refs = {}
    for flat in _checked_heads(B, H, Nk * d):
        s = (flat % H) % SRC
        if s not in refs:
            refs[s] = oracle.attention(q[:, s:s + 1], k[:, s:s + 1], v[:, s:s + 1], True, scale)
        o_ref, lse_ref = refs[s]
        compare(_head(o, flat, H).float().cpu().numpy()[None, None],
                _head(lse, flat, H).cpu().numpy()[None, None], o_ref, lse_ref,
                f"split-KV head {flat}")
    del qd, kd, vd, o, lse
