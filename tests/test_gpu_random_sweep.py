"""Seeded random sweep over the argument space of the forward, the split-KV
path and the backward (through the C ABI), every case checked against the
fp64 oracle with the tolerances the other parity tests use.

Drawn from a fixed seed, so every run checks the same cases: batch and head
counts, ragged sequence lengths (a third of them within one row of a tile
boundary), every head dimension the entry point takes, causal or not, bf16 or
fp16, the scale's sign and size (zero included), Q, K ~ N(0, s^2) with s up
to 3, and the memory layout: contiguous, [B, N, H, d] memory viewed as
[B, H, N, d], rows padded past d, and K, V shared by every head (head stride
0).  Each case is small enough for the oracle to finish in about a second."""
import math

import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import compare

pytestmark = pytest.mark.gpu

SEED = 20261202
LAYOUTS = ("contiguous", "bnhd", "padded", "shared_kv", "bnhd_out")


@pytest.fixture(scope="module")
def fa(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.load_library()
    return fa


def _near_boundary_n(rng, hi):
    """A sequence length, one time in three within one row of a multiple of 128."""
    if rng.random() < 1 / 3:
        base = 128 * int(rng.integers(1, max(2, hi // 128)))
        return max(1, base + int(rng.integers(-1, 2)))
    return int(rng.integers(1, hi))


def _fwd_cases(n=120):
    rng = np.random.Generator(np.random.PCG64(SEED))
    cases = []
    for i in range(n):
        d = int(rng.choice([16, 32, 48, 64, 80, 96, 112, 128, 256]))
        hi = 400 if d == 256 else 700
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        N = _near_boundary_n(rng, hi)
        causal = bool(rng.integers(0, 2))
        dtype = "f16" if rng.random() < 0.3 else "bf16"
        r = rng.random()
        scale = 0.0 if r < 0.05 else float((1 if r < 0.85 else -1) * rng.uniform(0.3, 1.5) / math.sqrt(d))
        qk_std = float(rng.choice([1.0, 1.5, 3.0]))
        layout = str(rng.choice(LAYOUTS))
        cases.append((i, B, H, N, d, causal, dtype, round(scale, 6), qk_std, layout))
    return cases


def _bwd_cases(n=40):
    rng = np.random.Generator(np.random.PCG64(SEED + 1))
    cases = []
    for i in range(n):
        d = int(rng.choice([16, 32, 64, 96, 128]))
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        N = _near_boundary_n(rng, 400)
        causal = bool(rng.integers(0, 2))
        dtype = "f16" if rng.random() < 0.3 else "bf16"
        scale = float(rng.uniform(0.5, 1.0) / math.sqrt(d))
        layout = str(rng.choice(("contiguous", "bnhd", "padded", "shared_kv")))
        cases.append((i, B, H, N, d, causal, dtype, round(scale, 6), layout))
    return cases


def _splitkv_cases(n=40):
    rng = np.random.Generator(np.random.PCG64(SEED + 2))
    cases = []
    for i in range(n):
        d = int(rng.choice([64, 128]))
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        Nq = int(rng.integers(1, 17))
        Nk = int(rng.integers(Nq, 5000))
        causal = bool(rng.integers(0, 2))
        splits = 0 if rng.random() < 0.5 else int(rng.integers(1, 25))
        scale = float(rng.uniform(0.5, 1.5) / math.sqrt(d))
        cases.append((i, B, H, Nq, Nk, d, causal, splits, round(scale, 6)))
    return cases


def _place(t, layout, d):
    """t (a contiguous [B, H, N, d] device tensor) in the given memory layout."""
    import torch

    if layout in ("bnhd", "bnhd_out"):
        return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    if layout == "padded":
        buf = torch.zeros(t.shape[:-1] + (d + 16,), dtype=t.dtype, device=t.device)
        buf[..., :d] = t
        return buf[..., :d]
    return t


def _inputs(B, H, N, d, seed, qk_std, dtype, shared_kv):
    q = workloads.generate_shape(B, H, N, d, seed=seed, qk_std=qk_std, dtype=dtype)[0]
    if shared_kv:
        _, k1, v1 = workloads.generate_shape(B, 1, N, d, seed=seed + 1, qk_std=qk_std, dtype=dtype)
        k, v = np.repeat(k1, H, axis=1), np.repeat(v1, H, axis=1)
        return q, k, v, (k1, v1)
    _, k, v = workloads.generate_shape(B, H, N, d, seed=seed + 1, qk_std=qk_std, dtype=dtype)
    return q, k, v, None


@pytest.mark.parametrize("case", _fwd_cases(), ids=lambda c: "f{0}_b{1}h{2}n{3}d{4}_c{5}_{6}_{9}".format(*c))
def test_forward_random_case(fa, cuda_device, case):
    import torch

    i, B, H, N, d, causal, dtype, scale, qk_std, layout = case
    q, k, v, kv1 = _inputs(B, H, N, d, 9000 + 7 * i, qk_std, dtype, layout == "shared_kv")
    dev = lambda a: workloads.as_torch(a, dtype).to(cuda_device)
    qd = _place(dev(q), layout, d)
    if kv1 is not None:
        kd, vd = (dev(a).expand(B, H, N, d) for a in kv1)
    else:
        kd, vd = (_place(dev(a), layout, d) for a in (k, v))
    elem = torch.float16 if dtype == "f16" else torch.bfloat16
    if layout == "bnhd_out":
        o = torch.empty((B, N, H, d), dtype=elem, device=cuda_device).permute(0, 2, 1, 3)
    else:
        o = torch.empty((B, H, N, d), dtype=elem, device=cuda_device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
    fa.fa_fwd(qd, kd, vd, o, lse, causal, scale)
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale, dtype=dtype)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"sweep case {case}")


@pytest.mark.parametrize("case", _splitkv_cases(), ids=lambda c: "s{0}_b{1}h{2}q{3}k{4}d{5}_c{6}_p{7}".format(*c))
def test_splitkv_random_case(fa, cuda_device, case):
    import torch

    i, B, H, Nq, Nk, d, causal, splits, scale = case
    q = workloads.generate_shape(B, H, Nq, d, seed=9500 + 7 * i, qk_std=1.5)[0]
    _, k, v = workloads.generate_shape(B, H, Nk, d, seed=9600 + 7 * i, qk_std=1.5)
    qd, kd, vd = (workloads.as_torch(a).to(cuda_device) for a in (q, k, v))
    o, lse = fa.attention_forward_splitkv(qd, kd, vd, causal=causal, scale=scale, num_splits=splits)
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"sweep case {case}")


@pytest.mark.parametrize("case", _bwd_cases(), ids=lambda c: "g{0}_b{1}h{2}n{3}d{4}_c{5}_{6}_{8}".format(*c))
def test_backward_random_case(fa, cuda_device, case):
    """Tolerance as the backward's own tests: |dX - ref| <= 3e-2 (1 + |ref|)
    elementwise and a relative Frobenius error <= 1e-2 (Q, K ~ N(0, 1.5^2)
    and a scale of at most 1/sqrt(d) here, where that bound is at least five
    standard deviations of the rounding model)."""
    import torch

    i, B, H, N, d, causal, dtype, scale, layout = case
    q, k, v, kv1 = _inputs(B, H, N, d, 9800 + 7 * i, 1.5, dtype, layout == "shared_kv")
    do = workloads.generate_shape(B, H, N, d, seed=9900 + 7 * i, dtype=dtype)[0]
    dev = lambda a: workloads.as_torch(a, dtype).to(cuda_device)
    qd, dod = _place(dev(q), layout, d), _place(dev(do), layout, d)
    if kv1 is not None:
        kd, vd = (dev(a).expand(B, H, N, d) for a in kv1)
    else:
        kd, vd = (_place(dev(a), layout, d) for a in (k, v))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    o = _place(o, layout, d)
    grads = [_place(torch.zeros_like(dev(q)), layout, d) for _ in range(3)]
    fa.fa_bwd(qd, kd, vd, o, lse, dod, *grads, causal, scale)
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    ref = oracle.attention_bwd(q, k, v, do, causal, scale, dtype=dtype)
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        got = g.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), f"{case} {name}: non-finite"
        err = np.abs(got - r)
        worst = float((err / (1.0 + np.abs(r))).max())
        fro = float(np.linalg.norm(err) / max(np.linalg.norm(r), math.sqrt(r.size)))
        assert worst <= 3e-2, f"{case} {name}: max |d|/(1+|ref|) = {worst:.3e}"
        assert fro <= 1e-2, f"{case} {name}: relative Frobenius error {fro:.3e}"
