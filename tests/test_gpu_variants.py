"""GPU parity of the forward's variants against the fp64 oracle, through the
C ABI (fa_fwd_strided): fp16 inputs, head dimensions that are multiples of 16
below the padded layout, and strided (non-contiguous) Q, K, V and O."""
import math

import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.load_library()
    return fa


def _run(fa, dev, q, k, v, causal, scale, dtype):
    import torch

    qd, kd, vd = (workloads.as_torch(a, dtype).to(dev) for a in (q, k, v))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize(dev)
    assert o.dtype == qd.dtype
    return o.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 129, 1000])
def test_fp16_matches_oracle(fa, cuda_device, N, d, causal):
    q, k, v = workloads.generate_shape(1, 2, N, d, seed=500 + N + d, qk_std=1.5, dtype="f16")
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, cuda_device, q, k, v, causal, scale, "f16")
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale, dtype="f16")
    compare(o, lse, o_ref, lse_ref, label=f"fp16 N{N} d{d} c{causal}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [16, 32, 48, 80, 96, 112])
def test_head_dims_match_oracle(fa, cuda_device, d, causal, dtype):
    N = 300
    q, k, v = workloads.generate_shape(2, 2, N, d, seed=600 + d, qk_std=1.5, dtype=dtype)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, cuda_device, q, k, v, causal, scale, dtype)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale, dtype=dtype)
    compare(o, lse, o_ref, lse_ref, label=f"d{d} c{causal} {dtype}")


def test_head_dim_outputs_stay_in_bounds(fa, cuda_device):
    """d = 80 into a row-padded output: the padding columns are untouched."""
    import torch

    B, H, N, d = 1, 2, 200, 80
    q, k, v = workloads.generate_shape(B, H, N, d, seed=650)
    qd, kd, vd = (workloads.as_torch(a).to(cuda_device) for a in (q, k, v))
    big = torch.full((B, H, N, d + 48), 7.0, dtype=torch.bfloat16, device=cuda_device)
    o = big[..., :d]
    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
    fa.fa_fwd(qd, kd, vd, o, lse, True, 0.11)
    torch.cuda.synchronize(cuda_device)
    assert bool((big[..., d:] == 7.0).all())
    o_ref, lse_ref = oracle.attention(q, k, v, True, 0.11)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, label="padded o")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 65, 129, 300, 1000])
def test_head_dim_256_matches_oracle(fa, cuda_device, N, causal, dtype):
    q, k, v = workloads.generate_shape(2, 2, N, 256, seed=680 + N, qk_std=1.5, dtype=dtype)
    scale = 1.0 / 16.0
    o, lse = _run(fa, cuda_device, q, k, v, causal, scale, dtype)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale, dtype=dtype)
    compare(o, lse, o_ref, lse_ref, label=f"d256 N{N} c{causal} {dtype}")


@pytest.mark.parametrize("scale", [0.0, -0.15])
def test_head_dim_256_unusual_scales(fa, cuda_device, scale):
    q, k, v = workloads.generate_shape(1, 2, 400, 256, seed=690)
    o, lse = _run(fa, cuda_device, q, k, v, True, scale, "bf16")
    o_ref, lse_ref = oracle.attention(q, k, v, True, scale)
    compare(o, lse, o_ref, lse_ref, label=f"d256 scale {scale}")


def test_head_dim_256_strided(fa, cuda_device):
    """[B, N, H, d] memory with d = 256, causal, more units than SMs."""
    import torch

    B, H, N, d = 2, 8, 1500, 256
    q, k, v = workloads.generate_shape(B, H, N, d, seed=695, qk_std=1.5)

    def bnhd(a):
        return workloads.as_torch(a).permute(0, 2, 1, 3).contiguous().to(cuda_device).permute(
            0, 2, 1, 3)

    qd, kd, vd = bnhd(q), bnhd(k), bnhd(v)
    o = torch.empty((B, N, H, d), dtype=qd.dtype, device=cuda_device).permute(0, 2, 1, 3)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
    fa.fa_fwd(qd, kd, vd, o, lse, True, 0.0625)
    torch.cuda.synchronize(cuda_device)
    rows = np.unique(np.concatenate([np.arange(0, N, 7), [N - 1]]))
    o_ref, lse_ref = oracle.attention(q, k, v, True, 0.0625, rows=rows)
    compare(o.float().cpu().numpy()[:, :, rows], lse.cpu().numpy()[:, :, rows], o_ref, lse_ref,
            label="d256 bnhd")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_strided_bnhd_layout(fa, cuda_device, dtype):
    """Q, K, V and O in [B, N, H, d] memory (heads interleaved within a row),
    viewed as [B, H, N, d]."""
    import torch

    B, H, N, d = 2, 3, 333, 64
    q, k, v = workloads.generate_shape(B, H, N, d, seed=700, qk_std=1.5, dtype=dtype)

    def bnhd(a):
        return workloads.as_torch(a, dtype).permute(0, 2, 1, 3).contiguous().to(
            cuda_device).permute(0, 2, 1, 3)

    qd, kd, vd = bnhd(q), bnhd(k), bnhd(v)
    assert not qd.is_contiguous()
    o = torch.empty((B, N, H, d), dtype=qd.dtype, device=cuda_device).permute(0, 2, 1, 3)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
    fa.fa_fwd(qd, kd, vd, o, lse, True, 0.125)
    torch.cuda.synchronize(cuda_device)
    o_ref, lse_ref = oracle.attention(q, k, v, True, 0.125, dtype=dtype)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, label=f"bnhd {dtype}")


def test_strided_padded_rows_and_shared_kv_head(fa, cuda_device):
    """Rows padded to d + 16 elements, and K, V shared by every query head
    (head stride 0)."""
    import torch

    B, H, N, d = 2, 4, 257, 128
    q, _, _ = workloads.generate_shape(B, H, N, d, seed=710)
    _, k1, v1 = workloads.generate_shape(B, 1, N, d, seed=711)

    def padded(a):
        t = workloads.as_torch(a)
        buf = torch.zeros(t.shape[:-1] + (d + 16,), dtype=t.dtype)
        buf[..., :d] = t
        return buf.to(cuda_device)[..., :d]

    qd = padded(q)
    kd = padded(k1).expand(B, H, N, d)
    vd = padded(v1).expand(B, H, N, d)
    assert kd.stride(1) == 0
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=cuda_device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
    fa.fa_fwd(qd, kd, vd, o, lse, False, 0.09)
    torch.cuda.synchronize(cuda_device)
    k = np.broadcast_to(k1, (B, H, N, d)).copy()
    v = np.broadcast_to(v1, (B, H, N, d)).copy()
    o_ref, lse_ref = oracle.attention(q, k, v, False, 0.09)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, label="padded/shared kv")


@pytest.mark.parametrize("name", [w.name for w in workloads.VARIANT_WORKLOADS])
def test_variant_workloads_sampled_rows(fa, cuda_device, name):
    w = workloads.by_name(name)
    q, k, v = workloads.generate(w)
    rows = workloads.sampled_rows(w)
    o, lse = _run(fa, cuda_device, q, k, v, w.causal, w.scale, w.dtype)
    o_ref, lse_ref = oracle.attention(q, k, v, w.causal, w.scale, rows=rows, dtype=w.dtype)
    compare(o[:, :, rows, :], lse[:, :, rows], o_ref, lse_ref, label=name)


def test_overlapping_output_rows_rejected(fa, cuda_device):
    import torch

    B, H, N, d = 1, 2, 64, 64
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device=cuda_device)
    buf = torch.empty(H * N * d, dtype=torch.bfloat16, device=cuda_device)
    o = buf.as_strided((B, H, N, d), (H * N * d, N * d, 32, 1))  # rows overlap
    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
    with pytest.raises(fa.FAError) as err:
        fa.fa_fwd(q, q, q, o, lse, False, 0.1)
    assert err.value.code == 13


def _growing_scores(B, H, N, d, seed, dtype):
    """Scores that jump up in the middle of key tiles: the scaled scores
    (base-2 exponent units) of head 0 rise by about 20 on keys 320..383 (the
    second half of key tile 2) and by about 20 more on keys 384..447 (the
    first half of key tile 3); those of head 1 climb by 4 to 6 every 64 keys.
    So a half tile's P sum against the reference of the keys before it
    exceeds 2^15 in either half of a key tile: the reference moves mid-tile
    as well as at tile starts."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, N, d)).astype(np.float32)
    k = rng.standard_normal((B, H, N, d)).astype(np.float32)
    v = rng.standard_normal((B, H, N, d)).astype(np.float32)
    q[..., 0] = 4.0
    k[..., 0] = 0.0
    k[:, 0, 320:384, 0] = 40.0
    k[:, 0, 384:448, 0] = 80.0
    if H > 1:
        k[:, 1, :, 0] = 8.0 * (np.arange(N) // 64)
    conv = workloads.f32_to_f16_bits if dtype == "f16" else workloads.f32_to_bf16_bits
    return conv(q), conv(k), conv(v)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_reference_moves_mid_tile(fa, cuda_device, d, causal, dtype):
    """Rows whose maximum grows inside a key tile (second half) and at the
    first half of the next, so the exponent reference moves after the first
    half of P has been computed and stored (that half is then rescaled in
    place): the result is still the oracle's."""
    N = 1000
    scale = 0.125 if d == 64 else 1.0 / math.sqrt(d)
    q, k, v = _growing_scores(1, 2, N, d, seed=690 + d, dtype=dtype)
    o, lse = _run(fa, cuda_device, q, k, v, causal, scale, dtype)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale, dtype=dtype)
    compare(o, lse, o_ref, lse_ref, label=f"moving reference d{d} c{causal} {dtype}")


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("offset,pad", [(0, 8), (8, 16)])
def test_output_rows_16_byte_aligned_only(fa, cuda_device, offset, pad, d):
    """O rows that are 16-byte but not 32-byte aligned (row stride d + 8
    elements, or the whole output shifted by 8 elements): the epilogue falls
    back to 16-byte stores, and the columns around each row stay untouched."""
    import torch

    B, H, N = 1, 2, 300
    q, k, v = workloads.generate_shape(B, H, N, d, seed=720 + offset)
    qd, kd, vd = (workloads.as_torch(a).to(cuda_device) for a in (q, k, v))
    big = torch.full((B, H, N, offset + d + pad), 5.0, dtype=torch.bfloat16, device=cuda_device)
    o = big[..., offset:offset + d]
    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
    fa.fa_fwd(qd, kd, vd, o, lse, True, 0.09)
    torch.cuda.synchronize(cuda_device)
    assert bool((big[..., :offset] == 5.0).all()) and bool((big[..., offset + d:] == 5.0).all())
    o_ref, lse_ref = oracle.attention(q, k, v, True, 0.09)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
            label=f"o offset {offset} pad {pad}")


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("bf16", 256)])
def test_host_buffers_match_oracle(fa, cuda_device, dtype, d, pinned):
    """fa_fwd_host: Q, K, V in host memory (page-locked or pageable), O and
    LSE written back to host memory; two calls in a row on one workspace."""
    import torch

    B, H, N = 1, 2, 300
    scale = 1.0 / math.sqrt(d)
    ws = torch.empty(fa.fa_fwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8,
                     device=cuda_device)
    for seed in (740, 741):
        q, k, v = workloads.generate_shape(B, H, N, d, seed=seed + d, qk_std=1.5, dtype=dtype)
        hq, hk, hv = (workloads.as_torch(a, dtype) for a in (q, k, v))
        ho = torch.empty_like(hq)
        hl = torch.empty((B, H, N), dtype=torch.float32)
        if pinned:
            hq, hk, hv, ho, hl = (t.pin_memory() for t in (hq, hk, hv, ho, hl))
        fa.fa_fwd_host(hq, hk, hv, ho, hl, True, scale, ws)
        torch.cuda.synchronize(cuda_device)
        o_ref, lse_ref = oracle.attention(q, k, v, True, scale, dtype=dtype)
        compare(ho.float().numpy(), hl.numpy(), o_ref, lse_ref,
                label=f"host {dtype} d{d} pinned={pinned} seed {seed}")
