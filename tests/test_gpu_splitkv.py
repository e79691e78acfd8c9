"""GPU parity of the split-KV path (short query block, long keys) against the
fp64 oracle, through the C ABI: all rows, several split counts, ragged key
counts, causal (end-aligned) and not."""
import math

import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import compare, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.load_library()
    return fa


def _inputs(B, H, Nq, Nk, d, seed, qk_std=1.0):
    q = workloads.generate_shape(B, H, Nq, d, seed=seed, qk_std=qk_std)[0]
    _, k, v = workloads.generate_shape(B, H, Nk, d, seed=seed + 1, qk_std=qk_std)
    return q, k, v


def _run(fa, dev, q, k, v, causal, scale, splits):
    import torch

    qd, kd, vd = (to_device(a, dev) for a in (q, k, v))
    o, lse = fa.attention_forward_splitkv(qd, kd, vd, causal=causal, scale=scale,
                                          num_splits=splits)
    torch.cuda.synchronize(dev)
    return o.float().cpu().numpy(), lse.cpu().numpy()


CASES = [
    # B, H, Nq, Nk, d, causal, splits
    (1, 2, 1, 1, 64, False, 0),
    (1, 2, 1, 100, 128, True, 0),
    (2, 3, 4, 1000, 128, True, 0),
    (1, 2, 16, 4097, 64, False, 5),
    (1, 4, 16, 300, 128, True, 1),
    (1, 2, 7, 129, 64, True, 64),
    (2, 8, 1, 16384, 128, False, 0),
    (1, 2, 3, 16000, 128, True, 7),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,splits", CASES)
def test_splitkv_matches_oracle(fa, cuda_device, B, H, Nq, Nk, d, causal, splits):
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=700 + Nq + Nk + d, qk_std=1.5)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, cuda_device, q, k, v, causal, scale, splits)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    compare(o, lse, o_ref, lse_ref, label=f"splitkv {B}x{H} Nq{Nq} Nk{Nk} d{d} c{causal} s{splits}")


def test_splitkv_equals_square_kernel_rows(fa, cuda_device):
    """With Nq == Nk the split path computes what fa_fwd computes."""
    import torch

    q, k, v = workloads.generate_shape(1, 2, 16, 128, seed=811)
    qd, kd, vd = (to_device(a, cuda_device) for a in (q, k, v))
    o1, l1 = fa.attention_forward(qd, kd, vd, causal=True, scale=0.09)
    o2, l2 = fa.attention_forward_splitkv(qd, kd, vd, causal=True, scale=0.09, num_splits=1)
    torch.cuda.synchronize(cuda_device)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_splitkv_workspace_too_small_is_rejected(fa, cuda_device):
    import torch

    q, k, v = _inputs(1, 2, 2, 1000, 64, seed=900)
    qd, kd, vd = (to_device(a, cuda_device) for a in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty((1, 2, 2), dtype=torch.float32, device=cuda_device)
    need = fa.fa_fwd_splitkv_workspace_bytes(1, 2, 2, 1000, 64, 3)
    ws = torch.empty(need - 16, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(fa.FAError) as err:
        fa.fa_fwd_splitkv(qd, kd, vd, o, lse, False, 0.125, 3, ws)
    assert err.value.code == 10


def test_splitkv_deterministic(fa, cuda_device):
    q, k, v = _inputs(2, 4, 5, 3000, 128, seed=950)
    a = _run(fa, cuda_device, q, k, v, True, 0.08, 0)
    b = _run(fa, cuda_device, q, k, v, True, 0.08, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("name", [w.name for w in workloads.DECODE_WORKLOADS])
def test_decode_workloads_full_size(fa, cuda_device, name):
    """The benchmark's decode workloads at full size, in the benchmark's
    launch configuration (automatic split count, caller workspace), every
    output checked."""
    import torch

    w = workloads.by_name(name)
    q, k, v = workloads.generate_decode(w)
    qd, kd, vd = (to_device(a, cuda_device) for a in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=cuda_device)
    ws = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, 0),
                     dtype=torch.uint8, device=cuda_device)
    fa.fa_fwd_splitkv(qd, kd, vd, o, lse, w.causal, w.scale, 0, ws)
    torch.cuda.synchronize(cuda_device)
    o_ref, lse_ref = oracle.attention(q, k, v, w.causal, w.scale)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, label=name)
