"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Order follows the small-to-large ladder of the pwwt.cn walkthrough §5.4:
tiny single-head cases first, then ragged lengths, then the five workloads
(the three large ones on sampled rows the oracle computes one by one).
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import check_against_oracle, run_cuda, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.load_library()
    return cuda_device


def test_workload_small(dev):
    w = workloads.WORKLOADS[0]
    q, k, v = workloads.generate(w)
    check_against_oracle(q, k, v, w.causal, w.scale, dev, label=w.name)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [64, 128, 256, 512, 2048])
def test_ladder(dev, N, d, causal):
    q, k, v = workloads.generate_shape(1, 1, N, d, seed=100 + N + d)
    check_against_oracle(q, k, v, causal, 1.0 / math.sqrt(d), dev, label=f"N{N} d{d} c{causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", workloads.RAGGED_N)
def test_ragged(dev, N, d, causal):
    q, k, v = workloads.generate_shape(1, 2, N, d, seed=200 + N + d, qk_std=1.5)
    check_against_oracle(q, k, v, causal, 1.0 / math.sqrt(d), dev, label=f"ragged N{N} d{d} c{causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("scale", [0.0, -0.2, 0.9])
def test_unusual_scales(dev, scale, d):
    q, k, v = workloads.generate_shape(2, 1, 300, d, seed=300)
    check_against_oracle(q, k, v, True, scale, dev, label=f"scale {scale}")
    check_against_oracle(q, k, v, False, scale, dev, label=f"scale {scale}")


def test_workload_b4h8n1024(dev):
    w = workloads.WORKLOADS[1]
    q, k, v = workloads.generate(w)
    check_against_oracle(q, k, v, w.causal, w.scale, dev, label=w.name)


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_workload_large_sampled_rows(dev, idx):
    w = workloads.WORKLOADS[idx]
    q, k, v = workloads.generate(w)
    rows = workloads.sampled_rows(w)
    check_against_oracle(q, k, v, w.causal, w.scale, dev, rows=rows, label=w.name)


def test_deterministic(dev):
    import torch

    w = workloads.WORKLOADS[1]
    q, k, v = workloads.generate(w)
    o1, l1 = run_cuda(q, k, v, True, w.scale, dev)
    o2, l2 = run_cuda(q, k, v, True, w.scale, dev)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_outputs_only_written_in_bounds(dev):
    """O and LSE of a ragged case are written exactly over [B,H,N,*]: a
    sentinel placed right after each output survives."""
    import torch

    import tiled_attention_forward_attn_gb300 as fa

    B, H, N, d = 1, 3, 200, 128
    q, k, v = workloads.generate_shape(B, H, N, d, seed=400)
    qd, kd, vd = (to_device(a, dev) for a in (q, k, v))
    o_buf = torch.full((B * H * N * d + 64,), 7.0, dtype=torch.bfloat16, device=dev)
    l_buf = torch.full((B * H * N + 16,), 7.0, dtype=torch.float32, device=dev)
    o = o_buf[: B * H * N * d].view(B, H, N, d)
    lse = l_buf[: B * H * N].view(B, H, N)
    fa.fa_fwd(qd, kd, vd, o, lse, True, 1.0 / math.sqrt(d))
    torch.cuda.synchronize(dev)
    assert torch.all(o_buf[B * H * N * d:] == 7.0)
    assert torch.all(l_buf[B * H * N:] == 7.0)
    o_ref, lse_ref = oracle.attention(q, k, v, True, 1.0 / math.sqrt(d))
    assert np.max(np.abs(o.float().cpu().numpy() - o_ref) / (1 + np.abs(o_ref))) <= 1e-2


def test_runs_on_a_side_stream(dev):
    import torch

    import tiled_attention_forward_attn_gb300 as fa

    q, k, v = workloads.generate_shape(1, 2, 384, 64, seed=500)
    qd, kd, vd = (to_device(a, dev) for a in (q, k, v))
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        o, lse = fa.attention_forward(qd, kd, vd, causal=True, scale=0.125)
    s.synchronize()
    o_ref, lse_ref = oracle.attention(q, k, v, True, 0.125)
    assert np.max(np.abs(o.float().cpu().numpy() - o_ref) / (1 + np.abs(o_ref))) <= 1e-2
    assert np.max(np.abs(lse.cpu().numpy() - lse_ref)) <= 1e-3
