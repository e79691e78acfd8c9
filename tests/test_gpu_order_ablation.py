"""GPU parity of the loop-order ablation kernels (fa_fwd_order_ablation,
orders 1 and 2) against the fp64 oracle, through the C ABI."""
import math

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


@pytest.mark.parametrize("order", [1, 2])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 63, 64, 65, 300, 1000])
def test_order_matches_oracle(fa, cuda_device, N, d, causal, order):
    import torch

    q, k, v = workloads.generate_shape(2, 2, N, d, seed=1400 + N + d, qk_std=2.0)
    qd, kd, vd = (to_device(a, cuda_device) for a in (q, k, v))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_forward_order_ablation(qd, kd, vd, causal, scale, order)
    torch.cuda.synchronize(cuda_device)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
            label=f"order{order} N{N} d{d} c{causal}")


@pytest.mark.parametrize("order", [1, 2])
def test_order_headline_sampled_rows(fa, cuda_device, order):
    import torch

    w = workloads.HEADLINE
    q, k, v = workloads.generate(w)
    qd, kd, vd = (to_device(a, cuda_device) for a in (q, k, v))
    o, lse = fa.attention_forward_order_ablation(qd, kd, vd, w.causal, w.scale, order)
    torch.cuda.synchronize(cuda_device)
    rows = workloads.sampled_rows(w)
    o_ref, lse_ref = oracle.attention(q, k, v, w.causal, w.scale, rows=rows)
    compare(o.float().cpu().numpy()[:, :, rows], lse.cpu().numpy()[:, :, rows], o_ref, lse_ref,
            label=f"{w.name} order {order}")
