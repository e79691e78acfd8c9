"""The torch.autograd wrapper (``attention``): its forward is fa_fwd and its
backward fa_bwd on the saved O and LSE, so through autograd both must equal
the direct calls bit for bit; a gradient that autograd hands over expanded
(a plain ``.sum()`` loss gives all-ones with zero strides) goes through the
same kernels after a contiguous copy, checked against the oracle."""
import math

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.load_library()
    return fa


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
def test_autograd_equals_direct_calls(fa, cuda_device, causal, dtype):
    import torch

    B, H, N, d = 2, 3, 300, 64
    scale = 1.0 / math.sqrt(d)
    q, k, v = workloads.generate_shape(B, H, N, d, seed=8100, qk_std=1.5, dtype=dtype)
    do = workloads.generate_shape(B, H, N, d, seed=8101, dtype=dtype)[0]
    qd, kd, vd, dod = (workloads.as_torch(a, dtype).to(cuda_device) for a in (q, k, v, do))
    leaves = [t.clone().requires_grad_(True) for t in (qd, kd, vd)]
    o = fa.attention(*leaves, causal=causal)
    o.backward(dod)
    o_ref, lse_ref = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    grads = fa.attention_backward(qd, kd, vd, o_ref, lse_ref, dod, causal=causal, scale=scale)
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    assert torch.equal(o.detach(), o_ref)
    for name, leaf, g in zip(("dQ", "dK", "dV"), leaves, grads):
        assert torch.equal(leaf.grad, g), name


def test_autograd_sum_loss_matches_oracle(fa, cuda_device):
    """loss = O.sum(): the incoming gradient is an expanded tensor of ones."""
    import torch

    B, H, N, d = 1, 2, 200, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = workloads.generate_shape(B, H, N, d, seed=8200, qk_std=1.5)
    leaves = [workloads.as_torch(a).to(cuda_device).requires_grad_(True) for a in (q, k, v)]
    o = fa.attention(*leaves, causal=True, scale=scale)
    o.sum().backward()
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    ones = workloads.torch_bf16_to_bits(torch.ones((B, H, N, d), dtype=torch.bfloat16))
    ref = oracle.attention_bwd(q, k, v, ones, True, scale)
    for name, leaf, r in zip(("dQ", "dK", "dV"), leaves, ref):
        got = leaf.grad.float().cpu().numpy().astype(np.float64)
        err = np.abs(got - r) / (1.0 + np.abs(r))
        assert float(err.max()) <= 3e-2, f"{name}: {float(err.max()):.3e}"
