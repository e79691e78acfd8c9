"""Secondary cross-check against PyTorch's scaled_dot_product_attention,
evaluated in fp32 on the GPU from the same 16-bit inputs ("pwwt.cn
FlashAttention/Triton walkthrough" §4.2 and §5.2 compare with PyTorch SDPA and
expect errors around 1e-2 with 16-bit inputs and fp32 accumulation).  The fp64
oracle stays the reference of record; this checks the kernels against code
that shares nothing with either.  Tolerances as the oracle comparisons:
|O - ref| <= 1e-2 (1 + |ref|), and 3e-2 (1 + |ref|) for the gradients."""
import math

import pytest

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.load_library()
    return fa


def _worst(a, ref):
    return float(((a.float() - ref).abs() / (1.0 + ref.abs())).max())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(333, 64), (1025, 128), (200, 96)])
def test_forward_and_backward_match_sdpa_fp32(fa, cuda_device, N, d, causal):
    import torch
    import torch.nn.functional as F

    B, H = 2, 3
    scale = 1.0 / math.sqrt(d)
    q, k, v = (workloads.as_torch(a).to(cuda_device)
               for a in workloads.generate_shape(B, H, N, d, seed=8300 + N + d, qk_std=1.5))
    do = workloads.as_torch(workloads.generate_shape(B, H, N, d, seed=8400 + N)[0]).to(cuda_device)
    o, lse = fa.attention_forward(q, k, v, causal=causal, scale=scale)
    grads = fa.attention_backward(q, k, v, o, lse, do, causal=causal, scale=scale)

    q32, k32, v32 = (t.float().requires_grad_(True) for t in (q, k, v))
    o32 = F.scaled_dot_product_attention(q32, k32, v32, is_causal=causal, scale=scale)
    o32.backward(do.float())
    s = torch.einsum("bhid,bhjd->bhij", q.float(), k.float()) * scale
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool, device=cuda_device).triu(1), float("-inf"))
    lse32 = torch.logsumexp(s, dim=-1)
    torch.cuda.synchronize(cuda_device)
    assert _worst(o, o32.detach()) <= 1e-2
    assert float((lse - lse32).abs().max()) <= 1e-3
    for name, g, r in zip(("dQ", "dK", "dV"), grads, (q32.grad, k32.grad, v32.grad)):
        assert _worst(g, r) <= 3e-2, name
