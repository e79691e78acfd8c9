"""The host-buffer entry points of the split-KV path and of the backward
(fa_fwd_splitkv_host, fa_bwd_host, through the C ABI): the same kernels as
the device-pointer entry points, so their results must equal those bit for
bit on the same inputs, and match the fp64 oracle within the usual
tolerances; page-locked and pageable host buffers both work."""
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


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("Nq,Nk,d,causal,splits", [(1, 4000, 128, False, 0), (16, 3000, 64, True, 0),
                                                   (5, 2000, 128, True, 12)])
def test_splitkv_host_equals_device_path(fa, cuda_device, Nq, Nk, d, causal, splits, pinned):
    import torch

    B, H = 2, 3
    q = workloads.generate_shape(B, H, Nq, d, seed=4300 + Nq, qk_std=1.5)[0]
    _, k, v = workloads.generate_shape(B, H, Nk, d, seed=4400 + Nk, qk_std=1.5)
    scale = 1.0 / math.sqrt(d)
    o_dev, lse_dev = fa.attention_forward_splitkv(*(to_device(a, cuda_device) for a in (q, k, v)),
                                                  causal=causal, scale=scale, num_splits=splits)

    def host(a):
        t = workloads.as_torch(a)
        return t.pin_memory() if pinned else t

    hq, hk, hv = host(q), host(k), host(v)
    ho = torch.empty((B, H, Nq, d), dtype=torch.bfloat16)
    hl = torch.empty((B, H, Nq), dtype=torch.float32)
    if pinned:
        ho, hl = ho.pin_memory(), hl.pin_memory()
    ws = torch.empty(fa.fa_fwd_splitkv_host_workspace_bytes(B, H, Nq, Nk, d, splits),
                     dtype=torch.uint8, device=cuda_device)
    fa.fa_fwd_splitkv_host(hq, hk, hv, ho, hl, causal, scale, splits, ws)
    torch.cuda.synchronize(cuda_device)
    assert torch.equal(ho, o_dev.cpu()) and torch.equal(hl, lse_dev.cpu())
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    compare(ho.float().numpy(), hl.numpy(), o_ref, lse_ref, "split-KV host")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(129, 64), (300, 128)])
def test_bwd_host_equals_device_path(fa, cuda_device, N, d, causal, dtype):
    import torch

    B, H = 1, 2
    q, k, v = workloads.generate_shape(B, H, N, d, seed=4500 + N + d, qk_std=1.5, dtype=dtype)
    do = workloads.generate_shape(B, H, N, d, seed=4600 + N + d, dtype=dtype)[0]
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = (workloads.as_torch(a, dtype).to(cuda_device) for a in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    grads_dev = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)

    hin = [workloads.as_torch(a, dtype).pin_memory() for a in (q, k, v)]
    ho, hl = o.cpu().pin_memory(), lse.cpu().pin_memory()
    hdo = workloads.as_torch(do, dtype).pin_memory()
    outs = [torch.empty_like(hin[0]).pin_memory() for _ in range(3)]
    ws = torch.empty(fa.fa_bwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8,
                     device=cuda_device)
    fa.fa_bwd_host(*hin, ho, hl, hdo, *outs, causal, scale, ws)
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    for name, h, g in zip(("dQ", "dK", "dV"), outs, grads_dev):
        assert torch.equal(h, g.cpu()), name
    ref = oracle.attention_bwd(q, k, v, do, causal, scale, dtype=dtype)
    for name, h, r in zip(("dQ", "dK", "dV"), outs, ref):
        err = np.abs(h.float().numpy().astype(np.float64) - r) / (1.0 + np.abs(r))
        assert float(err.max()) <= 3e-2, f"bwd host {name}: {float(err.max()):.3e}"
