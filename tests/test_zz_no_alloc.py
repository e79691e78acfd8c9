"""The allocation-free split-KV entry point (fa_fwd_splitkv_static) against
the workspace entry point (fa_fwd_splitkv), through the C ABI.

Kept in a file that pytest collects last: it must pass both alone in a fresh
process and after every other test has used the library."""
import ctypes
import math

import pytest

import workloads
from gpu_helpers import LSE_ATOL, O_ATOL, to_device

pytestmark = pytest.mark.gpu

FA_ERR_SCRATCH_LIMIT = 11


@pytest.fixture(scope="module")
def fa(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.load_library()
    return fa


def _inputs(B, H, Nq, Nk, d, seed):
    q = workloads.generate_shape(B, H, Nq, d, seed=seed, qk_std=1.5)[0]
    _, k, v = workloads.generate_shape(B, H, Nk, d, seed=seed + 1, qk_std=1.5)
    return q, k, v


def _both(fa, dev, B, H, Nq, Nk, d, causal, splits, seed):
    """Run the workspace entry point and the static one on the same inputs;
    return both results (O as fp32, LSE) on the host."""
    import torch

    q, k, v = (to_device(a, dev) for a in _inputs(B, H, Nq, Nk, d, seed))
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = fa.attention_forward_splitkv(q, k, v, causal=causal, scale=scale,
                                                  num_splits=splits)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=dev)
    lib = fa.load_library()
    stream = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.fa_fwd_splitkv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, Nq, Nk, d, int(causal), ctypes.c_float(scale),
                                   splits, stream or None)
    assert rc == 0, fa.fa_strerror(rc)
    torch.cuda.synchronize(dev)
    return (o.float().cpu(), lse.cpu()), (o_ref.float().cpu(), lse_ref.cpu())


def _close(got, ref):
    (o, lse), (o_ref, lse_ref) = got, ref
    assert bool(torch_isfinite(o)) and bool(torch_isfinite(lse))
    o_err = ((o - o_ref).abs() / (1.0 + o_ref.abs())).max().item()
    l_err = (lse - lse_ref).abs().max().item()
    assert o_err <= O_ATOL, o_err
    assert l_err <= LSE_ATOL, l_err


def torch_isfinite(t):
    import torch

    return torch.isfinite(t).all()


def test_static_scratch_matches_workspace_path_two_calls(fa, cuda_device):
    # Two calls in a row with different shapes: the second must not see the
    # first call's scratch contents.
    first = _both(fa, cuda_device, 2, 4, 5, 3000, 128, True, 0, seed=4100)
    _close(*first)
    second = _both(fa, cuda_device, 1, 8, 16, 1000, 64, False, 3, seed=4200)
    _close(*second)


def test_static_scratch_rejects_oversize_request(fa, cuda_device):
    import torch

    cap = fa.fa_fwd_splitkv_static_scratch_bytes()
    assert cap == 8 << 20
    # 256 ranges x 64 heads x 16 queries x (4*128 + 4) bytes > 8 MiB.
    B, H, Nq, Nk, d, splits = 1, 64, 16, 256 * 64, 128, 256
    assert fa.fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, splits) > cap
    q = torch.zeros((B, H, Nq, d), dtype=torch.bfloat16, device=cuda_device)
    k = torch.zeros((B, H, Nk, d), dtype=torch.bfloat16, device=cuda_device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=cuda_device)
    with pytest.raises(fa.FAError) as err:
        fa.fa_fwd_splitkv_static(q, k, k, o, lse, False, 0.1, splits)
    assert err.value.code == FA_ERR_SCRATCH_LIMIT
