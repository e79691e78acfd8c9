"""The allocation-free split-KV entry point (fa_fwd_splitkv_static), through
the C ABI: on two calls in a row its output must match the workspace entry
point (fa_fwd_splitkv) on the same inputs and the fp64 oracle, within the
acceptance tolerance of every other parity test, and a call must leave the
device's free memory unchanged.

Some callers cannot allocate device memory (all of it belongs to a pool or
arena they do not control, an allocation's implicit synchronisation or
failure is not acceptable mid-work, or a plug-in host gives them no
allocator); this entry point keeps its scratch in an array built into the
library instead.

Kept in a file that pytest collects last: it must pass both alone in a fresh
process and after every other test has used the library."""
import ctypes
import math

import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import LSE_ATOL, compare, to_device

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


def _static_call(fa, dev, qd, kd, vd, o, lse, causal, scale, splits):
    import torch

    B, H, Nq, d = qd.shape
    Nk = kd.shape[2]
    lib = fa.load_library()
    stream = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.fa_fwd_splitkv_static(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, Nq, Nk, d, int(causal),
                                   ctypes.c_float(scale), splits, stream or None)
    assert rc == 0, fa.fa_strerror(rc)
    torch.cuda.synchronize(dev)


def _check(fa, dev, B, H, Nq, Nk, d, causal, splits, seed):
    """Runs the static entry point (twice, checking that the second call
    changes no free-memory figure) and compares it with the workspace entry
    point and with the oracle."""
    import torch

    q, k, v = _inputs(B, H, Nq, Nk, d, seed)
    qd, kd, vd = (to_device(a, dev) for a in (q, k, v))
    scale = 1.0 / math.sqrt(d)
    o_ws, lse_ws = fa.attention_forward_splitkv(qd, kd, vd, causal=causal, scale=scale,
                                                num_splits=splits)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=dev)
    _static_call(fa, dev, qd, kd, vd, o, lse, causal, scale, splits)
    # A repeated call (the array's address is known by now) allocates nothing.
    free_before = torch.cuda.mem_get_info(dev)[0]
    _static_call(fa, dev, qd, kd, vd, o, lse, causal, scale, splits)
    assert torch.cuda.mem_get_info(dev)[0] == free_before

    o_np = o.float().cpu().numpy()
    lse_np = lse.cpu().numpy()
    # Against the workspace entry point: same arithmetic on the same inputs.
    compare(o_np, lse_np, o_ws.float().cpu().numpy().astype(np.float64),
            lse_ws.cpu().numpy().astype(np.float64), "static vs workspace")
    # Against the fp64 oracle (end-aligned causal mask for Nq < Nk).
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    worst_o, worst_l = compare(o_np, lse_np, o_ref, lse_ref, "static vs oracle")
    assert worst_l <= LSE_ATOL


def test_static_scratch_two_calls_match_workspace_path_and_oracle(fa, cuda_device):
    # Two calls in a row with different shapes: the second must not see the
    # first call's scratch contents.
    _check(fa, cuda_device, 2, 4, 5, 3000, 128, True, 0, seed=4100)
    _check(fa, cuda_device, 1, 8, 16, 1000, 64, False, 3, seed=4200)


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
