"""Failure path of the bounded waits, exercised without faulting the GPU.

A test hook makes every CTA skip one streamed-tile copy (the first V tile of
the forward kernels, the first K/V tile of the split-KV pass, the first
streamed stage of each backward pass), so the wait for it can never
complete.  With a short wait limit every kernel must give up, record
FA_DEVICE_STATUS_TIMEOUT, drain what it issued, free TMEM and exit; the
context must stay usable and the next normal call must be correct.
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import check_against_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.load_library()
    return fa


@pytest.mark.parametrize("d", [64, 128])
def test_timeout_is_reported_and_context_survives(fa, cuda_device, d):
    import torch

    q, k, v = workloads.generate_shape(1, 2, 300, d, seed=600 + d)
    qd, kd, vd = (to_device(a, cuda_device) for a in (q, k, v))
    fa.fa_clear_device_status()
    assert fa.fa_get_device_status() == 0
    fa.fa_set_wait_limit_ns(50_000_000)  # 50 ms
    fa.fa_set_fault_injection(fa.FA_INJECT_SKIP_FIRST_V_LOAD)
    try:
        fa.attention_forward(qd, kd, vd, causal=True, scale=1.0 / math.sqrt(d))
        torch.cuda.synchronize(cuda_device)
        status = fa.fa_get_device_status()
    finally:
        fa.fa_set_fault_injection(0)
        fa.fa_set_wait_limit_ns(0)
    assert status & fa.FA_DEVICE_STATUS_TIMEOUT
    fa.fa_clear_device_status()
    # The context is intact: a normal call afterwards is correct and clean.
    check_against_oracle(q, k, v, True, 1.0 / math.sqrt(d), cuda_device, label="after timeout")
    assert fa.fa_get_device_status() == 0


def _expect_timeout(fa, dev, call):
    """Runs `call` with the test hook on and a 50 ms wait limit; returns the
    device status word it left."""
    import torch

    fa.fa_clear_device_status()
    assert fa.fa_get_device_status() == 0
    fa.fa_set_wait_limit_ns(50_000_000)
    fa.fa_set_fault_injection(fa.FA_INJECT_SKIP_FIRST_V_LOAD)
    try:
        call()
        torch.cuda.synchronize(dev)
        status = fa.fa_get_device_status()
    finally:
        fa.fa_set_fault_injection(0)
        fa.fa_set_wait_limit_ns(0)
    fa.fa_clear_device_status()
    return status


def _close(got, ref, atol, label):
    got = np.asarray(got, dtype=np.float64)
    err = float((np.abs(got - ref) / (1.0 + np.abs(ref))).max())
    assert np.all(np.isfinite(got)) and err <= atol, f"{label}: {err:.3e}"


def test_timeout_head_dim_256(fa, cuda_device):
    import torch

    q, k, v = workloads.generate_shape(1, 2, 300, 256, seed=620)
    qd, kd, vd = (to_device(a, cuda_device) for a in (q, k, v))
    status = _expect_timeout(
        fa, cuda_device, lambda: fa.attention_forward(qd, kd, vd, causal=True, scale=0.0625))
    assert status & fa.FA_DEVICE_STATUS_TIMEOUT
    o, lse = fa.attention_forward(qd, kd, vd, causal=True, scale=0.0625)
    torch.cuda.synchronize(cuda_device)
    o_ref, lse_ref = oracle.attention(q, k, v, True, 0.0625)
    _close(o.float().cpu().numpy(), o_ref, 1e-2, "d256 after timeout")
    _close(lse.cpu().numpy(), lse_ref, 1e-3, "d256 LSE after timeout")
    assert fa.fa_get_device_status() == 0


@pytest.mark.parametrize("static", [False, True])
def test_timeout_split_kv(fa, cuda_device, static):
    """The clustered one-launch form and the two-pass form (the
    allocation-free entry point)."""
    import torch

    q = workloads.generate_shape(1, 2, 4, 128, seed=630)[0]
    _, k, v = workloads.generate_shape(1, 2, 3000, 128, seed=631)
    qd, kd, vd = (to_device(a, cuda_device) for a in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty((1, 2, 4), dtype=torch.float32, device=cuda_device)

    def run():
        if static:
            fa.fa_fwd_splitkv_static(qd, kd, vd, o, lse, True, 0.09)
        else:
            o2, lse2 = fa.attention_forward_splitkv(qd, kd, vd, causal=True, scale=0.09)
            o.copy_(o2)
            lse.copy_(lse2)

    assert _expect_timeout(fa, cuda_device, run) & fa.FA_DEVICE_STATUS_TIMEOUT
    run()
    torch.cuda.synchronize(cuda_device)
    o_ref, lse_ref = oracle.attention(q, k, v, True, 0.09)
    _close(o.float().cpu().numpy(), o_ref, 1e-2, "split-KV after timeout")
    _close(lse.cpu().numpy(), lse_ref, 1e-3, "split-KV LSE after timeout")
    assert fa.fa_get_device_status() == 0


def test_timeout_backward(fa, cuda_device):
    import torch

    q, k, v = workloads.generate_shape(1, 2, 300, 64, seed=640, qk_std=1.5)
    do = workloads.generate_shape(1, 2, 300, 64, seed=641)[0]
    qd, kd, vd, dod = (to_device(a, cuda_device) for a in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=True, scale=0.125)
    torch.cuda.synchronize(cuda_device)
    status = _expect_timeout(
        fa, cuda_device,
        lambda: fa.attention_backward(qd, kd, vd, o, lse, dod, causal=True, scale=0.125))
    assert status & fa.FA_DEVICE_STATUS_TIMEOUT
    grads = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=True, scale=0.125)
    torch.cuda.synchronize(cuda_device)
    refs = oracle.attention_bwd(q, k, v, do, True, 0.125)
    for name, g, r in zip(("dQ", "dK", "dV"), grads, refs):
        _close(g.float().cpu().numpy(), r, 3e-2, f"backward {name} after timeout")
    assert fa.fa_get_device_status() == 0
