"""Failure path of the bounded waits, exercised without faulting the GPU.

A test hook makes every CTA skip one V-tile copy, so the MMA warp's wait for
it can never complete.  With a short wait limit the kernel must give up,
record FA_DEVICE_STATUS_TIMEOUT, drain what it issued, free TMEM and exit;
the context must stay usable and the next normal call must be correct.
"""
import math

import pytest

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
