"""The guarded build (libfa_guarded.so: the same kernels compiled with
FA_GUARDED=1, every TMA tile origin, shared-memory destination, TMEM column
range and global store checked against its bounds before the access) over
the ragged ladder and the other paths: every result still matches the fp64
oracle, and the device status word stays 0 (no bounds check failed, no wait
ran out).  This stands in for a memory checker, which this test setup does
not run."""
import math

import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import check_against_oracle, compare, to_device
import test_gpu_random_sweep as sweep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.reload_library(fa.GUARDED_LIB_PATH)
    fa.fa_clear_device_status()
    yield fa
    fa.reload_library()


@pytest.fixture(autouse=True)
def clear_status(fa):
    """The status word is sticky: each test starts from 0."""
    fa.fa_clear_device_status()


def _status_clean(fa):
    st = fa.fa_get_device_status()
    assert st == 0, f"device status {st:#x} (bounds bit {fa.FA_DEVICE_STATUS_BOUNDS:#x})"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", workloads.RAGGED_N)
def test_guarded_forward_ragged_ladder(fa, cuda_device, N, d, causal):
    q, k, v = workloads.generate_shape(1, 2, N, d, seed=3000 + N + d, qk_std=1.5)
    check_against_oracle(q, k, v, causal, 1.0 / math.sqrt(d), cuda_device,
                         label=f"guarded N{N} d{d} c{causal}")
    _status_clean(fa)


@pytest.mark.parametrize("d", [16, 48, 96, 256])
def test_guarded_forward_other_head_dims(fa, cuda_device, d):
    q, k, v = workloads.generate_shape(1, 3, 333, d, seed=3100 + d, qk_std=1.5)
    check_against_oracle(q, k, v, True, 1.0 / math.sqrt(d), cuda_device, label=f"guarded d{d}")
    _status_clean(fa)


def test_guarded_forward_fp16_and_strided_output(fa, cuda_device):
    import torch

    B, H, N, d = 2, 3, 257, 128
    q, k, v = workloads.generate_shape(B, H, N, d, seed=3200, qk_std=1.5, dtype="f16")
    qd, kd, vd = (workloads.as_torch(a, "f16").to(cuda_device) for a in (q, k, v))
    # O in a [B, N, H, d] buffer (row stride H*d, head stride d).
    buf = torch.zeros((B, N, H, d), dtype=torch.float16, device=cuda_device)
    o = buf.permute(0, 2, 1, 3)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
    rc = fa.fa_fwd_strided(qd.data_ptr(), None, kd.data_ptr(), None, vd.data_ptr(), None,
                           o.data_ptr(), tuple(o.stride()[:3]), lse.data_ptr(), 1, B, H, N, d,
                           True, 0.1, torch.cuda.current_stream(cuda_device).cuda_stream)
    assert rc == 0, fa.fa_strerror(rc)
    torch.cuda.synchronize(cuda_device)
    o_ref, lse_ref = oracle.attention(q, k, v, True, 0.1, dtype="f16")
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "guarded fp16 strided")
    _status_clean(fa)


@pytest.mark.parametrize("Nq,Nk,d,causal,splits", [(1, 3000, 128, False, 0), (16, 5000, 64, True, 0),
                                                   (7, 1000, 128, True, 20)])
def test_guarded_splitkv(fa, cuda_device, Nq, Nk, d, causal, splits):
    q = workloads.generate_shape(2, 3, Nq, d, seed=3300 + Nq, qk_std=1.5)[0]
    _, k, v = workloads.generate_shape(2, 3, Nk, d, seed=3400 + Nk, qk_std=1.5)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_forward_splitkv(*(to_device(a, cuda_device) for a in (q, k, v)),
                                          causal=causal, scale=scale, num_splits=splits)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "guarded split-KV")
    _status_clean(fa)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [17, 129, 300])
def test_guarded_backward(fa, cuda_device, N, d, causal):
    import torch

    q, k, v = workloads.generate_shape(1, 2, N, d, seed=3500 + N + d, qk_std=1.5)
    do = workloads.generate_shape(1, 2, N, d, seed=3600 + N + d)[0]
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = (to_device(a, cuda_device) for a in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    grads = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize(cuda_device)
    ref = oracle.attention_bwd(q, k, v, do, causal, scale)
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        err = np.abs(g.float().cpu().numpy().astype(np.float64) - r) / (1.0 + np.abs(r))
        assert float(err.max()) <= 3e-2, f"guarded backward {name}: {float(err.max()):.3e}"
    _status_clean(fa)


def test_guarded_backward_strided(fa, cuda_device):
    """Every backward tensor in [B, N, H, d] memory, gradients included."""
    import torch

    B, H, N, d = 2, 3, 300, 64
    q, k, v = workloads.generate_shape(B, H, N, d, seed=3650, qk_std=1.5)
    do = workloads.generate_shape(B, H, N, d, seed=3651)[0]
    qd, kd, vd, dod = (to_device(a, cuda_device) for a in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=True, scale=0.125)

    def bnhd(t):
        return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)

    grads = [torch.empty((B, N, H, d), dtype=torch.bfloat16, device=cuda_device).permute(
        0, 2, 1, 3) for _ in range(3)]
    fa.fa_bwd(bnhd(qd), bnhd(kd), bnhd(vd), bnhd(o), lse, bnhd(dod), *grads, True, 0.125)
    torch.cuda.synchronize(cuda_device)
    ref = oracle.attention_bwd(q, k, v, do, True, 0.125)
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        err = np.abs(g.float().cpu().numpy().astype(np.float64) - r) / (1.0 + np.abs(r))
        assert float(err.max()) <= 3e-2, f"guarded strided backward {name}: {float(err.max()):.3e}"
    _status_clean(fa)


@pytest.mark.parametrize("order", [1, 2])
def test_guarded_loop_order_ablation(fa, cuda_device, order):
    q, k, v = workloads.generate_shape(1, 2, 300, 64, seed=3700, qk_std=1.5)
    scale = 0.125
    o, lse = fa.attention_forward_order_ablation(*(to_device(a, cuda_device) for a in (q, k, v)),
                                                 True, scale, order)
    o_ref, lse_ref = oracle.attention(q, k, v, True, scale)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"guarded order {order}")
    _status_clean(fa)


@pytest.mark.parametrize("case", sweep._fwd_cases()[:32], ids=lambda c: f"f{c[0]}")
def test_guarded_random_forward(fa, cuda_device, case):
    """The first cases of the random sweep (every layout, head dimension and
    element type among them) with every access bounds-checked."""
    sweep.test_forward_random_case(fa, cuda_device, case)
    _status_clean(fa)


@pytest.mark.parametrize("case", sweep._splitkv_cases()[:12], ids=lambda c: f"s{c[0]}")
def test_guarded_random_splitkv(fa, cuda_device, case):
    sweep.test_splitkv_random_case(fa, cuda_device, case)
    _status_clean(fa)


@pytest.mark.parametrize("case", sweep._bwd_cases()[:12], ids=lambda c: f"g{c[0]}")
def test_guarded_random_backward(fa, cuda_device, case):
    sweep.test_backward_random_case(fa, cuda_device, case)
    _status_clean(fa)
