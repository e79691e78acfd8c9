"""Pins for the oracle's backward (gradients of the attention forward), each
independent of the backward's own formulas: central finite differences of
a plain fp64 forward, fp64 autograd of the library's SDPA, and closed
forms."""
import numpy as np
import pytest

import oracle
import workloads


def _decoded(bits):
    return workloads.bf16_bits_to_f32(bits).astype(np.float64)


def _forward64(q, k, v, causal, scale):
    """softmax(scale q k^T [+ causal mask]) v for one head, fp64."""
    s = scale * q @ k.T
    if causal:
        s = np.where(np.tril(np.ones(s.shape, dtype=bool)), s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


@pytest.mark.parametrize("causal", [False, True])
def test_b1_matches_central_finite_differences(causal):
    N, d, scale = 6, 5, 0.7
    q, k, v = workloads.generate_shape(1, 1, N, d, seed=81, qk_std=1.5)
    do = workloads.generate_shape(1, 1, N, d, seed=82)[0]
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, scale)
    x = [_decoded(a)[0, 0] for a in (q, k, v)]
    g = _decoded(do)[0, 0]
    h = 1e-6
    for which, grad in enumerate((dq, dk, dv)):
        num = np.zeros((N, d))
        for i in range(N):
            for t in range(d):
                plus = [a.copy() for a in x]
                minus = [a.copy() for a in x]
                plus[which][i, t] += h
                minus[which][i, t] -= h
                lp = np.sum(g * _forward64(*plus, causal, scale))
                lm = np.sum(g * _forward64(*minus, causal, scale))
                num[i, t] = (lp - lm) / (2 * h)
        assert np.max(np.abs(grad[0, 0] - num)) <= 1e-7, ("dq", "dk", "dv")[which]


@pytest.mark.parametrize("causal", [False, True])
def test_b2_matches_sdpa_autograd(causal):
    torch = pytest.importorskip("torch")
    B, H, N, d, scale = 2, 2, 33, 16, 0.3
    q, k, v = workloads.generate_shape(B, H, N, d, seed=83, qk_std=2.0)
    do = workloads.generate_shape(B, H, N, d, seed=84)[0]
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, scale)
    qt, kt, vt = (torch.from_numpy(_decoded(a)).requires_grad_() for a in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal,
                                                           scale=scale)
    out.backward(torch.from_numpy(_decoded(do)))
    for got, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        assert np.max(np.abs(got - ref.numpy())) <= 1e-12


def test_b3_closed_forms():
    B, H, N, d = 1, 2, 10, 8
    q, k, v = workloads.generate_shape(B, H, N, d, seed=85)
    do = workloads.generate_shape(B, H, N, d, seed=86)[0]
    g = _decoded(do)
    # scale 0: dQ = dK = 0 exactly; P is uniform over the visible keys, so
    # dV_j = sum_i dO_i / N (all keys) or sum_{i >= j} dO_i / (i + 1) (causal).
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, False, 0.0)
    assert not dq.any() and not dk.any()
    assert np.max(np.abs(dv - g.sum(axis=2, keepdims=True) / N)) <= 1e-12
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, True, 0.0)
    w = g / np.arange(1, N + 1)[None, None, :, None]
    ref = np.flip(np.cumsum(np.flip(w, axis=2), axis=2), axis=2)
    assert not dq.any() and not dk.any()
    assert np.max(np.abs(dv - ref)) <= 1e-12
    # dO = 0: every gradient is 0.
    zero = np.zeros_like(do)
    for grad in oracle.attention_bwd(q, k, v, zero, True, 0.5):
        assert not grad.any()
    # all value rows equal: O does not depend on Q or K, so dQ = dK = 0.
    v_same = np.broadcast_to(v[:, :, :1, :], v.shape).copy()
    dq, dk, _ = oracle.attention_bwd(q, k, v_same, do, True, 0.5)
    assert np.max(np.abs(dq)) <= 1e-12 and np.max(np.abs(dk)) <= 1e-12
