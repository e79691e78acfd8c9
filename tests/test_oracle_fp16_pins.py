"""Pins for the oracle's fp16 input format (the fp16 variant of the forward:
"pwwt.cn FlashAttention/Triton walkthrough" §3.4 runs in fp16, §5 lists it
among the extensions)."""
import numpy as np
import pytest

import oracle
import workloads


def test_f1_f16_widening_matches_ieee_binary16_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = oracle.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)  # numpy's IEEE binary16
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero, the largest finite value, the smallest subnormal
    assert np.signbit(oracle.f16_to_f64(np.array([0x8000], np.uint16))[0])
    assert oracle.f16_to_f64(np.array([0x7BFF], np.uint16))[0] == 65504.0
    assert oracle.f16_to_f64(np.array([0x0001], np.uint16))[0] == 2.0 ** -24


@pytest.mark.parametrize("causal", [False, True])
def test_f2_f16_attention_matches_sdpa(causal):
    torch = pytest.importorskip("torch")
    q, k, v = workloads.generate_shape(1, 2, 37, 48, seed=61, qk_std=1.5, dtype="f16")
    O, L = oracle.attention(q, k, v, causal, 0.2, dtype="f16")
    qf, kf, vf = (torch.from_numpy(a.view(np.float16).astype(np.float64)) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, is_causal=causal,
                                                           scale=0.2)
    assert np.max(np.abs(O - ref.numpy())) <= 1e-12
    s = 0.2 * qf @ kf.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(37, 37, dtype=torch.bool).triu(1), float("-inf"))
    assert np.max(np.abs(L - torch.logsumexp(s, -1).numpy())) <= 1e-12


def test_f3_format_flag_is_honoured():
    # Small integers are exact in both formats: the results agree.  The same
    # bit patterns read as the other format give a different problem.
    rng = np.random.Generator(np.random.PCG64(5))
    ints = rng.integers(-3, 4, size=(3, 1, 9, 16)).astype(np.float32)
    f16 = ints.astype(np.float16).view(np.uint16)
    bf16 = workloads.f32_to_bf16_bits(ints)
    a = oracle.attention(f16[0], f16[1], f16[2], False, 0.25, dtype="f16")
    b = oracle.attention(bf16[0], bf16[1], bf16[2], False, 0.25, dtype="bf16")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    c = oracle.attention(f16[0], f16[1], f16[2], False, 0.25, dtype="bf16")
    assert not np.allclose(a[0], c[0])
    with pytest.raises(ValueError):
        oracle.attention(f16[0], f16[1], f16[2], False, 0.25, dtype="fp8")
