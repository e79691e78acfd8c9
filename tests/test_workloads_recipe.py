"""The seeded input recipe (no GPU): the same seed gives the same bits, the
draws have the stated spread, the bf16 and fp16 roundings are the nearest
representable values, the row samples hold the tiling's boundary rows, and
the workload table carries the shapes and nominal counts of the method's
evaluation."""
import math

import numpy as np
import pytest

import workloads


def test_same_seed_same_bits_other_seed_other_bits():
    a = workloads.generate_shape(1, 2, 64, 32, seed=11)
    b = workloads.generate_shape(1, 2, 64, 32, seed=11)
    c = workloads.generate_shape(1, 2, 64, 32, seed=12)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not np.array_equal(a[0], c[0])
    assert all(x.dtype == np.uint16 and x.shape == (1, 2, 64, 32) for x in a)


@pytest.mark.parametrize("qk_std", [1.0, 3.0])
def test_spread_of_the_draws(qk_std):
    q, k, v = workloads.generate_shape(1, 4, 512, 64, seed=5, qk_std=qk_std)
    for bits, std in ((q, qk_std), (k, qk_std), (v, 1.0)):
        x = workloads.bf16_bits_to_f32(bits).astype(np.float64)
        assert abs(x.mean()) < 0.02 * std
        assert abs(x.std() / std - 1.0) < 0.02


def test_bf16_rounding_is_nearest_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even
    # pattern (1.0); just above the halfway point rounds up.
    halfway = np.float32(1.0 + 2.0 ** -8)
    above = np.nextafter(halfway, np.float32(2.0))
    bits = workloads.f32_to_bf16_bits(np.array([halfway, above, -halfway], dtype=np.float32))
    assert list(bits) == [0x3F80, 0x3F81, 0xBF80]
    # Random values: within half a bf16 step (2^-8 relative) of the input,
    # and no farther than the truncated pattern or the one above it.
    rng = np.random.Generator(np.random.PCG64(3))
    x = rng.standard_normal(10000).astype(np.float32)
    y = workloads.bf16_bits_to_f32(workloads.f32_to_bf16_bits(x)).astype(np.float64)
    assert np.all(np.abs(y - x) <= np.abs(x) * 2.0 ** -8)
    trunc = (x.view(np.uint32) >> 16).astype(np.uint16)
    lo = workloads.bf16_bits_to_f32(trunc).astype(np.float64)
    hi = workloads.bf16_bits_to_f32(trunc + np.uint16(1)).astype(np.float64)
    assert np.all(np.abs(y - x) <= np.minimum(np.abs(lo - x), np.abs(hi - x)))


def test_fp16_variant_is_numpy_half():
    q16, _, _ = workloads.generate_shape(1, 1, 8, 16, seed=4, dtype="f16")
    rng = np.random.Generator(np.random.PCG64(4))
    x = rng.standard_normal(size=(1, 1, 8, 16), dtype=np.float32)
    assert np.array_equal(q16, x.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("w", workloads.WORKLOADS + workloads.VARIANT_WORKLOADS,
                         ids=lambda w: w.name)
def test_sampled_rows_hold_the_boundaries(w):
    rows = workloads.sampled_rows(w)
    assert rows.dtype == np.int64
    assert np.all(np.diff(rows) > 0) and rows[0] >= 0 and rows[-1] < w.N
    if w.rows == "all":
        assert rows.size == w.N
        return
    last_tile = ((w.N - 1) // 128) * 128
    for r in (0, 1, 127, 128, 255, 256, last_tile, w.N - 1):
        assert r in rows
    assert 512 <= rows.size <= 512 + 8


def test_workload_table():
    names = [w.name for w in workloads.WORKLOADS]
    assert names[2] == "b2h16n4096d128_causal" and workloads.HEADLINE is workloads.WORKLOADS[2]
    h = workloads.HEADLINE
    assert (h.B, h.H, h.N, h.d, h.causal) == (2, 16, 4096, 128, True)
    assert h.scale == pytest.approx(1.0 / math.sqrt(128))
    assert h.flops == pytest.approx(137.438953472e9)
    assert h.io_bytes == 4 * 2 * 16 * 4096 * 128 * 2 + 2 * 16 * 4096 * 4
    assert workloads.by_name("b1h32n8192d128_causal_qk3").qk_std == 3.0
    dec = workloads.by_name("decode_b4h16q16k16384d128_causal")
    assert (dec.B, dec.H, dec.Nq, dec.Nk, dec.d, dec.causal) == (4, 16, 16, 16384, 128, True)
    with pytest.raises(KeyError):
        workloads.by_name("no such workload")
