"""Pins for the oracle: it is checked against what the pages print and what
the mathematics fixes, never against itself.

P1  worked safe-softmax example (page "Online Softmax and FlashAttention")
P2  block-merge identity (page 1 eq. (20); same page 2 example)
P3  tile/concatenation equivalence of Q K^T, bit-exact on integers
P4  every probability row sums to 1
P5  causal mask: exact zeros for j > i; row 0 attends only to key 0
P6  closed forms (scale 0, V = 1, identical keys)
P7  library special case: torch SDPA in fp64 on the CPU
P8  the tiled online restatements reach the definition; each bug of the
    pwwt.cn walkthrough's catalogue (§4.1-§4.5), planted in the oracle's
    online restatement, is caught by the same comparison.
"""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
import workloads
from oracle import online

GOLDEN_DIR = os.path.join(os.path.dirname(__file__), "golden")
with open(os.path.join(GOLDEN_DIR, "worked_softmax.json")) as f:
    WORKED = json.load(f)


def _exp_decimal(x: float) -> Decimal:
    getcontext().prec = 50
    return Decimal(x).exp()


# ------------------------------------------------------------------ widening

def test_bf16_widening_known_patterns():
    # IEEE bf16 facts: sign/exponent/mantissa of a few patterns.
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3F81: 1.0078125, 0x0000: 0.0,
             0x7F7F: 3.3895313892515355e38, 0x0001: 2.0 ** -133}
    got = oracle.bf16_to_f64(np.array(list(cases), dtype=np.uint16))
    assert got.tolist() == list(cases.values())


def test_input_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(4096) * 10.0 ** rng.integers(-6, 6, 4096)).astype(np.float32)
    ours = workloads.f32_to_bf16_bits(x)
    ref = workloads.torch_bf16_to_bits(torch.from_numpy(x).to(torch.bfloat16))
    assert np.array_equal(ours, ref)
    # ties go to even: 1 + 2^-8 -> 1.0, 1 + 3*2^-8 -> 1 + 2^-6
    ties = workloads.f32_to_bf16_bits(np.array([1.00390625, 1.01171875], dtype=np.float32))
    assert ties.tolist() == [0x3F80, 0x3F82]


# ------------------------------------------------------------------ P1

def test_p1_worked_example():
    m, shifted, l, p = oracle.safe_softmax(WORKED["x"])
    assert m == WORKED["max"]
    assert shifted.tolist() == WORKED["shifted"]
    l_exact = sum(_exp_decimal(s) for s in WORKED["shifted"])
    assert abs(Decimal(l) - l_exact) <= Decimal("4e-16") * l_exact
    for pj, s in zip(p, WORKED["shifted"]):
        pj_exact = _exp_decimal(s) / l_exact
        assert abs(Decimal(pj) - pj_exact) <= Decimal("4e-16") * pj_exact
    # the largest shifted entry is exactly 0, so its exponent is exactly 1
    assert max(shifted) == 0.0


# ------------------------------------------------------------------ P2

def test_p2_block_merge_worked_example():
    (a, b) = WORKED["blocks"]
    m_a, _, l_a, _ = oracle.safe_softmax(a)
    m_b, _, l_b, _ = oracle.safe_softmax(b)
    assert [m_a, m_b] == WORKED["block_max"]
    m, l = online.merge_stats(m_a, l_a, m_b, l_b)
    assert m == WORKED["merged_max"]
    l_direct = sum(_exp_decimal(s) for s in WORKED["shifted"])
    assert abs(Decimal(float(l)) - l_direct) <= Decimal("1e-15") * l_direct
    # the element-at-a-time recurrence reaches the same state
    m_s, l_s = online.stream_stats(WORKED["x"])
    assert m_s == WORKED["merged_max"]
    assert abs(Decimal(float(l_s)) - l_direct) <= Decimal("1e-15") * l_direct


@pytest.mark.parametrize("seed", range(6))
def test_p2_block_merge_random(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 300))
    x = rng.standard_normal(n) * float(rng.choice([0.1, 1.0, 30.0]))
    cut = int(rng.integers(1, n))
    m_a, _, l_a, _ = oracle.safe_softmax(x[:cut])
    m_b, _, l_b, _ = oracle.safe_softmax(x[cut:])
    m, l = online.merge_stats(m_a, l_a, m_b, l_b)
    m_full, _, l_full, _ = oracle.safe_softmax(x)
    assert m == m_full == x.max()
    assert abs(l - l_full) <= 1e-13 * l_full
    # an independent evaluation of the exponent sum at 50 digits
    l_dec = sum(_exp_decimal(float(v) - float(x.max())) for v in x)
    assert abs(Decimal(l_full) - l_dec) <= Decimal("1e-13") * l_dec


# ------------------------------------------------------------------ P3

def _int_bf16(a):
    return workloads.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def test_p3_tile_concat_exact():
    rng = np.random.default_rng(7)
    Q = rng.integers(-3, 4, size=(4, 4))
    K = rng.integers(-3, 4, size=(5, 4))
    qb, kb = _int_bf16(Q), _int_bf16(K)
    S = oracle.scores(qb, kb)
    # the plain integer product, exact in int64
    assert np.array_equal(S, (Q.astype(np.int64) @ K.astype(np.int64).T).astype(np.float64))
    # two 2x4 query tiles, concatenated along the query (row) axis
    S_rows = np.vstack([oracle.scores(qb[:2], kb), oracle.scores(qb[2:], kb, row_offset=2)])
    assert np.array_equal(S_rows, S)
    # key tiles, concatenated along the key (column) axis
    S_cols = np.hstack([oracle.scores(qb, kb[:2]), oracle.scores(qb, kb[2:])])
    assert np.array_equal(S_cols, S)
    # causal masking in a tile uses absolute query indices
    Sc = oracle.scores(qb[2:], kb, causal=True, row_offset=2)
    for r in range(2):
        for j in range(5):
            if j > r + 2:
                assert Sc[r, j] == -math.inf
            else:
                assert Sc[r, j] == S[r + 2, j]


# ------------------------------------------------------------------ P4 / P5

def _widen(*arrs):
    return [workloads.bf16_bits_to_f32(a).astype(np.float64) for a in arrs]


@pytest.mark.parametrize("causal", [False, True])
def test_p4_rows_sum_to_one(causal):
    q, k, v = workloads.generate_shape(1, 2, 67, 16, seed=11, qk_std=2.0)
    _, _, P = oracle.attention(q, k, v, causal, 0.25, return_probs=True)
    assert np.max(np.abs(P.sum(-1) - 1.0)) <= 1e-12
    assert np.all(P >= 0.0)


def test_p5_causal_zeros_and_first_row():
    q, k, v = workloads.generate_shape(1, 2, 67, 16, seed=12)
    O, LSE, P = oracle.attention(q, k, v, True, 0.25, return_probs=True)
    N = 67
    future = np.triu(np.ones((N, N), dtype=bool), k=1)
    assert np.all(P[..., future] == 0.0)
    assert np.all(P[..., ~future] > 0.0)
    qf, kf, vf = _widen(q, k, v)
    # row 0 sees only key 0: weight 1, output v_0, LSE = s_00
    assert np.array_equal(O[0, :, 0, :], vf[0, :, 0, :])
    s00 = 0.25 * np.einsum("hd,hd->h", qf[0, :, 0, :], kf[0, :, 0, :])
    assert np.allclose(LSE[0, :, 0], s00, rtol=1e-15, atol=1e-15)


# ------------------------------------------------------------------ P6

@pytest.mark.parametrize("causal", [False, True])
def test_p6_scale_zero_is_uniform_average(causal):
    N = 50
    q, k, v = workloads.generate_shape(1, 1, N, 8, seed=13)
    O, LSE = oracle.attention(q, k, v, causal, 0.0)
    vf = _widen(v)[0][0, 0]
    if causal:
        expect = np.cumsum(vf, axis=0) / np.arange(1, N + 1)[:, None]
        lse = np.log(np.arange(1, N + 1))
    else:
        expect = np.broadcast_to(vf.mean(axis=0), (N, 8))
        lse = np.full(N, math.log(N))
    assert np.allclose(O[0, 0], expect, rtol=0, atol=1e-13)
    assert np.allclose(LSE[0, 0], lse, rtol=0, atol=1e-13)


def test_p6_values_all_ones_and_identical_keys():
    N = 40
    q, k, v = workloads.generate_shape(1, 1, N, 8, seed=14, qk_std=3.0)
    ones = workloads.f32_to_bf16_bits(np.ones((1, 1, N, 8), dtype=np.float32))
    O, _ = oracle.attention(q, k, ones, False, 0.5)
    assert np.max(np.abs(O - 1.0)) <= 1e-14
    # every key identical -> every score in a row equal -> uniform weights
    same_k = np.broadcast_to(k[:, :, :1, :], k.shape).copy()
    O_same, LSE_same = oracle.attention(q, same_k, v, False, 0.5)
    O_zero, _ = oracle.attention(q, k, v, False, 0.0)
    assert np.allclose(O_same, O_zero, rtol=0, atol=1e-13)
    qf, kf, _ = _widen(q, same_k, v)
    s_row = 0.5 * qf[0, 0] @ kf[0, 0, 0]
    assert np.allclose(LSE_same[0, 0], s_row + math.log(N), rtol=0, atol=1e-12)


# ------------------------------------------------------------------ P7

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 8), (37, 16), (96, 64)])
def test_p7_matches_torch_sdpa_fp64(causal, N, d):
    torch = pytest.importorskip("torch")
    q, k, v = workloads.generate_shape(2, 3, N, d, seed=N + d, qk_std=1.5)
    scale = 1.0 / math.sqrt(d)
    O, LSE = oracle.attention(q, k, v, causal, scale)
    qt, kt, vt = [torch.from_numpy(a) for a in _widen(q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
    assert np.max(np.abs(O - ref.numpy())) <= 1e-12
    s = scale * (qt @ kt.transpose(-1, -2))
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), -math.inf)
    assert np.max(np.abs(LSE - torch.logsumexp(s, dim=-1).numpy())) <= 1e-12


# ------------------------------------------------------------------ P8

def _one_head(N, d, seed, qk_std=1.0):
    q, k, v = workloads.generate_shape(1, 1, N, d, seed=seed, qk_std=qk_std)
    return (q, k, v), [a[0, 0] for a in _widen(q, k, v)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("blocks", [(1, 1), (3, 3), (7, 5), (64, 64), (64, 128), (128, 128), (131, 131)])
def test_p8_online_q_outer_reaches_definition(causal, blocks):
    bits, (q, k, v) = _one_head(131, 16, seed=21, qk_std=2.0)
    O_ref, LSE_ref = oracle.attention(*bits, causal, 0.3)
    O, LSE = online.attention_q_outer(q, k, v, 0.3, causal, *blocks)
    assert np.max(np.abs(O - O_ref[0, 0])) <= 1e-12
    assert np.max(np.abs(LSE - LSE_ref[0, 0])) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("blocks", [(1, 1), (4, 1), (5, 7), (64, 64), (131, 131)])
def test_p8_online_kv_outer_reaches_definition(causal, blocks):
    bits, (q, k, v) = _one_head(131, 16, seed=22, qk_std=2.0)
    O_ref, LSE_ref = oracle.attention(*bits, causal, 0.3)
    O, LSE = online.attention_kv_outer(q, k, v, 0.3, causal, *blocks)
    assert np.max(np.abs(O - O_ref[0, 0])) <= 1e-12
    assert np.max(np.abs(LSE - LSE_ref[0, 0])) <= 1e-12


def _max_before_alpha(m_old, s):
    m_new = np.maximum(m_old, s.max(axis=1))
    m_old = m_new  # bug: the max is replaced before alpha is taken
    return m_new, np.exp(m_old - m_new)


def _mask_without_padding(s, q_idx, k_idx, n_keys, causal):
    s = s.copy()  # bug: padding keys keep their score of 0
    if causal:
        s[k_idx[None, :] > q_idx[:, None]] = -np.inf
    return s


MUTATIONS = {
    # §4.1 / §4.4: running max initialised to 0 instead of -inf
    "max starts at 0": ("initial_max", lambda rows: np.zeros(rows)),
    # §4.2 / §4.5: padding filled with 0 instead of -inf
    "padding scored 0": ("mask_tile", _mask_without_padding),
    # §4.2: accumulator rescaled after the add instead of before
    "rescale after add": ("update_acc", lambda acc, a, p, v: (acc + p @ v) * a[:, None]),
    # §4.2: exponent sum updated in the wrong order
    "sum rescale order": ("update_sum", lambda l, a, p: (l + p.sum(axis=1)) * a),
    # §4.5: alpha computed after the max was updated
    "alpha after max update": ("max_and_alpha", _max_before_alpha),
    # §4.1: the 1/sqrt(d) scale forgotten
    "scale dropped": ("tile_scores", lambda qt, kt, scale: qt @ kt.T),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_p8_planted_bugs_are_caught(name, monkeypatch):
    attr, broken = MUTATIONS[name]
    N, d = 131, 16
    if name == "max starts at 0":
        # every score near -1000: exp underflows against a max of 0
        q = np.full((N, d), 8.0)
        k = np.full((N, d), -8.0)
        k[::2] = -7.75
        v = _widen(workloads.generate_shape(1, 1, N, d, seed=5)[2])[0][0, 0]
        bits = tuple(workloads.f32_to_bf16_bits(a.astype(np.float32)[None, None]) for a in (q, k, v))
        causal, scale = False, 1.0
    else:
        bits, (q, k, v) = _one_head(N, d, seed=23, qk_std=2.0)
        causal, scale = (name != "padding scored 0"), 0.3
    O_ref, LSE_ref = oracle.attention(*bits, causal, scale)
    ok = online.attention_q_outer(q, k, v, scale, causal, 32, 64)
    assert np.max(np.abs(ok[0] - O_ref[0, 0])) <= 1e-12  # the unbroken restatement passes
    monkeypatch.setattr(online, attr, broken)
    O, LSE = online.attention_q_outer(q, k, v, scale, causal, 32, 64)
    err = np.nan_to_num(np.abs(O - O_ref[0, 0]), nan=np.inf).max()
    err_lse = np.nan_to_num(np.abs(LSE - LSE_ref[0, 0]), nan=np.inf).max()
    assert max(err, err_lse) > 1e-3, f"mutation '{name}' was not caught"
