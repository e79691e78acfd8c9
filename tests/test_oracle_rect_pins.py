"""Pins for the oracle's rectangular form (Nq queries against Nk keys, causal
masking aligned to the end of the keys) and for the split-combine
restatement used by the split-KV path.

R1  torch SDPA in fp64 with an explicit end-aligned mask (library routine)
R2  a single query sees every key: causal equals non-causal exactly
R3  end alignment: the last Nq rows of square attention are the rectangular
    result for those queries, bit for bit
R4  combining results over disjoint key subsets (page 1 eq. (20) block merge)
    reproduces the full result, including subsets with no visible key
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from oracle import online


def _widen(*arrs):
    return [workloads.bf16_bits_to_f32(a).astype(np.float64) for a in arrs]


def _qkv(B, H, Nq, Nk, d, seed):
    q = workloads.generate_shape(B, H, Nq, d, seed=seed)[0]
    _, k, v = workloads.generate_shape(B, H, Nk, d, seed=seed + 1)
    return q, k, v


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 300), (5, 77), (64, 300), (40, 40)])
def test_r1_matches_sdpa_with_end_aligned_mask(Nq, Nk, causal):
    torch = pytest.importorskip("torch")
    d = 32
    q, k, v = _qkv(2, 2, Nq, Nk, d, seed=Nq * 7 + Nk)
    scale = 1.0 / math.sqrt(d)
    O, LSE = oracle.attention(q, k, v, causal, scale)
    qt, kt, vt = [torch.from_numpy(a) for a in _widen(q, k, v)]
    allowed = torch.ones(Nq, Nk, dtype=torch.bool)
    if causal:
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        allowed = j <= (Nk - Nq) + i
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=allowed, scale=scale)
    assert np.max(np.abs(O - ref.numpy())) <= 1e-12
    s = (scale * (qt @ kt.transpose(-1, -2))).masked_fill(~allowed, -math.inf)
    assert np.max(np.abs(LSE - torch.logsumexp(s, dim=-1).numpy())) <= 1e-12


def test_r2_single_query_sees_every_key():
    q, k, v = _qkv(1, 3, 1, 513, 64, seed=9)
    Oc, Lc = oracle.attention(q, k, v, True, 0.125)
    On, Ln = oracle.attention(q, k, v, False, 0.125)
    assert np.array_equal(Oc, On) and np.array_equal(Lc, Ln)


@pytest.mark.parametrize("Nq", [1, 7, 64])
def test_r3_end_alignment_matches_square_tail(Nq):
    N, d = 200, 32
    q, k, v = workloads.generate_shape(1, 2, N, d, seed=31)
    O_sq, L_sq = oracle.attention(q, k, v, True, 0.2)
    O_r, L_r = oracle.attention(np.ascontiguousarray(q[:, :, N - Nq:]), k, v, True, 0.2)
    assert np.array_equal(O_r, O_sq[:, :, N - Nq:])
    assert np.array_equal(L_r, L_sq[:, :, N - Nq:])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("bounds", [[0, 100], [0, 37, 100], [0, 1, 50, 64, 90, 100]])
def test_r4_combining_key_subsets_reproduces_the_whole(bounds, causal):
    Nq, Nk, d = 16, 100, 32
    q, k, v = _qkv(1, 2, Nq, Nk, d, seed=41)
    O, LSE, P = oracle.attention(q, k, v, causal, 0.3, return_probs=True)
    vf = _widen(v)[0]
    o_parts, lse_parts = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        mass = P[..., a:b].sum(-1)  # probability mass of the subset
        with np.errstate(divide="ignore", invalid="ignore"):
            o_s = np.einsum("bhqk,bhkd->bhqd", P[..., a:b], vf[:, :, a:b]) / mass[..., None]
            lse_s = LSE + np.log(mass)  # -inf where no key of the subset is visible
        o_parts.append(np.where(mass[..., None] > 0, o_s, 0.0))
        lse_parts.append(lse_s)
    if causal and len(bounds) > 3:
        assert np.isneginf(np.array(lse_parts)).any()  # an empty subset is exercised
    O_c, LSE_c = online.combine_partials(o_parts, lse_parts)
    assert np.max(np.abs(O_c - O)) <= 1e-12
    assert np.max(np.abs(LSE_c - LSE)) <= 1e-12
