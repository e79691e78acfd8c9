"""Tiled online-softmax attention in fp64 — TEST INFRASTRUCTURE (oracle side).

A second, independent restatement of the method, kept deliberately plain:
numpy fp64, no fusion beyond what the pages' algorithm states, every step a
module-level function so a test can replace one step with a deliberately
broken version (the bug catalogue of the pwwt.cn walkthrough, §4.1-§4.5) and
check that the comparison against the definition (``oracle.attention``)
catches it.

Two loop orders are restated:

* :func:`attention_q_outer` — query tiles outer, K/V tiles inner, an
  unnormalised accumulator divided by ``l`` once at the end.  Steps follow the
  forward pseudocode of the pwwt.cn walkthrough §2.2 and the loop order of
  "Online Softmax and FlashAttention" (course unit 12: "Q/O stay, K/V move"),
  including the causal tile classes of that page (fully-future tiles skipped,
  diagonal tiles masked element by element).
* :func:`attention_kv_outer` — K/V tiles outer, query tiles inner, the
  normalised output updated in place by eq. (37) of "Parsing FlashAttention
  (2): FlashAttention-v1 forward pass" §3.9-§3.12 (Algorithm 1, §4); with
  ``block_k == 1`` each step is the scalar update eq. (36) of §3.8.

Inputs are fp64 arrays ``q, k, v`` shaped ``[N, d]`` (one head).  Outputs are
``(O [N, d], LSE [N])`` with ``LSE = m + ln(l)``.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


# ---------------------------------------------------------------- statistics

def initial_max(rows: int) -> np.ndarray:
    """Running max starts at -inf (walkthrough §2.2; page 1 §4 init)."""
    return np.full(rows, NEG_INF)


def initial_sum(rows: int) -> np.ndarray:
    """Running exponent sum starts at 0."""
    return np.zeros(rows)


def merge_stats(m_a, l_a, m_b, l_b):
    """Block merge of two (max, exponent-sum) states onto a common base.

    page 1 eqs (17)-(20); "Online Softmax and FlashAttention", block-merge
    passage: m = max(m_a, m_b), l = l_a e^(m_a - m) + l_b e^(m_b - m).
    """
    m = np.maximum(m_a, m_b)
    return m, l_a * np.exp(m_a - m) + l_b * np.exp(m_b - m)


def combine_partials(o_parts, lse_parts):
    """Merge attention results computed over disjoint key subsets.

    o_parts[s] is the normalised output of subset s and lse_parts[s] its
    log-sum-exp (-inf for a subset with no visible key).  The block-merge
    identity (page 1 eq. (20); "Online Softmax and FlashAttention") with
    l_s = e^(LSE_s - m_s) gives LSE = ln sum_s e^(LSE_s) and
    O = sum_s e^(LSE_s - LSE) O_s.  Shapes: o_parts [S, ..., d],
    lse_parts [S, ...]; returns (O [..., d], LSE [...]).
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    w = np.exp(lse_parts - m)  # 0 for empty subsets
    total = w.sum(axis=0)
    lse = m + np.log(total)
    o = (np.where(w[..., None] > 0, o_parts, 0.0) * (w / total)[..., None]).sum(axis=0)
    return o, lse


def stream_stats(x):
    """Online max/sum over a vector one element at a time (the prefix
    recurrence of "Online Softmax and FlashAttention"): m_t = max(m_{t-1},
    x_t), l_t = l_{t-1} e^(m_{t-1} - m_t) + e^(x_t - m_t)."""
    m, l = NEG_INF, 0.0
    for xt in np.asarray(x, dtype=np.float64):
        m_new = max(m, xt)
        l = l * np.exp(m - m_new) + np.exp(xt - m_new)
        m = m_new
    return m, l


# ---------------------------------------------------------------- tile steps

def tile_scores(q_tile, k_tile, scale):
    """S_ij = scale * Q_i K_j^T for one tile pair (fp64)."""
    return scale * (q_tile @ k_tile.T)


def mask_tile(s, q_idx, k_idx, n_keys, causal):
    """-inf for padding keys past the end (walkthrough §4.2, §4.5: pad with
    -inf, never 0) and, when causal, for every future key j > i."""
    s = s.copy()
    s[:, k_idx >= n_keys] = NEG_INF
    if causal:
        s[k_idx[None, :] > q_idx[:, None]] = NEG_INF
    return s


def tile_is_future(q_start, q_end, k_start, causal):
    """A tile whose smallest key index is not below the query tile's end is
    entirely above the diagonal and is skipped (no load, no compute);
    half-open intervals [q_start, q_end), [k_start, k_end)."""
    return bool(causal) and k_start >= q_end


def max_and_alpha(m_old, s):
    """New running max and the rescale factor for the old state.  alpha is
    computed from the OLD max before the max is replaced (walkthrough
    §4.5)."""
    m_new = np.maximum(m_old, s.max(axis=1))
    alpha = np.exp(m_old - m_new)
    return m_new, alpha


def tile_probs(s, m_new):
    """Unnormalised probabilities P~ = exp(S - m_new) of the tile."""
    return np.exp(s - m_new[:, None])


def update_sum(l, alpha, p):
    """l <- l * alpha + rowsum(P~)."""
    return l * alpha + p.sum(axis=1)


def update_acc(acc, alpha, p, v_tile):
    """Rescale the accumulator first, then add the tile's P~ V (walkthrough
    §4.2: the rescale must precede the add)."""
    return acc * alpha[:, None] + p @ v_tile


def finish(acc, l, m):
    """O = acc / l and LSE = m + ln l."""
    return acc / l[:, None], m + np.log(l)


# ---------------------------------------------------------------- drivers

def _padded(x, block):
    n = x.shape[0]
    n_pad = -(-n // block) * block
    if n_pad == n:
        return x
    # Padding rows are zero, as a tile load past the end would read; their
    # scores are masked to -inf by mask_tile.
    out = np.zeros((n_pad,) + x.shape[1:], dtype=x.dtype)
    out[:n] = x
    return out


def attention_q_outer(q, k, v, scale, causal, block_q, block_k):
    """Q tiles outer, K/V tiles inner; unnormalised accumulator."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape
    kp, vp = _padded(k, block_k), _padded(v, block_k)
    o = np.zeros((n, d))
    lse = np.zeros(n)
    for q_start in range(0, n, block_q):
        q_end = min(q_start + block_q, n)
        q_idx = np.arange(q_start, q_end)
        q_tile = q[q_start:q_end]
        rows = q_end - q_start
        m = initial_max(rows)
        l = initial_sum(rows)
        acc = np.zeros((rows, d))
        for k_start in range(0, kp.shape[0], block_k):
            if tile_is_future(q_start, q_end, k_start, causal):
                continue
            k_idx = np.arange(k_start, k_start + block_k)
            s = tile_scores(q_tile, kp[k_start:k_start + block_k], scale)
            s = mask_tile(s, q_idx, k_idx, n, causal)
            m, alpha = max_and_alpha(m, s)
            p = tile_probs(s, m)
            l = update_sum(l, alpha, p)
            acc = update_acc(acc, alpha, p, vp[k_start:k_start + block_k])
        o[q_start:q_end], lse[q_start:q_end] = finish(acc, l, m)
    return o, lse


def attention_kv_outer(q, k, v, scale, causal, block_q, block_k):
    """K/V tiles outer, Q tiles inner; the normalised output and its (m, l)
    are read and rewritten on every inner step, eq. (37):

        m_new = max(m, m~),  l_new = e^(m - m_new) l + e^(m~ - m_new) l~
        O_i  <- diag(l_new)^-1 (diag(l) e^(m - m_new) O_i + e^(m~ - m_new) P~ V_j)

    where m~ = rowmax(S_ij), P~ = exp(S_ij - m~), l~ = rowsum(P~).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape
    kp, vp = _padded(k, block_k), _padded(v, block_k)
    o = np.zeros((n, d))
    l = np.zeros(n)
    m = np.full(n, NEG_INF)
    for k_start in range(0, kp.shape[0], block_k):
        k_idx = np.arange(k_start, k_start + block_k)
        k_tile = kp[k_start:k_start + block_k]
        v_tile = vp[k_start:k_start + block_k]
        for q_start in range(0, n, block_q):
            q_end = min(q_start + block_q, n)
            if tile_is_future(q_start, q_end, k_start, causal):
                continue
            q_idx = np.arange(q_start, q_end)
            s = mask_tile(tile_scores(q[q_start:q_end], k_tile, scale), q_idx, k_idx, n, causal)
            m_tilde = s.max(axis=1)
            # A row of this tile may be fully masked (all keys in its
            # future); it contributes nothing: its weights are exactly 0.
            live = m_tilde > NEG_INF
            p_tilde = np.zeros_like(s)
            p_tilde[live] = np.exp(s[live] - m_tilde[live, None])
            l_tilde = p_tilde.sum(axis=1)
            m_i, l_i, o_i = m[q_start:q_end], l[q_start:q_end], o[q_start:q_end]
            m_new = np.maximum(m_i, m_tilde)
            old = np.where(np.isneginf(m_i), 0.0, np.exp(m_i - m_new))
            new = np.where(live, np.exp(m_tilde - m_new), 0.0)
            l_new = old * l_i + new * l_tilde
            o_new = ((l_i * old)[:, None] * o_i + new[:, None] * (p_tilde @ v_tile)) / l_new[:, None]
            o[q_start:q_end] = o_new
            l[q_start:q_end] = l_new
            m[q_start:q_end] = m_new
    return o, m + np.log(l)
