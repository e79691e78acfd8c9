"""Seeded synthetic attention inputs shared by the tests, the benchmark and
the smoke check.

This module holds no attention arithmetic: it only draws Q, K, V and picks
the rows that large cases check one by one.  Both the oracle side and the
CUDA side receive the same bf16 bit patterns from here.

Recipe (the same on every machine): numpy ``PCG64(seed)``; Q, K, V drawn in
that order as fp32 ``standard_normal`` of shape ``[B, H, N, d]``; Q and K
multiplied by ``qk_std`` (3.0 for the large-dynamic-range case); each value
rounded to bf16 with round-to-nearest-even on its fp32 bits (or, for the
fp16 variants, to IEEE binary16 by numpy's nearest-even conversion).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    scale: float
    qk_std: float = 1.0
    seed: int = 0
    # "all": the oracle checks every row; "sampled": 512 seeded rows per head
    # plus the boundary rows of the tiling.
    rows: str = "all"
    dtype: str = "bf16"  # element type of Q, K, V, O: "bf16" or "f16"

    @property
    def flops(self) -> float:
        """Nominal attention-forward FLOPs: 4·B·H·N²·d, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V once (bf16), write O (bf16)
        and LSE (fp32) once."""
        return 4 * self.B * self.H * self.N * self.d * 2 + self.B * self.H * self.N * 4


# The five workloads of the method's evaluation, in order.  Index 0 is the
# small case the oracle finishes in well under a second; index 2 is the
# headline (B=2, H=16, N=4096, d=128, causal).
WORKLOADS = (
    Workload("b1h1n256d64", 1, 1, 256, 64, False, 1.0 / 8.0, seed=0, rows="all"),
    Workload("b4h8n1024d64", 4, 8, 1024, 64, False, 1.0 / 8.0, seed=1, rows="all"),
    Workload("b2h16n4096d128_causal", 2, 16, 4096, 128, True, 1.0 / math.sqrt(128), seed=2,
             rows="sampled"),
    Workload("b1h32n8192d128_causal_qk3", 1, 32, 8192, 128, True, 1.0 / math.sqrt(128),
             qk_std=3.0, seed=3, rows="sampled"),
    Workload("b1h16n16000d128_causal", 1, 16, 16000, 128, True, 1.0 / math.sqrt(128), seed=4,
             rows="sampled"),
)

HEADLINE = WORKLOADS[2]

# The headline shape in fp16, at head dimension 96 (a multiple of 16 below
# the 128-column layout), at head dimension 256 and at head dimension 64 (the
# 64-column layout): the element-type and head-dimension variants of the
# forward.
VARIANT_WORKLOADS = (
    Workload("b2h16n4096d128_causal_fp16", 2, 16, 4096, 128, True, 1.0 / math.sqrt(128), seed=7,
             rows="sampled", dtype="f16"),
    Workload("b2h16n4096d96_causal", 2, 16, 4096, 96, True, 1.0 / math.sqrt(96), seed=8,
             rows="sampled"),
    Workload("b2h16n4096d256_causal", 2, 16, 4096, 256, True, 1.0 / 16.0, seed=9,
             rows="sampled"),
    Workload("b2h16n4096d64_causal", 2, 16, 4096, 64, True, 1.0 / 8.0, seed=10,
             rows="sampled"),
)

# Sequence lengths that are not multiples of any tile size, checked at both
# head dimensions, causal and not (B=1, H=2).
RAGGED_N = (1, 17, 127, 129, 1000, 4097)


@dataclass(frozen=True)
class DecodeWorkload:
    """A short block of queries against a long key sequence (split-KV path).
    Causal masking, when set, is aligned to the end of the keys."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    scale: float
    seed: int = 0

    @property
    def flops(self) -> float:
        """4·B·H·Nq·Nk·d (the same count as the square workloads, unmasked)."""
        return 4.0 * self.B * self.H * self.Nq * self.Nk * self.d

    @property
    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V once (bf16), write O (bf16)
        and LSE (fp32) once."""
        bh = self.B * self.H
        return bh * (2 * self.Nq * self.d * 2 + 2 * self.Nk * self.d * 2 + self.Nq * 4)


# Decode: one (and sixteen) new queries per head against a 16384-key cache;
# K and V (268 MB) exceed L2, so the path is bound by HBM.
DECODE_WORKLOADS = (
    DecodeWorkload("decode_b4h16q1k16384d128", 4, 16, 1, 16384, 128, False,
                   1.0 / math.sqrt(128), seed=5),
    DecodeWorkload("decode_b4h16q16k16384d128_causal", 4, 16, 16, 16384, 128, True,
                   1.0 / math.sqrt(128), seed=6),
)


def by_name(name: str):
    for w in WORKLOADS + VARIANT_WORKLOADS + DECODE_WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def generate_decode(w: DecodeWorkload):
    """Return ``(q [B,H,Nq,d], k [B,H,Nk,d], v [B,H,Nk,d])`` as uint16 bf16
    bit patterns: one PCG64(seed) stream draws q, then k, then v (fp32
    standard normal, rounded to bf16)."""
    rng = np.random.Generator(np.random.PCG64(w.seed))
    out = []
    for n in (w.Nq, w.Nk, w.Nk):
        x = rng.standard_normal(size=(w.B, w.H, n, w.d), dtype=np.float32)
        out.append(f32_to_bf16_bits(x))
    return tuple(out)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16
    bit patterns.  Inputs must be finite."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (for display/tests)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to IEEE binary16 (numpy, nearest even); returns
    uint16 bit patterns."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def generate(w: Workload):
    """Return ``(q, k, v)`` as uint16 bit patterns ``[B, H, N, d]`` of the
    workload's element type."""
    return generate_shape(w.B, w.H, w.N, w.d, seed=w.seed, qk_std=w.qk_std, dtype=w.dtype)


def generate_shape(B: int, H: int, N: int, d: int, seed: int, qk_std: float = 1.0,
                   dtype: str = "bf16"):
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (B, H, N, d)
    to_bits = f32_to_f16_bits if dtype == "f16" else f32_to_bf16_bits
    out = []
    for mult in (qk_std, qk_std, 1.0):
        x = rng.standard_normal(size=shape, dtype=np.float32)
        if mult != 1.0:
            x *= np.float32(mult)
        out.append(to_bits(x))
    return tuple(out)


def sampled_rows(w: Workload, count: int = 512, tile: int = 128) -> np.ndarray:
    """Seeded random query rows (the same set for every head) plus the
    boundary rows: 0, 1, tile-1, tile, 2*tile-1, 2*tile, the first and last
    row of the last tile, and N-1.  Sorted, unique, all in [0, N)."""
    if w.rows == "all":
        return np.arange(w.N, dtype=np.int64)
    rng = np.random.Generator(np.random.PCG64(1000 + w.seed))
    picked = rng.permutation(w.N)[:count]
    last_tile = ((w.N - 1) // tile) * tile
    forced = [0, 1, tile - 1, tile, 2 * tile - 1, 2 * tile, last_tile, w.N - 1]
    rows = np.unique(np.concatenate([picked, [r for r in forced if 0 <= r < w.N]]))
    return rows.astype(np.int64)


def as_torch_bf16(bits: np.ndarray):
    """View uint16 bf16 bit patterns as a CPU ``torch.bfloat16`` tensor
    (no copy of the values' meaning; bits are reinterpreted)."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def as_torch(bits: np.ndarray, dtype: str = "bf16"):
    """View uint16 bit patterns as a CPU tensor of ``dtype`` ("bf16" or
    "f16"); the bits are reinterpreted, not converted."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def torch_bf16_to_bits(t) -> np.ndarray:
    """Inverse of :func:`as_torch_bf16` for a CPU tensor."""
    import torch

    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
