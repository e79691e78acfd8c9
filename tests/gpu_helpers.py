"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI on seeded inputs and compare with the oracle element by element."""
from __future__ import annotations

import numpy as np

import oracle
import workloads

# Acceptance tolerance for bf16 inputs, fp32 accumulation and bf16 output:
# |O_gpu - O_ref| <= 1e-2 * (1 + |O_ref|) elementwise, |LSE_gpu - LSE_ref| <= 1e-3.
O_ATOL = 1e-2
O_RTOL = 1e-2
LSE_ATOL = 1e-3


def to_device(bits, device):
    return workloads.as_torch_bf16(bits).to(device)


def run_cuda(q, k, v, causal, scale, device):
    import torch

    import tiled_attention_forward_attn_gb300 as fa

    qd, kd, vd = (to_device(a, device) for a in (q, k, v))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize(device)
    return o, lse


def compare(o_gpu, lse_gpu, o_ref, lse_ref, label=""):
    """Elementwise check; returns (max |dO| / (1+|O|), max |dLSE|)."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    assert np.all(np.isfinite(o_gpu)), f"{label}: non-finite O"
    assert np.all(np.isfinite(lse_gpu)), f"{label}: non-finite LSE"
    o_err = np.abs(o_gpu - o_ref) / (1.0 + np.abs(o_ref))
    lse_err = np.abs(lse_gpu - lse_ref)
    worst_o = float(o_err.max())
    worst_l = float(lse_err.max())
    assert worst_o <= O_ATOL, f"{label}: max |dO|/(1+|O|) = {worst_o:.3e}"
    assert worst_l <= LSE_ATOL, f"{label}: max |dLSE| = {worst_l:.3e}"
    return worst_o, worst_l


def check_against_oracle(q, k, v, causal, scale, device, rows=None, label=""):
    """Run the CUDA path on (q, k, v) and compare the given rows (all rows
    when None) of every head with the oracle."""
    o, lse = run_cuda(q, k, v, causal, scale, device)
    o_np = o.float().cpu().numpy()
    lse_np = lse.cpu().numpy()
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale, rows=rows)
    if rows is not None:
        o_np = o_np[:, :, rows, :]
        lse_np = lse_np[:, :, rows]
    return compare(o_np, lse_np, o_ref, lse_ref, label)
