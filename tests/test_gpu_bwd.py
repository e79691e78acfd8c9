"""GPU parity of the backward pass (fa_bwd, through the C ABI) against the
fp64 oracle's gradients.

Tolerance, from the arithmetic: the gradients are rounded to 16 bits and
are sums over up to N products whose one operand (P or dS) is rounded to
16 bits before the MMA, accumulated in fp32; dS = P (dP - D) also inherits,
through D, the rounding of the forward's O.  The rounding model below
(bwd_rounding_sigma) gives each element's standard deviation; for inputs
with Q, K ~ N(0, 1.5^2) or narrower its largest value relative to 1 + |ref|
is about 6e-3 (bf16), so the fixed bound |dX - ref| <= 3e-2 (1 + |ref|) is
at least five standard deviations there; with the relative Frobenius error
of each gradient (floored at the norm of an all-ones tensor) <= 1e-2.  With
Q, K ~ N(0, 3^2) the model's deviation reaches 1.6e-2 (1 + |ref|) for dQ
and dK (the D term), and those tests check each element against eight of
its own standard deviations instead, when that is larger."""
import math

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

G_ATOL = 3e-2
G_FRO = 1e-2


@pytest.fixture(scope="module")
def fa(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.load_library()
    return fa


def _grads(fa, dev, q, k, v, do, causal, scale, dtype="bf16"):
    import torch

    qd, kd, vd, dod = (workloads.as_torch(a, dtype).to(dev) for a in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize(dev)
    assert fa.fa_get_device_status() == 0
    return [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]


def check_grads(got, ref, label):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert g.shape == r.shape
        assert np.all(np.isfinite(g)), f"{label} {name}: non-finite"
        err = np.abs(g - r)
        worst = float((err / (1.0 + np.abs(r))).max())
        # relative to the reference's norm, floored at that of an all-ones
        # tensor (as the elementwise bound uses 1 + |ref|): with one key,
        # dQ and dK are exactly 0.
        fro = float(np.linalg.norm(err) / max(np.linalg.norm(r), math.sqrt(r.size)))
        assert worst <= G_ATOL, f"{label} {name}: max |d|/(1+|ref|) = {worst:.3e}"
        assert fro <= G_FRO, f"{label} {name}: relative Frobenius error {fro:.3e}"


# Rounding model of the backward (16-bit operands, fp32 accumulation): each
# gradient element is a sum of products one operand of which was rounded to
# 16 bits (P for dV, dS for dQ and dK; relative error at most u, 2^-9 for
# bf16, 2^-11 for fp16, modelled as independent and uniform, variance u^2/3),
# plus the error of D_i = rowsum(dO_i * O_i), which the GPU forms from the
# forward's 16-bit O (O carries the forward's own rounding of P before P.V
# and its final rounding to 16 bits): that error enters dS_ij = P_ij (dP_ij - D_i) as
# -P_ij dD_i, i.e. dQ_i as -scale dD_i (P K)_i and dK_j as
# -scale sum_i P_ij dD_i q_i, plus the final 16-bit rounding of the gradient.
# A value below the smallest normal number is rounded to a fixed spacing
# instead: an absolute error up to h (2^-25 for fp16, whose subnormals are
# 2^-24 apart; negligible for bf16), so x^2 u^2 becomes x^2 u^2 + h^2.
# Errors of P itself (fp32 scores, ex2.approx, fp32 LSE: ~1e-6 relative) and
# of the fp32 accumulation are far below u and left out.  The bound is
# Z_SIGMA standard deviations (or the fixed elementwise bound, if larger).
Z_SIGMA = 8.0


def bwd_rounding_sigma(q, k, v, do, causal, scale, dtype="bf16"):
    """Per-element standard deviation (dQ, dK, dV) of the model above, from
    the oracle's exact probabilities."""
    u = 2.0 ** -9 if dtype == "bf16" else 2.0 ** -11
    hh = 0.0 if dtype == "bf16" else (2.0 ** -25 / u) ** 2  # (h / u)^2
    dec = oracle.bf16_to_f64 if dtype == "bf16" else oracle.f16_to_f64
    Q, K, V, dO = (dec(a) for a in (q, k, v, do))
    _, _, P = oracle.attention(q, k, v, causal, scale, return_probs=True, dtype=dtype)
    O = P @ V
    dP = dO @ np.swapaxes(V, -1, -2)
    D = (dO * O).sum(-1)
    dS = P * (dP - D[..., None])
    # Variance of the error of the GPU's O_it: (u^2/3) (O_it^2 + sum_j P_ij^2 V_jt^2);
    # D_i's error is the sum over t of dO_it times it.
    var_o = (u * u / 3.0) * (O ** 2 + hh + (P ** 2 + hh) @ (V ** 2))
    var_d = ((dO ** 2) * var_o).sum(-1)  # [..., N]
    Pt, dSt = np.swapaxes(P, -1, -2), np.swapaxes(dS, -1, -2)
    dQ = scale * dS @ K
    dK = scale * dSt @ Q
    dV = Pt @ dO
    r = u * u / 3.0
    var_dq = (r * (scale ** 2 * (dS ** 2 + hh) @ (K ** 2) + dQ ** 2 + hh)
              + scale ** 2 * var_d[..., None] * (P @ K) ** 2)
    var_dk = (r * (scale ** 2 * (dSt ** 2 + hh) @ (Q ** 2) + dK ** 2 + hh)
              + scale ** 2 * ((Pt ** 2) * var_d[..., None, :]) @ (Q ** 2))
    var_dv = r * ((Pt ** 2 + hh) @ (dO ** 2) + dV ** 2 + hh)
    return [np.sqrt(x) for x in (var_dq, var_dk, var_dv)]


def check_grads_model(got, ref, sigma, label):
    """Elementwise |d| <= max(G_ATOL (1 + |ref|), Z_SIGMA sigma), and the
    relative Frobenius error as in check_grads."""
    for name, g, r, sg in zip(("dQ", "dK", "dV"), got, ref, sigma):
        assert g.shape == r.shape == sg.shape
        assert np.all(np.isfinite(g)), f"{label} {name}: non-finite"
        err = np.abs(g - r)
        bound = np.maximum(G_ATOL * (1.0 + np.abs(r)), Z_SIGMA * sg)
        worst = float((err / bound).max())
        fro = float(np.linalg.norm(err) / max(np.linalg.norm(r), math.sqrt(r.size)))
        assert worst <= 1.0, f"{label} {name}: max |d| / bound = {worst:.3f}"
        assert fro <= G_FRO, f"{label} {name}: relative Frobenius error {fro:.3e}"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 17, 128, 129, 300, 1000])
def test_bwd_matches_oracle(fa, cuda_device, N, d, causal):
    q, k, v = workloads.generate_shape(1, 2, N, d, seed=1000 + N + d, qk_std=1.5)
    do = workloads.generate_shape(1, 2, N, d, seed=1100 + N + d)[0]
    scale = 1.0 / math.sqrt(d)
    got = _grads(fa, cuda_device, q, k, v, do, causal, scale)
    ref = oracle.attention_bwd(q, k, v, do, causal, scale)
    check_grads(got, ref, f"N{N} d{d} c{causal}")


@pytest.mark.parametrize("causal", [True, False])
def test_bwd_headline_shape_on_four_heads(fa, cuda_device, causal):
    """B=2, H=16, N=4096, d=128 (causal, and without the mask): the GPU
    computes every head; four heads (two per batch) are checked against the
    oracle in full."""
    w = workloads.HEADLINE
    q, k, v = workloads.generate(w)
    do = workloads.generate_shape(w.B, w.H, w.N, w.d, seed=1200)[0]
    got = _grads(fa, cuda_device, q, k, v, do, causal, w.scale)
    heads = [(0, 0), (0, 9), (1, 4), (1, 15)]

    def pick(a):
        return np.stack([a[b, h] for b, h in heads])[None]

    ref = oracle.attention_bwd(pick(q), pick(k), pick(v), pick(do), causal, w.scale)
    check_grads([pick(g) for g in got], ref, f"{w.name} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_bwd_more_tiles_than_sms(fa, cuda_device, d, causal):
    """160 tiles per pass on 152 SMs: the persistent grids give some CTAs a
    second tile (the stationary tile reloaded, accumulators reused), every
    head checked in full."""
    q, k, v = workloads.generate_shape(1, 20, 1000, d, seed=1400 + d, qk_std=1.5)
    do = workloads.generate_shape(1, 20, 1000, d, seed=1500 + d)[0]
    scale = 1.0 / math.sqrt(d)
    got = _grads(fa, cuda_device, q, k, v, do, causal, scale)
    ref = oracle.attention_bwd(q, k, v, do, causal, scale)
    check_grads(got, ref, f"H20 N1000 d{d} causal={causal}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [16, 32, 48, 80, 96, 112])
@pytest.mark.parametrize("N", [129, 300])
def test_bwd_other_head_dims(fa, cuda_device, N, d, causal, dtype):
    """Head dimensions below 64 run in the D = 64 layout, those between 64
    and 128 in the D = 128 one: the columns past d arrive as zeros (they add
    nothing to S or dP) and are never stored."""
    q, k, v = workloads.generate_shape(1, 2, N, d, seed=1800 + N + d, qk_std=1.5, dtype=dtype)
    do = workloads.generate_shape(1, 2, N, d, seed=1900 + N + d, dtype=dtype)[0]
    scale = 1.0 / math.sqrt(d)
    got = _grads(fa, cuda_device, q, k, v, do, causal, scale, dtype=dtype)
    ref = oracle.attention_bwd(q, k, v, do, causal, scale, dtype=dtype)
    check_grads(got, ref, f"{dtype} N{N} d{d} c{causal}")


@pytest.mark.parametrize("d", [48, 96])
def test_bwd_narrow_rows_write_nothing_past_d(fa, cuda_device, d):
    """dQ, dK and dV placed at the very front of larger buffers holding a
    sentinel: the rows are d wide (not the layout's 64 or 128), so a store
    past column d of the last row would land in the sentinel."""
    import torch

    B, H, N = 1, 3, 200
    q, k, v = workloads.generate_shape(B, H, N, d, seed=2000 + d, qk_std=1.5)
    do = workloads.generate_shape(B, H, N, d, seed=2100 + d)[0]
    qd, kd, vd, dod = (workloads.as_torch(a).to(cuda_device) for a in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=True, scale=0.2)
    n = B * H * N * d
    bufs = [torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device=cuda_device)
            for _ in range(3)]
    dq, dk, dv = (b[:n].view(B, H, N, d) for b in bufs)
    fa.fa_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, True, 0.2)
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    for b in bufs:
        assert bool((b[n:] == 7.0).all())
    got = [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]
    check_grads(got, oracle.attention_bwd(q, k, v, do, True, 0.2), f"sentinel d{d}")


def test_bwd_deterministic_and_workspace_checked(fa, cuda_device):
    import torch

    q, k, v = workloads.generate_shape(2, 2, 500, 64, seed=1300)
    do = workloads.generate_shape(2, 2, 500, 64, seed=1301)[0]
    a = _grads(fa, cuda_device, q, k, v, do, True, 0.1)
    b = _grads(fa, cuda_device, q, k, v, do, True, 0.1)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    qd = workloads.as_torch(q).to(cuda_device)
    o, lse = fa.attention_forward(qd, qd, qd, causal=False, scale=0.1)
    grads = [torch.empty_like(qd) for _ in range(3)]
    small = torch.empty(fa.fa_bwd_workspace_bytes(2, 2, 500, 64) - 16, dtype=torch.uint8,
                        device=cuda_device)
    with pytest.raises(fa.FAError) as err:
        fa.fa_bwd(qd, qd, qd, o, lse, qd, *grads, False, 0.1, small)
    assert err.value.code == 10


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [17, 129, 1000])
def test_bwd_fp16_matches_oracle(fa, cuda_device, N, d, causal):
    """fp16 inputs (fa_bwd_ex with FA_DTYPE_FP16): the oracle decodes the
    same binary16 inputs exactly."""
    q, k, v = workloads.generate_shape(1, 2, N, d, seed=1600 + N + d, qk_std=1.5, dtype="f16")
    do = workloads.generate_shape(1, 2, N, d, seed=1700 + N + d, dtype="f16")[0]
    scale = 1.0 / math.sqrt(d)
    got = _grads(fa, cuda_device, q, k, v, do, causal, scale, dtype="f16")
    ref = oracle.attention_bwd(q, k, v, do, causal, scale, dtype="f16")
    check_grads(got, ref, f"fp16 N{N} d{d} c{causal}")


def test_bwd_fp16_headline_shape_on_two_heads(fa, cuda_device):
    """B=2, H=16, N=4096, d=128, causal, fp16: every head computed, two
    checked against the oracle in full."""
    w = workloads.by_name("b2h16n4096d128_causal_fp16")
    q, k, v = workloads.generate(w)
    do = workloads.generate_shape(w.B, w.H, w.N, w.d, seed=1800, dtype="f16")[0]
    got = _grads(fa, cuda_device, q, k, v, do, w.causal, w.scale, dtype="f16")
    heads = [(0, 3), (1, 12)]

    def pick(a):
        return np.stack([a[b, h] for b, h in heads])[None]

    ref = oracle.attention_bwd(pick(q), pick(k), pick(v), pick(do), w.causal, w.scale,
                               dtype="f16")
    check_grads([pick(g) for g in got], ref, w.name)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [300, 1000])
def test_bwd_large_score_range(fa, cuda_device, N, d, causal, dtype):
    """Q, K ~ N(0, 3^2): scaled scores with a standard deviation of about 9,
    as in the 8192-key forward workload that stresses the online softmax;
    P is nearly one-hot and D_i is large, so the error that D takes from the
    16-bit O (times |(P K)_i| ~ |k|) dominates dQ and dK.  Checked against
    the rounding model's per-element bound and the Frobenius bound."""
    q, k, v = workloads.generate_shape(1, 2, N, d, seed=2200 + N + d, qk_std=3.0, dtype=dtype)
    do = workloads.generate_shape(1, 2, N, d, seed=2300 + N + d, dtype=dtype)[0]
    scale = 1.0 / math.sqrt(d)
    got = _grads(fa, cuda_device, q, k, v, do, causal, scale, dtype=dtype)
    ref = oracle.attention_bwd(q, k, v, do, causal, scale, dtype=dtype)
    sigma = bwd_rounding_sigma(q, k, v, do, causal, scale, dtype=dtype)
    check_grads_model(got, ref, sigma, f"qk3 {dtype} N{N} d{d} c{causal}")


def _bnhd(t):
    """t's values in [B, N, H, d] memory, viewed as [B, H, N, d]."""
    return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("N,d", [(333, 64), (200, 128), (129, 96)])
def test_bwd_strided_equals_contiguous(fa, cuda_device, N, d, dtype):
    """Every tensor in [B, N, H, d] memory, and the gradients in row-padded
    buffers: the same kernels on the same values, so the gradients equal the
    contiguous call's bit for bit (and match the oracle); the padding between
    rows stays untouched."""
    import torch

    B, H = 2, 3
    scale = 1.0 / math.sqrt(d)
    q, k, v = workloads.generate_shape(B, H, N, d, seed=5100 + N + d, qk_std=1.5, dtype=dtype)
    do = workloads.generate_shape(B, H, N, d, seed=5200 + N + d, dtype=dtype)[0]
    qd, kd, vd, dod = (workloads.as_torch(a, dtype).to(cuda_device) for a in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=True, scale=scale)
    ref_grads = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=True, scale=scale)

    qs, ks, vs, os_, dos = (_bnhd(t) for t in (qd, kd, vd, o, dod))
    assert not qs.is_contiguous() and qs.stride(2) == H * d
    pads = [torch.full((B, H, N, d + 24), 5.0, dtype=qd.dtype, device=cuda_device)
            for _ in range(3)]
    grads = [pb[..., :d] for pb in pads]
    fa.fa_bwd(qs, ks, vs, os_, lse, dos, *grads, True, scale)
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref_grads):
        assert torch.equal(g, r), name
    for pb in pads:
        assert bool((pb[..., d:] == 5.0).all())
    got = [t.float().cpu().numpy().astype(np.float64) for t in grads]
    check_grads(got, oracle.attention_bwd(q, k, v, do, True, scale, dtype=dtype),
                f"strided N{N} d{d} {dtype}")


def test_bwd_strided_shared_kv_head(fa, cuda_device):
    """K and V shared by every query head (head stride 0): each head's dK and
    dV are that head's own share, equal bit for bit to the call with K and V
    copied into every head."""
    import torch

    B, H, N, d = 2, 4, 257, 128
    q, _, _ = workloads.generate_shape(B, H, N, d, seed=5300, qk_std=1.5)
    _, k1, v1 = workloads.generate_shape(B, 1, N, d, seed=5301, qk_std=1.5)
    do = workloads.generate_shape(B, H, N, d, seed=5302)[0]
    qd, dod = (workloads.as_torch(a).to(cuda_device) for a in (q, do))
    k1d, v1d = (workloads.as_torch(a).to(cuda_device) for a in (k1, v1))
    ke, ve = k1d.expand(B, H, N, d), v1d.expand(B, H, N, d)
    assert ke.stride(1) == 0
    kc, vc = ke.contiguous(), ve.contiguous()
    o, lse = fa.attention_forward(qd, kc, vc, causal=False, scale=0.1)
    want = fa.attention_backward(qd, kc, vc, o, lse, dod, causal=False, scale=0.1)
    got = [torch.empty_like(qd) for _ in range(3)]
    fa.fa_bwd(qd, ke, ve, o, lse, dod, *got, False, 0.1)
    torch.cuda.synchronize(cuda_device)
    assert fa.fa_get_device_status() == 0
    for name, g, w in zip(("dQ", "dK", "dV"), got, want):
        assert torch.equal(g, w), name
