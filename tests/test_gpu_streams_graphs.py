"""The entry points under concurrent use and inside CUDA graphs.

The library keeps no per-call state (tensor maps are built on the host for
each call and passed by value; the only shared device state is the status
word), so calls from several host threads on their own streams must give
exactly the results of the same calls made one after another, and a call
captured into a CUDA graph must give, on every replay, exactly what the call
gives eagerly on the inputs present at replay time."""
import math
import threading

import pytest

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import tiled_attention_forward_attn_gb300 as fa
    from tiled_attention_forward_attn_gb300 import _build

    _build.build()
    fa.load_library()
    return fa


def _qkv(dev, B, H, N, d, seed, dtype="bf16"):
    return [workloads.as_torch(a, dtype).to(dev)
            for a in workloads.generate_shape(B, H, N, d, seed=seed, qk_std=1.5, dtype=dtype)]


def test_forward_from_four_threads_on_four_streams(fa, cuda_device):
    """Four host threads, each with its own stream and inputs, call the
    forward eight times each, interleaved: every output equals the result of
    the same call made alone."""
    import torch

    shapes = [(1, 4, 1000, 128, True), (2, 3, 777, 64, False), (1, 2, 2048, 256, True),
              (2, 2, 513, 96, True)]
    inputs = [_qkv(cuda_device, B, H, N, d, 7000 + i) for i, (B, H, N, d, _) in enumerate(shapes)]
    expected = []
    for (B, H, N, d, causal), (q, k, v) in zip(shapes, inputs):
        o, lse = fa.attention_forward(q, k, v, causal=causal, scale=1.0 / math.sqrt(d))
        expected.append((o.clone(), lse.clone()))
    torch.cuda.synchronize(cuda_device)

    results = [None] * len(shapes)
    errors = []

    def worker(i):
        try:
            (B, H, N, d, causal), (q, k, v) = shapes[i], inputs[i]
            stream = torch.cuda.Stream(device=cuda_device)
            outs = []
            with torch.cuda.stream(stream):
                for _ in range(8):
                    o = torch.empty_like(q)
                    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
                    fa.fa_fwd(q, k, v, o, lse, causal, 1.0 / math.sqrt(d), stream=stream)
                    outs.append((o, lse))
            stream.synchronize()
            results[i] = outs
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert fa.fa_get_device_status() == 0
    for i, outs in enumerate(results):
        for o, lse in outs:
            assert torch.equal(o, expected[i][0]) and torch.equal(lse, expected[i][1]), shapes[i]


def test_forward_and_backward_in_a_cuda_graph(fa, cuda_device):
    """Forward and backward (four launches) captured once; each replay, on
    new values written into the captured input buffers, equals eager calls."""
    import torch

    B, H, N, d = 2, 3, 700, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = _qkv(cuda_device, B, H, N, d, 7100)
    do = _qkv(cuda_device, B, H, N, d, 7101)[0]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=cuda_device)

    def step():
        fa.fa_fwd(q, k, v, o, lse, True, scale)
        fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, True, scale, ws)

    side = torch.cuda.Stream(device=cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(side):
        step()  # first calls (function attributes set) outside the capture
    torch.cuda.current_stream(cuda_device).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for rep in range(3):
        nq, nk, nv = _qkv(cuda_device, B, H, N, d, 7200 + 3 * rep)
        ndo = _qkv(cuda_device, B, H, N, d, 7300 + rep)[0]
        for dst, src in ((q, nq), (k, nk), (v, nv), (do, ndo)):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize(cuda_device)
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        eo, else_ = fa.attention_forward(nq, nk, nv, causal=True, scale=scale)
        eg = fa.attention_backward(nq, nk, nv, eo, else_, ndo, causal=True, scale=scale)
        torch.cuda.synchronize(cuda_device)
        for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), got, (eo, else_) + tuple(eg)):
            assert torch.equal(a, b), f"replay {rep}: {name}"
    assert fa.fa_get_device_status() == 0


def test_splitkv_in_a_cuda_graph(fa, cuda_device):
    """A decode step (16 queries against 5000 keys, split-KV with a caller
    workspace) captured once and replayed on new queries."""
    import torch

    B, H, Nq, Nk, d = 2, 4, 16, 5000, 128
    scale = 1.0 / math.sqrt(d)
    q = _qkv(cuda_device, B, H, Nq, d, 7400)[0]
    _, k, v = _qkv(cuda_device, B, H, Nk, d, 7401)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=cuda_device)
    ws = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, 0), dtype=torch.uint8,
                     device=cuda_device)
    side = torch.cuda.Stream(device=cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(side):
        fa.fa_fwd_splitkv(q, k, v, o, lse, True, scale, 0, ws)
    torch.cuda.current_stream(cuda_device).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.fa_fwd_splitkv(q, k, v, o, lse, True, scale, 0, ws)
    for rep in range(3):
        nq = _qkv(cuda_device, B, H, Nq, d, 7500 + rep)[0]
        q.copy_(nq)
        graph.replay()
        torch.cuda.synchronize(cuda_device)
        got = (o.clone(), lse.clone())
        eo, else_ = fa.attention_forward_splitkv(nq, k, v, causal=True, scale=scale)
        torch.cuda.synchronize(cuda_device)
        assert torch.equal(got[0], eo) and torch.equal(got[1], else_), f"replay {rep}"
    assert fa.fa_get_device_status() == 0
