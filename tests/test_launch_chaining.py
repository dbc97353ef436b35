"""Back-to-back calls on one stream, with no synchronisation between them.

The library's kernels may be launched so that one starts its prologue while
the previous kernel in the stream finishes; each waits for that kernel before
reading or writing global memory.  These chains make every call depend on the
one before it -- reading its output (read after write) or overwriting a buffer
it reads (write after read) -- and compare with the same calls run with a
synchronisation after each: the results must be identical bit for bit."""
import pytest
import torch

from sdpa_inputs import make_qkv

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

# one-tile layout (few units at D=64), two-tile layout (D=128), a larger D=64
SHAPES = [(2, 4, 4, 256, 64), (1, 8, 2, 384, 128), (8, 16, 4, 1000, 64)]


def _qkv(seed, B, H, Hkv, S, D):
    x = make_qkv(seed, B, H, Hkv, S, S, D, "bf16")
    return (t.to(DEV) for t in (x.q, x.k, x.v))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_each_call_reads_the_previous_output(shape):
    from scaled_dot_product_05_gb300 import sdpa_fwd
    B, H, Hkv, S, D = shape
    q, k, v = _qkv(500 + D, *shape)
    if Hkv != H:                      # O has Hq heads: the chain needs K, V with as many
        k = k.repeat_interleave(H // Hkv, dim=2).contiguous()
        v = v.repeat_interleave(H // Hkv, dim=2).contiguous()
    n = 40
    chained = [q]
    for i in range(n):
        chained.append(sdpa_fwd(chained[-1], k, v, causal=(i % 2 == 0)))
    torch.cuda.synchronize()
    step = [q]
    for i in range(n):
        step.append(sdpa_fwd(step[-1], k, v, causal=(i % 2 == 0)))
        torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(chained, step))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_each_call_overwrites_what_the_previous_reads(shape):
    from scaled_dot_product_05_gb300 import sdpa_fwd
    B, H, Hkv, S, D = shape
    q, k, v = _qkv(600 + D, *shape)
    n = 40
    # call i reads bufs[i] and writes bufs[i + 1]'s successor slot, which
    # call i + 1 then overwrites while call i may still be reading bufs[i]
    srcs = [q * (1.0 + 0.01 * i) for i in range(n + 1)]
    bufs = [s.clone() for s in srcs]
    outs = [torch.empty_like(q) for _ in range(n)]
    for i in range(n):
        sdpa_fwd(bufs[i], k, v, outs[i], causal=True)
        if i + 1 < n:
            # overwrite the input of call i with another call's output, right behind it
            sdpa_fwd(bufs[i + 1], k, v, bufs[i], causal=False)
    torch.cuda.synchronize()
    ref = []
    for i in range(n):
        o = torch.empty_like(q)
        sdpa_fwd(srcs[i], k, v, o, causal=True)
        torch.cuda.synchronize()
        ref.append(o)
    assert all(torch.equal(a, b) for a, b in zip(outs, ref))


def test_backward_chain_of_short_calls():
    # short backward calls (their three kernels launched back to back with
    # programmatic serialization), each reading the previous call's dQ as its
    # dO: identical to the same calls with a synchronisation after each
    from scaled_dot_product_05_gb300 import sdpa_bwd, sdpa_fwd_ex
    B, H, S, D = 1, 4, 256, 64
    q, k, v = _qkv(700, B, H, H, S, D)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=DEV)
    sdpa_fwd_ex(q, k, v, o, lse, causal=True)
    n = 12
    g0 = torch.randn_like(q) * 0.1

    def run(sync):
        g = g0
        res = []
        for _ in range(n):
            dq, dk, dv = sdpa_bwd(q, k, v, o, g, lse, causal=True)
            if sync:
                torch.cuda.synchronize()
            res.append((dq, dk, dv))
            g = (dq / (dq.abs().max() + 1e-3)).contiguous()      # the next dO from this dQ
        torch.cuda.synchronize()
        return res
    a, b = run(False), run(True)
    assert all(torch.equal(x, y) for ra, rb in zip(a, b) for x, y in zip(ra, rb))


def test_cuda_graph_of_chained_calls():
    # the same chains captured in a CUDA graph (programmatic launches become
    # programmatic dependency edges) and replayed: identical to eager calls
    from scaled_dot_product_05_gb300 import sdpa_bwd, sdpa_fwd, sdpa_fwd_ex
    q, k, v = _qkv(800, 2, 4, 4, 256, 64)
    n = 8
    # eager chain, each call reading the previous output as its Q
    eager = [q]
    for i in range(n):
        eager.append(sdpa_fwd(eager[-1], k, v, causal=(i % 2 == 0)))
    torch.cuda.synchronize()
    # captured chain into preallocated outputs
    outs = [torch.empty_like(q) for _ in range(n)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        src = q
        for i in range(n):              # warm-up on the capture stream
            sdpa_fwd(src, k, v, outs[i], causal=(i % 2 == 0))
            src = outs[i]
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for o in outs:
        o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        src = q
        for i in range(n):
            sdpa_fwd(src, k, v, outs[i], causal=(i % 2 == 0))
            src = outs[i]
    g.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(eager[1:], outs))

    # a short backward call (its three kernels chained) in a graph
    B = 1
    qb, kb, vb = q[:B].contiguous(), k[:B].contiguous(), v[:B].contiguous()
    o = torch.empty_like(qb)
    lse = torch.empty((B, 4, 256), dtype=torch.float32, device=DEV)
    sdpa_fwd_ex(qb, kb, vb, o, lse, causal=True)
    do = (torch.randn_like(qb) * 0.1).contiguous()
    from scaled_dot_product_05_gb300 import bwd_workspace_bytes
    ws = torch.empty(bwd_workspace_bytes(B, 4, 256, 64), dtype=torch.uint8, device=DEV)
    ref = sdpa_bwd(qb, kb, vb, o, do, lse, causal=True, workspace=ws)
    torch.cuda.synchronize()
    grads = tuple(torch.empty_like(t) for t in ref)
    with torch.cuda.stream(side):
        sdpa_bwd(qb, kb, vb, o, do, lse, *grads, causal=True, workspace=ws)
    torch.cuda.synchronize()
    for t in grads:
        t.zero_()
    gb = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gb):
        sdpa_bwd(qb, kb, vb, o, do, lse, *grads, causal=True, workspace=ws)
    gb.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(ref, grads))
