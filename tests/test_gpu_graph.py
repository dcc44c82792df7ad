"""The calls captured into CUDA graphs.

rc_cache_write, rc_attend and rc_cache_delta_rotate launch only kernels, so a
run of them can be captured into a graph and launched later; the host-side
bookkeeping runs at capture time and the graph keeps each call's arguments.
Every graph here is launched once, in the order of capture -- in the pipelined
case the host captures step s + 1 while step s has not run yet, as the bench's
timed region does.  Captured calls must match the oracle with the bars of the
direct path, and leave the cache and the outputs bit for bit as the same calls
made directly do (the same kernels with the same arguments).
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity_util import check_attention, check_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rc():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_ring_kv_cache_gb300 as rc
    oracle.build()
    return rc


def captured(fn):
    """fn's launches as a CUDA graph (captured on a side stream, not launched)."""
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        g.capture_begin(capture_error_mode="thread_local")
        try:
            fn()
        finally:
            g.capture_end()
    return g


def warm(rc, D):
    """One direct call of each kind at this head_dim (kernel attributes are set then)."""
    c = rc.RingKVCache(1, 2, D, 300)
    k, v, q = (si.normal_bf16(16, 2, D, s, "cuda") for s in (1, 2, 3))
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    c.write(0, k, v, np.arange(16))
    c.attend(0, q, out)
    c.delta_rotate(-3)
    c.sync()
    c.close()


@pytest.mark.parametrize("seed", [1, 2])
def test_tiny_schedule_in_graphs(rc, seed):
    s = si.TINY
    warm(rc, s.head_dim)
    g = rc.RingKVCache(s.layers, s.heads, s.head_dim, s.slots)
    o = oracle.OracleCache(s.layers, s.heads, s.head_dim, s.slots)
    keep, step, q = [], 0, None
    for op in si.tiny_schedule():
        if op[0] == "write":
            _, layer, p0, n = op
            k, v, q = si.tiny_tensors(seed, step, "cuda")
            pos = np.arange(p0, p0 + n)
            keep.append(captured(lambda: g.write(layer, k, v, pos)))
            keep[-1].replay()
            o.write(layer, k.cpu(), v.cpu(), pos)
            g.sync()
            check_state(g.export(layer), o.export(layer), f"after captured write {step}")
            step += 1
        elif op[0] == "delta":
            keep.append(captured(lambda: g.delta_rotate(op[1])))
            keep[-1].replay()
            o.delta_rotate(op[1])
            g.sync()
            check_state(g.export(0), o.export(0), "after captured delta")
        else:
            layer = op[1]
            out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
            keep.append(captured(lambda: g.attend(layer, q, out)))
            keep[-1].replay()
            g.sync()
            st = g.export(layer)
            ref = oracle.attend_image(st["kcodes"], st["kscale"], st["vcodes"], st["vscale"], st["pos"], q.cpu(),
                                      o.last_positions(layer), 10000.0)
            check_attention(out.cpu().numpy(), ref, "captured attention")
    g.close()


@pytest.mark.parametrize("D", [128, 64])
def test_pipelined_steps_match_direct(rc, D):
    # steps of (write + attend in every layer, then a delta that moves the
    # window back by one write), as in the bench: the ring advances n slots a
    # step, so every step's arguments differ
    warm(rc, D)
    L, H, C, n, S = 2, 4, 700, 150, 4
    pos = np.arange(C - n, C)
    K = [[si.normal_bf16(n, H, D, 1000 + 10 * s + l, "cuda") for l in range(L)] for s in range(S)]
    V = [[si.normal_bf16(n, H, D, 2000 + 10 * s + l, "cuda") for l in range(L)] for s in range(S)]
    Q = [[si.normal_bf16(n, H, D, 3000 + 10 * s + l, "cuda") for l in range(L)] for s in range(S)]
    kp, vp = si.normal_bf16(C - n, H, D, 7, "cuda"), si.normal_bf16(C - n, H, D, 8, "cuda")
    caches, outs = [], []
    for _ in range(2):
        c = rc.RingKVCache(L, H, D, C, max_write=C)
        for l in range(L):
            c.write(l, kp, vp, np.arange(0, C - n))
        caches.append(c)
        outs.append([[torch.empty(n, H, D, dtype=torch.float32, device="cuda") for _ in range(L)]
                     for _ in range(S)])

    def step(c, out, s):
        for l in range(L):
            c.write(l, K[s][l], V[s][l], pos)
            c.attend(l, Q[s][l], out[s][l])
        c.delta_rotate(-n)

    for s in range(S):
        step(caches[0], outs[0], s)
    keep = [captured(lambda: step(caches[1], outs[1], 0))]
    for s in range(S):
        keep[-1].replay()
        if s + 1 < S:
            keep.append(captured(lambda: step(caches[1], outs[1], s + 1)))
    torch.cuda.synchronize()
    for c in caches:
        c.sync()
    for l in range(L):
        a, b = caches[0].export(l), caches[1].export(l)
        for key in a:
            assert np.array_equal(a[key], b[key]), f"layer {l}: {key} differs between captured and direct calls"
    for s in range(S):
        for l in range(L):
            assert torch.equal(outs[0][s][l], outs[1][s][l]), f"step {s} layer {l}: attention output differs"
    for c in caches:
        c.close()
