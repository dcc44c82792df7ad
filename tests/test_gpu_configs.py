"""Parity of the full-chunk, reset-stress and sustained workloads (through the C ABI).

Each operation is checked on its own: before a write or a delta rotation the
oracle is re-seeded with the GPU's exported state, so a code that rounds one
step differently cannot compound into later comparisons.  Attention is compared
against the oracle's attention on the GPU's own exported cache, on sampled
heads.  Bars: slots / positions / write serials bit-exact, scales within 1e-6,
codes >= 99.99 % identical and otherwise one step, attention max-abs <= 3e-2 and
mean-abs <= 3e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity_util import check_attention, check_state

pytestmark = pytest.mark.gpu

N, H, D, C, PREFILL = si.PROD_NEW, si.PROD_HEADS, si.PROD_DIM, si.PROD_SLOTS, si.PROD_PREFILL


@pytest.fixture(scope="module")
def rc():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_ring_kv_cache_gb300 as rc
    oracle.build()
    return rc


def _sampled_attention(st, q, qpos, out, heads, what):
    hs = list(heads)
    ref = oracle.attend_image(st["kcodes"][hs], st["kscale"][hs], st["vcodes"][hs], st["vscale"][hs], st["pos"],
                              q[:, hs].cpu(), qpos)
    return check_attention(out[:, hs].cpu().numpy(), ref, what)


class Gpu:
    """The GPU cache plus what the tests need to mirror it: the handle-wide
    write serial (one per write, over all layers) and each layer's last positions."""

    def __init__(self, rc, L, heads):
        self.g = rc.RingKVCache(L, heads, D, C, max_write=C)
        self.writes = 0
        self.last = [np.zeros(0, np.int64)] * L

    def write(self, layer, k, v, pos):
        self.g.write(layer, k, v, pos)
        self.writes += 1
        self.last[layer] = np.asarray(pos, np.int64)


class Mirror:
    """One oracle layer that follows one GPU layer one operation at a time."""

    def __init__(self, heads):
        self.o = oracle.OracleCache(1, heads, D, C)

    def sync_from(self, st, last_pos, delta_total, next_gid):
        self.o.import_layer(0, st, last_pos, delta_total, next_gid)


def test_chunk_workload_sampled_layers(rc):
    # 60 layers, prefill, then two chunks of 4 passes x 60 layers (write 757 +
    # attend) with the window advancing by 757 after each chunk; layers 0, 31
    # and 59 are followed by the oracle
    seed, L = 21, si.PROD_LAYERS
    sampled = (0, 31, 59)
    gp = Gpu(rc, L, H)
    g = gp.g
    mult = si.outlier_mask(H, D, seed)
    kp = si.normal_bf16(PREFILL, H, D, si.subseed(seed, 7), "cuda", mult)
    vp = si.normal_bf16(PREFILL, H, D, si.subseed(seed, 8), "cuda", mult)
    mirrors = {layer: Mirror(H) for layer in sampled}
    for layer in range(L):
        if layer in mirrors:
            mirrors[layer].sync_from(mirrors[layer].o.export(0), np.zeros(0, np.int64), 0, gp.writes)
            mirrors[layer].o.write(0, kp.cpu(), vp.cpu(), np.arange(0, PREFILL))
        gp.write(layer, kp, vp, np.arange(0, PREFILL))
    g.sync()
    for layer in sampled:
        check_state(g.export(layer), mirrors[layer].o.export(0), f"layer {layer} prefill")
    chunk_pos = np.arange(PREFILL, PREFILL + N)
    out = torch.empty(N, H, D, dtype=torch.float32, device="cuda")
    for chunk in range(2):
        for pas in range(si.PROD_PASSES):
            for layer in range(L):
                k, v, q = si.chunk_tensors(seed, chunk, pas, layer, "cuda", mult=mult)
                if layer in mirrors and pas == si.PROD_PASSES - 1:
                    g.sync()
                    m = mirrors[layer]
                    m.sync_from(g.export(layer), gp.last[layer], g.delta_total, gp.writes)
                    m.o.write(0, k.cpu(), v.cpu(), chunk_pos)
                gp.write(layer, k, v, chunk_pos)
                g.attend(layer, q, out)
                if layer in mirrors and pas == si.PROD_PASSES - 1:
                    g.sync()
                    st = g.export(layer)
                    check_state(st, mirrors[layer].o.export(0), f"chunk {chunk} layer {layer} write")
                    if chunk == 1:
                        _sampled_attention(st, q, chunk_pos, out, (0, 17, 40), f"chunk {chunk} layer {layer}")
        # the window restarts: every layer rotates by -757
        g.sync()
        before = {layer: g.export(layer) for layer in sampled}
        g.delta_rotate(-N)
        g.sync()
        for layer in sampled:
            m = mirrors[layer]
            m.sync_from(before[layer], gp.last[layer], g.delta_total + N, gp.writes)
            m.o.delta_rotate(-N)
            check_state(g.export(layer), m.o.export(0), f"chunk {chunk} layer {layer} rotation")
    assert g.delta_total == -2 * N
    g.close()


def test_reset_stress_and_drift(rc):
    # a full ring at positions up to 200,000; 100 x (delta ~ U[-200000, 0],
    # write 757 at the next positions, attend).  Every step is checked against
    # the oracle; separately the stored keys are compared with the exact fp64
    # rotation of their original bf16 rows, by the number of rotations survived.
    seed, Hs = 31, 8
    gp = Gpu(rc, 1, Hs)
    g = gp.g
    m = Mirror(Hs)
    top = 200_000
    p_first = top - C + 1
    k0 = si.normal_bf16(C, Hs, D, si.subseed(seed, 1), "cuda")
    v0 = si.normal_bf16(C, Hs, D, si.subseed(seed, 2), "cuda")
    gp.write(0, k0, v0, np.arange(p_first, top + 1))
    m.o.write(0, k0.cpu(), v0.cpu(), np.arange(p_first, top + 1))
    g.sync()
    check_state(g.export(0), m.o.export(0), "stress fill")
    # per slot: the original bf16 key row and the number of rotations since its write
    korig = np.zeros((C, Hs, D), np.float64)
    age = np.zeros(C, np.int64)
    kk = k0.float().cpu().numpy().astype(np.float64)
    for t in range(C):
        korig[m.o.slot_of(p_first + t)] = kk[t]
    drift = {}
    out = torch.empty(N, Hs, D, dtype=torch.float32, device="cuda")
    next_pos = top + 1
    for step, delta in enumerate(si.stress_deltas(seed, 100)):
        st = g.export(0)
        m.sync_from(st, gp.last[0], g.delta_total, gp.writes)
        g.delta_rotate(delta)
        m.o.delta_rotate(delta)
        g.sync()
        st = g.export(0)
        check_state(st, m.o.export(0), f"stress step {step} rotation")
        age += 1
        next_pos += delta
        if step % 10 == 0:
            # drift of the stored keys against exact re-rotation of their original rows
            occ = st["pos"] != oracle.EMPTY
            exact = oracle.rope_rows(korig[occ].reshape(-1, D), np.repeat(st["pos"][occ], Hs)).reshape(-1, Hs, D)
            got = st["kcodes"][:, occ].transpose(1, 0, 2)
            sc = st["kscale"][:, occ].T[:, :, None].astype(np.float64)
            deq = oracle.e4m3_decode_all()[got] * sc
            # error in units of the group's largest magnitude (448 x its scale)
            rel = np.abs(deq - exact) / (448.0 * sc)
            for a in np.unique(age[occ]):
                sel = age[occ] == a
                r = rel[sel]
                d = drift.setdefault(int(a), [0.0, 0.0, 0])
                d[0] = max(d[0], float(r.max()))
                d[1] += float((r ** 2).sum())
                d[2] += r.size
        k = si.normal_bf16(N, Hs, D, si.subseed(seed, 10, step, 1), "cuda")
        v = si.normal_bf16(N, Hs, D, si.subseed(seed, 10, step, 2), "cuda")
        q = si.normal_bf16(N, Hs, D, si.subseed(seed, 10, step, 3), "cuda")
        pos = np.arange(next_pos, next_pos + N)
        next_pos += N
        m.sync_from(st, gp.last[0], g.delta_total, gp.writes)
        m.o.write(0, k.cpu(), v.cpu(), pos)
        gp.write(0, k, v, pos)
        g.attend(0, q, out)
        g.sync()
        st = g.export(0)
        check_state(st, m.o.export(0), f"stress step {step} write")
        kn = k.float().cpu().numpy().astype(np.float64)
        for t in range(N):
            s = m.o.slot_of(pos[t])
            korig[s] = kn[t]
            age[s] = 0
        if step % 20 == 19:
            _sampled_attention(st, q, pos, out, (0, 5), f"stress step {step}")
    # drift report, in units of the group's largest magnitude: the write and
    # each requantisation add at most half an E4M3 step of the top binade
    # (16/448), measured against a group maximum that a rotation can move by a
    # factor of at most sqrt(2)
    print("rotations survived: max error, rms error (units of the group's largest magnitude)")
    for a in sorted(drift):
        mx, ss, cnt = drift[a]
        print(f"  {a:3d}: {mx:.4f} {np.sqrt(ss / cnt):.5f}")
        assert mx <= (a + 1) * (16.0 / 448.0) * np.sqrt(2.0) + 1e-9
    g.close()


def test_sustained_per_head_std(rc):
    # per-head std U[0.5, 4] for Q, K and V; three chunks of 4 passes on 2 layers
    # with the window restarting at 0 (delta = -oldest position) after each chunk
    seed, L = 41, 2
    std = si.head_std(L, H, seed)
    gp = Gpu(rc, L, H)
    g = gp.g
    mirrors = [Mirror(H) for _ in range(L)]
    for layer in range(L):
        kp = si.normal_bf16(PREFILL, H, D, si.subseed(seed, layer, 7), "cuda", std[layer].view(H, 1))
        vp = si.normal_bf16(PREFILL, H, D, si.subseed(seed, layer, 8), "cuda", std[layer].view(H, 1))
        mirrors[layer].sync_from(mirrors[layer].o.export(0), np.zeros(0, np.int64), 0, gp.writes)
        mirrors[layer].o.write(0, kp.cpu(), vp.cpu(), np.arange(0, PREFILL))
        gp.write(layer, kp, vp, np.arange(0, PREFILL))
    chunk_pos = np.arange(PREFILL, PREFILL + N)
    out = torch.empty(N, H, D, dtype=torch.float32, device="cuda")
    for chunk in range(3):
        for pas in range(si.PROD_PASSES):
            for layer in range(L):
                k, v, q = si.chunk_tensors(seed, chunk, pas, layer, "cuda", std=std[layer])
                g.sync()
                mm = mirrors[layer]
                mm.sync_from(g.export(layer), gp.last[layer], g.delta_total, gp.writes)
                mm.o.write(0, k.cpu(), v.cpu(), chunk_pos)
                gp.write(layer, k, v, chunk_pos)
                g.attend(layer, q, out)
                g.sync()
                st = g.export(layer)
                check_state(st, mm.o.export(0), f"chunk {chunk} pass {pas} layer {layer}")
                if pas == si.PROD_PASSES - 1:
                    _sampled_attention(st, q, chunk_pos, out, (int(torch.argmax(std[layer])), 3),
                                       f"chunk {chunk} layer {layer}")
        befores = [g.export(layer) for layer in range(L)]
        oldest = min(int(b["pos"][b["pos"] != oracle.EMPTY].min()) for b in befores)
        dt = g.delta_total
        g.delta_rotate(-oldest)
        g.sync()
        for layer in range(L):
            mm = mirrors[layer]
            mm.sync_from(befores[layer], gp.last[layer], dt, gp.writes)
            mm.o.delta_rotate(-oldest)
            check_state(g.export(layer), mm.o.export(0), f"chunk {chunk} layer {layer} reset")
    g.close()
