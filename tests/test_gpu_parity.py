"""Parity of the CUDA path (through the C ABI) against the oracle.

Write and delta rotation are compared state against state (slots, positions
and write serials bit-exact; scales within 1e-6; codes >= 99.99 % identical and
otherwise one step).  Attention is compared against the oracle's attention on
the GPU's own exported cache (the same dequantised cache), max-abs <= 3e-2 and
mean-abs <= 3e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity_util import check_attention, check_codes, check_scales, check_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rc():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_ring_kv_cache_gb300 as rc
    oracle.build()
    return rc


def gpu_attend_vs_oracle(cache, layer, Q, qpos, heads=None):
    out = torch.empty(Q.shape, dtype=torch.float32, device="cuda")
    cache.attend(layer, Q, out)
    cache.sync()
    st = cache.export(layer)
    hs = slice(None) if heads is None else heads
    ref = oracle.attend_image(st["kcodes"][hs], st["kscale"][hs], st["vcodes"][hs], st["vscale"][hs], st["pos"],
                              Q[:, hs].cpu(), qpos, cache_base(cache))
    return check_attention(out[:, hs].cpu().numpy(), ref)


def cache_base(cache):
    return 10000.0


class Pair:
    """The GPU cache and the oracle state machine driven in lockstep."""

    def __init__(self, rc, L, H, D, C, max_write=None, readtime=False):
        self.g = rc.RingKVCache(L, H, D, C, max_write=max_write, readtime_ablation=readtime)
        self.o = oracle.OracleCache(L, H, D, C)
        self.L, self.H, self.D, self.C = L, H, D, C

    def write(self, layer, K, V, pos):
        self.g.write(layer, K, V, pos)
        self.o.write(layer, K.cpu(), V.cpu(), pos)

    def delta(self, d):
        self.g.delta_rotate(d)
        self.o.delta_rotate(d)

    def check(self, layer, what):
        self.g.sync()
        return check_state(self.g.export(layer), self.o.export(layer), what)

    def attend_check(self, layer, Q, heads=None):
        return gpu_attend_vs_oracle(self.g, layer, Q, self.o.last_positions(layer), heads)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_tiny_schedule(rc, seed):
    s = si.TINY
    pr = Pair(rc, s.layers, s.heads, s.head_dim, s.slots)
    step, q = 0, None
    for op in si.tiny_schedule():
        if op[0] == "write":
            _, layer, p0, n = op
            k, v, q = si.tiny_tensors(seed, step, "cuda")
            pr.write(layer, k, v, np.arange(p0, p0 + n))
            pr.check(layer, f"after write {step}")
            assert pr.g.occupancy(0) == min(16 * (step + 1), s.slots)
            step += 1
        elif op[0] == "delta":
            pr.delta(op[1])
            pr.check(0, "after delta")
            assert pr.g.delta_total == op[1]
        else:
            pr.attend_check(op[1], q)


@pytest.mark.parametrize("D", [64, 128])
def test_ragged_partial_ring(rc, D):
    # C not a multiple of 128, partially filled ring (masked path), n not a multiple of 128
    H, C = 3, 300
    pr = Pair(rc, 2, H, D, C, max_write=260)
    p = 10
    for i, n in enumerate([1, 17, 200, 31, 260]):
        layer = i % 2
        k = si.normal_bf16(n, H, D, 500 + i, "cuda")
        v = si.normal_bf16(n, H, D, 600 + i, "cuda")
        qq = si.normal_bf16(n, H, D, 700 + i, "cuda")
        pr.write(layer, k, v, np.arange(p, p + n))
        p += n
        pr.check(layer, f"write {i}")
        pr.attend_check(layer, qq)


@pytest.mark.parametrize("D", [64, 128])
def test_split_tiles(rc, D):
    # A full 8-tile ring written as runs whose ends fall at columns 1, 31, 32,
    # 33, 64, 96 and 127 of tiles 0..6 (two write groups per tile), with tile 7
    # holding three groups; neighbouring runs differ 8x in K and 4x in V
    # magnitude, so the two groups of a tile carry different scales.  Then a
    # write that wraps onto slots 0..199 (tile 1 split at column 72) and a
    # delta rotation.
    H, C = 4, 1024
    cuts = [0, 1, 128 + 31, 256 + 32, 384 + 33, 512 + 64, 640 + 96, 768 + 127, 896 + 10, 896 + 70, 1024]
    pr = Pair(rc, 1, H, D, C, max_write=C)
    for i in range(len(cuts) - 1):
        n = cuts[i + 1] - cuts[i]
        ks, vs = (0.25, 0.5) if i % 2 == 0 else (2.0, 2.0)
        k = si.normal_bf16(n, H, D, 900 + i, "cuda", torch.full((H, 1), ks))
        v = si.normal_bf16(n, H, D, 950 + i, "cuda", torch.full((H, 1), vs))
        pr.write(0, k, v, np.arange(cuts[i], cuts[i + 1]))
    pr.check(0, "split runs")
    n_last = cuts[-1] - cuts[-2]
    pr.attend_check(0, si.normal_bf16(n_last, H, D, 990, "cuda"))
    k = si.normal_bf16(200, H, D, 991, "cuda", torch.full((H, 1), 4.0))
    v = si.normal_bf16(200, H, D, 992, "cuda")
    pr.write(0, k, v, np.arange(C, C + 200))
    pr.check(0, "wrapped write")
    q = si.normal_bf16(200, H, D, 993, "cuda")
    pr.attend_check(0, q)
    pr.delta(-C)
    pr.check(0, "after delta")
    pr.attend_check(0, q)


def _rolled(st: dict, r: int) -> dict:
    """An exported layer state with its slot axis rotated: slot s takes slot (s + r) mod C."""
    out = {}
    for k, v in st.items():
        out[k] = np.roll(v, -r, axis=1 if k in ("kcodes", "kscale", "vcodes", "vscale") else 0)
    return out


@pytest.mark.parametrize("D", [64, 128])
def test_copy_window(rc, D):
    # The copy-based window: shifts of the slot axis (k = 37, 123, C - 1, C)
    # between writes (one that wraps), a delta and attends.  The GPU state is
    # the oracle's with the slot axis rotated by the sum of the shifts, and
    # attention equals the oracle's.  C = 300 is not a multiple of 16, so the
    # shifted V chunks straddle the ring's end and its padding.
    H, C = 3, 300
    g = rc.RingKVCache(2, H, D, C, max_write=C, copy_window=True)
    o = oracle.OracleCache(2, H, D, C)
    shift = 0

    def write(layer, p0, n, seed):
        k = si.normal_bf16(n, H, D, seed, "cuda")
        v = si.normal_bf16(n, H, D, seed + 1, "cuda")
        g.write(layer, k, v, np.arange(p0, p0 + n))
        o.write(layer, k.cpu(), v.cpu(), np.arange(p0, p0 + n))

    def check(what):
        g.sync()
        for layer in range(2):
            check_state(g.export(layer), _rolled(o.export(layer), shift % C), f"{what}, layer {layer}")

    def attend(layer, seed):
        q = si.normal_bf16(len(o.last_positions(layer)), H, D, seed, "cuda")
        gpu_attend_vs_oracle(g, layer, q, o.last_positions(layer))

    def window_shift(k):
        nonlocal shift
        g.window_shift(k)
        shift += k

    write(0, 0, 200, 1100)
    write(1, 0, 150, 1110)
    check("first writes")
    attend(0, 1120)
    window_shift(37)
    check("shift 37")
    attend(0, 1121)
    write(0, 200, 100, 1130)
    check("write after shift")
    attend(0, 1131)
    window_shift(123)
    write(1, 150, 271, 1140)   # wraps and overwrites the oldest slots
    check("wrapping write after shift 123")
    attend(1, 1141)
    g.delta_rotate(-100)
    o.delta_rotate(-100)
    check("delta")
    attend(0, 1150)
    window_shift(C - 1)
    write(0, 300, 57, 1160)
    check("write after shift C - 1")
    attend(0, 1161)
    window_shift(C)            # moves nothing
    check("shift C")
    attend(1, 1170)
    g.close()


def test_production_call(rc):
    t = si.production_tensors(11, "cuda")
    C = si.PROD_SLOTS
    pr = Pair(rc, 1, si.PROD_HEADS, si.PROD_DIM, C)
    pr.write(0, t["k_prefill"], t["v_prefill"], np.arange(0, si.PROD_PREFILL))
    pr.write(0, t["k_new"], t["v_new"], np.arange(si.PROD_PREFILL, C))
    pr.check(0, "production state")
    assert pr.g.occupancy(0) == C
    res = pr.attend_check(0, t["q"])
    print("production attention error", res)


@pytest.mark.parametrize("seed", [12, 13])
def test_production_call_sampled_heads(rc, seed):
    t = si.production_tensors(seed, "cuda")
    C = si.PROD_SLOTS
    g = rc.RingKVCache(1, si.PROD_HEADS, si.PROD_DIM, C)
    g.write(0, t["k_prefill"], t["v_prefill"], np.arange(0, si.PROD_PREFILL))
    g.write(0, t["k_new"], t["v_new"], np.arange(si.PROD_PREFILL, C))
    # heads carrying the most outlier channels, and two ordinary ones
    counts = (t["mult"] > 1).sum(1)
    heads = sorted(set(torch.argsort(counts, descending=True)[:4].tolist() + [0, 47]))
    gpu_attend_vs_oracle(g, 0, t["q"], np.arange(si.PROD_PREFILL, C), heads)


def test_delta_one_step_multilayer(rc):
    # three layers, several live write groups (one partly overwritten), then a reset;
    # the oracle runs the delta on the GPU's own pre-rotation state
    L, H, D, C = 3, 4, 128, 1000
    g = rc.RingKVCache(L, H, D, C)
    o = oracle.OracleCache(L, H, D, C)
    p = 0
    for i, n in enumerate([300, 500, 250, 120]):
        for layer in range(L):
            k = si.normal_bf16(n, H, D, 1000 + 10 * i + layer, "cuda", mult=torch.full((H, 1), 1.0 + i))
            v = si.normal_bf16(n, H, D, 2000 + 10 * i + layer, "cuda")
            g.write(layer, k, v, np.arange(p, p + n))
            o.write(layer, k.cpu(), v.cpu(), np.arange(p, p + n))
        p += n
    g.sync()
    before = [g.export(layer) for layer in range(L)]
    for layer in range(L):
        check_state(before[layer], o.export(layer), f"layer {layer} before")
        o.import_layer(layer, before[layer], o.last_positions(layer), o.delta_total, 4)
    for delta in (-137, -99999, 5):
        g.delta_rotate(delta)
        o.delta_rotate(delta)
        g.sync()
        for layer in range(L):
            st = g.export(layer)
            check_state(st, o.export(layer), f"layer {layer} after delta {delta}")
            # re-seed the oracle with the GPU's state: each step is checked on its own
            o.import_layer(layer, st, o.last_positions(layer), o.delta_total, 4)
    assert g.delta_total == -137 - 99999 + 5


@pytest.mark.parametrize("D,C", [(128, 6144), (128, 6200), (64, 10240), (64, 10300)])
def test_delta_both_rotation_kernels(rc, D, C):
    # A CTA of the rotation's cluster of 8 stages its share of a head's tiles
    # in shared memory while that share is at most 6 tiles (D = 128) or 10
    # (D = 64): rings of up to 6,144 / 10,240 slots.  Larger rings take the
    # two-pass kernel.  Both sides of each limit, with a wrapping write and
    # groups of different scales, checked one step at a time.
    H = 2
    g = rc.RingKVCache(1, H, D, C, max_write=C)
    o = oracle.OracleCache(1, H, D, C)
    p = 0
    for i, n in enumerate([C - 700, 900, 450]):
        k = si.normal_bf16(n, H, D, 3000 + i, "cuda", mult=torch.full((H, 1), 0.5 + i))
        v = si.normal_bf16(n, H, D, 3100 + i, "cuda")
        g.write(0, k, v, np.arange(p, p + n))
        o.write(0, k.cpu(), v.cpu(), np.arange(p, p + n))
        p += n
    g.sync()
    st = g.export(0)
    check_state(st, o.export(0), f"C={C} before")
    o.import_layer(0, st, o.last_positions(0), o.delta_total, 4)
    for delta in (-4321, 77):
        g.delta_rotate(delta)
        o.delta_rotate(delta)
        g.sync()
        st = g.export(0)
        check_state(st, o.export(0), f"C={C} after delta {delta}")
        o.import_layer(0, st, o.last_positions(0), o.delta_total, 4)


def test_memory_stable_across_write_sizes(rc):
    C = si.PROD_SLOTS
    g = rc.RingKVCache(1, 8, 128, C)
    torch.cuda.synchronize()
    kmax = si.normal_bf16(C, 8, 128, 1, "cuda")
    qmax = si.normal_bf16(C, 8, 128, 2, "cuda")
    out = torch.empty(C, 8, 128, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    p = 0
    for rep in range(2):
        for n in (1, 17, 489, 757, 5031, C):
            g.write(0, kmax[:n], kmax[:n], np.arange(p, p + n))
            g.attend(0, qmax[:n], out[:n])
            p += n
    g.sync()
    assert torch.cuda.mem_get_info()[0] == free0


def test_errors(rc):
    g = rc.RingKVCache(2, 2, 64, 64, max_write=32)
    k = si.normal_bf16(33, 2, 64, 1, "cuda")
    out = torch.empty(33, 2, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(rc.RcError) as e:
        g.write(0, k, k, np.arange(33))                  # n > max_write
    assert e.value.status == rc.RC_ERR_ARG
    with pytest.raises(rc.RcError) as e:
        g.write(0, k[:2], k[:2], [0, 64])                # same slot twice
    assert e.value.status == rc.RC_ERR_ARG
    with pytest.raises(rc.RcError) as e:
        g.write(2, k[:2], k[:2], [0, 1])                 # no such layer
    assert e.value.status == rc.RC_ERR_ARG
    with pytest.raises(rc.RcError) as e:
        g.attend(0, k[:4], out[:4])                      # nothing written
    assert e.value.status == rc.RC_ERR_STATE
    g.write(0, k[:4], k[:4], np.arange(4))
    with pytest.raises(rc.RcError) as e:
        g.attend(0, k[:5], out[:5])                      # n differs from the last write
    assert e.value.status == rc.RC_ERR_STATE
    with pytest.raises(rc.RcError) as e:
        g.attend_readtime(0, k[:4], out[:4])             # ablation store not kept
    assert e.value.status == rc.RC_ERR_STATE
    g.attend(0, k[:4], out[:4])
    g.sync()
    assert g.occupancy(0) == 4 and g.occupancy(1) == 0


def test_readtime_ablation(rc):
    H, D, C = 4, 128, 700
    g = rc.RingKVCache(1, H, D, C, readtime_ablation=True)
    o = oracle.OracleCache(1, H, D, C)
    kraw = torch.zeros(H, C, D, dtype=torch.bfloat16)
    vraw = torch.zeros(H, C, D, dtype=torch.bfloat16)
    p = 0
    for i, n in enumerate([400, 200, 300]):   # the last write wraps and overwrites
        k = si.normal_bf16(n, H, D, 3000 + i, "cuda", mult=torch.full((H, 1), 1.0 + 2 * i))
        v = si.normal_bf16(n, H, D, 4000 + i, "cuda")
        q = si.normal_bf16(n, H, D, 5000 + i, "cuda")
        pos = np.arange(p, p + n)
        g.write(0, k, v, pos)
        o.write(0, k.cpu(), v.cpu(), pos)
        slots = [o.slot_of(x) for x in pos]
        kraw[:, slots] = k.cpu().permute(1, 0, 2)
        vraw[:, slots] = v.cpu().permute(1, 0, 2)
        p += n
        out_rt = torch.empty(n, H, D, dtype=torch.float32, device="cuda")
        out_wt = torch.empty(n, H, D, dtype=torch.float32, device="cuda")
        g.attend_readtime(0, q, out_rt)
        g.attend(0, q, out_wt)
        g.sync()
        img = g.export_readtime()
        want = oracle.readtime_image(kraw, vraw, o.export(0)["pos"])
        occ = o.export(0)["pos"] != oracle.EMPTY
        check_codes(img["kcodes"][:, occ], want["kcodes"][:, occ], "read-time K codes")
        check_codes(img["vcodes"][:, occ], want["vcodes"][:, occ], "read-time V codes")
        check_scales(img["kscale"][:, occ], want["kscale"][:, occ], "read-time K scales")
        check_scales(img["vscale"][:, occ], want["vscale"][:, occ], "read-time V scales")
        ref = oracle.attend_image(img["kcodes"], img["kscale"], img["vcodes"], img["vscale"],
                                  o.export(0)["pos"], q.cpu(), pos)
        check_attention(out_rt.cpu().numpy(), ref, "read-time attention")
        assert torch.isfinite(out_wt).all()


@pytest.mark.parametrize("D", [128, 64])
def test_readtime_after_resets(rc, D):
    """The read-time ablation after position resets: every key of the whole
    cache is rotated at its slot's CURRENT position in each call.  Sequence:
    write, delta, a write that wraps, read-time attention, a second delta (the
    window restarts at 0), read-time attention again; the read-time ring and
    the output are compared with the oracle's read-time image built from the
    unrotated keys at the positions the oracle's state machine holds."""
    H, C = 4, 700
    g = rc.RingKVCache(1, H, D, C, readtime_ablation=True)
    o = oracle.OracleCache(1, H, D, C)
    kraw = torch.zeros(H, C, D, dtype=torch.bfloat16)
    vraw = torch.zeros(H, C, D, dtype=torch.bfloat16)

    def write(p0, n, seed):
        k = si.normal_bf16(n, H, D, seed, "cuda", mult=torch.full((H, 1), 1.5))
        v = si.normal_bf16(n, H, D, seed + 1, "cuda")
        pos = np.arange(p0, p0 + n)
        g.write(0, k, v, pos)
        o.write(0, k.cpu(), v.cpu(), pos)
        slots = [o.slot_of(x) for x in pos]
        kraw[:, slots] = k.cpu().permute(1, 0, 2)
        vraw[:, slots] = v.cpu().permute(1, 0, 2)
        return pos

    def check(q, what):
        n = q.shape[0]
        out = torch.empty(n, H, D, dtype=torch.float32, device="cuda")
        g.attend_readtime(0, q, out)
        g.sync()
        img = g.export_readtime()
        st = o.export(0)
        assert np.array_equal(g.export(0)["pos"], st["pos"]), f"{what}: positions"
        want = oracle.readtime_image(kraw, vraw, st["pos"])
        occ = st["pos"] != oracle.EMPTY
        check_codes(img["kcodes"][:, occ], want["kcodes"][:, occ], f"{what}: read-time K codes")
        check_codes(img["vcodes"][:, occ], want["vcodes"][:, occ], f"{what}: read-time V codes")
        check_scales(img["kscale"][:, occ], want["kscale"][:, occ], f"{what}: read-time K scales")
        check_scales(img["vscale"][:, occ], want["vscale"][:, occ], f"{what}: read-time V scales")
        ref = oracle.attend_image(img["kcodes"], img["kscale"], img["vcodes"], img["vscale"], st["pos"],
                                  q.cpu(), o.last_positions(0))
        check_attention(out.cpu().numpy(), ref, f"{what}: read-time attention")

    write(0, 500, 7100)
    g.delta_rotate(-123_457)
    o.delta_rotate(-123_457)
    pos = write(500 - 123_457, 450, 7200)          # wraps onto slots 0..249
    check(si.normal_bf16(len(pos), H, D, 7300, "cuda"), "after one reset")
    oldest = int(o.export(0)["pos"][o.export(0)["pos"] != oracle.EMPTY].min())
    g.delta_rotate(-oldest)
    o.delta_rotate(-oldest)
    check(si.normal_bf16(len(pos), H, D, 7400, "cuda"), "after the window restart")
    g.close()
