"""Parity of the bf16 ring (RC_F_BF16_CACHE) against the oracle's bf16 cache.

The non-FP8 side of the FP8-versus-bf16 cache comparison (cpdf.ai blog,
section "Blackwell, escalabilidade e limites do decodificador").  The GPU cache
and oracle.OracleBf16Cache are driven in lockstep from the same seeded inputs;
neither sees the other's state.

  positions, write serials                   : bit-exact
  V bits                                     : bit-exact with the oracle's V
                                               rounded to fp16 (the ring stores
                                               V in fp16; exact for every
                                               2^-17 <= |v| < 65520)
  K bits                                     : >= 99.9 % identical; each of the
                                               rest within one bf16 step of the
                                               oracle plus 2^-21 of its RoPE
                                               pair's norm (the fp32 rotation's
                                               absolute error) after a write; and
                                               after k delta rotations, plus k
                                               steps of the pair's norm more
  attention output                           : |error| <= 1e-3 + 2^-11 vmax for
                                               each (head, channel), vmax the
                                               largest |V| stored there; mean-abs
                                               <= 1e-3

The kernel rotates in fp32 and the oracle in fp64, each rounding once to bf16,
so a rounding decision near a tie can go the other way (about once in 10^4
elements).  Where x cos - y sin cancels, the fp32 result's absolute error, a
few 2^-24 of the pair's norm, can exceed the small result's own bf16 step.  A
key that differs by a step before a delta carries that difference, a step of
the pair's larger component at most, into both elements of its pair, which for
a small element is many of its own steps: hence the bounds in units of the
pair's norm.

The attention bar follows from the kernel's arithmetic: the queries keep ~16
significant bits (two bf16 pieces), the scores accumulate in fp32, P is rounded
to fp16 (relative error <= 2^-12) and V is held in fp16 (exact but for
|v| < 2^-17, off by < 2^-25 there); O divides
sum_i p~_i v_i by l = sum_i p_i, so its error is at most 2^-12 of the largest
|v| in the channel, plus the far smaller effects of the query's residual bits
and of the rare key differences.  The bar takes twice that, plus 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si

pytestmark = pytest.mark.gpu

KEY_SAME_FRAC = 0.999
ATTN_ABS = 1e-3
ATTN_V_REL = 2.0 ** -11
ATTN_MEAN_ABS = 1e-3


@pytest.fixture(scope="module")
def rc():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_ring_kv_cache_gb300 as rc
    oracle.build()
    return rc


def bf16_value(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_step(x: np.ndarray) -> np.ndarray:
    """The bf16 spacing at |x| (8 significant bits; 2^-133 below the normal range)."""
    m = np.abs(x)
    e = np.floor(np.log2(np.where(m > 0, m, 1.0)))
    return np.where(m >= 2.0 ** -126, np.exp2(e - 7), 2.0 ** -133)


def as_f16_bits(vbits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns rounded to fp16 and returned as bf16 bit patterns."""
    t = torch.from_numpy(vbits.astype(np.int16)).view(torch.bfloat16)
    return t.to(torch.float16).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def check_keys(got: np.ndarray, want: np.ndarray, deltas: int, what: str) -> dict:
    g, w = bf16_value(got), bf16_value(want)
    diff = np.abs(g - w)
    norm = np.repeat(np.hypot(w[..., 0::2], w[..., 1::2]), 2, axis=-1)  # the RoPE pair's norm
    bound = bf16_step(w) + (1 + deltas) * 2.0 ** -21 * norm + deltas * bf16_step(norm)
    frac = float((got == want).mean()) if got.size else 1.0
    bad = diff > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} keys beyond the bound, worst {float((diff - bound).max()):.3g}"
    assert frac >= KEY_SAME_FRAC, f"{what}: only {frac:.6f} identical"
    return dict(identical=frac)


def check_out(got: np.ndarray, want: np.ndarray, vbits: np.ndarray, what: str) -> dict:
    """got, want [n][H][d]; vbits [H][slots][d], the stored values of the occupied slots."""
    err = np.abs(got.astype(np.float64) - want)
    vmax = np.abs(bf16_value(vbits)).max(axis=1)          # [H][d]
    bound = ATTN_ABS + ATTN_V_REL * vmax[None]
    mx, mean = float(err.max()), float(err.mean())
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    worst = float((err / bound).max())
    assert worst <= 1.0, f"{what}: error {worst:.3f} x the bound (max-abs {mx:.4g})"
    assert mean <= ATTN_MEAN_ABS, f"{what}: mean-abs {mean:.4g} > {ATTN_MEAN_ABS}"
    return dict(max_abs=mx, mean_abs=mean, of_bound=worst)


class Pair:
    """The GPU bf16 cache and the oracle's bf16 cache driven in lockstep."""

    def __init__(self, rc, L, H, D, C, max_write=None):
        self.g = rc.RingKVCache(L, H, D, C, max_write=max_write, bf16_cache=True)
        self.o = oracle.OracleBf16Cache(L, H, D, C)
        self.deltas = 0

    def write(self, layer, K, V, pos):
        self.g.write(layer, K, V, pos)
        self.o.write(layer, K.cpu(), V.cpu(), pos)

    def delta(self, d):
        self.g.delta_rotate(d)
        self.o.delta_rotate(d)
        self.deltas += 1

    def check(self, layer, what):
        self.g.sync()
        got, want = self.g.export(layer), self.o.export(layer)
        assert np.array_equal(got["pos"], want["pos"]), f"{what}: positions differ"
        assert np.array_equal(got["gid"], want["gid"]), f"{what}: write serials differ"
        occ = want["pos"] != oracle.EMPTY
        assert np.array_equal(got["vbits"][:, occ], as_f16_bits(want["vbits"][:, occ])), f"{what}: V bits differ"
        return check_keys(got["kbits"][:, occ], want["kbits"][:, occ], self.deltas, f"{what} K bits")

    def attend_check(self, layer, Q, what="attention"):
        out = torch.empty(Q.shape, dtype=torch.float32, device="cuda")
        self.g.attend(layer, Q, out)
        self.g.sync()
        st = self.o.export(layer)
        occ = st["pos"] != oracle.EMPTY
        return check_out(out.cpu().numpy(), self.o.attend(layer, Q.cpu()), st["vbits"][:, occ], what)


@pytest.mark.parametrize("seed", [1, 2])
def test_bf16_tiny_schedule(rc, seed):
    s = si.TINY
    pr = Pair(rc, s.layers, s.heads, s.head_dim, s.slots)
    step, q = 0, None
    for op in si.tiny_schedule():
        if op[0] == "write":
            _, layer, p0, n = op
            k, v, q = si.tiny_tensors(seed, step, "cuda")
            pr.write(layer, k, v, np.arange(p0, p0 + n))
            pr.check(layer, f"after write {step}")
            step += 1
        elif op[0] == "delta":
            pr.delta(op[1])
            pr.check(0, "after delta")
        else:
            pr.attend_check(op[1], q, f"attention after write {step}")


@pytest.mark.parametrize("D", [64, 128])
def test_bf16_ragged_partial_ring(rc, D):
    # C not a multiple of 128; a partially filled ring (masked tiles), write
    # sizes that are not multiples of the CTA's 64 tokens or 128 query rows;
    # the last write wraps and overwrites the oldest slots
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
        pr.attend_check(layer, qq, f"attention {i}")


@pytest.mark.parametrize("D", [64, 128])
def test_bf16_full_ring_delta_multilayer(rc, D):
    # full 8-tile rings on three layers (every tile takes the fast path), a
    # wrapping write, one delta rotation of every layer, attention after it
    L, H, C = 3, 4, 1024
    pr = Pair(rc, L, H, D, C, max_write=C)
    p = 0
    for i, n in enumerate([700, 324, 200]):
        for layer in range(L):
            k = si.normal_bf16(n, H, D, 1000 + 10 * i + layer, "cuda", mult=torch.full((H, 1), 1.0 + i))
            v = si.normal_bf16(n, H, D, 2000 + 10 * i + layer, "cuda")
            pr.write(layer, k, v, np.arange(p, p + n))
        p += n
    for layer in range(L):
        pr.check(layer, f"layer {layer} before the delta")
    q = si.normal_bf16(200, H, D, 3000, "cuda")
    pr.attend_check(1, q, "attention before the delta")
    pr.delta(-p)
    for layer in range(L):
        pr.check(layer, f"layer {layer} after the delta")
    pr.attend_check(2, q, "attention after the delta")


@pytest.mark.parametrize("seed", [12])
def test_bf16_production_call_sampled_heads(rc, seed):
    # the production call (5,788 slots, 757 new tokens, head_dim 128) on the
    # GPU with all 48 heads; the oracle runs the heads carrying the most
    # outlier channels and two ordinary ones (heads are independent)
    t = si.production_tensors(seed, "cuda")
    C, H, D = si.PROD_SLOTS, si.PROD_HEADS, si.PROD_DIM
    g = rc.RingKVCache(1, H, D, C, bf16_cache=True)
    g.write(0, t["k_prefill"], t["v_prefill"], np.arange(0, si.PROD_PREFILL))
    g.write(0, t["k_new"], t["v_new"], np.arange(si.PROD_PREFILL, C))
    out = torch.empty(t["q"].shape, dtype=torch.float32, device="cuda")
    g.attend(0, t["q"], out)
    g.sync()
    counts = (t["mult"] > 1).sum(1)
    heads = sorted(set(torch.argsort(counts, descending=True)[:3].tolist() + [0, 47]))
    o = oracle.OracleBf16Cache(1, len(heads), D, C)
    o.write(0, t["k_prefill"][:, heads].cpu(), t["v_prefill"][:, heads].cpu(), np.arange(0, si.PROD_PREFILL))
    o.write(0, t["k_new"][:, heads].cpu(), t["v_new"][:, heads].cpu(), np.arange(si.PROD_PREFILL, C))
    st = g.export(0)
    want = o.export(0)
    assert np.array_equal(st["vbits"][heads], as_f16_bits(want["vbits"]))
    check_keys(st["kbits"][heads], want["kbits"], 0, "production K bits")
    res = check_out(out[:, heads].cpu().numpy(), o.attend(0, t["q"][:, heads].cpu()), want["vbits"],
                    "production attention")
    print("bf16 production attention error", res)


def test_bf16_flags_and_errors(rc):
    with pytest.raises(rc.RcError) as e:
        rc.RingKVCache(1, 2, 64, 64, bf16_cache=True, readtime_ablation=True)
    assert e.value.status == rc.RC_ERR_UNSUPPORTED
    with pytest.raises(rc.RcError) as e:
        rc.RingKVCache(1, 2, 64, 64, bf16_cache=True, copy_window=True)
    assert e.value.status == rc.RC_ERR_UNSUPPORTED
    g = rc.RingKVCache(1, 2, 64, 64, bf16_cache=True)
    k = si.normal_bf16(4, 2, 64, 1, "cuda")
    g.write(0, k, k, np.arange(4))
    with pytest.raises(rc.RcError) as e:
        rc.rc_cache_export(g.handle, 0, 2, 64, 64)       # FP8 export of a bf16 ring
    assert e.value.status == rc.RC_ERR_STATE
    with pytest.raises(rc.RcError) as e:
        g.window_shift(3)
    assert e.value.status == rc.RC_ERR_STATE
    f = rc.RingKVCache(1, 2, 64, 64)
    with pytest.raises(rc.RcError) as e:
        rc.rc_cache_export_bf16(f.handle, 0, 2, 64, 64)  # bf16 export of an FP8 ring
    assert e.value.status == rc.RC_ERR_STATE
    g.sync()
