"""Parity of the write fused into the K/V projection (rc_cache_write_fused)
against the oracle's orc_write_proj, which forms the products exactly in fp64.

  positions, write serials, occupancy            : bit-exact
  per-slot scales                                : within 2e-5 relative
  E4M3 codes                                     : >= 99.99 % identical, the rest
                                                   one step apart
  attention on the GPU's exported cache          : max-abs <= 3e-2, mean-abs <= 3e-3

The bars follow from the arithmetic: the kernel's products are sums of
hidden / 32 MMA partial sums accumulated in fp32 in TMEM, where the oracle's
fp64 sums are exact; for the 192 steps of hidden = 6,144 that bounds the
relative error of a dominant-sign sum, a head's amax among them, by about
192 x 2^-24 = 1.1e-5 (the bar takes 2e-5; measured: below 1e-6).  A code
changes only where the fp32 quotient lies that close to a boundary between
two E4M3 values (relative spacing 1/8 to 1/16), a few elements in 10^5, and
then by one step.  Everything after the product is the write's own
arithmetic, checked bit for bit by the write's parity tests.
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity_util import check_attention, code_ordinal

pytestmark = pytest.mark.gpu

FUSED_SCALE_REL = 2e-5
FUSED_CODE_SAME = 0.9999


@pytest.fixture(scope="module")
def rc():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_ring_kv_cache_gb300 as rc
    oracle.build()
    return rc


def check_fused_state(gpu: dict, ora: dict, what: str, heads=None) -> dict:
    assert np.array_equal(gpu["pos"], ora["pos"]), f"{what}: positions differ"
    assert np.array_equal(gpu["gid"], ora["gid"]), f"{what}: write serials differ"
    occ = ora["pos"] != oracle.EMPTY
    hs = slice(None) if heads is None else heads
    res = {}
    for kind in ("k", "v"):
        g, o = gpu[kind + "codes"][hs][:, occ], ora[kind + "codes"][:, occ]
        og, oo = code_ordinal(g), code_ordinal(o)
        d = np.abs(og - oo)
        same = float((d == 0).mean())
        assert int(d.max(initial=0)) <= 1, f"{what}: {kind} codes more than one step apart"
        assert same >= FUSED_CODE_SAME, f"{what}: only {same:.5f} of {kind} codes identical"
        sg = gpu[kind + "scale"][hs][:, occ].astype(np.float64)
        so = ora[kind + "scale"][:, occ].astype(np.float64)
        rel = float((np.abs(sg - so) / so).max())
        assert rel <= FUSED_SCALE_REL, f"{what}: {kind} scales {rel:.3g} apart"
        res[kind] = dict(identical=same, scale_rel=rel)
    return res


def attend_check(g, layer, q, qpos, heads=None, what="attention"):
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    g.attend(layer, q, out)
    g.sync()
    st = g.export(layer)
    hs = slice(None) if heads is None else heads
    ref = oracle.attend_image(st["kcodes"][hs], st["kscale"][hs], st["vcodes"][hs], st["vscale"][hs], st["pos"],
                              q[:, hs].cpu(), qpos, 10000.0)
    return check_attention(out[:, hs].cpu().numpy(), ref, what)


@pytest.mark.parametrize("D", [128, 64])
def test_fused_writes_and_delta(rc, D):
    # two writes over 1 and 2 blocks of 256 rows (clusters of 1 and 2), the
    # second wrapping over the ring's end; then a delta and a third write
    H, C, hidden = 4, 600, 256
    g = rc.RingKVCache(2, H, D, C, max_write=C)
    o = oracle.OracleCache(2, H, D, C)
    p = 100
    for i, (layer, n) in enumerate([(0, 200), (0, 460), (1, 257)]):
        x, xs, wk, wks, wv, wvs = si.proj_operands(30 + i, n, hidden, H * D, "cuda")
        pos = np.arange(p, p + n)
        g.write_fused(layer, x, xs, wk, wks, wv, wvs, pos)
        o.write_proj(layer, x.cpu(), xs, wk.cpu(), wks, wv.cpu(), wvs, pos)
        p += n
        g.sync()
        print(f"write {i}:", check_fused_state(g.export(layer), o.export(layer), f"write {i}"))
        q = si.normal_bf16(n, H, D, 40 + i, "cuda")
        attend_check(g, layer, q, pos, what=f"attention {i}")
        if i == 1:
            g.delta_rotate(-300)
            o.delta_rotate(-300)
            p -= 300


def test_fused_single_token_and_permuted_positions(rc):
    H, D, C, hidden = 2, 128, 300, 128
    g = rc.RingKVCache(1, H, D, C, max_write=C)
    o = oracle.OracleCache(1, H, D, C)
    x, xs, wk, wks, wv, wvs = si.proj_operands(50, 1, hidden, H * D, "cuda")
    g.write_fused(0, x, xs, wk, wks, wv, wvs, [7])
    o.write_proj(0, x.cpu(), xs, wk.cpu(), wks, wv.cpu(), wvs, [7])
    g.sync()
    check_fused_state(g.export(0), o.export(0), "one token")
    rng = np.random.default_rng(51)
    pos = 1000 + rng.permutation(150)
    x, xs, wk, wks, wv, wvs = si.proj_operands(52, 150, hidden, H * D, "cuda")
    g.write_fused(0, x, xs, wk, wks, wv, wvs, pos)
    o.write_proj(0, x.cpu(), xs, wk.cpu(), wks, wv.cpu(), wvs, pos)
    g.sync()
    check_fused_state(g.export(0), o.export(0), "permuted positions")
    attend_check(g, 0, si.normal_bf16(150, H, D, 53, "cuda"), pos, what="attention after permuted write")


def test_fused_production_write_sampled_heads(rc):
    # 757 tokens, 48 heads x 128, hidden 6,144 (three blocks of rows: a
    # cluster of 3); the oracle forms the products of five heads
    H, D, C, n, hidden = si.PROD_HEADS, si.PROD_DIM, si.PROD_SLOTS, si.PROD_NEW, si.PROD_HIDDEN
    x, xs, wk, wks, wv, wvs = si.proj_operands(60, n, hidden, H * D, "cuda")
    g = rc.RingKVCache(1, H, D, C, max_write=C)
    pos = np.arange(si.PROD_PREFILL, C)
    g.write_fused(0, x, xs, wk, wks, wv, wvs, pos)
    g.sync()
    heads = [0, 13, 26, 39, 47]
    rows = np.concatenate([np.arange(h * D, (h + 1) * D) for h in heads])
    o = oracle.OracleCache(1, len(heads), D, C)
    o.write_proj(0, x.cpu(), xs, wk.cpu()[rows], wks, wv.cpu()[rows], wvs, pos)
    res = check_fused_state(g.export(0), o.export(0), "production fused write", heads)
    print("production fused write:", res)
    attend_check(g, 0, si.normal_bf16(n, H, D, 61, "cuda"), pos, heads, "production attention after fused write")


def test_fused_errors(rc):
    x, xs, wk, wks, wv, wvs = si.proj_operands(70, 8, 128, 2 * 64, "cuda")
    g = rc.RingKVCache(1, 2, 64, 64)
    with pytest.raises(rc.RcError) as e:
        g.write_fused(0, x[:, :96].contiguous(), xs, wk[:, :96].contiguous(), wks, wv[:, :96].contiguous(), wvs,
                      np.arange(8))                                   # hidden not a multiple of 64
    assert e.value.status == rc.RC_ERR_ARG
    with pytest.raises(rc.RcError) as e:
        g.write_fused(0, x, -1.0, wk, wks, wv, wvs, np.arange(8))    # scale not positive
    assert e.value.status == rc.RC_ERR_ARG
    for kw in (dict(bf16_cache=True), dict(readtime_ablation=True)):
        b = rc.RingKVCache(1, 2, 64, 64, **kw)
        with pytest.raises(rc.RcError) as e:
            b.write_fused(0, x, xs, wk, wks, wv, wvs, np.arange(8))
        assert e.value.status == rc.RC_ERR_UNSUPPORTED
    g.sync()


def test_fused_wait_runs_out_then_recovers(rc):
    """Wait limit 0 on the fused write: its first wait whose phase is not
    complete gives up, every CTA still passes the cluster barriers, drains its
    copies and MMAs and frees its tensor memory, and rc_cache_sync reports
    RC_ERR_TIMEOUT.  The write's slots are then undefined; written again with
    the limit restored they match the oracle (which made the same write twice,
    so the write serials agree)."""
    H, D, C, hidden, n = 4, 128, 1200, 512, 700
    g = rc.RingKVCache(1, H, D, C, max_write=C)
    o = oracle.OracleCache(1, H, D, C)
    x, xs, wk, wks, wv, wvs = si.proj_operands(80, n, hidden, H * D, "cuda")
    pos = np.arange(300, 300 + n)
    g.set_wait_limit(0)
    g.write_fused(0, x, xs, wk, wks, wv, wvs, pos)
    with pytest.raises(rc.RcError) as e:
        g.sync()
    assert e.value.status == rc.RC_ERR_TIMEOUT
    g.sync()  # the record was cleared
    g.set_wait_limit(2_000_000_000)
    g.write_fused(0, x, xs, wk, wks, wv, wvs, pos)
    for _ in range(2):
        o.write_proj(0, x.cpu(), xs, wk.cpu(), wks, wv.cpu(), wvs, pos)
    g.sync()
    check_fused_state(g.export(0), o.export(0), "fused write after a timed-out one")
    attend_check(g, 0, si.normal_bf16(n, H, D, 81, "cuda"), pos, what="attention after recovery")
