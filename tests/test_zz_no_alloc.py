"""rc_ring_write_noalloc against rc_cache_write, through the C ABI.

Some callers cannot call cudaMalloc: a process whose device memory is all
reserved by another allocator (a framework's caching allocator or a fixed
arena), or a latency-critical loop that must never pay for cudaMalloc/cudaFree,
which can synchronise the device.  rc_ring_write_noalloc writes into a ring the
caller owns and keeps its only scratch (the RoPE table) in a static device
array.  Here the test itself allocates that caller-owned ring with torch, makes
two writes in a row with both entry points on the same inputs, and compares
codes, scales and groups with the tolerances of the other parity tests --
against rc_cache_write and, for the consecutive-position writes, against the
oracle's write as well.
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity_util import check_codes, check_scales

pytestmark = pytest.mark.gpu


def _koff(row, col, D):
    x = (row & 7) if D == 128 else ((row >> 1) & 3)
    return row * D + ((((col >> 4) ^ x) << 4) | (col & 15))


def _voff(drow, slot):
    return drow * 128 + ((((slot >> 4) ^ (drow & 7)) << 4) | (slot & 15))


def _canonical(ring, H, D, C):
    """Caller-owned ring buffers -> [H][C][D] codes and [H][C] scales (the layout rc.h documents)."""
    T = (C + 127) // 128
    kc = ring["kcodes"].cpu().numpy().reshape(H, T, 128 * D)
    vc = ring["vcodes"].cpu().numpy().reshape(H, T, 128 * D)
    s = np.arange(C)
    d = np.arange(D)
    kidx = _koff((s % 128)[:, None], d[None, :], D)           # [C][D]
    vidx = _voff(d[None, :], (s % 128)[:, None])              # [C][D]
    tiles = (s // 128)[:, None]
    out = dict(kcodes=kc[:, tiles, kidx], vcodes=vc[:, tiles, vidx],
               kscale=ring["kscale"].cpu().numpy().reshape(H, T * 128)[:, :C],
               vscale=ring["vscale"].cpu().numpy().reshape(H, T * 128)[:, :C],
               group=ring["group"].cpu().numpy()[:C])
    return out


def _new_ring(H, D, C):
    T = (C + 127) // 128
    return dict(kcodes=torch.zeros(H * T * 128 * D, dtype=torch.uint8, device="cuda"),
                vcodes=torch.zeros(H * T * 128 * D, dtype=torch.uint8, device="cuda"),
                kscale=torch.zeros(H * T * 128, dtype=torch.float32, device="cuda"),
                vscale=torch.zeros(H * T * 128, dtype=torch.float32, device="cuda"),
                group=torch.full((T * 128,), -1, dtype=torch.int32, device="cuda"),
                heads=H, head_dim=D, slots=C)


@pytest.mark.parametrize("D", [128, 64])
def test_noalloc_write_matches_cache_write(D):
    import fp8_ring_kv_cache_gb300 as rc
    from fp8_ring_kv_cache_gb300._binding import rc_ring_write_noalloc

    H, C = 8, 1000
    oracle.build()
    cache = rc.RingKVCache(1, H, D, C)
    ora = oracle.OracleCache(1, H, D, C)
    ring = _new_ring(H, D, C)
    writes = [(0, 600, 0.5), (600, 500, 3.0)]   # the second write wraps onto slots 0..99
    inputs = []
    for i, (p0, n, scale) in enumerate(writes):
        k = si.normal_bf16(n, H, D, 9100 + i, "cuda", mult=torch.full((H, 1), scale))
        v = si.normal_bf16(n, H, D, 9200 + i, "cuda")
        inputs.append((k, v, np.arange(p0, p0 + n)))
    torch.cuda.synchronize()
    for i, (k, v, pos) in enumerate(inputs):
        cache.write(0, k, v, pos)
        ora.write(0, k.cpu(), v.cpu(), pos)
        free_before = torch.cuda.mem_get_info()[0]
        rc_ring_write_noalloc(ring, k, v, pos, delta_total=0, group=i)
        torch.cuda.synchronize()
        if i > 0:
            # after the first call's one-time set-up, a call takes no device memory
            assert torch.cuda.mem_get_info()[0] == free_before
        want = cache.export(0)
        got = _canonical(ring, H, D, C)
        occ = want["pos"] != rc.EMPTY
        check_codes(got["kcodes"][:, occ], want["kcodes"][:, occ], f"write {i} K codes")
        check_codes(got["vcodes"][:, occ], want["vcodes"][:, occ], f"write {i} V codes")
        check_scales(got["kscale"][:, occ], want["kscale"][:, occ], f"write {i} K scales")
        check_scales(got["vscale"][:, occ], want["vscale"][:, occ], f"write {i} V scales")
        # the slots of write j carry group j; untouched slots stay empty
        assert np.array_equal(got["group"][occ], want["gid"][occ].astype(np.int32))
        assert (got["group"][~occ] == -1).all()
        # and the oracle's write of the same tokens
        ref = ora.export(0)
        assert np.array_equal(ref["pos"] != oracle.EMPTY, occ)
        check_codes(got["kcodes"][:, occ], ref["kcodes"][:, occ], f"write {i} K codes vs oracle")
        check_codes(got["vcodes"][:, occ], ref["vcodes"][:, occ], f"write {i} V codes vs oracle")
        check_scales(got["kscale"][:, occ], ref["kscale"][:, occ], f"write {i} K scales vs oracle")
        check_scales(got["vscale"][:, occ], ref["vscale"][:, occ], f"write {i} V scales vs oracle")
    cache.close()


def test_noalloc_rejects_oversize():
    import fp8_ring_kv_cache_gb300 as rc
    from fp8_ring_kv_cache_gb300._binding import RC_NOALLOC_MAX_TOKENS, rc_ring_write_noalloc

    H, D, C = 2, 64, RC_NOALLOC_MAX_TOKENS + 8
    ring = _new_ring(H, D, C)
    n = RC_NOALLOC_MAX_TOKENS + 1
    k = torch.zeros(n, H, D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rc.RcError) as e:
        rc_ring_write_noalloc(ring, k, k, np.arange(n), delta_total=0, group=0)
    assert e.value.status == rc.RC_ERR_ARG


@pytest.mark.parametrize("D", [128, 64])
def test_noalloc_permuted_positions_after_reset(D):
    """A write whose positions are not an arithmetic run (they are copied into
    the static array) into a ring whose positions were reset (nonzero
    delta_total), against rc_cache_write after the same reset.  The caller-owned
    ring has no delta rotation, so the comparison covers the slots of the write
    made after the reset."""
    import fp8_ring_kv_cache_gb300 as rc
    from fp8_ring_kv_cache_gb300._binding import rc_ring_write_noalloc

    H, C, delta = 6, 900, -100_003
    cache = rc.RingKVCache(1, H, D, C)
    ring = _new_ring(H, D, C)
    k0 = si.normal_bf16(700, H, D, 9300, "cuda")
    v0 = si.normal_bf16(700, H, D, 9301, "cuda")
    cache.write(0, k0, v0, np.arange(0, 700))
    rc_ring_write_noalloc(ring, k0, v0, np.arange(0, 700), delta_total=0, group=0)
    cache.delta_rotate(delta)
    rng = np.random.default_rng(9302)
    for i, (p0, n) in enumerate([(700 + delta, 500), (1200 + delta, 333)]):
        pos = rng.permutation(np.arange(p0, p0 + n))      # wraps past slot 899 in the first write
        k = si.normal_bf16(n, H, D, 9310 + i, "cuda", mult=torch.full((H, 1), 2.0))
        v = si.normal_bf16(n, H, D, 9320 + i, "cuda")
        cache.write(0, k, v, pos)
        rc_ring_write_noalloc(ring, k, v, pos, delta_total=delta, group=1 + i)
        torch.cuda.synchronize()
        want = cache.export(0)
        got = _canonical(ring, H, D, C)
        slots = (pos - delta) % C
        check_codes(got["kcodes"][:, slots], want["kcodes"][:, slots], f"write {i} K codes")
        check_codes(got["vcodes"][:, slots], want["vcodes"][:, slots], f"write {i} V codes")
        check_scales(got["kscale"][:, slots], want["kscale"][:, slots], f"write {i} K scales")
        check_scales(got["vscale"][:, slots], want["vscale"][:, slots], f"write {i} V scales")
        assert (got["group"][slots] == 1 + i).all()
        assert np.array_equal(want["pos"][slots], pos)
    cache.close()
