"""Failure paths without a GPU fault (the failure-detection forms of the test
strategy): a bounded device wait made to run out, and host-side fault
injection of allocations and launches.  Every case checks a clean status, no
leaked device memory, and that the cache (or a fresh one) still matches the
oracle afterwards."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity_util import check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rc():
    import fp8_ring_kv_cache_gb300 as m
    oracle.build()
    return m


def _write_attend_check(rc, cache, H, D, C, n_pre, n_new, seed):
    """Prefill + a write + an attention call on `cache`, checked against the oracle."""
    o = oracle.OracleCache(1, H, D, C)
    kp = si.normal_bf16(n_pre, H, D, seed, "cuda")
    vp = si.normal_bf16(n_pre, H, D, seed + 1, "cuda")
    kn = si.normal_bf16(n_new, H, D, seed + 2, "cuda")
    vn = si.normal_bf16(n_new, H, D, seed + 3, "cuda")
    q = si.normal_bf16(n_new, H, D, seed + 4, "cuda")
    for k, v, pos in ((kp, vp, np.arange(n_pre)), (kn, vn, np.arange(n_pre, n_pre + n_new))):
        cache.write(0, k, v, pos)
        o.write(0, k.cpu(), v.cpu(), pos)
    out = torch.empty(n_new, H, D, dtype=torch.float32, device="cuda")
    cache.attend(0, q, out)
    cache.sync()
    st = cache.export(0)
    ref = oracle.attend_image(st["kcodes"], st["kscale"], st["vcodes"], st["vscale"], st["pos"], q.cpu(),
                              np.arange(n_pre, n_pre + n_new))
    check_attention(out.cpu().numpy(), ref, "attention")
    return q


def test_wait_runs_out_then_recovers(rc):
    """Wait limit 0: the first wait whose phase is not complete gives up, the
    kernel frees its tensor memory and returns, and rc_cache_sync reports
    RC_ERR_TIMEOUT.  The same handle (limit restored) and a fresh one then give
    oracle-exact attention."""
    H, D, C = 4, 128, 1500
    cache = rc.RingKVCache(1, H, D, C)
    q = _write_attend_check(rc, cache, H, D, C, 1000, 300, 500)
    out = torch.empty(300, H, D, dtype=torch.float32, device="cuda")
    cache.set_wait_limit(0)
    cache.attend(0, q, out)
    with pytest.raises(rc.RcError) as e:
        cache.sync()
    assert e.value.status == rc.RC_ERR_TIMEOUT
    cache.sync()  # the record was cleared; nothing else is pending
    # the same handle, limit restored: the ring was not modified by the call that gave up
    cache.set_wait_limit(2_000_000_000)
    cache.attend(0, q, out)
    cache.sync()
    st = cache.export(0)
    ref = oracle.attend_image(st["kcodes"], st["kscale"], st["vcodes"], st["vscale"], st["pos"], q.cpu(),
                              np.arange(1000, 1300))
    check_attention(out.cpu().numpy(), ref, "attention on the same handle after the timeout")
    cache.close()
    fresh = rc.RingKVCache(1, H, D, C)
    _write_attend_check(rc, fresh, H, D, C, 1100, 200, 600)
    fresh.close()
    again = rc.RingKVCache(1, H, D, C)
    _write_attend_check(rc, again, H, D, C, 900, 300, 700)
    again.close()


def test_injected_allocation_failures_leak_nothing(rc, monkeypatch):
    """RC_FAULT_INJECT=alloc:K for every allocation rc_cache_create makes: the
    call fails with RC_ERR_OOM and the device's free memory is unchanged."""
    H, D, C = 4, 64, 700
    rc.RingKVCache(1, H, D, C, readtime_ablation=True).close()  # module and context set-up happen once
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    failed = 0
    for k in range(1, 40):
        monkeypatch.setenv("RC_FAULT_INJECT", f"alloc:{k}")
        try:
            c = rc.RingKVCache(1, H, D, C, readtime_ablation=(k % 2 == 0))
        except rc.RcError as e:
            assert e.status == rc.RC_ERR_OOM
            failed += 1
            assert torch.cuda.mem_get_info()[0] == free0, f"allocation {k}: device memory leaked"
            continue
        c.close()  # k past the last allocation: the cache was built
        assert torch.cuda.mem_get_info()[0] == free0
    assert failed >= 20  # every allocation index of a plain and an ablation cache was hit
    monkeypatch.delenv("RC_FAULT_INJECT")
    c = rc.RingKVCache(1, H, D, C)
    _write_attend_check(rc, c, H, D, C, 400, 200, 800)
    c.close()


def test_injected_launch_failures_change_nothing(rc, monkeypatch):
    """RC_FAULT_INJECT=launch: write, attend and delta rotation each return
    RC_ERR_CUDA without touching the cache; once the injection is gone the same
    cache gives oracle-exact results."""
    H, D, C = 4, 128, 1200
    cache = rc.RingKVCache(1, H, D, C)
    o = oracle.OracleCache(1, H, D, C)
    k = si.normal_bf16(800, H, D, 900, "cuda")
    v = si.normal_bf16(800, H, D, 901, "cuda")
    q = si.normal_bf16(800, H, D, 902, "cuda")
    cache.write(0, k, v, np.arange(800))
    o.write(0, k.cpu(), v.cpu(), np.arange(800))
    before = cache.export(0)
    launches = cache.launch_count
    out = torch.empty(800, H, D, dtype=torch.float32, device="cuda")
    monkeypatch.setenv("RC_FAULT_INJECT", "launch")
    for call in (lambda: cache.write(0, k, v, np.arange(800, 1600)), lambda: cache.attend(0, q, out),
                 lambda: cache.delta_rotate(-77)):
        with pytest.raises(rc.RcError) as e:
            call()
        assert e.value.status == rc.RC_ERR_CUDA
    monkeypatch.delenv("RC_FAULT_INJECT")
    assert cache.launch_count == launches and cache.delta_total == 0
    after = cache.export(0)
    for key in before:
        assert np.array_equal(before[key], after[key]), key
    cache.attend(0, q, out)
    cache.sync()
    st = cache.export(0)
    ref = oracle.attend_image(st["kcodes"], st["kscale"], st["vcodes"], st["vscale"], st["pos"], q.cpu(),
                              np.arange(800))
    check_attention(out.cpu().numpy(), ref, "attention after injected failures")
    cache.close()
