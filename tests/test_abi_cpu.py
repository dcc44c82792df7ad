"""The C-ABI library loads and exports every entry point include/rc.h declares.

No compute call is made here: without a GPU, rc_cache_create must fail with an
error status instead of falling back to anything."""
import ctypes
import re

import pytest
import torch


@pytest.fixture(scope="module")
def rc():
    import __graft_entry__
    __graft_entry__.build()
    import fp8_ring_kv_cache_gb300 as rc
    return rc


def test_every_declared_symbol_is_exported(rc):
    declared = rc.declared_symbols()
    assert "rc_cache_create" in declared and "rc_attend" in declared
    missing = [s for s in declared if not hasattr(rc.lib, s)]
    assert not missing, missing


def test_header_declarations_are_the_abi(rc):
    # every declared function is extern "C" in the library (no C++ mangling)
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", rc._binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (rc_\w+)$", out, flags=re.M))
    assert set(rc.declared_symbols()) <= exported


def test_bounds_checked_build_has_the_same_abi(rc):
    # librc_bounds.so (-DRC_BOUNDS_CHECK) exports every declared entry point
    # and says so through rc_build_flags; librc.so reports no checks
    import os
    import subprocess
    here = os.path.dirname(rc._binding.__file__)
    flags = {}
    for name in ("librc.so", "librc_bounds.so"):
        path = os.path.join(here, name)
        out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
        exported = set(re.findall(r"\bT (rc_\w+)$", out, flags=re.M))
        assert set(rc.declared_symbols()) <= exported, name
        lib = ctypes.CDLL(path)
        lib.rc_build_flags.restype = ctypes.c_uint
        flags[name] = lib.rc_build_flags()
    assert flags == {"librc.so": 0, "librc_bounds.so": rc.RC_BUILD_BOUNDS_CHECK}


def test_status_strings(rc):
    for st in (rc.RC_OK, rc.RC_ERR_ARG, rc.RC_ERR_STATE, rc.RC_ERR_CUDA, rc.RC_ERR_OOM, rc.RC_ERR_TIMEOUT,
               rc.RC_ERR_UNSUPPORTED, rc.RC_ERR_BOUNDS):
        s = rc.rc_status_string(st)
        assert s and s != "unknown status"
    assert rc.rc_status_string(12345) == "unknown status"


def test_bad_config_rejected_before_device_work(rc):
    cfg = rc._binding.rc_config(1, 2, 96, 64, 64, 10000.0, 0)      # head_dim 96 unsupported
    h = ctypes.c_void_p()
    st = rc.lib.rc_cache_create(ctypes.byref(cfg), 0, ctypes.byref(h))
    assert st == rc.RC_ERR_UNSUPPORTED and not h.value
    cfg = rc._binding.rc_config(1, 2, 64, 64, 65, 10000.0, 0)      # max_write > slots
    assert rc.lib.rc_cache_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == rc.RC_ERR_ARG
    assert rc.lib.rc_cache_create(None, 0, ctypes.byref(h)) == rc.RC_ERR_ARG
    cfg = rc._binding.rc_config(1, 2, 64, 64, 64, 10000.0, rc.RC_F_READTIME_ABLATION | rc.RC_F_COPY_WINDOW)
    assert rc.lib.rc_cache_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == rc.RC_ERR_UNSUPPORTED


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure path")
def test_no_gpu_fails_loudly(rc):
    with pytest.raises(rc.RcError):
        rc.RingKVCache(1, 2, 64, 64)


def test_null_handle_calls_are_rejected(rc):
    assert rc.lib.rc_cache_write(None, 0, None, None, None, 1, None) == rc.RC_ERR_ARG
    assert rc.lib.rc_attend(None, 0, None, None, 1, None) == rc.RC_ERR_ARG
    assert rc.lib.rc_cache_delta_rotate(None, 5, None) == rc.RC_ERR_ARG
    assert rc.lib.rc_cache_window_shift(None, 5, None) == rc.RC_ERR_ARG
    assert rc.lib.rc_cache_sync(None) == rc.RC_ERR_ARG
    rc.lib.rc_cache_destroy(None)
