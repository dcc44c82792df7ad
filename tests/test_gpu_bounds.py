"""The GPU parity tests again, on the bounds-checked build.

compute-sanitizer is closed on this machine; librc_bounds.so (the same sources
compiled with -DRC_BOUNDS_CHECK) stands in for it.  There the write, rotation, read-time
and attention kernels test the index of each checked global access against
its buffer before making it (a failed check skips the access and records the
site in the status word; nothing traps), and every device buffer sits between
two guard zones that rc_cache_sync checks.  The GPU suites run in a child
process with RC_BOUNDS_CHECK=1, so they load that build: a failed check fails
the test whose sync reports it, and tests/conftest.py fails any test that left
a cache with an unreported failure when it was closed.  Their shapes include
ragged rings (C not a multiple of 128), partly filled rings, single-token and
wrapping writes, split tiles, both rotation kernels and head_dim 64 and 128.
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_child(args, timeout):
    env = dict(os.environ, RC_BOUNDS_CHECK="1")
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


@pytest.fixture(scope="module")
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()


def test_child_loads_the_bounds_checked_build(built):
    r = run_child(["-c", "import fp8_ring_kv_cache_gb300 as rc, sys; "
                         "sys.exit(0 if rc.rc_build_flags() & rc.RC_BUILD_BOUNDS_CHECK else 3)"], 300)
    assert r.returncode == 0, r.stdout + r.stderr


# the 16-bit and fused-write kernels have no index checks; their suites still
# run here for the guard zones, which catch a write past either end of any buffer
@pytest.mark.parametrize("suite", ["tests/test_gpu_parity.py", "tests/test_gpu_graph.py", "tests/test_gpu_bf16.py",
                                   "tests/test_gpu_fused.py"])
def test_parity_suite_on_bounds_checked_build(built, suite):
    r = run_child(["-m", "pytest", suite, "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider"], 1500)
    tail = (r.stdout[-4000:] + r.stderr[-2000:])
    assert r.returncode == 0, tail
    print(tail.strip().splitlines()[-1])
