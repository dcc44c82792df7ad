"""The oracle still reproduces its committed tiny-workload fixture.

tests/golden/tiny_seed1.txt was written by tests/golden/make_golden.py, which
calls only the oracle; the pages print no worked example of their own."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))


def test_tiny_fixture(oracle_mod):
    import make_golden
    want = open(os.path.join(HERE, "golden", "tiny_seed1.txt")).read().splitlines()[1:]
    got = make_golden.run(1)
    assert len(want) == len(got)
    for w, g in zip(want, got):
        if w.startswith("attend"):
            a = np.array(w.split()[2:], dtype=np.float64)
            b = np.array(g.split()[2:], dtype=np.float64)
            assert np.max(np.abs(a - b)) < 1e-12
        else:
            assert w == g
