"""Host logic that picks the attention kernel's softmax path per KV tile
(rc_tile_kinds, the function the attention call itself uses), against a
classifier written from the definition: a tile is uniform when one write group
holds all of its slots; a full tile is a two-run tile when its slots form
exactly two runs of occupied slots, [0, b) and [b, 128), of different groups."""
import numpy as np
import pytest

import fp8_ring_kv_cache_gb300 as rc


def expected(grp):
    grp = list(grp)
    C = len(grp)
    uniform = np.zeros(4, np.uint64)
    split = np.zeros(256, np.uint8)
    for t in range(min((C + 127) // 128, 256)):
        seg = grp[128 * t:min(128 * t + 128, C)]
        runs = []  # (group, length)
        for g in seg:
            if runs and runs[-1][0] == g:
                runs[-1][1] += 1
            else:
                runs.append([g, 1])
        if any(g < 0 for g, _ in runs):
            continue
        if len(runs) == 1:
            uniform[t // 64] |= np.uint64(1) << np.uint64(t % 64)
        elif len(runs) == 2 and len(seg) == 128:
            split[t] = runs[0][1]
    return uniform, split


def from_runs(lengths, groups):
    return np.concatenate([np.full(n, g, np.int32) for n, g in zip(lengths, groups)])


def check(grp):
    u, s = rc.rc_tile_kinds(grp)
    eu, es = expected(grp)
    assert np.array_equal(u, eu), (u, eu)
    assert np.array_equal(s, es), np.nonzero(s != es)


@pytest.mark.parametrize("b", [1, 31, 32, 33, 64, 96, 127])
def test_split_column(b):
    # tile 1 split at b, tiles 0 and 2 uniform
    grp = from_runs([128 + b, 256 - b], [3, 8])
    u, s = rc.rc_tile_kinds(grp)
    assert s[1] == b and s[0] == 0 and s[2] == 0
    assert int(u[0]) == 0b101
    check(grp)


def test_special_tiles():
    check(np.full(1, 0, np.int32))                               # one slot
    check(np.full(300, -1, np.int32))                            # empty ring
    check(from_runs([128, 100, 72], [1, 2, 2]))                  # run ends exactly at a tile edge
    check(from_runs([40, 40, 48], [1, 2, 1]))                    # A B A: three runs, two groups
    check(from_runs([64, 64], [5, -1]))                          # second run empty: not two-run
    check(from_runs([64, 64], [-1, 5]))                          # first slot empty
    check(from_runs([128, 28], [1, 1]))                          # partial last tile, one group
    check(from_runs([128, 10, 18], [1, 1, 2]))                   # partial last tile, two groups
    check(from_runs([5788], [0]))                                # the production ring after one write
    check(from_runs([5031, 757], [0, 1]))                        # the production call


def test_random_layouts():
    rng = np.random.default_rng(7)
    for _ in range(300):
        C = int(rng.choice([1, 64, 127, 128, 129, 300, 1024, 5788, 32768]))
        lengths, total = [], 0
        while total < C:
            n = int(min(C - total, rng.integers(1, 400)))
            lengths.append(n)
            total += n
        groups = rng.integers(-1, 6, len(lengths))
        check(from_runs(lengths, groups))


def test_steady_state_chunk_ring():
    # the chunk workload's ring once the window has restarted: runs of 757
    # starting at a moving offset; 8 of 46 tiles hold two runs, none needs the
    # general path
    C, N = 5788, 757
    grp = np.zeros(C, np.int32)
    for k in range(8):
        for p in range(5031 + k * N, 5031 + (k + 1) * N):
            grp[p % C] = k + 1
    u, s = rc.rc_tile_kinds(grp)
    n_uni = sum(bin(int(w)).count("1") for w in u)
    assert n_uni + int((s > 0).sum()) == 46
    check(grp)


def test_arguments_rejected():
    g = np.zeros(10, np.int32)
    with pytest.raises(rc.RcError):
        rc.rc_tile_kinds(np.zeros(0, np.int32))
    with pytest.raises(rc.RcError):
        rc.rc_tile_kinds(np.zeros(32769, np.int32))
    assert rc.lib.rc_tile_kinds(None, 10, None, None) == rc.RC_ERR_ARG
    u, s = rc.rc_tile_kinds(g)
    assert int(u[0]) == 1 and not s.any()
