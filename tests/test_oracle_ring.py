"""Pins of the oracle's ring-slot state machine.

Against an independent sliding-window model (a Python deque holding the most
recent C tokens in write order): the stored positions and data equal the
model's window, occupancy is min(total written, C), a reset moves positions but
not slots, rewriting the same positions reuses the same slots, and bad writes
are rejected."""
import collections

import numpy as np
import pytest
import torch

import synth_inputs as si


def _kv(n, H, d, seed):
    return (si.normal_bf16(n, H, d, seed), si.normal_bf16(n, H, d, seed + 1))


def test_window_matches_deque_model(oracle_mod):
    L, H, d, C = 1, 1, 8, 37
    oc = oracle_mod.OracleCache(L, H, d, C)
    window = collections.deque(maxlen=C)
    rng = np.random.default_rng(0)
    p = 0
    total = 0
    for step in range(40):
        n = int(rng.integers(1, C + 1))
        k, v = _kv(n, H, d, 100 + step)
        pos = np.arange(p, p + n)
        oc.write(0, k, v, pos)
        for t in range(n):
            window.append((int(pos[t]), step, t))
        p += n
        total += n
        st = oc.export(0)
        occ = st["pos"] != oracle_mod.EMPTY
        assert occ.sum() == min(total, C)
        assert sorted(st["pos"][occ].tolist()) == sorted(w[0] for w in window)
        # every stored position carries the gid (write serial) the model says
        where = {w[0]: w[1] for w in window}
        for s in np.nonzero(occ)[0]:
            assert st["gid"][s] == where[int(st["pos"][s])]


def test_slot_formula_and_reset(oracle_mod):
    oc = oracle_mod.OracleCache(1, 1, 4, 10)
    assert [oc.slot_of(p) for p in (0, 9, 10, -1, -11)] == [0, 9, 0, 9, 9]
    k, v = _kv(10, 1, 4, 1)
    oc.write(0, k, v, np.arange(100, 110))
    before = oc.export(0)["pos"].copy()
    oc.delta_rotate(-100)
    after = oc.export(0)["pos"]
    # same slots, positions moved by the delta
    assert np.array_equal(after, before - 100)
    for s in range(10):
        assert oc.slot_of(after[s]) == s


def test_rewrite_same_positions_same_slots(oracle_mod):
    oc = oracle_mod.OracleCache(1, 2, 8, 16)
    for pas in range(4):
        k, v = _kv(6, 2, 8, 10 * pas)
        oc.write(0, k, v, np.arange(3, 9))
        st = oc.export(0)
        assert np.array_equal(np.nonzero(st["pos"] != oracle_mod.EMPTY)[0], np.arange(3, 9))
        assert set(st["gid"][3:9].tolist()) == {pas}


def test_rejects_bad_writes(oracle_mod):
    oc = oracle_mod.OracleCache(1, 1, 4, 8)
    k, v = _kv(2, 1, 4, 3)
    with pytest.raises(ValueError):
        oc.write(0, k, v, [0, 8])          # both on slot 0
    with pytest.raises(ValueError):
        oc.write(1, k, v, [0, 1])          # no such layer
    k9, v9 = _kv(9, 1, 4, 4)
    with pytest.raises(ValueError):
        oc.write(0, k9, v9, np.arange(9))  # n > C
    with pytest.raises(RuntimeError):
        oc.attend(0, k)                    # nothing written yet
    oc.write(0, k, v, [0, 1])
    k3, _ = _kv(3, 1, 4, 5)
    with pytest.raises(RuntimeError):
        oc.attend(0, k3)                   # n differs from the last write


def test_tiny_schedule_tables(oracle_mod):
    s = si.TINY
    oc = oracle_mod.OracleCache(s.layers, s.heads, s.head_dim, s.slots)
    window = collections.deque(maxlen=s.slots)
    step = 0
    for op in si.tiny_schedule():
        if op[0] == "write":
            _, layer, p0, n = op
            k, v, q = si.tiny_tensors(1, step, "cpu")
            oc.write(layer, k, v, np.arange(p0, p0 + n))
            window.extend(range(p0, p0 + n))
            step += 1
        elif op[0] == "delta":
            oc.delta_rotate(op[1])
            window = collections.deque((p + op[1] for p in window), maxlen=s.slots)
        st = oc.export(0)
        occ = st["pos"] != oracle_mod.EMPTY
        assert sorted(st["pos"][occ].tolist()) == sorted(window)
    # after the reset and two wrapping writes: positions 24..55 sit in slots 0..31
    st = oc.export(0)
    assert st["pos"][:32].tolist() == list(range(24, 56))
    assert st["pos"][32:].tolist() == list(range(-8, 24))
