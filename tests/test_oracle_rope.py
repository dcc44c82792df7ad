"""Pins of the oracle's rotary position embedding (fp64).

Composition R(a)R(b) = R(a+b) (so a delta rotation equals re-rotation from the
unrotated keys), R(0) = I, pair norms, relative-position invariance of the
score, and an independent complex-number formulation that fixes the pairing
and the sign of the rotation."""
import numpy as np
import pytest

D = 64
BASE = 10000.0


def _rand(n, d=D, seed=0):
    return np.random.default_rng(seed).standard_normal((n, d))


def test_theta_endpoints(oracle_mod):
    assert oracle_mod.rope_theta(0, D, BASE) == 1.0
    th = [oracle_mod.rope_theta(i, D, BASE) for i in range(D // 2)]
    assert all(a > b for a, b in zip(th, th[1:]))
    # theta_i * base^(2i/d) == 1 for every i
    for i, t in enumerate(th):
        assert abs(t * BASE ** (2 * i / D) - 1.0) < 1e-14


def test_d2_closed_form(oracle_mod):
    # with d = 2 the only frequency is 1: (1, 0) at position p -> (cos p, sin p)
    for p in (0, 1, 2, 7, -3, 200000):
        y = oracle_mod.rope_rows(np.array([[1.0, 0.0]]), [p], BASE)[0]
        assert abs(y[0] - np.cos(p)) < 1e-12 and abs(y[1] - np.sin(p)) < 1e-12


def test_identity_at_zero(oracle_mod):
    x = _rand(5)
    assert np.array_equal(oracle_mod.rope_rows(x, [0] * 5, BASE), x)


def test_composition(oracle_mod):
    x = _rand(6, seed=1)
    for a, b in [(3, 11), (200000, -137), (-199999, 5031), (5787, 5788)]:
        two = oracle_mod.rope_rows(oracle_mod.rope_rows(x, [a] * 6, BASE), [b] * 6, BASE)
        one = oracle_mod.rope_rows(x, [a + b] * 6, BASE)
        assert np.max(np.abs(two - one)) < 1e-12 * max(1, abs(a) + abs(b)) ** 0.5 * 10


def test_delta_equals_rerotation(oracle_mod):
    # keys stored rotated at p, then rotated by delta, equal keys rotated at p + delta
    rng = np.random.default_rng(2)
    k = _rand(32, seed=3)
    p = rng.integers(0, 200000, size=32)
    delta = -123457
    stored = oracle_mod.rope_rows(k, p, BASE)
    moved = oracle_mod.rope_rows(stored, [delta] * 32, BASE)
    direct = oracle_mod.rope_rows(k, p + delta, BASE)
    assert np.max(np.abs(moved - direct)) < 1e-10


def test_pair_norms_preserved(oracle_mod):
    x = _rand(8, seed=4)
    y = oracle_mod.rope_rows(x, np.arange(8) * 977, BASE)
    nx = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
    ny = y[:, 0::2] ** 2 + y[:, 1::2] ** 2
    assert np.max(np.abs(nx - ny)) < 1e-12


def test_relative_position_invariance(oracle_mod):
    q, k = _rand(1, seed=5), _rand(1, seed=6)
    def score(p, r):
        return float(oracle_mod.rope_rows(q, [p], BASE)[0] @ oracle_mod.rope_rows(k, [r], BASE)[0])
    base_score = score(100, 37)
    for t in (-5000, 1, 4096, 199000):
        assert abs(score(100 + t, 37 + t) - base_score) < 1e-10


def test_complex_formulation(oracle_mod):
    # pair (x_2i, x_2i+1) as the complex number x_2i + i x_2i+1 multiplied by
    # exp(i p theta_i), with theta_i = base^(-2i/d)
    x = _rand(4, seed=8)
    pos = np.array([0, 1, 5031, -40])
    y = oracle_mod.rope_rows(x, pos, BASE)
    i = np.arange(D // 2)
    theta = np.exp(-(2.0 * i / D) * np.log(BASE))
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * pos[:, None] * theta[None, :])
    assert np.max(np.abs(y[:, 0::2] - z.real)) < 1e-10
    assert np.max(np.abs(y[:, 1::2] - z.imag)) < 1e-10
