"""Pins of the oracle's attention.

Brute force against torch's fp64 scaled_dot_product_attention, closed-form
special cases (one slot, identical keys, zero query), relative-position
invariance, and agreement of the state machine's attend with the image form."""
import numpy as np
import pytest
import torch

import synth_inputs as si


def test_matches_torch_sdpa(oracle_mod):
    rng = np.random.default_rng(0)
    for n, m, d in [(1, 1, 8), (5, 17, 16), (33, 70, 64)]:
        q = rng.standard_normal((n, d)) * 2
        k = rng.standard_normal((m, d))
        v = rng.standard_normal((m, d)) * 3
        got = oracle_mod.attention_rows(q, k, v)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None]
        )[0].numpy()
        assert np.max(np.abs(got - ref)) < 1e-12


def test_special_cases(oracle_mod):
    rng = np.random.default_rng(1)
    d = 16
    v = rng.standard_normal((9, d))
    q = rng.standard_normal((3, d))
    # one slot: the output is that slot's value
    assert np.allclose(oracle_mod.attention_rows(q, v[:1] * 0 + 1, v[:1]), np.repeat(v[:1], 3, 0), atol=0, rtol=1e-15)
    # identical keys, or a zero query: the mean of the values
    k_same = np.repeat(rng.standard_normal((1, d)), 9, 0)
    assert np.max(np.abs(oracle_mod.attention_rows(q, k_same, v) - v.mean(0))) < 1e-13
    k = rng.standard_normal((9, d))
    assert np.max(np.abs(oracle_mod.attention_rows(np.zeros((2, d)), k, v) - v.mean(0))) < 1e-13


def test_relative_position_invariance(oracle_mod):
    rng = np.random.default_rng(2)
    d, m, n = 32, 40, 6
    k, v, q = rng.standard_normal((m, d)), rng.standard_normal((m, d)), rng.standard_normal((n, d))
    kp = rng.integers(0, 5000, m)
    qp = rng.integers(0, 5000, n)
    out0 = oracle_mod.attention_rows(oracle_mod.rope_rows(q, qp), oracle_mod.rope_rows(k, kp), v)
    for delta in (-4999, 17, 190000):
        out1 = oracle_mod.attention_rows(oracle_mod.rope_rows(q, qp + delta),
                                         oracle_mod.rope_rows(k, kp + delta), v)
        assert np.max(np.abs(out1 - out0)) < 1e-9


def test_state_machine_attend_equals_image(oracle_mod):
    H, d, C = 2, 16, 24
    oc = oracle_mod.OracleCache(1, H, d, C)
    K, V = si.normal_bf16(20, H, d, 1), si.normal_bf16(20, H, d, 2)
    oc.write(0, K, V, np.arange(20))
    K2, V2, Q = si.normal_bf16(8, H, d, 3), si.normal_bf16(8, H, d, 4), si.normal_bf16(8, H, d, 5)
    oc.write(0, K2, V2, np.arange(20, 28))      # wraps onto slots 20..23, 0..3
    out = oc.attend(0, Q)
    st = oc.export(0)
    img = oracle_mod.attend_image(st["kcodes"], st["kscale"], st["vcodes"], st["vscale"],
                                  st["pos"], Q, np.arange(20, 28))
    assert np.array_equal(out, img)
    # and against torch SDPA on the dequantised cache, head by head
    dec = np.vectorize(oracle_mod.e4m3_decode)
    occ = st["pos"] != oracle_mod.EMPTY
    for h in range(H):
        kh = dec(st["kcodes"][h][occ]) * st["kscale"][h][occ][:, None]
        vh = dec(st["vcodes"][h][occ]) * st["vscale"][h][occ][:, None]
        qh = oracle_mod.rope_rows(Q[:, h, :].to(torch.float64).numpy(), np.arange(20, 28))
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qh)[None], torch.from_numpy(kh)[None], torch.from_numpy(vh)[None])[0].numpy()
        assert np.max(np.abs(out[:, h, :] - ref)) < 1e-12
    # after a reset the output is unchanged up to requantisation of the keys
    oc.delta_rotate(-1000)
    out2 = oc.attend(0, Q)
    assert np.max(np.abs(out2 - out)) < 0.25


def test_partial_ring_ignores_empty_slots(oracle_mod):
    H, d, C, n = 2, 16, 32, 10
    oc = oracle_mod.OracleCache(1, H, d, C)
    K, V, Q = si.normal_bf16(n, H, d, 7), si.normal_bf16(n, H, d, 8), si.normal_bf16(n, H, d, 9)
    pos = np.arange(100, 100 + n)
    oc.write(0, K, V, pos)
    out = oc.attend(0, Q)
    st = oc.export(0)
    occ = st["pos"] != oracle_mod.EMPTY
    assert occ.sum() == n
    dec = np.vectorize(oracle_mod.e4m3_decode)
    for h in range(H):
        kh = dec(st["kcodes"][h][occ]) * st["kscale"][h][occ][:, None]
        vh = dec(st["vcodes"][h][occ]) * st["vscale"][h][occ][:, None]
        qh = oracle_mod.rope_rows(Q[:, h, :].to(torch.float64).numpy(), pos)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qh)[None], torch.from_numpy(kh)[None], torch.from_numpy(vh)[None])[0].numpy()
        assert np.max(np.abs(out[:, h, :] - ref)) < 1e-12
