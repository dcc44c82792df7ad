"""Pins of the oracle's write-time quantisation.

An independent restatement built from torch's E4M3 conversion and numpy complex
rotation must give the same codes and scales for a write; every group with a
non-zero amax holds a code of magnitude 448; an all-zero group has scale 1 and
zero codes; and the delta rotation requantises with a fresh group scale."""
import numpy as np
import pytest
import torch

import synth_inputs as si


def _independent_write(K, positions, base=10000.0):
    """Codes and scales of one head-major write, from torch + numpy only."""
    x = K.to(torch.float64).numpy()          # [n][H][d]
    n, H, d = x.shape
    i = np.arange(d // 2)
    theta = np.exp(-(2.0 * i / d) * np.log(base))
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * np.asarray(positions)[:, None, None] * theta)
    y = np.empty_like(x)
    y[..., 0::2], y[..., 1::2] = z.real, z.imag
    codes = np.zeros((H, n, d), np.uint8)
    scales = np.zeros(H, np.float32)
    for h in range(H):
        amax = np.abs(y[:, h, :]).max()
        s = np.float32(amax / 448.0) if amax > 0 else np.float32(1.0)
        scales[h] = s
        q = torch.from_numpy(y[:, h, :] / np.float64(s)).to(torch.float32)   # fp32 quotient
        codes[h] = q.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, scales


def test_write_matches_independent_restatement(oracle_mod):
    H, d, C, n = 3, 16, 32, 20
    g = torch.Generator().manual_seed(5)
    K = (torch.randn(n, H, d, generator=g) * torch.tensor([1.0, 3.0, 0.25]).view(1, H, 1)).to(torch.bfloat16)
    V = torch.randn(n, H, d, generator=g).to(torch.bfloat16)
    pos = np.arange(1000, 1000 + n)
    oc = oracle_mod.OracleCache(1, H, d, C)
    oc.write(0, K, V, pos)
    st = oc.export(0)
    slots = [oc.slot_of(p) for p in pos]
    codes, scales = _independent_write(K, pos)
    vcodes, vscales = _independent_write(V, np.zeros(n, np.int64))
    for h in range(H):
        assert st["kscale"][h, slots[0]] == scales[h]
        assert st["vscale"][h, slots[0]] == vscales[h]
        # codes are the E4M3 rounding of the fp32 quotient: identical
        assert np.array_equal(st["kcodes"][h, slots], codes[h])
        assert np.array_equal(st["vcodes"][h, slots], vcodes[h])


def test_every_group_reaches_448(oracle_mod):
    H, d, C = 4, 32, 100
    oc = oracle_mod.OracleCache(1, H, d, C)
    p = 0
    for w, n in enumerate((30, 50, 40, 25)):
        K, V = si.normal_bf16(n, H, d, 10 + w), si.normal_bf16(n, H, d, 20 + w)
        oc.write(0, K, V, np.arange(p, p + n))
        p += n
    oc.delta_rotate(-777)
    st = oc.export(0)
    occ = st["pos"] != oracle_mod.EMPTY
    for h in range(H):
        for g in np.unique(st["gid"][occ]):
            rows = np.nonzero(occ & (st["gid"] == g))[0]
            for key in ("kcodes", "vcodes"):
                mags = st[key][h, rows] & 0x7F
                assert (mags == 0x7E).any()
            # one scale per (head, group)
            assert len(np.unique(st["kscale"][h, rows])) == 1


def test_zero_group(oracle_mod):
    oc = oracle_mod.OracleCache(1, 1, 8, 8)
    z = torch.zeros(3, 1, 8, dtype=torch.bfloat16)
    oc.write(0, z, z, [0, 1, 2])
    st = oc.export(0)
    # +0 and -0 are the same value (a rotated zero may come out as -0)
    assert ((st["kcodes"][0, :3] & 0x7F) == 0).all() and (st["kscale"][0, :3] == 1.0).all()
    assert (st["vcodes"][0, :3] == 0).all() and (st["vscale"][0, :3] == 1.0).all()


def test_scale_formula(oracle_mod):
    for amax in (1.0, 448.0, 3.7e-3, 80.25, 1e-30):
        s = oracle_mod.scale_from_amax(amax)
        assert abs(s - amax / 448.0) <= 1e-6 * amax / 448.0
    assert oracle_mod.scale_from_amax(0.0) == 1.0


def test_delta_rotation_requantises_groups(oracle_mod):
    # after a delta the dequantised keys are close to the re-rotated originals
    H, d, C, n = 2, 16, 16, 16
    K = si.normal_bf16(n, H, d, 31)
    V = si.normal_bf16(n, H, d, 32)
    oc = oracle_mod.OracleCache(1, H, d, C)
    pos = np.arange(n)
    oc.write(0, K, V, pos)
    before_v = oc.export(0)["vcodes"].copy()
    oc.delta_rotate(-12345)
    st = oc.export(0)
    assert np.array_equal(st["vcodes"], before_v)      # values are never rotated
    dq = np.vectorize(oracle_mod.e4m3_decode)(st["kcodes"]) * st["kscale"][..., None]
    for h in range(H):
        exact = oracle_mod.rope_rows(K[:, h, :].to(torch.float64).numpy(), pos - 12345)
        err = np.abs(dq[h] - exact).max() / np.abs(exact).max()
        assert err < 2 * 2.0 ** -4   # two E4M3 roundings, each <= half a step (relative 2^-4)


def test_readtime_image_matches_write_time_when_one_group(oracle_mod):
    # a cache filled by ONE write: the read-time image (one scale per head over
    # the whole cache) equals the write-time state exactly
    H, d, C = 3, 16, 40
    K, V = si.normal_bf16(C, H, d, 41), si.normal_bf16(C, H, d, 42)
    pos = np.arange(500, 500 + C)
    oc = oracle_mod.OracleCache(1, H, d, C)
    oc.write(0, K, V, pos)
    st = oc.export(0)
    slots = np.array([oc.slot_of(p) for p in pos])
    kraw = torch.zeros(H, C, d, dtype=torch.bfloat16)
    vraw = torch.zeros(H, C, d, dtype=torch.bfloat16)
    kraw[:, slots] = K.permute(1, 0, 2)
    vraw[:, slots] = V.permute(1, 0, 2)
    img = oracle_mod.readtime_image(kraw, vraw, st["pos"])
    for k in ("kcodes", "kscale", "vcodes", "vscale"):
        assert np.array_equal(img[k], st[k]), k


def test_readtime_image_whole_cache_scale(oracle_mod):
    # two writes with very different magnitudes: read time uses one scale per head
    H, d, C = 2, 8, 20
    oc = oracle_mod.OracleCache(1, H, d, C)
    K1 = si.normal_bf16(10, H, d, 1, mult=torch.full((H, 1), 10.0))
    K2 = si.normal_bf16(10, H, d, 2)
    oc.write(0, K1, K1, np.arange(10))
    oc.write(0, K2, K2, np.arange(10, 20))
    st = oc.export(0)
    assert st["kscale"][0, 0] != st["kscale"][0, 15]
    kraw = torch.cat([K1, K2]).permute(1, 0, 2).contiguous()
    img = oracle_mod.readtime_image(kraw, kraw, st["pos"])
    assert len(np.unique(img["kscale"][0])) == 1
    x = oracle_mod.rope_rows(kraw[0].to(torch.float64).numpy(), st["pos"])
    assert abs(img["kscale"][0, 0] - np.abs(x).max() / 448) <= 1e-6 * np.abs(x).max() / 448
