"""Pins of the oracle's write fused into the K/V projection (orc_write_proj).

The fused write is the projection K = xs wks X Wk^T, V = xs wvs X Wv^T of
E4M3 operands followed by the write.  Pinned against: (1) the already pinned
bf16 write, which it must equal bit for bit when every row of X selects one
weight column (one-hot X: the products are E4M3 values, which bf16 holds
exactly); (2) an independent torch + numpy restatement (numpy fp64 product of
torch-decoded codes, complex RoPE, torch's E4M3 cast); (3) the exactness of
the fp64 sum, checked with Python integers (every E4M3 value is a multiple of
2^-9)."""
import numpy as np
import torch

from test_oracle_quant import _independent_write


def _codes(rng, shape, top=0x70):
    """Random E4M3 codes of both signs with magnitude codes below `top` (no NaN)."""
    mag = rng.integers(0, top, shape, dtype=np.uint8)
    sign = rng.integers(0, 2, shape, dtype=np.uint8) << 7
    return (mag | sign).astype(np.uint8)


def _decode(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_one_hot_projection_equals_the_bf16_write(oracle_mod):
    H, d, C, n, hidden = 2, 16, 40, 24, 32
    rng = np.random.default_rng(7)
    Wk = _codes(rng, (H * d, hidden))
    Wv = _codes(rng, (H * d, hidden))
    pick = rng.integers(0, hidden, n)
    X = np.zeros((n, hidden), np.uint8)
    X[np.arange(n), pick] = 0x38                      # E4M3 1.0
    pos = np.arange(500, 500 + n)
    a = oracle_mod.OracleCache(1, H, d, C)
    a.write_proj(0, X, 1.0, Wk, 1.0, Wv, 0.5, pos)
    K = torch.from_numpy(_decode(Wk)[:, pick].T.reshape(n, H, d)).to(torch.bfloat16)
    V = torch.from_numpy(0.5 * _decode(Wv)[:, pick].T.reshape(n, H, d)).to(torch.bfloat16)
    assert torch.equal(K.to(torch.float64), torch.from_numpy(_decode(Wk)[:, pick].T.reshape(n, H, d)))
    b = oracle_mod.OracleCache(1, H, d, C)
    b.write(0, K, V, pos)
    sa, sb = a.export(0), b.export(0)
    for key in ("kcodes", "kscale", "vcodes", "vscale", "pos", "gid"):
        assert np.array_equal(sa[key], sb[key]), key


def test_projection_matches_independent_restatement(oracle_mod):
    H, d, C, n, hidden = 3, 16, 64, 40, 96
    rng = np.random.default_rng(8)
    X = _codes(rng, (n, hidden))
    Wk = _codes(rng, (H * d, hidden), top=0x60)
    Wv = _codes(rng, (H * d, hidden), top=0x60)
    xs, wks, wvs = 0.03125, 0.5, 2.0
    pos = np.arange(77, 77 + n)
    oc = oracle_mod.OracleCache(1, H, d, C)
    oc.write_proj(0, X, xs, Wk, wks, Wv, wvs, pos)
    st = oc.export(0)
    K = torch.from_numpy((_decode(X) @ _decode(Wk).T * xs * wks).reshape(n, H, d))
    V = torch.from_numpy((_decode(X) @ _decode(Wv).T * xs * wvs).reshape(n, H, d))
    codes, scales = _independent_write(K, pos)
    vcodes, vscales = _independent_write(V, np.zeros(n, np.int64))
    slots = [oc.slot_of(p) for p in pos]
    for h in range(H):
        assert st["kscale"][h, slots[0]] == scales[h]
        assert st["vscale"][h, slots[0]] == vscales[h]
        assert np.array_equal(st["kcodes"][h, slots], codes[h])
        assert np.array_equal(st["vcodes"][h, slots], vcodes[h])


def test_fp64_projection_sum_is_exact():
    # every E4M3 value is an integer multiple of 2^-9, so a product is a
    # multiple of 2^-18 and a 6,144-term sum an integer times 2^-18 that needs
    # under 53 bits: the fp64 dot product (any order) equals the exact one
    rng = np.random.default_rng(9)
    hidden = 6144
    x = _decode(_codes(rng, (4, hidden), top=0x7F))
    w = _decode(_codes(rng, (4, hidden), top=0x7F))
    got = x @ w.T
    for i in range(4):
        for j in range(4):
            xi = [int(v * 512) for v in x[i]]
            wj = [int(v * 512) for v in w[j]]
            assert all(a == v * 512 for a, v in zip(xi, x[i]))
            exact = sum(a * b for a, b in zip(xi, wj))
            assert got[i, j] * 2.0 ** 18 == exact
