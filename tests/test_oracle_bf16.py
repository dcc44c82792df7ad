"""Pins of the oracle's bf16 cache (the non-FP8 cache of the comparison the
pages draw, cpdf.ai blog, section "Blackwell, escalabilidade e limites do
decodificador"), each against something other than the oracle: an exact
rational rounding, torch's float32 -> bfloat16 cast, an independent complex
formulation of RoPE, torch fp64 attention, the FP8 oracle's bookkeeping and
closed forms."""
import math
from fractions import Fraction

import numpy as np
import torch

import oracle


def bf16_exact(x: float) -> float:
    """x rounded to bf16 (8 significant bits, ties to even, subnormal step 2^-133), exactly."""
    if x == 0.0:
        return x
    a = Fraction(abs(x))
    e = math.frexp(abs(x))[1]
    step = Fraction(2) ** max(e - 8, -133)
    q = a / step
    r = math.floor(q)
    rem = q - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    return math.copysign(float(r * step), x)


def bits_to_float(b: int) -> float:
    return float(np.array([b << 16], np.uint32).view(np.float32)[0])


def test_bf16_encode_exact_rounding():
    rng = np.random.default_rng(3)
    vals = list(rng.standard_normal(3000) * np.exp2(rng.integers(-140, 120, 3000)))
    # ties in several binades, both parities, and the subnormal range
    for e in (-130, -20, 0, 7, 60):
        for m in (1, 3, 5, 255):
            vals.append(math.ldexp(2 * m + 1, e - 9))
    vals += [0.0, -0.0, 2.0 ** -133, 3 * 2.0 ** -134, 1.0, -448.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]
    for x in vals:
        got = bits_to_float(oracle.bf16_encode(x))
        want = bf16_exact(float(x))
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (x, got, want)


def test_bf16_encode_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_encode(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, want)


def rope_complex(x: np.ndarray, pos, d: int, base: float = 10000.0) -> np.ndarray:
    """RoPE as a complex rotation of the pairs (x[2i] + i x[2i+1]) by p theta_i."""
    z = x[..., 0::2] + 1j * x[..., 1::2]
    theta = base ** (-2.0 * np.arange(d // 2) / d)
    z = z * np.exp(1j * np.asarray(pos, np.float64)[:, None, None] * theta)
    out = np.empty(x.shape, np.float64)
    out[..., 0::2], out[..., 1::2] = z.real, z.imag
    return out


def bf16_round_array(x: np.ndarray) -> np.ndarray:
    return np.vectorize(bf16_exact)(x)


def ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    def ordered(b):
        b = b.astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def to_bits(x: np.ndarray) -> np.ndarray:
    return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def test_write_stores_rounded_rotated_keys_and_exact_values():
    H, d, C, n = 2, 16, 40, 12
    o = oracle.OracleBf16Cache(1, H, d, C)
    k, v = _bf16((n, H, d), 1, 3.0), _bf16((n, H, d), 2)
    pos = np.arange(100, 100 + n)
    o.write(0, k, v, pos)
    st = o.export(0)
    slots = pos % C
    want = to_bits(bf16_round_array(rope_complex(k.double().numpy(), pos, d)))
    got = st["kbits"][:, slots].transpose(1, 0, 2)
    du = ulp_diff(got, want)
    assert du.max() <= 1 and (du == 0).mean() >= 0.999
    vb = v.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(st["vbits"][:, slots].transpose(1, 0, 2), vb)


def test_delta_rounds_the_rerotated_keys():
    H, d, C = 2, 16, 32
    o = oracle.OracleBf16Cache(1, H, d, C)
    o.write(0, _bf16((20, H, d), 5, 2.0), _bf16((20, H, d), 6), np.arange(0, 20))
    before = o.export(0)
    o.delta_rotate(-7)
    after = o.export(0)
    occ = before["pos"] != oracle.EMPTY
    x = np.vectorize(bits_to_float)(before["kbits"][:, occ].transpose(1, 0, 2).astype(np.int64))
    want = to_bits(bf16_round_array(rope_complex(x, np.full(occ.sum(), -7), d)))
    du = ulp_diff(after["kbits"][:, occ].transpose(1, 0, 2), want)
    assert du.max() <= 1 and (du == 0).mean() >= 0.999
    assert np.array_equal(after["vbits"], before["vbits"])
    assert np.array_equal(after["pos"][occ], before["pos"][occ] - 7)


def test_attention_is_sdpa_over_the_stored_values():
    H, d, C, n = 2, 16, 24, 8
    o = oracle.OracleBf16Cache(1, H, d, C)
    o.write(0, _bf16((16, H, d), 7), _bf16((16, H, d), 8), np.arange(0, 16))
    q = _bf16((n, H, d), 9)
    k, v = _bf16((n, H, d), 10), _bf16((n, H, d), 11)
    pos = np.arange(16, 16 + n)
    o.write(0, k, v, pos)
    out = o.attend(0, q)
    st = o.export(0)
    occ = st["pos"] != oracle.EMPTY
    dec = np.vectorize(bits_to_float)
    K = torch.from_numpy(dec(st["kbits"][:, occ].astype(np.int64)))
    V = torch.from_numpy(dec(st["vbits"][:, occ].astype(np.int64)))
    Q = torch.from_numpy(rope_complex(q.double().numpy(), pos, d)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V).permute(1, 0, 2).numpy()
    assert np.abs(out - ref).max() < 1e-12


def test_one_slot_gives_its_value():
    H, d = 1, 8
    o = oracle.OracleBf16Cache(1, H, d, 4)
    v = _bf16((1, H, d), 12)
    o.write(0, _bf16((1, H, d), 13), v, [5])
    out = o.attend(0, _bf16((1, H, d), 14))
    assert np.array_equal(out[0, 0], v.double().numpy()[0, 0])


def test_bookkeeping_matches_the_fp8_cache():
    H, d, C = 1, 8, 50
    b = oracle.OracleBf16Cache(2, H, d, C)
    f = oracle.OracleCache(2, H, d, C)
    rng = np.random.default_rng(15)
    p = [0, 0]
    for i in range(25):
        layer = int(rng.integers(0, 2))
        n = int(rng.integers(1, 30))
        k, v = _bf16((n, H, d), 100 + i), _bf16((n, H, d), 200 + i)
        pos = np.arange(p[layer], p[layer] + n)
        p[layer] += n
        b.write(layer, k, v, pos)
        f.write(layer, k, v, pos)
        if i % 7 == 6:
            delta = int(rng.integers(-60, 10))
            b.delta_rotate(delta)
            f.delta_rotate(delta)
        for layer in range(2):
            sb, sf = b.export(layer), f.export(layer)
            assert np.array_equal(sb["pos"], sf["pos"]) and np.array_equal(sb["gid"], sf["gid"])
            assert np.array_equal(b.last_positions(layer), f.last_positions(layer))
