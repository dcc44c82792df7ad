"""Comparison helpers for the CUDA path against the oracle (acceptance bars).

  slots / occupancy / positions / write serials : bit-exact
  per-slot scales                               : within 1e-6 relative
  E4M3 codes                                    : >= 99.99 % identical, the rest
                                                  one step apart in signed-magnitude
                                                  order with +0 == -0
  attention output                              : max-abs <= 3e-2, mean-abs <= 3e-3
"""
import numpy as np

ATTN_MAX_ABS = 3e-2
ATTN_MEAN_ABS = 3e-3
SCALE_REL = 1e-6
CODE_SAME_FRAC = 0.9999


def code_ordinal(c: np.ndarray) -> np.ndarray:
    c = c.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def check_codes(got: np.ndarray, want: np.ndarray, what: str = "codes") -> dict:
    assert got.shape == want.shape, what
    og, ow = code_ordinal(got), code_ordinal(want)
    same = og == ow
    frac = float(same.mean()) if same.size else 1.0
    far = np.abs(og - ow) > 1
    assert not far.any(), f"{what}: {int(far.sum())} codes more than one step apart"
    assert frac >= CODE_SAME_FRAC, f"{what}: only {frac:.6f} identical"
    return dict(identical=frac, one_step=int((~same).sum()))


def check_scales(got: np.ndarray, want: np.ndarray, what: str = "scales") -> float:
    got = got.astype(np.float64)
    want = want.astype(np.float64)
    den = np.where(want == 0, 1.0, np.abs(want))
    rel = np.abs(got - want) / den
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= SCALE_REL, f"{what}: worst relative difference {worst:.3g}"
    return worst


def check_attention(got: np.ndarray, want: np.ndarray, what: str = "attention") -> dict:
    err = np.abs(got.astype(np.float64) - want)
    mx, mean = float(err.max()), float(err.mean())
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert mx <= ATTN_MAX_ABS, f"{what}: max-abs {mx:.4g} > {ATTN_MAX_ABS}"
    assert mean <= ATTN_MEAN_ABS, f"{what}: mean-abs {mean:.4g} > {ATTN_MEAN_ABS}"
    return dict(max_abs=mx, mean_abs=mean)


def check_state(gpu: dict, ora: dict, what: str = "state") -> dict:
    """Compare exported layer states (GPU vs oracle)."""
    assert np.array_equal(gpu["pos"], ora["pos"]), f"{what}: positions differ"
    assert np.array_equal(gpu["gid"], ora["gid"]), f"{what}: write serials differ"
    occ = ora["pos"] != np.iinfo(np.int64).min
    res = {}
    res["k"] = check_codes(gpu["kcodes"][:, occ], ora["kcodes"][:, occ], what + " K codes")
    res["v"] = check_codes(gpu["vcodes"][:, occ], ora["vcodes"][:, occ], what + " V codes")
    res["sk"] = check_scales(gpu["kscale"][:, occ], ora["kscale"][:, occ], what + " K scales")
    res["sv"] = check_scales(gpu["vscale"][:, occ], ora["vscale"][:, occ], what + " V scales")
    return res
