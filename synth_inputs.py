"""Seeded synthetic inputs for the ring-cache workloads.

This module only draws random numbers with the shapes, distributions and
schedules of the workloads: bf16 K, V, Q tensors ([n][H][d], token-major),
position vectors, outlier channel masks, per-head standard deviations and the
operation schedules of each workload.  It holds none of the cache's
arithmetic, and both the CUDA path and the oracle take their inputs from it.

Workloads (shapes from the pages: 757 new tokens over a 5,788-slot cache, 240
attention calls per chunk = 4 denoising passes x 60 layers; 48 heads x 128):
  tiny       1 layer, 2 heads, d 64, 64 slots, six 16-token writes (the last
             two wrap), one position reset by -40, N(0,1) data.
  production 48 heads, d 128, 5,788 slots; a 5,031-token prefill, a 757-token
             write, one attention call; K and V N(0,1) with 1 % of the
             (head, channel) pairs scaled by 20.
  chunk      60 layers; the production prefill, then chunks of 4 passes x 60
             layers of (write 757 at the chunk's positions, attend).
  stress     the ring full at positions up to 200,000; 100 x (reset by a delta
             drawn from [-200000, 0], write, attend).
  sustained  3,600 chunks; per (layer, head) std drawn from U[0.5, 4] for Q, K
             and V; a reset every 300 chunks to restart positions at 0.
"""
from __future__ import annotations

import dataclasses

import torch

PROD_HEADS, PROD_DIM, PROD_SLOTS, PROD_NEW, PROD_PREFILL = 48, 128, 5788, 757, 5031
PROD_LAYERS, PROD_PASSES = 60, 4


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def subseed(seed: int, *keys: int) -> int:
    """A deterministic sub-seed for (seed, keys...)."""
    s = int(seed) * 1_000_003 + 12345
    for k in keys:
        s = (s * 6364136223846793005 + int(k) + 1442695040888963407) & 0xFFFFFFFFFFFF
    return s


def outlier_mask(heads: int, dim: int, seed: int, frac: float = 0.01,
                 factor: float = 20.0) -> torch.Tensor:
    """[H][d] fp32 multipliers: round(frac*H*d) (head, channel) pairs get `factor`."""
    g = _gen(subseed(seed, 0xA11), "cpu")
    k = int(round(frac * heads * dim))
    m = torch.ones(heads * dim, dtype=torch.float32)
    idx = torch.randperm(heads * dim, generator=g)[:k]
    m[idx] = factor
    return m.view(heads, dim)


def head_std(layers: int, heads: int, seed: int, lo: float = 0.5, hi: float = 4.0) -> torch.Tensor:
    """[L][H] fp32 standard deviations drawn from U[lo, hi]."""
    g = _gen(subseed(seed, 0x57D), "cpu")
    return lo + (hi - lo) * torch.rand(layers, heads, generator=g)


def normal_bf16(n: int, heads: int, dim: int, seed: int, device="cpu",
                mult: torch.Tensor | None = None) -> torch.Tensor:
    """[n][H][d] bf16 N(0,1) samples, times an optional [H][d] or [H][1] multiplier."""
    g = _gen(seed, device)
    x = torch.randn(n, heads, dim, generator=g, device=device, dtype=torch.float32)
    if mult is not None:
        x = x * mult.to(device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def arange_positions(start: int, n: int) -> torch.Tensor:
    return torch.arange(start, start + n, dtype=torch.int64)


@dataclasses.dataclass
class Shape:
    layers: int
    heads: int
    head_dim: int
    slots: int
    rope_base: float = 10000.0


TINY = Shape(1, 2, 64, 64)
PRODUCTION = Shape(1, PROD_HEADS, PROD_DIM, PROD_SLOTS)
CHUNK = Shape(PROD_LAYERS, PROD_HEADS, PROD_DIM, PROD_SLOTS)


def tiny_schedule():
    """Operations of the tiny workload: ('write', layer, first_position, n),
    ('delta', delta), ('attend', layer).  Writes at 0..63 fill the ring, a
    reset by -40 moves the stored positions to -40..23, and two more writes at
    24..39 and 40..55 wrap onto the oldest slots.  Attention follows every write."""
    ops = []
    for p0 in (0, 16, 32, 48):
        ops += [("write", 0, p0, 16), ("attend", 0)]
    ops.append(("delta", -40))
    for p0 in (24, 40):
        ops += [("write", 0, p0, 16), ("attend", 0)]
    return ops


def tiny_tensors(seed: int, step: int, device="cpu"):
    """K, V, Q for write number `step` of the tiny workload."""
    s = TINY
    k = normal_bf16(16, s.heads, s.head_dim, subseed(seed, step, 1), device)
    v = normal_bf16(16, s.heads, s.head_dim, subseed(seed, step, 2), device)
    q = normal_bf16(16, s.heads, s.head_dim, subseed(seed, step, 3), device)
    return k, v, q


def production_tensors(seed: int, device="cpu", n_prefill: int = PROD_PREFILL,
                       n_new: int = PROD_NEW, heads: int = PROD_HEADS, dim: int = PROD_DIM):
    """Prefill K, V; new K, V; queries for the production call (outliers on K and V)."""
    mult = outlier_mask(heads, dim, seed)
    kp = normal_bf16(n_prefill, heads, dim, subseed(seed, 1), device, mult)
    vp = normal_bf16(n_prefill, heads, dim, subseed(seed, 2), device, mult)
    kn = normal_bf16(n_new, heads, dim, subseed(seed, 3), device, mult)
    vn = normal_bf16(n_new, heads, dim, subseed(seed, 4), device, mult)
    q = normal_bf16(n_new, heads, dim, subseed(seed, 5), device)
    return dict(k_prefill=kp, v_prefill=vp, k_new=kn, v_new=vn, q=q, mult=mult)


def chunk_tensors(seed: int, chunk: int, pas: int, layer: int, device="cpu",
                  n: int = PROD_NEW, heads: int = PROD_HEADS, dim: int = PROD_DIM,
                  mult: torch.Tensor | None = None, std: torch.Tensor | None = None):
    """K, V, Q for (chunk, pass, layer) of the chunk / sustained workloads.

    `mult` ([H][d]) multiplies K and V (outliers); `std` ([H]) multiplies Q, K
    and V alike (per-head standard deviation)."""
    km = mult
    qm = None
    if std is not None:
        s = std.view(heads, 1)
        km = s if km is None else km * s
        qm = s
    k = normal_bf16(n, heads, dim, subseed(seed, chunk, pas, layer, 1), device, km)
    v = normal_bf16(n, heads, dim, subseed(seed, chunk, pas, layer, 2), device, km)
    q = normal_bf16(n, heads, dim, subseed(seed, chunk, pas, layer, 3), device, qm)
    return k, v, q


def stress_deltas(seed: int, count: int = 100, lo: int = -200000, hi: int = 0) -> list[int]:
    """Reset deltas drawn uniformly from the integers in [lo, hi]."""
    g = _gen(subseed(seed, 0xDE17A), "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (count,), generator=g)]


PROD_HIDDEN = 6144  # projection input width (48 heads x 128)


def proj_operands(seed: int, n: int, hidden: int, features: int, device="cpu"):
    """E4M3 operands of the K/V projection: X [n][hidden] from N(0, 1) and Wk,
    Wv [features][hidden] from N(0, 1/hidden), each encoded with one scale
    (amax / 448) by torch's E4M3 cast.  Returns (X, x_scale, Wk, wk_scale, Wv,
    wv_scale), the codes as uint8 tensors on `device`."""
    g = _gen(subseed(seed, 0x9E0), "cpu")

    def enc(t: torch.Tensor):
        s = float(t.abs().max()) / 448.0
        codes = (t / s).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        return codes.to(device), s

    x, xs = enc(torch.randn(n, hidden, generator=g))
    wk, wks = enc(torch.randn(features, hidden, generator=g) / hidden ** 0.5)
    wv, wvs = enc(torch.randn(features, hidden, generator=g) / hidden ** 0.5)
    return x, xs, wk, wks, wv, wvs
