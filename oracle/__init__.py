"""Oracle for the write-time FP8 ring KV cache -- TEST INFRASTRUCTURE ONLY.

A plain fp64 C implementation (``rc_oracle.c``) of what the cache computes:
the ring-slot map, write-time RoPE and per-head E4M3 quantisation, the delta
rotation on a position reset, and softmax attention over the dequantised cache
(``OracleCache``); and the same ring with bf16 storage, the non-FP8 cache of
the pages' comparison (``OracleBf16Cache``).  This module compiles it with gcc
and wraps it with ctypes.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
and imports nothing from it.

Sources: the pages about "Runway Characters: Serving a 57B Video Diffusion
Transformer for Real-Time Conversation" (arXiv 2611.05642): the paperdot
abstract mirror (the cache as a ring; keys quantised to FP8 after RoPE a
single time, at write; stored keys rotated by the difference when positions reset; 757 new
tokens among 5,788 slots) and the cpdf.ai
blog sections "Como rodar 57B em tempo real com batch size 1" (write time
instead of read time, ring without copies) and "Blackwell, escalabilidade e
limites do decodificador" (per-head scales).  The readings of what the pages
leave open are listed at the top of ``rc_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rc_oracle.c")
_LIB = os.path.join(_HERE, "librc_oracle.so")
EMPTY = np.iinfo(np.int64).min

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile rc_oracle.c into librc_oracle.so (gcc, -O2, OpenMP, strict IEEE)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_decode.restype = f64
        lib.orc_e4m3_encode.argtypes = [f64]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_rope_theta.argtypes = [i32, i32, f64]
        lib.orc_rope_theta.restype = f64
        lib.orc_rope_rows.argtypes = [P, i32, i32, P, f64]
        lib.orc_rope_rows.restype = None
        lib.orc_scale_from_amax.argtypes = [f64]
        lib.orc_scale_from_amax.restype = ctypes.c_float
        lib.orc_attention_rows.argtypes = [P, i32, P, P, i32, i32, P]
        lib.orc_attention_rows.restype = None
        lib.orc_create.argtypes = [i32, i32, i32, i32, f64]
        lib.orc_create.restype = P
        lib.orc_destroy.argtypes = [P]
        lib.orc_destroy.restype = None
        lib.orc_slot_of.argtypes = [P, i64]
        lib.orc_slot_of.restype = i64
        lib.orc_write.argtypes = [P, i32, P, P, P, i32]
        lib.orc_write.restype = i32
        lib.orc_write_proj.argtypes = [P, i32, P, f64, P, f64, P, f64, i32, P, i32]
        lib.orc_write_proj.restype = i32
        lib.orc_delta_rotate.argtypes = [P, i64]
        lib.orc_delta_rotate.restype = None
        lib.orc_attend.argtypes = [P, i32, P, i32, P]
        lib.orc_attend.restype = i32
        lib.orc_attend_image.argtypes = [i32, i32, i32, f64, P, P, P, P, P, P, P, i32, P]
        lib.orc_attend_image.restype = i32
        lib.orc_readtime_image.argtypes = [i32, i32, i32, f64, P, P, P, P, P, P, P]
        lib.orc_readtime_image.restype = None
        lib.orc_export.argtypes = [P, i32, P, P, P, P, P, P]
        lib.orc_export.restype = None
        lib.orc_import.argtypes = [P, i32, P, P, P, P, P, P, P, i32]
        lib.orc_import.restype = None
        lib.orc_set_counters.argtypes = [P, i64, i64]
        lib.orc_set_counters.restype = None
        lib.orc_delta_total.argtypes = [P]
        lib.orc_delta_total.restype = i64
        lib.orc_last_n.argtypes = [P, i32]
        lib.orc_last_n.restype = i32
        lib.orc_last_pos.argtypes = [P, i32, P]
        lib.orc_last_pos.restype = None
        # the bf16 cache
        lib.orc_bf16_encode.argtypes = [f64]
        lib.orc_bf16_encode.restype = ctypes.c_uint16
        lib.orc_b_create.argtypes = [i32, i32, i32, i32, f64]
        lib.orc_b_create.restype = P
        lib.orc_b_destroy.argtypes = [P]
        lib.orc_b_destroy.restype = None
        lib.orc_b_write.argtypes = [P, i32, P, P, P, i32]
        lib.orc_b_write.restype = i32
        lib.orc_b_delta_rotate.argtypes = [P, i64]
        lib.orc_b_delta_rotate.restype = None
        lib.orc_b_attend.argtypes = [P, i32, P, i32, P]
        lib.orc_b_attend.restype = i32
        lib.orc_b_export.argtypes = [P, i32, P, P, P, P]
        lib.orc_b_export.restype = None
        lib.orc_b_last_n.argtypes = [P, i32]
        lib.orc_b_last_n.restype = i32
        lib.orc_b_last_pos.argtypes = [P, i32, P]
        lib.orc_b_last_pos.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u8(x) -> np.ndarray:
    """uint8 codes as a contiguous numpy array (accepts a torch uint8 tensor or a numpy array)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint8
        return np.ascontiguousarray(x)
    return np.ascontiguousarray(x.detach().cpu().contiguous().numpy())


def _bf16_bits(x) -> np.ndarray:
    """bf16 data as uint16 bit patterns (accepts a torch bf16 tensor or uint16 array)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # local: only for accepting torch inputs
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


# ------------------------------------------------------------------ primitives

def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(x: float) -> int:
    return int(_load().orc_e4m3_encode(float(x)))


def e4m3_decode_all() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def bf16_encode(x: float) -> int:
    """bf16 bits of x rounded once from fp64, to nearest with ties to even."""
    return int(_load().orc_bf16_encode(float(x)))


def rope_theta(i: int, d: int, base: float = 10000.0) -> float:
    return _load().orc_rope_theta(i, d, base)


def rope_rows(x: np.ndarray, positions, base: float = 10000.0) -> np.ndarray:
    """Return a rotated copy of x ([n][d] fp64); row t rotated by positions[t]."""
    x = np.array(x, dtype=np.float64, order="C", copy=True)
    n, d = x.shape
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
    assert pos.shape == (n,)
    _load().orc_rope_rows(_ptr(x), n, d, _ptr(pos), base)
    return x


def scale_from_amax(amax: float) -> float:
    return float(_load().orc_scale_from_amax(float(amax)))


def attention_rows(q: np.ndarray, khat: np.ndarray, vhat: np.ndarray) -> np.ndarray:
    """Softmax attention of rotated queries q [n][d] over khat, vhat [m][d] (fp64)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    khat = np.ascontiguousarray(khat, dtype=np.float64)
    vhat = np.ascontiguousarray(vhat, dtype=np.float64)
    n, d = q.shape
    m = khat.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    _load().orc_attention_rows(_ptr(q), n, _ptr(khat), _ptr(vhat), m, d, _ptr(out))
    return out


def attend_image(kc, sk, vc, sv, pos, Q, qpos, base: float = 10000.0) -> np.ndarray:
    """Attention over an explicit cache image of one layer.

    kc, vc: uint8 [H][C][d]; sk, sv: float32 [H][C]; pos: int64 [C] (EMPTY = free);
    Q: bf16 [n][H][d]; qpos: int64 [n].  Returns fp64 [n][H][d].
    """
    kc = np.ascontiguousarray(kc, dtype=np.uint8)
    vc = np.ascontiguousarray(vc, dtype=np.uint8)
    sk = np.ascontiguousarray(sk, dtype=np.float32)
    sv = np.ascontiguousarray(sv, dtype=np.float32)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    qb = _bf16_bits(Q)
    qpos = np.ascontiguousarray(qpos, dtype=np.int64)
    H, C, d = kc.shape
    n = qb.shape[0]
    assert qb.shape == (n, H, d) and qpos.shape == (n,)
    out = np.zeros((n, H, d), dtype=np.float64)
    m = _load().orc_attend_image(H, d, C, base, _ptr(kc), _ptr(sk), _ptr(vc), _ptr(sv),
                                 _ptr(pos), _ptr(qb), _ptr(qpos), n, _ptr(out))
    if m < 0:
        raise ValueError("attention over an empty cache")
    return out


def readtime_image(kraw, vraw, pos, base: float = 10000.0) -> dict:
    """Read-time quantisation of a whole layer: one scale per head over every occupied slot.

    kraw, vraw: bf16 [H][C][d] (the unrotated rows of every slot); pos: int64 [C].
    """
    kb, vb = _bf16_bits(kraw), _bf16_bits(vraw)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    H, C, d = kb.shape
    st = dict(kcodes=np.zeros((H, C, d), np.uint8), kscale=np.zeros((H, C), np.float32),
              vcodes=np.zeros((H, C, d), np.uint8), vscale=np.zeros((H, C), np.float32))
    _load().orc_readtime_image(H, d, C, base, _ptr(kb), _ptr(vb), _ptr(pos), _ptr(st["kcodes"]),
                               _ptr(st["kscale"]), _ptr(st["vcodes"]), _ptr(st["vscale"]))
    return st


# ------------------------------------------------------------------ state machine

class OracleCache:
    """The cache state machine: write / delta_rotate / attend, all in fp64."""

    def __init__(self, layers: int, heads: int, head_dim: int, slots: int,
                 rope_base: float = 10000.0):
        self._lib = _load()
        self.L, self.H, self.d, self.C = layers, heads, head_dim, slots
        self.base = rope_base
        self._h = self._lib.orc_create(layers, heads, head_dim, slots, rope_base)
        if not self._h:
            raise ValueError("bad oracle cache shape")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.orc_destroy(h)
            self._h = None

    def slot_of(self, p: int) -> int:
        return int(self._lib.orc_slot_of(self._h, int(p)))

    def write(self, layer: int, K, V, positions) -> None:
        kb, vb = _bf16_bits(K), _bf16_bits(V)
        pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
        n = pos.shape[0]
        assert kb.shape == (n, self.H, self.d) and vb.shape == kb.shape
        rc = self._lib.orc_write(self._h, layer, _ptr(kb), _ptr(vb), _ptr(pos), n)
        if rc != 0:
            raise ValueError("oracle write rejected (layer, n or duplicate slot)")

    def write_proj(self, layer: int, X, xs: float, Wk, wks: float, Wv, wvs: float, positions) -> None:
        """The write fused into the K/V projection: X [n][hidden], Wk and Wv
        [H*d][hidden] uint8 E4M3 codes with one scale each (see orc_write_proj)."""
        x = _u8(X)
        wk, wv = _u8(Wk), _u8(Wv)
        pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
        n, hidden = x.shape
        assert n == pos.shape[0] and wk.shape == (self.H * self.d, hidden) and wv.shape == wk.shape
        rc = self._lib.orc_write_proj(self._h, layer, _ptr(x), float(xs), _ptr(wk), float(wks), _ptr(wv),
                                      float(wvs), hidden, _ptr(pos), n)
        if rc != 0:
            raise ValueError("oracle write rejected (layer, n or duplicate slot)")

    def delta_rotate(self, delta: int) -> None:
        self._lib.orc_delta_rotate(self._h, int(delta))

    def attend(self, layer: int, Q) -> np.ndarray:
        qb = _bf16_bits(Q)
        n = qb.shape[0]
        out = np.zeros((n, self.H, self.d), dtype=np.float64)
        rc = self._lib.orc_attend(self._h, layer, _ptr(qb), n, _ptr(out))
        if rc == -1:
            raise ValueError("bad attend arguments")
        if rc == -2:
            raise RuntimeError("attend: query count differs from the last write, or layer empty")
        return out

    def export(self, layer: int) -> dict:
        H, C, d = self.H, self.C, self.d
        st = dict(kcodes=np.zeros((H, C, d), np.uint8), kscale=np.zeros((H, C), np.float32),
                  vcodes=np.zeros((H, C, d), np.uint8), vscale=np.zeros((H, C), np.float32),
                  pos=np.zeros(C, np.int64), gid=np.zeros(C, np.int64))
        self._lib.orc_export(self._h, layer, _ptr(st["kcodes"]), _ptr(st["kscale"]),
                             _ptr(st["vcodes"]), _ptr(st["vscale"]), _ptr(st["pos"]), _ptr(st["gid"]))
        return st

    def import_layer(self, layer: int, st: dict, last_pos, delta_total: int, next_gid: int) -> None:
        lp = np.ascontiguousarray(np.asarray(last_pos, dtype=np.int64))
        arrs = [np.ascontiguousarray(st[k]) for k in ("kcodes", "kscale", "vcodes", "vscale", "pos", "gid")]
        assert arrs[0].dtype == np.uint8 and arrs[1].dtype == np.float32
        assert arrs[4].dtype == np.int64 and arrs[5].dtype == np.int64
        self._lib.orc_import(self._h, layer, *[_ptr(a) for a in arrs], _ptr(lp), int(lp.shape[0]))
        self._lib.orc_set_counters(self._h, int(delta_total), int(next_gid))

    @property
    def delta_total(self) -> int:
        return int(self._lib.orc_delta_total(self._h))

    def last_positions(self, layer: int) -> np.ndarray:
        n = self._lib.orc_last_n(self._h, layer)
        out = np.zeros(n, np.int64)
        if n:
            self._lib.orc_last_pos(self._h, layer, _ptr(out))
        return out


class OracleBf16Cache:
    """The same ring with bf16 storage (the non-FP8 cache): a write stores
    RoPE(K) rounded once to bf16 and V as given; a delta rotation re-rotates
    every stored key in fp64 and rounds it back to bf16; attention reads the
    stored values.  Slots, positions and write serials as in OracleCache."""

    def __init__(self, layers: int, heads: int, head_dim: int, slots: int, rope_base: float = 10000.0):
        self._lib = _load()
        self.L, self.H, self.d, self.C = layers, heads, head_dim, slots
        self.base = rope_base
        self._h = self._lib.orc_b_create(layers, heads, head_dim, slots, rope_base)
        if not self._h:
            raise ValueError("bad oracle cache shape")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.orc_b_destroy(h)
            self._h = None

    def write(self, layer: int, K, V, positions) -> None:
        kb, vb = _bf16_bits(K), _bf16_bits(V)
        pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
        n = pos.shape[0]
        assert kb.shape == (n, self.H, self.d) and vb.shape == kb.shape
        if self._lib.orc_b_write(self._h, layer, _ptr(kb), _ptr(vb), _ptr(pos), n) != 0:
            raise ValueError("oracle write rejected (layer, n or duplicate slot)")

    def delta_rotate(self, delta: int) -> None:
        self._lib.orc_b_delta_rotate(self._h, int(delta))

    def attend(self, layer: int, Q) -> np.ndarray:
        qb = _bf16_bits(Q)
        n = qb.shape[0]
        out = np.zeros((n, self.H, self.d), dtype=np.float64)
        rc = self._lib.orc_b_attend(self._h, layer, _ptr(qb), n, _ptr(out))
        if rc == -1:
            raise ValueError("bad attend arguments")
        if rc == -2:
            raise RuntimeError("attend: query count differs from the last write, or layer empty")
        return out

    def export(self, layer: int) -> dict:
        H, C, d = self.H, self.C, self.d
        st = dict(kbits=np.zeros((H, C, d), np.uint16), vbits=np.zeros((H, C, d), np.uint16),
                  pos=np.zeros(C, np.int64), gid=np.zeros(C, np.int64))
        self._lib.orc_b_export(self._h, layer, _ptr(st["kbits"]), _ptr(st["vbits"]), _ptr(st["pos"]),
                               _ptr(st["gid"]))
        return st

    def last_positions(self, layer: int) -> np.ndarray:
        n = self._lib.orc_b_last_n(self._h, layer)
        out = np.zeros(n, np.int64)
        if n:
            self._lib.orc_b_last_pos(self._h, layer, _ptr(out))
        return out
