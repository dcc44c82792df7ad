"""ctypes binding of librc.so (include/rc.h): argument marshalling only.

Every function here has the name of the C entry point it calls.  Tensors are
passed as their device addresses; positions are passed as a host int64 array.
There is no fallback: if the library is missing, importing raises.  With
RC_BOUNDS_CHECK=1 in the environment the bounds-checked build librc_bounds.so
is loaded instead (same entry points; see rc_build_flags).
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librc_bounds.so" if os.environ.get("RC_BOUNDS_CHECK") == "1" else "librc.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "rc.h")

RC_OK = 0
RC_ERR_ARG = -1
RC_ERR_STATE = -2
RC_ERR_CUDA = -3
RC_ERR_OOM = -4
RC_ERR_TIMEOUT = -5
RC_ERR_UNSUPPORTED = -6
RC_ERR_BOUNDS = -7
RC_BUILD_BOUNDS_CHECK = 1
RC_F_READTIME_ABLATION = 1
RC_F_COPY_WINDOW = 2
RC_F_BF16_CACHE = 4
EMPTY = np.iinfo(np.int64).min
# bounds-checked build: caches whose index checks or guards failed, found when closed
BOUNDS_FAILURES: list[str] = []


class RcError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {rc_status_string(status)} ({status})")


class rc_config(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("slots", ctypes.c_int), ("max_write", ctypes.c_int), ("rope_base", ctypes.c_double),
                ("flags", ctypes.c_uint)]


class rc_ring_view(ctypes.Structure):
    _fields_ = [("kcodes", ctypes.c_void_p), ("vcodes", ctypes.c_void_p), ("kscale", ctypes.c_void_p),
                ("vscale", ctypes.c_void_p), ("group", ctypes.c_void_p), ("heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("slots", ctypes.c_int)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run fp8_ring_kv_cache_gb300.build.build() (nvcc, sm_103a) first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    sig = {
        "rc_cache_create": ([ctypes.POINTER(rc_config), I, ctypes.POINTER(P)], I),
        "rc_cache_write": ([P, I, P, P, P, I, P], I),
        "rc_cache_delta_rotate": ([P, I64, P], I),
        "rc_cache_window_shift": ([P, I64, P], I),
        "rc_attend": ([P, I, P, P, I, P], I),
        "rc_attend_readtime": ([P, I, P, P, I, P], I),
        "rc_cache_destroy": ([P], None),
        "rc_status_string": ([I], ctypes.c_char_p),
        "rc_cache_sync": ([P], I),
        "rc_build_flags": ([], ctypes.c_uint),
        "rc_cache_export": ([P, I, P, P, P, P, P, P], I),
        "rc_cache_export_readtime": ([P, P, P, P, P], I),
        "rc_cache_export_bf16": ([P, I, P, P, P, P], I),
        "rc_cache_write_fused": ([P, I, P, ctypes.c_float, P, ctypes.c_float, P, ctypes.c_float, I, P, I, P], I),
        "rc_cache_occupancy": ([P, I], I),
        "rc_cache_delta_total": ([P], I64),
        "rc_cache_launch_count": ([P], I64),
        "rc_cache_set_wait_limit": ([P, ctypes.c_uint64], I),
        "rc_tile_kinds": ([P, I, P, P], I),
        "rc_ring_write_noalloc": ([ctypes.POINTER(rc_ring_view), P, P, P, I, I64, ctypes.c_int32,
                                   ctypes.c_double, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


def declared_symbols() -> list[str]:
    """Names of the functions include/rc.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rc_\w+)\s*\(", text)))


def _check(st: int, what: str) -> None:
    if st != RC_OK:
        raise RcError(st, what)


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev_ptr(t, dtype, shape, what: str) -> ctypes.c_void_p:
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def rc_status_string(status: int) -> str:
    return lib.rc_status_string(int(status)).decode()


def rc_build_flags() -> int:
    return int(lib.rc_build_flags())


def rc_cache_create(layers: int, heads: int, head_dim: int, slots: int, max_write: int | None = None,
                    rope_base: float = 10000.0, flags: int = 0, device: int = 0) -> ctypes.c_void_p:
    cfg = rc_config(layers, heads, head_dim, slots, slots if max_write is None else max_write, rope_base, flags)
    h = ctypes.c_void_p()
    _check(lib.rc_cache_create(ctypes.byref(cfg), int(device), ctypes.byref(h)), "rc_cache_create")
    return h


def rc_cache_destroy(h) -> None:
    lib.rc_cache_destroy(h)


def rc_cache_write(h, layer: int, K, V, positions, heads: int, head_dim: int, stream=None) -> None:
    import torch
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
    n = int(pos.shape[0])
    shape = (n, heads, head_dim)
    kp = _dev_ptr(K, torch.bfloat16, shape, "K")
    vp = _dev_ptr(V, torch.bfloat16, shape, "V")
    _check(lib.rc_cache_write(h, int(layer), kp, vp, pos.ctypes.data_as(ctypes.c_void_p), n, _stream_ptr(stream)),
           "rc_cache_write")


def rc_cache_write_fused(h, layer: int, X, x_scale: float, Wk, wk_scale: float, Wv, wv_scale: float, positions,
                         heads: int, head_dim: int, stream=None) -> None:
    """X: CUDA uint8 [n][hidden] E4M3 codes; Wk, Wv: CUDA uint8 [heads*head_dim][hidden]."""
    import torch
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
    n = pos.shape[0]
    hidden = X.shape[1]
    xp = _dev_ptr(X, torch.uint8, (n, hidden), "X")
    kp = _dev_ptr(Wk, torch.uint8, (heads * head_dim, hidden), "Wk")
    vp = _dev_ptr(Wv, torch.uint8, (heads * head_dim, hidden), "Wv")
    _check(lib.rc_cache_write_fused(h, int(layer), xp, float(x_scale), kp, float(wk_scale), vp, float(wv_scale),
                                    int(hidden), _np_ptr(pos), n, _stream_ptr(stream)), "rc_cache_write_fused")


def rc_cache_delta_rotate(h, delta: int, stream=None) -> None:
    _check(lib.rc_cache_delta_rotate(h, int(delta), _stream_ptr(stream)), "rc_cache_delta_rotate")


def rc_cache_window_shift(h, k: int, stream=None) -> None:
    _check(lib.rc_cache_window_shift(h, int(k), _stream_ptr(stream)), "rc_cache_window_shift")


def rc_attend(h, layer: int, Q, out, heads: int, head_dim: int, stream=None) -> None:
    import torch
    n = int(Q.shape[0])
    qp = _dev_ptr(Q, torch.bfloat16, (n, heads, head_dim), "Q")
    op = _dev_ptr(out, torch.float32, (n, heads, head_dim), "out")
    _check(lib.rc_attend(h, int(layer), qp, op, n, _stream_ptr(stream)), "rc_attend")


def rc_attend_readtime(h, layer: int, Q, out, heads: int, head_dim: int, stream=None) -> None:
    import torch
    n = int(Q.shape[0])
    qp = _dev_ptr(Q, torch.bfloat16, (n, heads, head_dim), "Q")
    op = _dev_ptr(out, torch.float32, (n, heads, head_dim), "out")
    _check(lib.rc_attend_readtime(h, int(layer), qp, op, n, _stream_ptr(stream)), "rc_attend_readtime")


def rc_cache_sync(h) -> None:
    _check(lib.rc_cache_sync(h), "rc_cache_sync")


def _np_ptr(a: np.ndarray) -> ctypes.c_void_p:
    return a.ctypes.data_as(ctypes.c_void_p)


def rc_cache_export(h, layer: int, heads: int, head_dim: int, slots: int) -> dict:
    st = dict(kcodes=np.zeros((heads, slots, head_dim), np.uint8), kscale=np.zeros((heads, slots), np.float32),
              vcodes=np.zeros((heads, slots, head_dim), np.uint8), vscale=np.zeros((heads, slots), np.float32),
              pos=np.zeros(slots, np.int64), gid=np.zeros(slots, np.int64))
    _check(lib.rc_cache_export(h, int(layer), *[_np_ptr(st[k]) for k in
                                                ("kcodes", "kscale", "vcodes", "vscale", "pos", "gid")]),
           "rc_cache_export")
    return st


def rc_cache_export_readtime(h, heads: int, head_dim: int, slots: int) -> dict:
    st = dict(kcodes=np.zeros((heads, slots, head_dim), np.uint8), kscale=np.zeros((heads, slots), np.float32),
              vcodes=np.zeros((heads, slots, head_dim), np.uint8), vscale=np.zeros((heads, slots), np.float32))
    _check(lib.rc_cache_export_readtime(h, *[_np_ptr(st[k]) for k in ("kcodes", "kscale", "vcodes", "vscale")]),
           "rc_cache_export_readtime")
    return st


def rc_cache_export_bf16(h, layer: int, heads: int, head_dim: int, slots: int) -> dict:
    st = dict(kbits=np.zeros((heads, slots, head_dim), np.uint16), vbits=np.zeros((heads, slots, head_dim), np.uint16),
              pos=np.zeros(slots, np.int64), gid=np.zeros(slots, np.int64))
    _check(lib.rc_cache_export_bf16(h, int(layer), *[_np_ptr(st[k]) for k in ("kbits", "vbits", "pos", "gid")]),
           "rc_cache_export_bf16")
    return st


def rc_tile_kinds(grp) -> tuple[np.ndarray, np.ndarray]:
    """(uniform [4] uint64 bitmask, split [256] uint8) of a ring's slot groups."""
    g = np.ascontiguousarray(np.asarray(grp, dtype=np.int32))
    uniform = np.zeros(4, np.uint64)
    split = np.zeros(256, np.uint8)
    _check(lib.rc_tile_kinds(_np_ptr(g), int(g.shape[0]), _np_ptr(uniform), _np_ptr(split)), "rc_tile_kinds")
    return uniform, split


def rc_cache_occupancy(h, layer: int) -> int:
    v = lib.rc_cache_occupancy(h, int(layer))
    if v < 0:
        raise RcError(v, "rc_cache_occupancy")
    return v


def rc_cache_delta_total(h) -> int:
    return int(lib.rc_cache_delta_total(h))


def rc_cache_launch_count(h) -> int:
    return int(lib.rc_cache_launch_count(h))


def rc_cache_set_wait_limit(h, ns: int) -> None:
    _check(lib.rc_cache_set_wait_limit(h, int(ns)), "rc_cache_set_wait_limit")


class RingKVCache:
    """Owns one rc_cache handle; methods forward to the C entry points."""

    def __init__(self, layers: int, heads: int, head_dim: int, slots: int, max_write: int | None = None,
                 rope_base: float = 10000.0, readtime_ablation: bool = False, device: int = 0,
                 copy_window: bool = False, bf16_cache: bool = False):
        self.layers, self.heads, self.head_dim, self.slots = layers, heads, head_dim, slots
        self.max_write = slots if max_write is None else max_write
        flags = ((RC_F_READTIME_ABLATION if readtime_ablation else 0) | (RC_F_COPY_WINDOW if copy_window else 0) |
                 (RC_F_BF16_CACHE if bf16_cache else 0))
        self.bf16_cache = bf16_cache
        self.handle = rc_cache_create(layers, heads, head_dim, slots, self.max_write, rope_base, flags, device)

    def close(self) -> None:
        if getattr(self, "handle", None):
            if lib.rc_build_flags() & RC_BUILD_BOUNDS_CHECK:
                # the bounds-checked build: a failed index check or guard that
                # no sync reported yet is recorded before the handle goes
                st = lib.rc_cache_sync(self.handle)
                if st == RC_ERR_BOUNDS:
                    BOUNDS_FAILURES.append(f"{self.layers}x{self.heads}x{self.head_dim}, {self.slots} slots")
            rc_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        self.close()

    def write(self, layer, K, V, positions, stream=None):
        rc_cache_write(self.handle, layer, K, V, positions, self.heads, self.head_dim, stream)

    def write_fused(self, layer, X, x_scale, Wk, wk_scale, Wv, wv_scale, positions, stream=None):
        rc_cache_write_fused(self.handle, layer, X, x_scale, Wk, wk_scale, Wv, wv_scale, positions, self.heads,
                             self.head_dim, stream)

    def delta_rotate(self, delta, stream=None):
        rc_cache_delta_rotate(self.handle, delta, stream)

    def window_shift(self, k, stream=None):
        rc_cache_window_shift(self.handle, k, stream)

    def attend(self, layer, Q, out, stream=None):
        rc_attend(self.handle, layer, Q, out, self.heads, self.head_dim, stream)

    def attend_readtime(self, layer, Q, out, stream=None):
        rc_attend_readtime(self.handle, layer, Q, out, self.heads, self.head_dim, stream)

    def sync(self):
        rc_cache_sync(self.handle)

    def export(self, layer):
        if self.bf16_cache:
            return rc_cache_export_bf16(self.handle, layer, self.heads, self.head_dim, self.slots)
        return rc_cache_export(self.handle, layer, self.heads, self.head_dim, self.slots)

    def export_readtime(self):
        return rc_cache_export_readtime(self.handle, self.heads, self.head_dim, self.slots)

    def occupancy(self, layer):
        return rc_cache_occupancy(self.handle, layer)

    @property
    def delta_total(self):
        return rc_cache_delta_total(self.handle)

    @property
    def launch_count(self):
        return rc_cache_launch_count(self.handle)

    def set_wait_limit(self, ns):
        rc_cache_set_wait_limit(self.handle, ns)


RC_NOALLOC_MAX_TOKENS = 4096


def rc_ring_write_noalloc(ring: dict, K, V, positions, delta_total: int, group: int,
                          rope_base: float = 10000.0, stream=None) -> None:
    """Write into caller-owned ring tensors without any device allocation.

    ring: dict of torch CUDA tensors kcodes, vcodes (uint8), kscale, vscale
    (float32), group (int32) laid out as include/rc.h describes, plus ints
    heads, head_dim, slots."""
    import torch
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
    n = int(pos.shape[0])
    H, Dh, C = int(ring["heads"]), int(ring["head_dim"]), int(ring["slots"])
    T = (C + 127) // 128
    view = rc_ring_view(
        _dev_ptr(ring["kcodes"], torch.uint8, (H * T * 128 * Dh,), "kcodes").value,
        _dev_ptr(ring["vcodes"], torch.uint8, (H * T * 128 * Dh,), "vcodes").value,
        _dev_ptr(ring["kscale"], torch.float32, (H * T * 128,), "kscale").value,
        _dev_ptr(ring["vscale"], torch.float32, (H * T * 128,), "vscale").value,
        _dev_ptr(ring["group"], torch.int32, (T * 128,), "group").value, H, Dh, C)
    kp = _dev_ptr(K, torch.bfloat16, (n, H, Dh), "K")
    vp = _dev_ptr(V, torch.bfloat16, (n, H, Dh), "V")
    _check(lib.rc_ring_write_noalloc(ctypes.byref(view), kp, vp, pos.ctypes.data_as(ctypes.c_void_p), n,
                                     int(delta_total), int(group), float(rope_base), _stream_ptr(stream)),
           "rc_ring_write_noalloc")
