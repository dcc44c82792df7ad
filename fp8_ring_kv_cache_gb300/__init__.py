"""Write-time FP8 ring KV cache for one GB300 (sm_103a).

The compute path is the CUDA library librc.so (C ABI in include/rc.h); this
package only binds it.  Build it with ``python fp8_ring_kv_cache_gb300/build.py`` (or ``__graft_entry__.build()``).

Use (K, V, Q: CUDA bf16 tensors [n][heads][head_dim]; out: CUDA fp32, same shape)::

    import numpy as np, torch
    import fp8_ring_kv_cache_gb300 as rc

    cache = rc.RingKVCache(layers=60, heads=48, head_dim=128, slots=5788)
    cache.write(layer, K, V, np.arange(p0, p0 + n))  # RoPE + per-head E4M3, once
    cache.attend(layer, Q, out)                      # Q = the last write's tokens
    cache.delta_rotate(-757)                         # positions reset: keys re-rotated in place
    cache.sync()                                     # raises RcError on a kernel error

``RingKVCache(..., bf16_cache=True)`` keeps the same ring in bf16 (no scales):
the non-FP8 side of the FP8-versus-bf16 cache comparison.

Every call is stream-ordered on torch's current stream (or ``stream=``); no
call after construction allocates device memory.
"""
from ._binding import (  # noqa: F401
    EMPTY, RC_BUILD_BOUNDS_CHECK, RC_ERR_ARG, RC_ERR_BOUNDS, RC_ERR_CUDA, RC_ERR_OOM, RC_ERR_STATE, RC_ERR_TIMEOUT,
    RC_ERR_UNSUPPORTED, rc_build_flags,
    RC_F_BF16_CACHE, RC_F_COPY_WINDOW, RC_F_READTIME_ABLATION, RC_OK, RcError, RingKVCache, declared_symbols, lib, rc_attend, rc_attend_readtime,
    rc_cache_create, rc_cache_delta_rotate, rc_cache_delta_total, rc_cache_destroy, rc_cache_export,
    rc_cache_export_bf16, rc_cache_export_readtime, rc_cache_launch_count, rc_cache_occupancy, rc_cache_set_wait_limit, rc_cache_sync,
    rc_cache_write, rc_cache_write_fused,
    rc_cache_window_shift, rc_tile_kinds,
    rc_status_string,
)
