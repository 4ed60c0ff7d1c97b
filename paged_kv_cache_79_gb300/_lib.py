"""ctypes declarations of libpagedkv.so (see include/pagedkv.h)."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

c_int, c_size_t, c_float, c_void_p = ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
c_int64_p = ctypes.POINTER(ctypes.c_int64)
c_int32_p = ctypes.POINTER(ctypes.c_int32)
c_int_p = ctypes.POINTER(ctypes.c_int)

# name: (restype, argtypes)
SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [c_int]),
    "pa_last_cuda_error": (c_int, []),
    "pa_decode": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_int,
                          c_int, c_float, c_int, c_int, c_int, c_int, c_int, c_int, c_void_p,
                          c_size_t, c_void_p]),
    "pa_decode_append": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_int, c_void_p, c_int, c_int, c_float, c_int, c_int, c_int, c_int,
                                 c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "pa_decode_shared": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_int, c_void_p, c_void_p, c_int, c_int, c_float, c_int, c_int, c_int,
                                 c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "pa_decode_plan_bytes": (c_size_t, [c_int] * 7),
    "pa_decode_plan": (c_int, [c_void_p, c_size_t, c_void_p, c_int, c_void_p, c_int, c_int, c_int, c_int,
                               c_int, c_int]),
    "pa_decode_planned": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_int, c_void_p, c_int, c_int, c_float, c_int, c_int, c_int, c_int,
                                  c_int, c_void_p, c_size_t, c_void_p, c_size_t, c_void_p]),
    "pa_decode_shared_workspace_size": (c_size_t, [c_int] * 6),
    "pa_decode_shared_plan_bytes": (c_size_t, [c_int] * 7),
    "pa_decode_shared_plan": (c_int, [c_void_p, c_size_t, c_void_p, c_int, c_void_p, c_void_p, c_int, c_int,
                                      c_int, c_int, c_int, c_int]),
    "pa_decode_shared_planned": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_float, c_int,
                                         c_int, c_int, c_int, c_int, c_void_p, c_size_t, c_void_p, c_size_t,
                                         c_void_p]),
    "pa_share_groups": (c_int, [c_void_p, c_int, c_int, c_void_p, c_int, c_int, c_void_p]),
    "pa_decode_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p,
                                  c_int, c_int, c_float, c_int, c_int, c_int, c_int, c_int, c_int,
                                  c_void_p]),
    "pa_decode_partition_size": (c_int, [c_int] * 7),
    "pa_decode_workspace_size": (c_size_t, [c_int] * 7),
    "pa_reshape_and_cache": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                     c_int, c_int, c_int, c_int, c_void_p]),
    "pa_copy_blocks": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_size_t, c_void_p]),
    "pa_device_errors": (c_int, [ctypes.POINTER(ctypes.c_uint), c_void_p]),
    "pa_set_wait_limit_ns": (ctypes.c_ulonglong, [ctypes.c_ulonglong]),
    "pa_alloc_create": (c_int, [ctypes.POINTER(c_void_p), c_int, c_int, c_void_p]),
    "pa_alloc_destroy": (None, [c_void_p]),
    "pa_alloc_new_seq": (c_int, [c_void_p, c_int_p]),
    "pa_alloc_fork": (c_int, [c_void_p, c_int, c_int_p]),
    "pa_alloc_append": (c_int, [c_void_p, c_int, c_int64_p, c_int32_p, c_int32_p]),
    "pa_alloc_append_n": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_int_p, c_int_p]),
    "pa_alloc_free_seq": (c_int, [c_void_p, c_int]),
    "pa_alloc_block_table": (c_int, [c_void_p, c_int, c_void_p, c_int, c_int_p]),
    "pa_alloc_seq_len": (c_int, [c_void_p, c_int, c_int_p]),
    "pa_alloc_refcount": (c_int, [c_void_p, c_int]),
    "pa_alloc_num_free": (c_int, [c_void_p]),
    "pa_alloc_free_list": (c_int, [c_void_p, c_void_p, c_int, c_int_p]),
    "pa_alloc_set_host_pool": (c_int, [c_void_p, c_int]),
    "pa_alloc_usage_stats": (c_int, [c_void_p, c_void_p]),
    "pa_alloc_swap_out": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int_p]),
    "pa_alloc_swap_in": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int_p]),
    "pa_alloc_is_swapped": (c_int, [c_void_p, c_int]),
    "pa_alloc_host_refcount": (c_int, [c_void_p, c_int]),
    "pa_alloc_num_free_host": (c_int, [c_void_p]),
    "pa_alloc_host_free_list": (c_int, [c_void_p, c_void_p, c_int, c_int_p]),
    "pa_swap_blocks": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                               c_size_t, c_void_p]),
    "pa_gather_blocks": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p, c_size_t,
                                 c_void_p]),
    "pa_scatter_blocks": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_size_t,
                                  c_void_p]),
    "pa_kv_transfer_worthwhile": (c_int, [ctypes.c_longlong, ctypes.c_longlong]),
}


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libpagedkv.so, building it first if it is missing or stale.

    Raises if the library cannot be built or loaded: there is no fallback path."""
    global _lib
    with _lock:
        if _lib is None:
            if not _build.up_to_date():
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"libpagedkv.so missing at {_build.LIB}")
            L = ctypes.CDLL(_build.LIB)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib
