"""ctypes view of libtlpa.so (the C ABI of include/tl_paged_attn.h).

Loading fails loudly when the library has not been built: there is no other
implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

i32, i64, u32p, vp, sz, f32 = (ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_size_t, ctypes.c_float)

SIGNATURES = {
    "tl_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "tl_version": ([], i32),
    "tl_get_device_error": ([vp, vp, i32, vp], ctypes.c_int),
    "tl_decode_trace_reset": ([], ctypes.c_int),
    "tl_decode_trace_read": ([vp, i32], ctypes.c_int),
    "tl_prefill_trace_reset": ([], ctypes.c_int),
    "tl_prefill_trace_read": ([vp, i32], ctypes.c_int),
    "tl_kv_cache_write": ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_int, u32p, vp],
                          ctypes.c_int),
    "tl_kv_cache_write_fp8": ([vp, vp, ctypes.c_int, vp, vp, vp, i32, i32, i32, i32, i32, u32p,
                               vp], ctypes.c_int),
    "tl_kv_cache_write_int8": ([vp, vp, ctypes.c_int, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                u32p, vp], ctypes.c_int),
    "tl_paged_attn_decode_workspace_size": ([i32, i32, i32, i32], sz),
    "tl_paged_attn_decode_int8": ([vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                   i32, i32, f32, vp, sz, u32p, vp], ctypes.c_int),
    "tl_paged_attn_decode_write_int8": ([vp, vp, vp, ctypes.c_int, vp, i32, vp, vp, vp, vp, vp,
                                         i32, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp,
                                         sz, u32p, vp], ctypes.c_int),
    "tl_paged_attn_decode": ([vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                              ctypes.c_int, vp, sz, u32p, vp], ctypes.c_int),
    "tl_paged_attn_decode_write": ([vp, vp, vp, ctypes.c_int, vp, i32, vp, vp, vp, i32, vp, vp,
                                    i32, i32, i32, i32, i32, i32, i32, f32, ctypes.c_int, vp, sz,
                                    u32p, vp], ctypes.c_int),
    "tl_paged_attn_decode_noalloc": ([vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                      i32, f32, ctypes.c_int, u32p, vp], ctypes.c_int),
    "tl_paged_attn_prefill_workspace_size": ([i32, i32, i32, i32, i32, i32, i32], sz),
    "tl_paged_attn_prefill": ([vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                               i32, f32, ctypes.c_int, vp, sz, u32p, vp], ctypes.c_int),
    "tl_paged_attn_decode_ring": ([vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                   i32, i32, f32, ctypes.c_int, vp, sz, u32p, vp], ctypes.c_int),
    "tl_paged_attn_prefill_ring_workspace_size": ([i32, i32, i32, i32, i32, i32, i32, i32], sz),
    "tl_paged_attn_decode_multi_workspace_size": ([i32, i32, i32, i32, i32], sz),
    "tl_paged_attn_prefill_workspace_size_keys": ([i32, i32, i32, i32, i32, i32, ctypes.c_int],
                                                  sz),
    "tl_paged_attn_prefill_workspace_size_ex": ([i32, i32, i32, i32, i32, i32, i32, i32,
                                                 ctypes.c_int], sz),
    "tl_paged_attn_decode_multi": ([vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                    i32, i32, f32, ctypes.c_int, vp, sz, u32p, vp], ctypes.c_int),
    "tl_paged_attn_decode_write_ring": ([vp, vp, vp, ctypes.c_int, vp, i32, vp, vp, vp, i32, vp,
                                         vp, i32, i32, i32, i32, i32, i32, i32, i32, f32,
                                         ctypes.c_int, vp, sz, u32p, vp], ctypes.c_int),
    "tl_paged_attn_decode_multi_int8": ([vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                         i32, i32, i32, i32, f32, vp, sz, u32p, vp],
                                        ctypes.c_int),
    "tl_paged_attn_decode_ring_int8": ([vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                        i32, i32, i32, i32, f32, vp, sz, u32p, vp], ctypes.c_int),
    "tl_paged_attn_prefill_ring_int8": ([vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                         i32, i32, i32, i32, i32, f32, vp, sz, u32p, vp],
                                        ctypes.c_int),
    "tl_paged_attn_prefill_int8": ([vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                    i32, i32, i32, f32, vp, sz, u32p, vp], ctypes.c_int),
    "tl_paged_attn_prefill_ring": ([vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                    i32, i32, i32, f32, ctypes.c_int, vp, sz, u32p, vp],
                                   ctypes.c_int),
}


class TLNotBuilt(RuntimeError):
    pass


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False, path: str = None):
    """The loaded library; with build_if_missing, compile it first if needed.
    path: load that build of the library instead (a variant from
    build.build_variant, e.g. the decode trace build), before any other
    call of the process has loaded one."""
    global _lib
    if _lib is not None:  # loaded: no lock needed to read it
        if path is not None and getattr(_lib, "_name", None) != path:
            raise RuntimeError(f"{_lib._name} is already loaded in this process")
        return _lib
    with _lock:
        if _lib is None:
            if path is None:
                if build_if_missing:
                    _build.build()
                path = _build.LIB
                if not os.path.exists(path):
                    raise TLNotBuilt(
                        f"{path} is missing: build it with "
                        "`python -c 'import __graft_entry__ as g; g.build()'` "
                        "(or python -m paged_kv_attention_cache_gb300.build)")
            lib = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib
