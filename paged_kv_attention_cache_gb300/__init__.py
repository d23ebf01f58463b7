"""Paged attention over a block-table KV cache, for GB300 (sm_103a).

The compute path is the C-ABI library libtlpa.so (hand-written CUDA kernels,
declared in include/tl_paged_attn.h); this package builds it in-tree and binds
it with the same names.  There is no CPU or framework fallback: calling an op
without the built library, or without a CUDA device, raises.
"""
from .api import (TL_BF16, TL_FP8_E4M3, tl_kv_cache_write_fp8, TL_DEVERR_CONTEXT_RANGE, TL_DEVERR_PAGE_RANGE,  # noqa: F401
                  TL_DEVERR_SLOT_RANGE, TL_DEVERR_TIMEOUT, TL_DEVERR_VALUE_RANGE, TL_ERR_CUDA, TL_ERR_INVALID_ARG, TL_ERR_UNSUPPORTED,
                  TL_ERR_WORKSPACE, TL_ERR_DEVICE_BOUNDS, TL_ERR_DEVICE_TIMEOUT,
                  TL_DEVERR_PLAN_CAPACITY, TL_F32, TL_OK, TLError, alloc_workspace,
                  tl_get_device_error,
                  TL_DECODE_NOALLOC_SCRATCH_BYTES, tl_kv_cache_write, tl_paged_attn_decode,
                  tl_paged_attn_decode_noalloc, tl_paged_attn_decode_workspace_size,
                  tl_paged_attn_decode_write, tl_kv_cache_write_int8, tl_paged_attn_decode_int8,
                  tl_paged_attn_decode_write_int8, tl_paged_attn_prefill_int8, TL_INT8,
                  tl_paged_attn_prefill, tl_paged_attn_prefill_workspace_size, tl_status_string,
                  tl_paged_attn_decode_ring, tl_paged_attn_prefill_ring,
                  tl_paged_attn_decode_ring_int8, tl_paged_attn_prefill_ring_int8,
                  tl_paged_attn_decode_multi_int8, tl_paged_attn_decode_write_ring,
                  tl_paged_attn_prefill_ring_workspace_size, tl_paged_attn_decode_multi,
                  tl_paged_attn_decode_multi_workspace_size,
                  tl_paged_attn_prefill_workspace_size_ex,
                  tl_paged_attn_prefill_workspace_size_keys,
                  tl_version)
from . import build as _build_module


def build_library(force: bool = False) -> str:
    """Compile libtlpa.so in-tree if it is missing or stale; returns its path."""
    return _build_module.build(force=force)

__all__ = [
    "tl_kv_cache_write", "tl_kv_cache_write_fp8", "tl_kv_cache_write_int8",
    "tl_paged_attn_decode", "tl_paged_attn_decode_int8", "tl_paged_attn_decode_write_int8",
    "tl_paged_attn_decode_noalloc", "tl_paged_attn_prefill_int8",
    "tl_paged_attn_prefill",
    "tl_paged_attn_decode_workspace_size", "tl_paged_attn_prefill_workspace_size",
    "tl_paged_attn_decode_ring", "tl_paged_attn_prefill_ring",
    "tl_paged_attn_decode_ring_int8", "tl_paged_attn_prefill_ring_int8",
    "tl_paged_attn_decode_multi_int8", "tl_paged_attn_decode_write_ring",
    "tl_paged_attn_prefill_ring_workspace_size", "tl_paged_attn_decode_multi",
    "tl_paged_attn_decode_multi_workspace_size", "tl_paged_attn_prefill_workspace_size_keys",
    "tl_status_string", "tl_version", "tl_get_device_error", "TLError", "build_library", "alloc_workspace",
]
