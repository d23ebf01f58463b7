"""Python binding of the C ABI, with the same names.

Argument marshalling only: every function checks that the tensors are CUDA,
contiguous and of the expected dtype, passes their device pointers and sizes to
libtlpa.so, and raises TLError on a non-TL_OK status.  No arithmetic of the
path happens here; torch provides the device memory and the stream.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib

TL_OK, TL_ERR_INVALID_ARG, TL_ERR_UNSUPPORTED, TL_ERR_CUDA, TL_ERR_WORKSPACE = range(5)
TL_F32, TL_BF16, TL_FP8_E4M3 = 0, 1, 2
TL_DEVERR_SLOT_RANGE, TL_DEVERR_PAGE_RANGE, TL_DEVERR_CONTEXT_RANGE = 1, 2, 4
TL_DEVERR_TIMEOUT, TL_DEVERR_VALUE_RANGE = 8, 16

_DTYPES = {torch.float32: TL_F32, torch.bfloat16: TL_BF16, torch.float8_e4m3fn: TL_FP8_E4M3}


def _query_dtype(cache_dtype):
    """Queries against an e4m3 pool are bf16; otherwise the pool's dtype."""
    return torch.bfloat16 if cache_dtype == torch.float8_e4m3fn else cache_dtype


class TLError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tl_status_string(status)}")


def tl_status_string(status: int) -> str:
    return _lib.load().tl_status_string(int(status)).decode()


def tl_version() -> int:
    return int(_lib.load().tl_version())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _check(status: int, where: str):
    if status != TL_OK:
        raise TLError(status, where)


def tl_kv_cache_write(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                      error_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """In place: cache row slot_mapping[t] = new[t] for every t with slot != -1.
    k_new/v_new [N, H_kv, d]; caches [num_pages, page_size, H_kv, d]."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n)
    _need(slot_mapping, "slot_mapping", torch.int64)
    P, ps, hkv, d = k_cache.shape
    st = _lib.load().tl_kv_cache_write(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
        slot_mapping.numel(), P, ps, hkv, d, _DTYPES.get(k_cache.dtype, -1), _ptr(error_word),
        _stream(stream))
    _check(st, "tl_kv_cache_write")


def tl_kv_cache_write_fp8(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                          error_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """In place: the e4m3 codes of new[t] (f32 or bf16, [N, H_kv, d]) into the
    fp8 pools (torch.float8_e4m3fn [num_pages, page_size, H_kv, d]) at slot[t],
    for every t with slot != -1; values clamp to +-448."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, n)
    _need(k_cache, "k_cache", torch.float8_e4m3fn)
    _need(v_cache, "v_cache", torch.float8_e4m3fn)
    _need(slot_mapping, "slot_mapping", torch.int64)
    P, ps, hkv, d = k_cache.shape
    st = _lib.load().tl_kv_cache_write_fp8(
        _ptr(k_new), _ptr(v_new), _DTYPES.get(k_new.dtype, -1), _ptr(k_cache), _ptr(v_cache),
        _ptr(slot_mapping), slot_mapping.numel(), P, ps, hkv, d, _ptr(error_word),
        _stream(stream))
    _check(st, "tl_kv_cache_write_fp8")


def _need_int8_pools(k_codes, v_codes, k_scales, v_scales):
    _need(k_codes, "k_codes", torch.int8)
    _need(v_codes, "v_codes", torch.int8)
    _need(k_scales, "k_scales", torch.float32)
    _need(v_scales, "v_scales", torch.float32)
    P, ps, hkv, d = k_codes.shape
    if v_codes.shape != k_codes.shape or tuple(k_scales.shape) != (P, hkv, ps) or \
            v_scales.shape != k_scales.shape:
        raise ValueError("int8 pools: codes [num_pages, page_size, H_kv, d], "
                         "scales [num_pages, H_kv, page_size]")
    return P, ps, hkv, d


def tl_kv_cache_write_int8(k_new: torch.Tensor, v_new: torch.Tensor, k_codes: torch.Tensor,
                           v_codes: torch.Tensor, k_scales: torch.Tensor, v_scales: torch.Tensor,
                           slot_mapping: torch.Tensor, error_word: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    """In place: for every t with slot != -1 and every KV head, the row of
    new[t] (f32 or bf16 [N, H_kv, d]) as int8 codes (pool int8 [num_pages,
    page_size, H_kv, d]) and its scale max |x| / 127 (float32 [num_pages,
    H_kv, page_size]); codes are x / scale rounded half to even."""
    _need(k_new, "k_new")
    _need(v_new, "v_new", k_new.dtype)
    _need(slot_mapping, "slot_mapping", torch.int64)
    P, ps, hkv, d = _need_int8_pools(k_codes, v_codes, k_scales, v_scales)
    st = _lib.load().tl_kv_cache_write_int8(
        _ptr(k_new), _ptr(v_new), _DTYPES.get(k_new.dtype, -1), _ptr(k_codes), _ptr(v_codes),
        _ptr(k_scales), _ptr(v_scales), _ptr(slot_mapping), slot_mapping.numel(), P, ps, hkv, d,
        _ptr(error_word), _stream(stream))
    _check(st, "tl_kv_cache_write_int8")


def tl_paged_attn_decode_int8(q: torch.Tensor, k_codes: torch.Tensor, v_codes: torch.Tensor,
                              k_scales: torch.Tensor, v_scales: torch.Tensor,
                              block_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                              window: int = 0, out: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None,
                              error_word: Optional[torch.Tensor] = None,
                              stream=None) -> torch.Tensor:
    """tl_paged_attn_decode over int8 pools (bf16 q): out[B, H_q, d] float32,
    every K/V element read as code x its row's scale."""
    _need(q, "q", torch.bfloat16)
    _need(block_table, "block_table", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    P, ps, hkv, _ = _need_int8_pools(k_codes, v_codes, k_scales, v_scales)
    B, hq, d = q.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        workspace = alloc_workspace(tl_paged_attn_decode_workspace_size(B, hq, hkv, d), q.device)
    st = _lib.load().tl_paged_attn_decode_int8(
        _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(block_table),
        block_table.shape[1], _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window),
        float(scale), _ptr(workspace), workspace.numel(), _ptr(error_word), _stream(stream))
    _check(st, "tl_paged_attn_decode_int8")
    return out


def tl_paged_attn_decode_write_int8(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                    slot_mapping: torch.Tensor, k_codes: torch.Tensor,
                                    v_codes: torch.Tensor, k_scales: torch.Tensor,
                                    v_scales: torch.Tensor, block_table: torch.Tensor,
                                    context_lens: torch.Tensor, scale: float, window: int = 0,
                                    out: Optional[torch.Tensor] = None,
                                    workspace: Optional[torch.Tensor] = None,
                                    error_word: Optional[torch.Tensor] = None,
                                    stream=None) -> torch.Tensor:
    """tl_kv_cache_write_int8 of the new rows (f32 or bf16 [N, H_kv, d] at
    slot_mapping [N], -1 = padding), then tl_paged_attn_decode_int8, in one
    call: out[B, H_q, d] float32; the pools are updated in place."""
    _need(q, "q", torch.bfloat16)
    _need(k_new, "k_new")
    _need(v_new, "v_new", k_new.dtype)
    _need(slot_mapping, "slot_mapping", torch.int64)
    _need(block_table, "block_table", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    P, ps, hkv, _ = _need_int8_pools(k_codes, v_codes, k_scales, v_scales)
    B, hq, d = q.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        workspace = alloc_workspace(tl_paged_attn_decode_workspace_size(B, hq, hkv, d), q.device)
    st = _lib.load().tl_paged_attn_decode_write_int8(
        _ptr(q), _ptr(k_new), _ptr(v_new), _DTYPES.get(k_new.dtype, -1), _ptr(slot_mapping),
        slot_mapping.numel(), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales),
        _ptr(block_table), block_table.shape[1], _ptr(context_lens), _ptr(out), B, hq, hkv, d,
        P, ps, int(window), float(scale), _ptr(workspace), workspace.numel(), _ptr(error_word),
        _stream(stream))
    _check(st, "tl_paged_attn_decode_write_int8")
    return out


def tl_paged_attn_prefill_workspace_size_ex(B: int, T: int, h_q: int, h_kv: int, d: int,
                                            max_pages_per_seq: int, page_size: int,
                                            ring_pages: int, dtype: int) -> int:
    return int(_lib.load().tl_paged_attn_prefill_workspace_size_ex(
        B, T, h_q, h_kv, d, max_pages_per_seq, page_size, ring_pages, dtype))


def tl_paged_attn_decode_workspace_size(B: int, h_q: int, h_kv: int, d: int) -> int:
    return int(_lib.load().tl_paged_attn_decode_workspace_size(B, h_q, h_kv, d))


def tl_paged_attn_prefill_workspace_size(B: int, T: int, h_q: int, h_kv: int, d: int,
                                         max_pages_per_seq: int, page_size: int) -> int:
    return int(_lib.load().tl_paged_attn_prefill_workspace_size(B, T, h_q, h_kv, d,
                                                                 max_pages_per_seq, page_size))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A device byte buffer (torch allocations are 256-byte aligned)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def tl_paged_attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         block_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                         window: int = 0, out: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None,
                         error_word: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[B, H_q, d] (float32): one query per sequence, causal length context_lens[b]."""
    _need(q, "q", _query_dtype(k_cache.dtype))
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", k_cache.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    B, hq, d = q.shape
    P, ps, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        workspace = alloc_workspace(tl_paged_attn_decode_workspace_size(B, hq, hkv, d), q.device)
    st = _lib.load().tl_paged_attn_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window), float(scale),
        _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), workspace.numel(), _ptr(error_word),
        _stream(stream))
    _check(st, "tl_paged_attn_decode")
    return out


def tl_paged_attn_decode_write(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                               slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                               v_cache: torch.Tensor, block_table: torch.Tensor,
                               context_lens: torch.Tensor, scale: float, window: int = 0,
                               out: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None,
                               error_word: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """The write of the new rows k_new / v_new [N, H_kv, d] at slot_mapping
    [N] (int64, -1 = padding) into the pools (in place; e4m3 pools take bf16
    or f32 rows and convert them), then decode as tl_paged_attn_decode, in
    one call: out[B, H_q, d] (float32)."""
    _need(q, "q", _query_dtype(k_cache.dtype))
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", k_cache.dtype)
    _need(k_new, "k_new")
    _need(v_new, "v_new", k_new.dtype)
    _need(slot_mapping, "slot_mapping", torch.int64)
    _need(block_table, "block_table", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    B, hq, d = q.shape
    P, ps, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        workspace = alloc_workspace(tl_paged_attn_decode_workspace_size(B, hq, hkv, d), q.device)
    st = _lib.load().tl_paged_attn_decode_write(
        _ptr(q), _ptr(k_new), _ptr(v_new), _DTYPES.get(k_new.dtype, -1), _ptr(slot_mapping),
        slot_mapping.numel(), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window),
        float(scale), _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), workspace.numel(),
        _ptr(error_word), _stream(stream))
    _check(st, "tl_paged_attn_decode_write")
    return out


TL_DECODE_NOALLOC_SCRATCH_BYTES = 32 << 20


def tl_paged_attn_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                 block_table: torch.Tensor, context_lens: torch.Tensor,
                                 scale: float, out: torch.Tensor, window: int = 0,
                                 error_word: Optional[torch.Tensor] = None,
                                 stream=None) -> torch.Tensor:
    """Decode into a caller-provided `out` without any device allocation: the
    scratch is a fixed array inside the library (see the C header); calls on a
    device share it, so calls that overlap on the GPU must be serialised."""
    _need(q, "q", _query_dtype(k_cache.dtype))
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", k_cache.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    _need(out, "out", torch.float32)
    B, hq, d = q.shape
    P, ps, hkv, _ = k_cache.shape
    st = _lib.load().tl_paged_attn_decode_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window), float(scale),
        _DTYPES.get(k_cache.dtype, -1), _ptr(error_word), _stream(stream))
    _check(st, "tl_paged_attn_decode_noalloc")
    return out


def tl_paged_attn_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          block_table: torch.Tensor, positions: torch.Tensor, scale: float,
                          window: int = 0, out: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None,
                          error_word: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """out[B, T, H_q, d] (float32): right-aligned batched prefill, padding at position -1."""
    _need(q, "q", _query_dtype(k_cache.dtype))
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", k_cache.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(positions, "positions", torch.int32)
    B, T, hq, d = q.shape
    P, ps, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty((B, T, hq, d), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        workspace = alloc_workspace(
            tl_paged_attn_prefill_workspace_size_ex(B, T, hq, hkv, d, block_table.shape[1], ps, 0,
                                                    _DTYPES.get(k_cache.dtype, -1)), q.device)
    st = _lib.load().tl_paged_attn_prefill(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(positions), _ptr(out), B, T, hq, hkv, d, P, ps, int(window), float(scale),
        _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), workspace.numel(), _ptr(error_word),
        _stream(stream))
    _check(st, "tl_paged_attn_prefill")
    return out


def tl_paged_attn_decode_ring(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                              block_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                              window: int, ring_pages: int, out: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None,
                              error_word: Optional[torch.Tensor] = None,
                              stream=None) -> torch.Tensor:
    """Decode over a ring: the first ring_pages entries of each table row hold
    the sequence's ring (logical block k on entry k % ring_pages)."""
    _need(q, "q", _query_dtype(k_cache.dtype))
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", k_cache.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    B, hq, d = q.shape
    P, ps, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        workspace = alloc_workspace(tl_paged_attn_decode_workspace_size(B, hq, hkv, d), q.device)
    st = _lib.load().tl_paged_attn_decode_ring(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window), int(ring_pages),
        float(scale), _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), workspace.numel(),
        _ptr(error_word), _stream(stream))
    _check(st, "tl_paged_attn_decode_ring")
    return out


def tl_paged_attn_prefill_ring_workspace_size(B: int, T: int, h_q: int, h_kv: int, d: int,
                                              max_pages_per_seq: int, page_size: int,
                                              ring_pages: int) -> int:
    return int(_lib.load().tl_paged_attn_prefill_ring_workspace_size(
        B, T, h_q, h_kv, d, max_pages_per_seq, page_size, ring_pages))


def tl_paged_attn_prefill_ring(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_table: torch.Tensor, positions: torch.Tensor, scale: float,
                               window: int, ring_pages: int, out: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None,
                               error_word: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """Batched prefill over rings (see tl_paged_attn_decode_ring)."""
    _need(q, "q", _query_dtype(k_cache.dtype))
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", k_cache.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(positions, "positions", torch.int32)
    B, T, hq, d = q.shape
    P, ps, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty((B, T, hq, d), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        workspace = alloc_workspace(tl_paged_attn_prefill_workspace_size_ex(
            B, T, hq, hkv, d, block_table.shape[1], ps, ring_pages,
            _DTYPES.get(k_cache.dtype, -1)), q.device)
    st = _lib.load().tl_paged_attn_prefill_ring(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(positions), _ptr(out), B, T, hq, hkv, d, P, ps, int(window), int(ring_pages),
        float(scale), _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), workspace.numel(),
        _ptr(error_word), _stream(stream))
    _check(st, "tl_paged_attn_prefill_ring")
    return out


def tl_paged_attn_decode_multi_workspace_size(B: int, q_len: int, h_q: int, h_kv: int,
                                              d: int) -> int:
    return int(_lib.load().tl_paged_attn_decode_multi_workspace_size(B, q_len, h_q, h_kv, d))


def tl_paged_attn_decode_multi(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_table: torch.Tensor, context_lens: torch.Tensor,
                               scale: float, window: int = 0, out: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None,
                               error_word: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """out[B, q_len, H_q, d] (float32): q_len query tokens at positions
    L - q_len .. L - 1 of each sequence (L = context_lens[b])."""
    _need(q, "q", _query_dtype(k_cache.dtype))
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", k_cache.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    B, q_len, hq, d = q.shape
    P, ps, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty((B, q_len, hq, d), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        workspace = alloc_workspace(
            tl_paged_attn_decode_multi_workspace_size(B, q_len, hq, hkv, d), q.device)
    st = _lib.load().tl_paged_attn_decode_multi(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(context_lens), _ptr(out), B, q_len, hq, hkv, d, P, ps, int(window), float(scale),
        _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), workspace.numel(), _ptr(error_word),
        _stream(stream))
    _check(st, "tl_paged_attn_decode_multi")
    return out
