"""Python binding of the C ABI, with the same names.

Argument marshalling only: every function checks that the tensors are CUDA,
contiguous and of the expected dtype, passes their device pointers and sizes to
libtlpa.so, and raises TLError on a non-TL_OK status.  No arithmetic of the
path happens here; torch provides the device memory and the stream.
"""
from __future__ import annotations

import functools
from typing import Optional

import torch

from . import _lib

# torch's own fast paths for the current device and stream (a call costs
# ~0.1 us against ~3 us for torch.cuda.current_stream()); the public calls
# stand in where a build lacks them
_current_device = getattr(torch._C, "_cuda_getDevice", None)
_current_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)

(TL_OK, TL_ERR_INVALID_ARG, TL_ERR_UNSUPPORTED, TL_ERR_CUDA, TL_ERR_DEVICE_BOUNDS,
 TL_ERR_WORKSPACE, TL_ERR_DEVICE_TIMEOUT) = range(7)
TL_F32, TL_BF16, TL_FP8_E4M3, TL_INT8 = 0, 1, 2, 3
TL_DEVERR_SLOT_RANGE, TL_DEVERR_PAGE_RANGE, TL_DEVERR_CONTEXT_RANGE = 1, 2, 4
TL_DEVERR_TIMEOUT, TL_DEVERR_VALUE_RANGE, TL_DEVERR_PLAN_CAPACITY = 8, 16, 32

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


def _need(t: torch.Tensor, name: str, dtype=None, shape=None, device=None):
    """A contiguous CUDA tensor of the given dtype and shape (None entries of
    `shape` match any size) on `device`."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None:
        ts = t.shape
        bad = len(ts) != len(shape)
        if not bad:
            for a, w in zip(ts, shape):
                if w is not None and a != w:
                    bad = True
                    break
        if bad:
            raise ValueError(f"{name} must have shape {tuple(shape)} (None: any), got {tuple(ts)}")
    if device is not None and t.get_device() != device.index:
        raise ValueError(f"{name} is on {t.device}, the call's tensors are on {device}")


def _check(status: int, where: str):
    if status != TL_OK:
        raise TLError(status, where)


def _run(where: str, device, stream, *args):
    """Call the entry point `where` with `args` and the stream, with `device`
    current (the library launches on the current device)."""
    fn = getattr(_lib.load(), where)
    idx = device.index
    if _current_device is not None and _current_raw_stream is not None and \
            _current_device() == idx:
        st = fn(*args, _current_raw_stream(idx) if stream is None else _stream(stream))
    else:
        with torch.cuda.device(device):
            st = fn(*args, _stream(stream))
    _check(st, where)


def _need_table(block_table, lens, B, device, lens_name="context_lens"):
    """block_table [B, max_pages] int32 and a per-sequence length vector [B] int32."""
    _need(block_table, "block_table", torch.int32, (B, None), device)
    if block_table.shape[1] < 1:
        raise ValueError("block_table needs at least one column")
    _need(lens, lens_name, torch.int32, (B,), device)


def _need_pools(k_cache, v_cache, device, dtype=None):
    """k_cache / v_cache [num_pages, page_size, H_kv, d] of one dtype and shape."""
    _need(k_cache, "k_cache", dtype, (None, None, None, None), device)
    _need(v_cache, "v_cache", k_cache.dtype, tuple(k_cache.shape), device)
    return k_cache.shape


def _need_new_rows(k_new, v_new, slot_mapping, hkv, d, device, dtype=None):
    """k_new / v_new [N, H_kv, d] of one dtype and slot_mapping [N] int64."""
    _need(k_new, "k_new", dtype, (None, hkv, d), device)
    _need(v_new, "v_new", k_new.dtype, tuple(k_new.shape), device)
    _need(slot_mapping, "slot_mapping", torch.int64, (k_new.shape[0],), device)


def tl_get_device_error(error_word: torch.Tensor, clear: bool = False, stream=None) -> int:
    """The TL_DEVERR_* bits of a device error word once the work enqueued on
    the stream before this call has finished (synchronises the stream); with
    clear, the word is zeroed afterwards.  Returns the bits; the C call's
    status (TL_OK, TL_ERR_DEVICE_BOUNDS or TL_ERR_DEVICE_TIMEOUT) follows
    from them."""
    import ctypes
    _need(error_word, "error_word", None, (1,))
    if error_word.element_size() != 4:
        raise TypeError("error_word must be a 4-byte integer tensor")
    bits = ctypes.c_uint32(0)
    with torch.cuda.device(error_word.device):
        st = _lib.load().tl_get_device_error(_ptr(error_word), ctypes.byref(bits), int(bool(clear)),
                                             _stream(stream))
    if st not in (TL_OK, TL_ERR_DEVICE_BOUNDS, TL_ERR_DEVICE_TIMEOUT):
        raise TLError(st, "tl_get_device_error")
    return int(bits.value)


def _err_word(error_word, device):
    if error_word is not None:
        _need(error_word, "error_word", None, (1,), device)
        if error_word.element_size() != 4:
            raise TypeError("error_word must be a 4-byte integer tensor")
    return _ptr(error_word)


def tl_kv_cache_write(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                      error_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """In place: cache row slot_mapping[t] = new[t] for every t with slot != -1.
    k_new/v_new [N, H_kv, d]; caches [num_pages, page_size, H_kv, d]."""
    dev = k_cache.device
    P, ps, hkv, d = _need_pools(k_cache, v_cache, dev)
    _need_new_rows(k_new, v_new, slot_mapping, hkv, d, dev, k_cache.dtype)
    _run("tl_kv_cache_write", dev, stream,
         _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
         slot_mapping.numel(), P, ps, hkv, d, _DTYPES.get(k_cache.dtype, -1),
         _err_word(error_word, dev))


def tl_kv_cache_write_fp8(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                          error_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """In place: the e4m3 codes of new[t] (f32 or bf16, [N, H_kv, d]) into the
    fp8 pools (torch.float8_e4m3fn [num_pages, page_size, H_kv, d]) at slot[t],
    for every t with slot != -1; values clamp to +-448."""
    dev = k_cache.device
    P, ps, hkv, d = _need_pools(k_cache, v_cache, dev, torch.float8_e4m3fn)
    _need_new_rows(k_new, v_new, slot_mapping, hkv, d, dev)
    _run("tl_kv_cache_write_fp8", dev, stream,
         _ptr(k_new), _ptr(v_new), _DTYPES.get(k_new.dtype, -1), _ptr(k_cache), _ptr(v_cache),
         _ptr(slot_mapping), slot_mapping.numel(), P, ps, hkv, d, _err_word(error_word, dev))


def _need_int8_pools(k_codes, v_codes, k_scales, v_scales, device):
    _need(k_codes, "k_codes", torch.int8, (None, None, None, None), device)
    _need(v_codes, "v_codes", torch.int8, tuple(k_codes.shape), device)
    P, ps, hkv, d = k_codes.shape
    _need(k_scales, "k_scales", torch.float32, (P, hkv, ps), device)
    _need(v_scales, "v_scales", torch.float32, (P, hkv, ps), device)
    return P, ps, hkv, d


def tl_kv_cache_write_int8(k_new: torch.Tensor, v_new: torch.Tensor, k_codes: torch.Tensor,
                           v_codes: torch.Tensor, k_scales: torch.Tensor, v_scales: torch.Tensor,
                           slot_mapping: torch.Tensor, error_word: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    """In place: for every t with slot != -1 and every KV head, the row of
    new[t] (f32 or bf16 [N, H_kv, d]) as int8 codes (pool int8 [num_pages,
    page_size, H_kv, d]) and its scale max |x| / 127 (float32 [num_pages,
    H_kv, page_size]); codes are x / scale rounded half to even."""
    dev = k_codes.device
    P, ps, hkv, d = _need_int8_pools(k_codes, v_codes, k_scales, v_scales, dev)
    _need_new_rows(k_new, v_new, slot_mapping, hkv, d, dev)
    _run("tl_kv_cache_write_int8", dev, stream,
         _ptr(k_new), _ptr(v_new), _DTYPES.get(k_new.dtype, -1), _ptr(k_codes), _ptr(v_codes),
         _ptr(k_scales), _ptr(v_scales), _ptr(slot_mapping), slot_mapping.numel(), P, ps, hkv, d,
         _err_word(error_word, dev))


def _decode_out(out, shape, device):
    if out is None:
        return torch.empty(shape, dtype=torch.float32, device=device)
    _need(out, "out", torch.float32, shape, device)
    return out


def _workspace(workspace, nbytes, device):
    if workspace is None:
        return alloc_workspace(nbytes, device)
    _need(workspace, "workspace", None, None, device)
    return workspace


def _ws_bytes(workspace):
    return workspace.numel() * workspace.element_size()


def tl_paged_attn_decode_int8(q: torch.Tensor, k_codes: torch.Tensor, v_codes: torch.Tensor,
                              k_scales: torch.Tensor, v_scales: torch.Tensor,
                              block_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                              window: int = 0, out: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None,
                              error_word: Optional[torch.Tensor] = None,
                              stream=None) -> torch.Tensor:
    """tl_paged_attn_decode over int8 pools (bf16 q): out[B, H_q, d] float32,
    every K/V element read as code x its row's scale."""
    dev = q.device
    P, ps, hkv, d = _need_int8_pools(k_codes, v_codes, k_scales, v_scales, dev)
    _need(q, "q", torch.bfloat16, (None, None, d), dev)
    B, hq, _ = q.shape
    _need_table(block_table, context_lens, B, dev)
    out = _decode_out(out, (B, hq, d), dev)
    workspace = _workspace(workspace, tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    _run("tl_paged_attn_decode_int8", dev, stream,
         _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(block_table),
         block_table.shape[1], _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window),
         float(scale), _ptr(workspace), _ws_bytes(workspace), _err_word(error_word, dev))
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
    dev = q.device
    P, ps, hkv, d = _need_int8_pools(k_codes, v_codes, k_scales, v_scales, dev)
    _need(q, "q", torch.bfloat16, (None, None, d), dev)
    _need_new_rows(k_new, v_new, slot_mapping, hkv, d, dev)
    B, hq, _ = q.shape
    _need_table(block_table, context_lens, B, dev)
    out = _decode_out(out, (B, hq, d), dev)
    workspace = _workspace(workspace, tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    _run("tl_paged_attn_decode_write_int8", dev, stream,
         _ptr(q), _ptr(k_new), _ptr(v_new), _DTYPES.get(k_new.dtype, -1), _ptr(slot_mapping),
         slot_mapping.numel(), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales),
         _ptr(block_table), block_table.shape[1], _ptr(context_lens), _ptr(out), B, hq, hkv, d,
         P, ps, int(window), float(scale), _ptr(workspace), _ws_bytes(workspace),
         _err_word(error_word, dev))
    return out


def tl_paged_attn_prefill_workspace_size_ex(B: int, T: int, h_q: int, h_kv: int, d: int,
                                            max_pages_per_seq: int, page_size: int,
                                            ring_pages: int, dtype: int) -> int:
    return int(_lib.load().tl_paged_attn_prefill_workspace_size_ex(
        B, T, h_q, h_kv, d, max_pages_per_seq, page_size, ring_pages, dtype))


def tl_paged_attn_prefill_workspace_size_keys(B: int, T: int, h_q: int, h_kv: int, d: int,
                                              max_row_keys: int, dtype: int = TL_BF16) -> int:
    """Workspace of a prefill call whose rows each read at most max_row_keys
    keys (from the first key a row's first token sees to its last position);
    independent of the table's width."""
    return int(_lib.load().tl_paged_attn_prefill_workspace_size_keys(B, T, h_q, h_kv, d,
                                                                      max_row_keys, dtype))


@functools.lru_cache(maxsize=1024)
def tl_paged_attn_decode_workspace_size(B: int, h_q: int, h_kv: int, d: int) -> int:
    return int(_lib.load().tl_paged_attn_decode_workspace_size(B, h_q, h_kv, d))


def tl_paged_attn_prefill_workspace_size(B: int, T: int, h_q: int, h_kv: int, d: int,
                                         max_pages_per_seq: int, page_size: int) -> int:
    return int(_lib.load().tl_paged_attn_prefill_workspace_size(B, T, h_q, h_kv, d,
                                                                 max_pages_per_seq, page_size))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A device byte buffer (torch allocations are 256-byte aligned)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _decode_args(q, k_cache, v_cache, block_table, context_lens, q_tokens=False):
    """Shapes of a decode call: q [B, H_q, d] (or [B, q_len, H_q, d]) in the
    pools' query dtype, the pools, the table and the lengths, all on q's device."""
    dev = q.device
    P, ps, hkv, d = _need_pools(k_cache, v_cache, dev)
    _need(q, "q", _query_dtype(k_cache.dtype), (None, None, None, d) if q_tokens else
          (None, None, d), dev)
    _need_table(block_table, context_lens, q.shape[0], dev)
    return dev, P, ps, hkv, d


def tl_paged_attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         block_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                         window: int = 0, out: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None,
                         error_word: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[B, H_q, d] (float32): one query per sequence, causal length context_lens[b]."""
    dev, P, ps, hkv, d = _decode_args(q, k_cache, v_cache, block_table, context_lens)
    B, hq, _ = q.shape
    out = _decode_out(out, (B, hq, d), dev)
    workspace = _workspace(workspace, tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    _run("tl_paged_attn_decode", dev, stream,
         _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
         _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window), float(scale),
         _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), _ws_bytes(workspace),
         _err_word(error_word, dev))
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
    dev, P, ps, hkv, d = _decode_args(q, k_cache, v_cache, block_table, context_lens)
    _need_new_rows(k_new, v_new, slot_mapping, hkv, d, dev)
    B, hq, _ = q.shape
    out = _decode_out(out, (B, hq, d), dev)
    workspace = _workspace(workspace, tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    _run("tl_paged_attn_decode_write", dev, stream,
         _ptr(q), _ptr(k_new), _ptr(v_new), _DTYPES.get(k_new.dtype, -1), _ptr(slot_mapping),
         slot_mapping.numel(), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
         block_table.shape[1], _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window),
         float(scale), _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), _ws_bytes(workspace),
         _err_word(error_word, dev))
    return out


TL_DECODE_NOALLOC_SCRATCH_BYTES = 32 << 20


def tl_paged_attn_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                 block_table: torch.Tensor, context_lens: torch.Tensor,
                                 scale: float, out: torch.Tensor, window: int = 0,
                                 error_word: Optional[torch.Tensor] = None,
                                 stream=None) -> torch.Tensor:
    """Decode into a caller-provided `out` without any device allocation: the
    scratch is a fixed array inside the library (see the C header); calls on a
    device share it, so calls that overlap on the GPU must be serialised.  The
    call runs with q's device current (the array of that device is used)."""
    dev, P, ps, hkv, d = _decode_args(q, k_cache, v_cache, block_table, context_lens)
    B, hq, _ = q.shape
    if out is None:
        raise ValueError("out is required: this entry point allocates nothing")
    _need(out, "out", torch.float32, (B, hq, d), dev)
    _run("tl_paged_attn_decode_noalloc", dev, stream,
         _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
         _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window), float(scale),
         _DTYPES.get(k_cache.dtype, -1), _err_word(error_word, dev))
    return out


def _prefill_args(q, k_cache, v_cache, block_table, positions):
    dev = q.device
    P, ps, hkv, d = _need_pools(k_cache, v_cache, dev)
    _need(q, "q", _query_dtype(k_cache.dtype), (None, None, None, d), dev)
    B, T = q.shape[0], q.shape[1]
    _need(block_table, "block_table", torch.int32, (B, None), dev)
    if block_table.shape[1] < 1:
        raise ValueError("block_table needs at least one column")
    _need(positions, "positions", torch.int32, (B, T), dev)
    return dev, P, ps, hkv, d


def tl_paged_attn_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          block_table: torch.Tensor, positions: torch.Tensor, scale: float,
                          window: int = 0, out: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None,
                          error_word: Optional[torch.Tensor] = None,
                          stream=None, max_row_keys: Optional[int] = None) -> torch.Tensor:
    """out[B, T, H_q, d] (float32): right-aligned batched prefill, padding at
    position -1.  Without a workspace, one is allocated: as wide as the table,
    or, with max_row_keys, as wide as rows reading at most that many keys."""
    dev, P, ps, hkv, d = _prefill_args(q, k_cache, v_cache, block_table, positions)
    B, T, hq, _ = q.shape
    out = _decode_out(out, (B, T, hq, d), dev)
    dt = _DTYPES.get(k_cache.dtype, -1)
    workspace = _workspace(workspace, tl_paged_attn_prefill_workspace_size_keys(
        B, T, hq, hkv, d, max_row_keys, dt) if max_row_keys else
        tl_paged_attn_prefill_workspace_size_ex(B, T, hq, hkv, d, block_table.shape[1], ps, 0,
                                                dt), dev)
    _run("tl_paged_attn_prefill", dev, stream,
         _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
         _ptr(positions), _ptr(out), B, T, hq, hkv, d, P, ps, int(window), float(scale),
         _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), _ws_bytes(workspace),
         _err_word(error_word, dev))
    return out


def tl_paged_attn_prefill_int8(q: torch.Tensor, k_codes: torch.Tensor, v_codes: torch.Tensor,
                               k_scales: torch.Tensor, v_scales: torch.Tensor,
                               block_table: torch.Tensor, positions: torch.Tensor, scale: float,
                               window: int = 0, out: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None,
                               error_word: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """tl_paged_attn_prefill over int8 pools (bf16 q [B, T, H_q, d]): out
    [B, T, H_q, d] float32, every K/V element read as code x its row's scale."""
    dev = q.device
    P, ps, hkv, d = _need_int8_pools(k_codes, v_codes, k_scales, v_scales, dev)
    _need(q, "q", torch.bfloat16, (None, None, None, d), dev)
    B, T, hq, _ = q.shape
    _need(block_table, "block_table", torch.int32, (B, None), dev)
    if block_table.shape[1] < 1:
        raise ValueError("block_table needs at least one column")
    _need(positions, "positions", torch.int32, (B, T), dev)
    out = _decode_out(out, (B, T, hq, d), dev)
    workspace = _workspace(workspace, tl_paged_attn_prefill_workspace_size_ex(
        B, T, hq, hkv, d, block_table.shape[1], ps, 0, TL_INT8), dev)
    _run("tl_paged_attn_prefill_int8", dev, stream,
         _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(block_table),
         block_table.shape[1], _ptr(positions), _ptr(out), B, T, hq, hkv, d, P, ps, int(window),
         float(scale), _ptr(workspace), _ws_bytes(workspace), _err_word(error_word, dev))
    return out


def tl_paged_attn_decode_ring(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                              block_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                              window: int, ring_pages: int, out: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None,
                              error_word: Optional[torch.Tensor] = None,
                              stream=None) -> torch.Tensor:
    """Decode over a ring: the first ring_pages entries of each table row hold
    the sequence's ring (logical block k on entry k % ring_pages)."""
    dev, P, ps, hkv, d = _decode_args(q, k_cache, v_cache, block_table, context_lens)
    B, hq, _ = q.shape
    out = _decode_out(out, (B, hq, d), dev)
    workspace = _workspace(workspace, tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    _run("tl_paged_attn_decode_ring", dev, stream,
         _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
         _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window), int(ring_pages),
         float(scale), _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), _ws_bytes(workspace),
         _err_word(error_word, dev))
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
    dev, P, ps, hkv, d = _prefill_args(q, k_cache, v_cache, block_table, positions)
    B, T, hq, _ = q.shape
    out = _decode_out(out, (B, T, hq, d), dev)
    workspace = _workspace(workspace, tl_paged_attn_prefill_workspace_size_ex(
        B, T, hq, hkv, d, block_table.shape[1], ps, ring_pages,
        _DTYPES.get(k_cache.dtype, -1)), dev)
    _run("tl_paged_attn_prefill_ring", dev, stream,
         _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
         _ptr(positions), _ptr(out), B, T, hq, hkv, d, P, ps, int(window), int(ring_pages),
         float(scale), _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), _ws_bytes(workspace),
         _err_word(error_word, dev))
    return out


def tl_paged_attn_decode_write_ring(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                    slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                                    v_cache: torch.Tensor, block_table: torch.Tensor,
                                    context_lens: torch.Tensor, scale: float, window: int,
                                    ring_pages: int, out: Optional[torch.Tensor] = None,
                                    workspace: Optional[torch.Tensor] = None,
                                    error_word: Optional[torch.Tensor] = None,
                                    stream=None) -> torch.Tensor:
    """tl_paged_attn_decode_write over rings: the new rows at their ring slots
    (slot_mapping follows the ring rule), then tl_paged_attn_decode_ring."""
    dev, P, ps, hkv, d = _decode_args(q, k_cache, v_cache, block_table, context_lens)
    _need_new_rows(k_new, v_new, slot_mapping, hkv, d, dev)
    B, hq, _ = q.shape
    out = _decode_out(out, (B, hq, d), dev)
    workspace = _workspace(workspace, tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    _run("tl_paged_attn_decode_write_ring", dev, stream,
         _ptr(q), _ptr(k_new), _ptr(v_new), _DTYPES.get(k_new.dtype, -1), _ptr(slot_mapping),
         slot_mapping.numel(), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
         block_table.shape[1], _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window),
         int(ring_pages), float(scale), _DTYPES.get(k_cache.dtype, -1), _ptr(workspace),
         _ws_bytes(workspace), _err_word(error_word, dev))
    return out


def tl_paged_attn_decode_ring_int8(q: torch.Tensor, k_codes: torch.Tensor, v_codes: torch.Tensor,
                                   k_scales: torch.Tensor, v_scales: torch.Tensor,
                                   block_table: torch.Tensor, context_lens: torch.Tensor,
                                   scale: float, window: int, ring_pages: int,
                                   out: Optional[torch.Tensor] = None,
                                   workspace: Optional[torch.Tensor] = None,
                                   error_word: Optional[torch.Tensor] = None,
                                   stream=None) -> torch.Tensor:
    """tl_paged_attn_decode_ring over int8 pools (bf16 q): out[B, H_q, d]
    float32."""
    dev = q.device
    P, ps, hkv, d = _need_int8_pools(k_codes, v_codes, k_scales, v_scales, dev)
    _need(q, "q", torch.bfloat16, (None, None, d), dev)
    B, hq, _ = q.shape
    _need_table(block_table, context_lens, B, dev)
    out = _decode_out(out, (B, hq, d), dev)
    workspace = _workspace(workspace, tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    _run("tl_paged_attn_decode_ring_int8", dev, stream,
         _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(block_table),
         block_table.shape[1], _ptr(context_lens), _ptr(out), B, hq, hkv, d, P, ps, int(window),
         int(ring_pages), float(scale), _ptr(workspace), _ws_bytes(workspace),
         _err_word(error_word, dev))
    return out


def tl_paged_attn_prefill_ring_int8(q: torch.Tensor, k_codes: torch.Tensor,
                                    v_codes: torch.Tensor, k_scales: torch.Tensor,
                                    v_scales: torch.Tensor, block_table: torch.Tensor,
                                    positions: torch.Tensor, scale: float, window: int,
                                    ring_pages: int, out: Optional[torch.Tensor] = None,
                                    workspace: Optional[torch.Tensor] = None,
                                    error_word: Optional[torch.Tensor] = None,
                                    stream=None) -> torch.Tensor:
    """tl_paged_attn_prefill_ring over int8 pools (bf16 q [B, T, H_q, d]):
    out [B, T, H_q, d] float32."""
    dev = q.device
    P, ps, hkv, d = _need_int8_pools(k_codes, v_codes, k_scales, v_scales, dev)
    _need(q, "q", torch.bfloat16, (None, None, None, d), dev)
    B, T, hq, _ = q.shape
    _need(block_table, "block_table", torch.int32, (B, None), dev)
    if block_table.shape[1] < 1:
        raise ValueError("block_table needs at least one column")
    _need(positions, "positions", torch.int32, (B, T), dev)
    out = _decode_out(out, (B, T, hq, d), dev)
    workspace = _workspace(workspace, tl_paged_attn_prefill_workspace_size_ex(
        B, T, hq, hkv, d, block_table.shape[1], ps, ring_pages, TL_INT8), dev)
    _run("tl_paged_attn_prefill_ring_int8", dev, stream,
         _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(block_table),
         block_table.shape[1], _ptr(positions), _ptr(out), B, T, hq, hkv, d, P, ps, int(window),
         int(ring_pages), float(scale), _ptr(workspace), _ws_bytes(workspace),
         _err_word(error_word, dev))
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
    dev, P, ps, hkv, d = _decode_args(q, k_cache, v_cache, block_table, context_lens,
                                      q_tokens=True)
    B, q_len, hq, _ = q.shape
    out = _decode_out(out, (B, q_len, hq, d), dev)
    workspace = _workspace(
        workspace, tl_paged_attn_decode_multi_workspace_size(B, q_len, hq, hkv, d), dev)
    _run("tl_paged_attn_decode_multi", dev, stream,
         _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
         _ptr(context_lens), _ptr(out), B, q_len, hq, hkv, d, P, ps, int(window), float(scale),
         _DTYPES.get(k_cache.dtype, -1), _ptr(workspace), _ws_bytes(workspace),
         _err_word(error_word, dev))
    return out


def tl_paged_attn_decode_multi_int8(q: torch.Tensor, k_codes: torch.Tensor,
                                    v_codes: torch.Tensor, k_scales: torch.Tensor,
                                    v_scales: torch.Tensor, block_table: torch.Tensor,
                                    context_lens: torch.Tensor, scale: float, window: int = 0,
                                    out: Optional[torch.Tensor] = None,
                                    workspace: Optional[torch.Tensor] = None,
                                    error_word: Optional[torch.Tensor] = None,
                                    stream=None) -> torch.Tensor:
    """tl_paged_attn_decode_multi over int8 pools (bf16 q [B, q_len, H_q, d]):
    out [B, q_len, H_q, d] float32."""
    dev = q.device
    P, ps, hkv, d = _need_int8_pools(k_codes, v_codes, k_scales, v_scales, dev)
    _need(q, "q", torch.bfloat16, (None, None, None, d), dev)
    B, q_len, hq, _ = q.shape
    _need_table(block_table, context_lens, B, dev)
    out = _decode_out(out, (B, q_len, hq, d), dev)
    workspace = _workspace(
        workspace, tl_paged_attn_decode_multi_workspace_size(B, q_len, hq, hkv, d), dev)
    _run("tl_paged_attn_decode_multi_int8", dev, stream,
         _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(block_table),
         block_table.shape[1], _ptr(context_lens), _ptr(out), B, q_len, hq, hkv, d, P, ps,
         int(window), float(scale), _ptr(workspace), _ws_bytes(workspace),
         _err_word(error_word, dev))
    return out
