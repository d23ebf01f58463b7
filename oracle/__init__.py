"""Plain CPU oracle for paged KV-cache attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library never
imports, links or calls anything here, and nothing here imports the CUDA
library.

The arithmetic lives in ``oracle.c`` (plain C, double precision, one output at a
time); this module compiles it with gcc on first use and marshals numpy /
torch-CPU arrays to it.  What each function computes, and which passage of the
pages defines it, is stated in ``oracle.c``:

* ``kv_cache_write``  -- "How serving works in Tlaloc", sections 1-2
  (KV_CACHE_WRITE: scatter by slot, slot -1 never written);
* ``paged_decode`` / ``paged_prefill(blockwise=False)`` -- same page, section 2
  (PAGED_ATTENTION: gather through the block table, dot, masked softmax, dot;
  causal length = position + 1) and section 3 (sliding window p-W+1..p);
* ``paged_prefill(blockwise=True)`` -- same page, section 2 "Blockwise
  attention" (online softmax folded over 2,048-key blocks);
* ``kv_bytes_per_token`` -- "Serving Models", "Count KV heads and distinct
  stored tensors" (M = 2 L H_kv d q);
* ``kv_cache_write_fp8`` / ``fp8_value`` / ``fp8_code`` -- "How serving works
  in Tlaloc", the FP8 KV cache paragraph (e4m3fn codes, clamp to +-448, ties
  to even);
* ``kv_cache_write_int8`` / ``paged_decode_int8`` / ``paged_prefill_int8`` --
  same page: int8 KV pools
  are named as a next step without a format, read here from its "Int8 weights
  (opt-in)" paragraph (one f32 scale per row, max |x| / 127, codes rounded
  half to even; a value is code x scale).

Every function here is pinned by ``tests/test_oracle_pins.py`` (int8:
``tests/test_oracle_int8.py``) against facts the pages or the mathematics fix;
none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F32, BF16, FP8 = 0, 1, 2
DEFAULT_KEY_BLOCK = 2048

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, f64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.oracle_kv_cache_write.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64]
            lib.oracle_kv_cache_write.restype = ctypes.c_int
            lib.oracle_paged_decode.argtypes = [vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32,
                                                i32, i32, i32, i32, f64, vp, i32, vp, i32]
            lib.oracle_paged_decode.restype = ctypes.c_int
            lib.oracle_paged_prefill.argtypes = [vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32,
                                                 i32, i32, i32, i32, i32, f64, i32, i32, vp, i64,
                                                 vp, i32]
            lib.oracle_paged_prefill.restype = ctypes.c_int
            lib.oracle_ring_pages.argtypes = [i64, i64, i64]
            lib.oracle_fp8_value.argtypes = [i32]
            lib.oracle_fp8_value.restype = f64
            lib.oracle_fp8_code.argtypes = [f64]
            lib.oracle_fp8_code.restype = i32
            lib.oracle_kv_cache_write_fp8.argtypes = [vp, vp, i32, vp, vp, vp, i64, i64, i64, i64,
                                                      i64]
            lib.oracle_kv_cache_write_fp8.restype = ctypes.c_int
            lib.oracle_kv_cache_write_int8.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, i64, i64,
                                                       i64, i64, i64, vp]
            lib.oracle_kv_cache_write_int8.restype = ctypes.c_int
            lib.oracle_paged_decode_int8.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32,
                                                     i32, i32, i32, i32, i32, i32, f64, vp, i32,
                                                     vp, i32]
            lib.oracle_paged_decode_int8.restype = ctypes.c_int
            lib.oracle_paged_prefill_int8.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32,
                                                      i32, i32, i32, i32, i32, i32, i32, f64, i32,
                                                      i32, vp, i64, vp, i32]
            lib.oracle_paged_prefill_int8.restype = ctypes.c_int
            lib.oracle_ring_pages.restype = i64
            lib.oracle_kv_bytes_per_token.argtypes = [i64, i64, i64, i64]
            lib.oracle_kv_bytes_per_token.restype = i64
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _np(x):
    """numpy view of a numpy array or a CPU torch tensor (bf16 -> uint16 bits)."""
    if isinstance(x, np.ndarray):
        return x
    import torch  # local: only for callers that hand torch tensors in

    if isinstance(x, torch.Tensor):
        x = x.detach()
        if x.device.type != "cpu":
            raise OracleError("the oracle takes host arrays")
        if x.dtype == torch.bfloat16:
            return x.contiguous().view(torch.int16).numpy().view(np.uint16)
        if x.dtype == torch.float8_e4m3fn:
            return x.contiguous().view(torch.uint8).numpy()
        return x.contiguous().numpy()
    return np.asarray(x)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype in (np.uint16, np.int16):
        return BF16
    if a.dtype == np.uint8:
        return FP8
    raise OracleError(f"unsupported element type {a.dtype} (float32, bf16 or e4m3 bits)")


def _query_code(kv_code: int) -> int:
    """The query of an fp8 pool is bf16."""
    return BF16 if kv_code == FP8 else kv_code


def _c(a: np.ndarray, dtype=None) -> np.ndarray:
    if dtype is not None:
        a = np.asarray(a, dtype=dtype)
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def kv_cache_write(k_new, v_new, k_cache, v_cache, slot_mapping) -> None:
    """In place: cache[slot[t]] = new[t] for every t with slot[t] != -1."""
    lib = _load()
    kn, vn = _c(_np(k_new)), _c(_np(v_new))
    kc, vc = _np(k_cache), _np(v_cache)
    if not (kc.flags.c_contiguous and vc.flags.c_contiguous):
        raise OracleError("caches must be contiguous (written in place)")
    sm = _c(_np(slot_mapping), np.int64)
    P, ps, hkv, d = kc.shape
    if kn.shape != (sm.shape[0], hkv, d) or vn.shape != kn.shape or vc.shape != kc.shape:
        raise OracleError("shape mismatch")
    rc = lib.oracle_kv_cache_write(_ptr(kn), _ptr(vn), _ptr(kc), _ptr(vc), _ptr(sm), sm.shape[0],
                                   P, ps, hkv, d, kc.itemsize)
    if rc != 0:
        raise OracleError(f"oracle_kv_cache_write failed ({rc})")


def fp8_value(code: int) -> float:
    """Value of one e4m3fn code."""
    return float(_load().oracle_fp8_value(int(code)))


def fp8_code(x: float) -> int:
    """The e4m3fn code of x: nearest, ties to even mantissa, clamped to +-448."""
    return int(_load().oracle_fp8_code(float(x)))


def kv_cache_write_fp8(k_new, v_new, k_cache, v_cache, slot_mapping) -> None:
    """In place: the e4m3fn codes of new[t] into the fp8 pools (uint8 or
    torch.float8_e4m3fn, CPU) at slot[t], for every t with slot[t] != -1."""
    lib = _load()
    kn, vn = _c(_np(k_new)), _c(_np(v_new))
    kc, vc = _np(k_cache), _np(v_cache)
    if kc.dtype != np.uint8 or vc.dtype != np.uint8:
        raise OracleError("fp8 pools hold e4m3 codes (uint8)")
    if not (kc.flags.c_contiguous and vc.flags.c_contiguous):
        raise OracleError("caches must be contiguous (written in place)")
    sm = _c(_np(slot_mapping), np.int64)
    P, ps, hkv, d = kc.shape
    if kn.shape != (sm.shape[0], hkv, d) or vn.shape != kn.shape or vc.shape != kc.shape:
        raise OracleError("shape mismatch")
    rc = lib.oracle_kv_cache_write_fp8(_ptr(kn), _ptr(vn), _dtype_code(kn), _ptr(kc), _ptr(vc),
                                       _ptr(sm), sm.shape[0], P, ps, hkv, d)
    if rc != 0:
        raise OracleError(f"oracle_kv_cache_write_fp8 failed ({rc})")


def kv_cache_write_int8(k_new, v_new, k_codes, v_codes, k_scales, v_scales,
                        slot_mapping) -> int:
    """In place: the int8 codes and per-(token, KV head) scales of new[t] into
    the int8 pools (codes int8 [P, ps, H_kv, d], scales float32 [P, H_kv, ps])
    at slot[t], for every t with slot[t] != -1.  Returns the number of
    non-finite new values (written as code 0)."""
    lib = _load()
    kn, vn = _c(_np(k_new)), _c(_np(v_new))
    kc, vc, ks, vs = _np(k_codes), _np(v_codes), _np(k_scales), _np(v_scales)
    if kc.dtype != np.int8 or vc.dtype != np.int8 or ks.dtype != np.float32 or \
            vs.dtype != np.float32:
        raise OracleError("int8 pools: int8 codes and float32 scales")
    if not all(a.flags.c_contiguous for a in (kc, vc, ks, vs)):
        raise OracleError("pools must be contiguous (written in place)")
    sm = _c(_np(slot_mapping), np.int64)
    P, ps, hkv, d = kc.shape
    if kn.shape != (sm.shape[0], hkv, d) or vn.shape != kn.shape or vc.shape != kc.shape or \
            ks.shape != (P, hkv, ps) or vs.shape != ks.shape:
        raise OracleError("shape mismatch")
    bad = np.zeros(1, dtype=np.int64)
    rc = lib.oracle_kv_cache_write_int8(_ptr(kn), _ptr(vn), _dtype_code(kn), _ptr(kc), _ptr(vc),
                                        _ptr(ks), _ptr(vs), _ptr(sm), sm.shape[0], P, ps, hkv, d,
                                        _ptr(bad))
    if rc != 0:
        raise OracleError(f"oracle_kv_cache_write_int8 failed ({rc})")
    return int(bad[0])


def paged_decode_int8(q, k_codes, v_codes, k_scales, v_scales, block_table, context_lens, scale,
                      window=0, seqs=None, threads=0, ring_pages=0) -> np.ndarray:
    """paged_decode over int8 pools: each element read as code x its row's scale."""
    lib = _load()
    qa = _c(_np(q))
    kc, vc = _c(_np(k_codes)), _c(_np(v_codes))
    ks, vs = _c(_np(k_scales)), _c(_np(v_scales))
    bt = _c(_np(block_table), np.int32)
    cl = _c(_np(context_lens), np.int32)
    B, hq, d = qa.shape
    P, ps, hkv, d2 = kc.shape
    if _dtype_code(qa) != BF16 or kc.dtype != np.int8 or vc.shape != kc.shape or d2 != d or \
            ks.dtype != np.float32 or ks.shape != (P, hkv, ps) or vs.shape != ks.shape or \
            bt.shape[0] != B:
        raise OracleError("shape / dtype mismatch")
    sq = _c(np.arange(B) if seqs is None else np.asarray(seqs), np.int32)
    out = np.zeros((sq.shape[0], hq, d), dtype=np.float64)
    rc = lib.oracle_paged_decode_int8(_ptr(qa), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt),
                                      bt.shape[1], _ptr(cl), B, hq, hkv, d, P, ps, int(window),
                                      int(ring_pages), float(scale), _ptr(sq), sq.shape[0],
                                      _ptr(out), int(threads))
    if rc != 0:
        raise OracleError(f"oracle_paged_decode_int8 failed ({rc})")
    return out


def paged_decode(q, k_cache, v_cache, block_table, context_lens, scale, window=0, seqs=None,
                 threads=0, ring_pages=0) -> np.ndarray:
    """out[i, h, :] for sequence seqs[i] (all sequences by default), float64 [n, H_q, d].
    ring_pages > 0: the table's first ring_pages entries are each sequence's ring."""
    lib = _load()
    qa, kc, vc = _c(_np(q)), _c(_np(k_cache)), _c(_np(v_cache))
    bt = _c(_np(block_table), np.int32)
    cl = _c(_np(context_lens), np.int32)
    B, hq, d = qa.shape
    P, ps, hkv, d2 = kc.shape
    dt = _dtype_code(kc)
    if _dtype_code(qa) != _query_code(dt) or vc.shape != kc.shape or d2 != d or bt.shape[0] != B:
        raise OracleError("shape / dtype mismatch")
    sq = _c(np.arange(B) if seqs is None else np.asarray(seqs), np.int32)
    out = np.zeros((sq.shape[0], hq, d), dtype=np.float64)
    rc = lib.oracle_paged_decode(_ptr(qa), _ptr(kc), _ptr(vc), dt, _ptr(bt), bt.shape[1],
                                 _ptr(cl), B, hq, hkv, d, P, ps, int(window), int(ring_pages),
                                 float(scale), _ptr(sq), sq.shape[0], _ptr(out), int(threads))
    if rc != 0:
        raise OracleError(f"oracle_paged_decode failed ({rc})")
    return out


def paged_prefill(q, k_cache, v_cache, block_table, positions, scale, window=0,
                  blockwise=True, key_block=DEFAULT_KEY_BLOCK, tokens=None,
                  threads=0, ring_pages=0) -> np.ndarray:
    """out[i, h, :] for flat token tokens[i] = b*T + t (all by default), float64.
    ring_pages > 0: the table's first ring_pages entries are each row's ring."""
    lib = _load()
    qa, kc, vc = _c(_np(q)), _c(_np(k_cache)), _c(_np(v_cache))
    bt = _c(_np(block_table), np.int32)
    pos = _c(_np(positions), np.int32)
    B, T, hq, d = qa.shape
    P, ps, hkv, d2 = kc.shape
    dt = _dtype_code(kc)
    if _dtype_code(qa) != _query_code(dt) or vc.shape != kc.shape or d2 != d or \
            pos.shape != (B, T):
        raise OracleError("shape / dtype mismatch")
    tk = _c(np.arange(B * T) if tokens is None else np.asarray(tokens), np.int64)
    out = np.zeros((tk.shape[0], hq, d), dtype=np.float64)
    rc = lib.oracle_paged_prefill(_ptr(qa), _ptr(kc), _ptr(vc), dt, _ptr(bt), bt.shape[1],
                                  _ptr(pos), B, T, hq, hkv, d, P, ps, int(window), int(ring_pages),
                                  float(scale), 1 if blockwise else 0, int(key_block), _ptr(tk),
                                  tk.shape[0],
                                  _ptr(out), int(threads))
    if rc != 0:
        raise OracleError(f"oracle_paged_prefill failed ({rc})")
    return out


def paged_prefill_int8(q, k_codes, v_codes, k_scales, v_scales, block_table, positions, scale,
                       window=0, blockwise=True, key_block=DEFAULT_KEY_BLOCK, tokens=None,
                       threads=0, ring_pages=0) -> np.ndarray:
    """paged_prefill over int8 pools: each element read as code x its row's scale."""
    lib = _load()
    qa = _c(_np(q))
    kc, vc = _c(_np(k_codes)), _c(_np(v_codes))
    ks, vs = _c(_np(k_scales)), _c(_np(v_scales))
    bt = _c(_np(block_table), np.int32)
    pos = _c(_np(positions), np.int32)
    B, T, hq, d = qa.shape
    P, ps, hkv, d2 = kc.shape
    if _dtype_code(qa) != BF16 or kc.dtype != np.int8 or vc.shape != kc.shape or d2 != d or \
            ks.dtype != np.float32 or ks.shape != (P, hkv, ps) or vs.shape != ks.shape or \
            pos.shape != (B, T) or bt.shape[0] != B:
        raise OracleError("shape / dtype mismatch")
    tk = _c(np.arange(B * T) if tokens is None else np.asarray(tokens), np.int64)
    out = np.zeros((tk.shape[0], hq, d), dtype=np.float64)
    rc = lib.oracle_paged_prefill_int8(_ptr(qa), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt),
                                       bt.shape[1], _ptr(pos), B, T, hq, hkv, d, P, ps,
                                       int(window), int(ring_pages), float(scale),
                                       1 if blockwise else 0, int(key_block), _ptr(tk),
                                       tk.shape[0], _ptr(out), int(threads))
    if rc != 0:
        raise OracleError(f"oracle_paged_prefill_int8 failed ({rc})")
    return out


def kv_bytes_per_token(layers: int, h_kv: int, d_head: int, bytes_per_elem: int) -> int:
    """M_KV/token = 2 * layers * H_kv * d_head * q."""
    return int(_load().oracle_kv_bytes_per_token(layers, h_kv, d_head, bytes_per_elem))


def ring_pages(window: int, chunk: int, page_size: int) -> int:
    """Ring pages for calls of up to `chunk` tokens with window `window`:
    ceil((window - 1 + chunk) / page_size)."""
    return int(_load().oracle_ring_pages(window, chunk, page_size))
