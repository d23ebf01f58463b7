"""The C-ABI library loads and exports every entry point its header declares;
host-side argument checks refuse bad calls before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tl_paged_attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tl_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("tl_kv_cache_write", "tl_paged_attn_decode", "tl_paged_attn_prefill"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"{name} has no binding"


def test_status_strings(lib):
    for s in range(7):
        assert lib.tl_status_string(s).decode().startswith("TL_")
    assert lib.tl_status_string(99).decode() == "unknown tl_status"
    assert tl.tl_version() >= 10100


def test_status_and_error_bit_values_follow_the_header():
    """The binding's constants are the header's: TL_ERR_DEVICE_BOUNDS is 4 and
    TL_ERR_WORKSPACE 5; the TL_DEVERR_* bits are distinct powers of two."""
    from paged_kv_attention_cache_gb300 import api
    text = open(HEADER).read()
    statuses = {k: int(v) for k, v in re.findall(r"\b(TL_(?:OK|ERR_[A-Z_]+))\s*=\s*(\d+)", text)}
    assert statuses == {"TL_OK": 0, "TL_ERR_INVALID_ARG": 1, "TL_ERR_UNSUPPORTED": 2,
                        "TL_ERR_CUDA": 3, "TL_ERR_DEVICE_BOUNDS": 4, "TL_ERR_WORKSPACE": 5,
                        "TL_ERR_DEVICE_TIMEOUT": 6}
    for name, v in statuses.items():
        assert getattr(api, name) == v, name
    bits = {k: int(v) for k, v in re.findall(r"#define (TL_DEVERR_[A-Z_]+) (\d+)u", text)}
    assert len(bits) == 6
    for name, v in bits.items():
        assert getattr(api, name) == v, name
        assert v & (v - 1) == 0
    assert len(set(bits.values())) == len(bits)


def test_device_error_query_refuses_a_bad_word_before_any_cuda_call(lib):
    assert lib.tl_get_device_error(None, None, 0, None) == tl.TL_ERR_INVALID_ARG
    assert lib.tl_get_device_error(4098, None, 1, None) == tl.TL_ERR_INVALID_ARG  # misaligned


def align256(x):
    return (x + 255) // 256 * 256


def test_workspace_sizes(lib):
    assert tl.tl_paged_attn_decode_workspace_size(64, 32, 8, 128) > 0
    assert tl.tl_paged_attn_decode_workspace_size(64, 30, 8, 128) == 0  # h_q % h_kv
    assert tl.tl_paged_attn_decode_workspace_size(0, 32, 8, 128) == 0
    # the work counter (256 B), two int32 arrays over the B * n_pairs query-tile
    # pairs (n_pairs = 2048 / (2 * 128 / 4) = 32, each array rounded to 256 B),
    # the rows' first keys (B int32, rounded to 256 B), a flag per 64 keys of
    # each row (8 * 8192 / 64 int32) and per row (rounded to 256 B), then the
    # fp16 copy of V: B * h_kv * (max_pages_per_seq * page_size) * d * 2
    assert tl.tl_paged_attn_prefill_workspace_size(8, 2048, 32, 8, 128, 512, 16) == \
        256 + 2 * 1024 + 256 + 4096 + 256 + 8 * 8 * 512 * 16 * 128 * 2
    # over a ring of 257 pages the copy holds align_up(257 * 16, 128) + 256 keys
    # per row (70 flags of 64 keys per row: 2240 B, rounded to 2304)
    assert tl.tl_paged_attn_prefill_ring_workspace_size(8, 2048, 32, 8, 128, 512, 16, 257) == \
        256 + 2 * 1024 + 256 + 2304 + 256 + 8 * 8 * (4224 + 256) * 128 * 2
    assert tl.tl_paged_attn_prefill_ring_workspace_size(8, 2048, 32, 8, 128, 512, 16, 0) == 0
    assert tl.tl_paged_attn_prefill_workspace_size(8, 2048, 32, 8, 128, 0, 16) == 0
    # sized by the rows' keys instead of the table: the same layout with the
    # copy holding align_up(max_row_keys, 128) + 256 keys per row, whatever the
    # table's width (8192 keys -> 8448; 8448 / 64 = 132 flags per row)
    assert tl.tl_paged_attn_prefill_workspace_size_keys(8, 2048, 32, 8, 128, 8192, 1) == \
        256 + 2 * 1024 + 256 + align256(8 * 132 * 4) + 256 + 8 * 8 * 8448 * 128 * 2
    assert tl.tl_paged_attn_prefill_workspace_size_keys(8, 2048, 32, 8, 128, 0, 1) == 0
    # e4m3 and int8 pools add the bf16 copy of K (int8: and three scale arrays)
    kv = 8 * 8 * 8448
    assert tl.tl_paged_attn_prefill_workspace_size_keys(8, 2048, 32, 8, 128, 8192, 2) == \
        tl.tl_paged_attn_prefill_workspace_size_keys(8, 2048, 32, 8, 128, 8192, 1) + kv * 256
    assert tl.tl_paged_attn_prefill_workspace_size_keys(8, 2048, 32, 8, 128, 8192, 3) == \
        tl.tl_paged_attn_prefill_workspace_size_keys(8, 2048, 32, 8, 128, 8192, 2) + 3 * kv * 4
    # the decode bound grows with B and h_q but not with context length
    a = tl.tl_paged_attn_decode_workspace_size(64, 32, 8, 128)
    b = tl.tl_paged_attn_decode_workspace_size(128, 32, 8, 128)
    assert b > a


def test_host_validation_refuses_before_any_launch(lib):
    i = _lib
    # negative token count / null pointers: refused on the host
    assert lib.tl_kv_cache_write(None, None, None, None, None, -1, 4, 16, 8, 128, 1, None, None) == tl.TL_ERR_INVALID_ARG
    assert lib.tl_kv_cache_write(None, None, None, None, None, 3, 4, 16, 8, 128, 1, None, None) == tl.TL_ERR_INVALID_ARG
    # zero tokens is a no-op, even with null pointers
    assert lib.tl_kv_cache_write(None, None, None, None, None, 0, 4, 16, 8, 128, 1, None, None) == tl.TL_OK
    # misaligned pointers
    assert lib.tl_kv_cache_write(8, 16, 32, 48, 64, 1, 4, 16, 8, 128, 1, None, None) == tl.TL_ERR_INVALID_ARG
    # decode: null pointers, h_q % h_kv, unsupported head size, missing workspace
    args = dict(q=256, k=512, v=768, bt=1024, maxp=4, cl=1280, out=1536, B=2, hq=8, hkv=2,
                d=128, P=8, ps=16, w=0, sc=0.1, dt=1, ws=None, wsb=0, err=None, st=None)

    def dec(**kw):
        a = dict(args, **kw)
        return lib.tl_paged_attn_decode(a["q"], a["k"], a["v"], a["bt"], a["maxp"], a["cl"],
                                        a["out"], a["B"], a["hq"], a["hkv"], a["d"], a["P"],
                                        a["ps"], a["w"], a["sc"], a["dt"], a["ws"], a["wsb"],
                                        a["err"], a["st"])
    assert dec(q=None) == tl.TL_ERR_INVALID_ARG
    assert dec(hq=7) == tl.TL_ERR_INVALID_ARG
    assert dec(d=96) == tl.TL_ERR_UNSUPPORTED
    assert dec(dt=7) == tl.TL_ERR_UNSUPPORTED
    assert dec(hq=34, hkv=2) == tl.TL_ERR_UNSUPPORTED  # group 17 > 16
    assert dec(w=-1) == tl.TL_ERR_INVALID_ARG
    assert dec() == tl.TL_ERR_WORKSPACE
    assert dec(ws=2048 + 16, wsb=1 << 30) == tl.TL_ERR_WORKSPACE  # not 256-byte aligned

    # decode that writes its new rows first: the write's own checks, before
    # any launch (a 256-aligned fake workspace passes the size check)
    def decw(nk=2304, nv=2560, nd=1, sm=2816, n=2, **kw):
        a = dict(args, ws=4096, wsb=1 << 30, **kw)
        return lib.tl_paged_attn_decode_write(a["q"], nk, nv, nd, sm, n, a["k"], a["v"], a["bt"],
                                              a["maxp"], a["cl"], a["out"], a["B"], a["hq"],
                                              a["hkv"], a["d"], a["P"], a["ps"], a["w"], a["sc"],
                                              a["dt"], a["ws"], a["wsb"], a["err"], a["st"])
    assert decw(n=-1) == tl.TL_ERR_INVALID_ARG
    assert decw(nk=None) == tl.TL_ERR_INVALID_ARG
    assert decw(sm=2820) == tl.TL_ERR_INVALID_ARG  # slots not 8-byte aligned
    assert decw(nk=2312) == tl.TL_ERR_INVALID_ARG  # new rows not 16-byte aligned
    assert decw(nd=0) == tl.TL_ERR_UNSUPPORTED  # f32 rows into bf16 pools
    assert decw(nd=2, dt=2) == tl.TL_ERR_UNSUPPORTED  # e4m3 rows into e4m3 pools

    # int8 pools: the write's and the decode's own checks
    def w8(kn=2304, vn=2560, sd=1, ks=12288, vs=16384, sm=2816, n=2, d=128):
        return lib.tl_kv_cache_write_int8(kn, vn, sd, 4096, 8192, ks, vs, sm, n, 4, 16, 8, d,
                                          None, None)
    assert w8(n=-1) == tl.TL_ERR_INVALID_ARG
    assert w8(n=0, kn=None) == tl.TL_OK  # no rows: a no-op
    assert w8(sd=2) == tl.TL_ERR_UNSUPPORTED  # e4m3 rows
    assert w8(d=2048) == tl.TL_ERR_UNSUPPORTED
    assert w8(ks=None) == tl.TL_ERR_INVALID_ARG
    assert w8(ks=12290) == tl.TL_ERR_INVALID_ARG  # scales not 4-byte aligned
    assert w8(kn=2312) == tl.TL_ERR_INVALID_ARG  # new rows not 16-byte aligned
    assert w8(sm=2820) == tl.TL_ERR_INVALID_ARG  # slots not 8-byte aligned

    def d8(ks=12288, vs=16384, **kw):
        a = dict(args, ws=4096, wsb=1 << 30, **kw)
        return lib.tl_paged_attn_decode_int8(a["q"], a["k"], a["v"], ks, vs, a["bt"], a["maxp"],
                                             a["cl"], a["out"], a["B"], a["hq"], a["hkv"], a["d"],
                                             a["P"], a["ps"], a["w"], a["sc"], a["ws"], a["wsb"],
                                             a["err"], a["st"])
    assert d8(ks=None) == tl.TL_ERR_INVALID_ARG
    assert d8(vs=16392) == tl.TL_ERR_INVALID_ARG  # scales not 16-byte aligned
    assert d8(ps=24) == tl.TL_ERR_UNSUPPORTED  # a chunk's scales would span pages
    assert d8(d=64) == tl.TL_ERR_UNSUPPORTED
    assert d8(q=None) == tl.TL_ERR_INVALID_ARG

    def d8w(nd=1, sm=2816, n=2, ks=12288, **kw):
        a = dict(args, ws=4096, wsb=1 << 30, **kw)
        return lib.tl_paged_attn_decode_write_int8(a["q"], 2304, 2560, nd, sm, n, a["k"], a["v"],
                                                   ks, 16384, a["bt"], a["maxp"], a["cl"],
                                                   a["out"], a["B"], a["hq"], a["hkv"], a["d"],
                                                   a["P"], a["ps"], a["w"], a["sc"], a["ws"],
                                                   a["wsb"], a["err"], a["st"])
    assert d8w(ks=None) == tl.TL_ERR_INVALID_ARG
    assert d8w(n=-1) == tl.TL_ERR_INVALID_ARG
    assert d8w(sm=2820) == tl.TL_ERR_INVALID_ARG  # slots not 8-byte aligned
    assert d8w(nd=2) == tl.TL_ERR_UNSUPPORTED  # e4m3 rows into int8 pools
    assert d8w(ps=24) == tl.TL_ERR_UNSUPPORTED

    def pre(**kw):
        a = dict(args, **kw)
        return lib.tl_paged_attn_prefill(a["q"], a["k"], a["v"], a["bt"], a["maxp"], a["cl"],
                                         a["out"], a["B"], 4, a["hq"], a["hkv"], a["d"], a["P"],
                                         a["ps"], a["w"], a["sc"], a["dt"], a["ws"], a["wsb"],
                                         a["err"], a["st"])
    assert pre(q=None) == tl.TL_ERR_INVALID_ARG
    assert pre(dt=0) == tl.TL_ERR_UNSUPPORTED  # prefill is bf16 only
    assert pre(d=64) == tl.TL_ERR_UNSUPPORTED
    assert pre(ps=12) == tl.TL_ERR_UNSUPPORTED


def test_ops_refuse_cpu_tensors():
    import torch
    x = torch.zeros(4, 2, 8)
    with pytest.raises(TypeError):
        tl.tl_kv_cache_write(x, x, torch.zeros(2, 4, 2, 8), torch.zeros(2, 4, 2, 8),
                             torch.zeros(4, dtype=torch.int64))


def test_the_default_library_has_no_decode_trace(lib):
    """The trace calls exist in every build; the default one answers that the
    option is absent, before any CUDA call."""
    buf = (ctypes.c_uint64 * 8)()
    assert lib.tl_decode_trace_reset() == tl.TL_ERR_UNSUPPORTED
    assert lib.tl_decode_trace_read(buf, 8) == tl.TL_ERR_UNSUPPORTED


def test_the_default_library_has_no_prefill_trace(lib):
    buf = (ctypes.c_uint64 * 7)()
    assert lib.tl_prefill_trace_reset() == tl.TL_ERR_UNSUPPORTED
    assert lib.tl_prefill_trace_read(buf, 1) == tl.TL_ERR_UNSUPPORTED
