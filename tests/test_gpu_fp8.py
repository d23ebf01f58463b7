"""The fp8 (e4m3fn) KV cache on the GPU ("How serving works in Tlaloc", the
FP8 KV cache paragraph of its quantisation section): the converting write is
bit-exact against the oracle, and decode over e4m3 pools matches the oracle
reading the same codes.  The pools handed to both sides are built on the host
(torch's float8 conversion of seeded values, the oracle's write for the new
rows), so no oracle input comes from the CUDA path."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import workloads as wl
from tests.gpu_util import assert_decode_all, sub_pool
from tests.parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("src", [torch.bfloat16, torch.float32])
def test_fp8_write_is_bit_exact(src):
    g = torch.Generator().manual_seed(71)
    P, ps, hkv, d, N = 40, 16, 8, 128, 300
    kn = torch.randn((N, hkv, d), generator=g) * torch.exp(torch.randn((N, hkv, d), generator=g) * 3)
    vn = torch.randn((N, hkv, d), generator=g) * 50
    # exact ties between codes, the clamp, NaN, infinities, signed zeros
    codes = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double()
    mids = ((codes[:-1] + codes[1:]) / 2).float()
    kn.view(-1)[:mids.numel()] = mids
    kn.view(-1)[mids.numel():mids.numel() + 8] = torch.tensor(
        [448.0, 460.0, 464.0, 1e9, -1e9, float("inf"), float("-inf"), -0.0])
    vn.view(-1)[:3] = torch.tensor([float("nan"), -float("nan"), 0.0])
    kn, vn = kn.to(src), vn.to(src)
    slots = torch.randperm(P * ps, generator=g)[:N].to(torch.int64)
    slots[::7] = -1  # pads
    kc0 = torch.randint(0, 256, (P, ps, hkv, d), generator=g, dtype=torch.uint8)
    vc0 = torch.randint(0, 256, (P, ps, hkv, d), generator=g, dtype=torch.uint8)
    kc_ref, vc_ref = kc0.clone().numpy(), vc0.clone().numpy()
    oracle.kv_cache_write_fp8(kn, vn, kc_ref, vc_ref, slots)
    kc = kc0.to(DEV).view(torch.float8_e4m3fn)
    vc = vc0.to(DEV).view(torch.float8_e4m3fn)
    err = _err()
    tl.tl_kv_cache_write_fp8(kn.to(DEV), vn.to(DEV), kc, vc, slots.to(DEV), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(kc.view(torch.uint8).cpu().numpy(), kc_ref)
    assert np.array_equal(vc.view(torch.uint8).cpu().numpy(), vc_ref)


def _fp8_case(case):
    """Host e4m3 pools of a bf16 case (torch's conversion of the stored
    values), the new rows written by the oracle; then on the GPU."""
    k8 = case.k_cache.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    v8 = case.v_cache.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    oracle.kv_cache_write_fp8(case.k_new, case.v_new, k8, v8, case.slot_mapping)
    return (torch.from_numpy(k8).view(torch.float8_e4m3fn), torch.from_numpy(v8).view(torch.float8_e4m3fn))


def _decode_fp8(case, k8, v8, rows, window=None, ring=0):
    w = case.window if window is None else window
    dev = lambda t: t.to(DEV)
    err = _err()
    if ring:
        out = tl.tl_paged_attn_decode_ring(dev(case.q), dev(k8), dev(v8), dev(case.block_table),
                                           dev(case.context_lens), case.scale, w, ring,
                                           error_word=err)
    else:
        out = tl.tl_paged_attn_decode(dev(case.q), dev(k8), dev(v8), dev(case.block_table),
                                      dev(case.context_lens), case.scale, window=w,
                                      error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ps = case.page_size
    lens = case.context_lens.tolist()
    n_pages = [ring] * len(rows) if ring else [(max(lens[b], 0) + ps - 1) // ps for b in rows]
    kc, vc, bt = sub_pool(k8.view(torch.uint8), v8.view(torch.uint8), case.block_table, rows,
                          n_pages)
    ref = oracle.paged_decode(case.q[rows], kc.numpy(), vc.numpy(), bt, case.context_lens[rows],
                              case.scale, window=w, ring_pages=ring)
    return out, ref


@pytest.mark.parametrize("maker", [wl.llama8b_decode, lambda **k: wl.swa_decode(layer=0, **k),
                                   lambda **k: wl.swa_decode(layer=1, **k), wl.longctx_decode])
def test_fp8_decode_full_size_every_sequence(maker):
    """The full-size workloads over e4m3 pools, every sequence against the
    oracle's e4m3 form.  The pools are torch's float8_e4m3fn conversion of
    the seeded bf16 values (the conversion the oracle's e4m3 encoder is
    pinned against), not the library's write."""
    case = maker(seed=0, device=DEV)
    g = wl.to_device(case, DEV)
    k8 = torch.empty(g.k_cache.shape, dtype=torch.float8_e4m3fn, device=DEV)
    v8 = torch.empty_like(k8)
    for src, dst in ((g.k_cache, k8), (v_cache := g.v_cache, v8)):
        for p0 in range(0, src.shape[0], 4096):
            dst[p0:p0 + 4096] = src[p0:p0 + 4096].float().to(torch.float8_e4m3fn)
    del g.k_cache, g.v_cache, v_cache
    err = _err()
    out = tl.tl_paged_attn_decode(g.q, k8, v8, g.block_table, g.context_lens, g.scale,
                                  window=g.window, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_decode_all(out, g.q, k8, v8, g.block_table, g.context_lens, g.scale, window=g.window,
                      what="fp8 decode")


@pytest.mark.parametrize("window", [0, 1, 16, 100])
def test_fp8_decode_edge_lengths(window):
    case = wl.decode_case([1, 15, 16, 17, 100, 257, 1000], Hq=32, Hkv=8, d=128, seed=72,
                          window=window)
    k8, v8 = _fp8_case(case)
    rows = list(range(case.B))
    out, ref = _decode_fp8(case, k8, v8, rows)
    assert_close(out, ref, f"fp8 decode window {window}")


@pytest.mark.parametrize("page_size", [8, 24, 32, 40])
@pytest.mark.parametrize("window", [0, 37])
def test_fp8_decode_page_sizes(page_size, window):
    """e4m3 pipeline stages hold two 16-key chunks; pages that are not a
    multiple of 16 keys (8, 24, 40) take the per-key page lookup, a page size
    that is not a power of two the division path; lengths around chunk, stage
    and page boundaries."""
    lens = [1, 15, 16, 17, 31, 32, 33, 47, 48, 49, 95, 96, 97, 300, 1000]
    case = wl.decode_case(lens, Hq=16, Hkv=4, d=128, page_size=page_size, seed=74,
                          window=window, nan_unused=True)  # dead rows hold NaN codes
    k8, v8 = _fp8_case(case)
    rows = list(range(case.B))
    out, ref = _decode_fp8(case, k8, v8, rows)
    assert_close(out, ref, f"fp8 decode page {page_size} window {window}")


@pytest.mark.parametrize("shape", ["many_short", "one_long", "mixed"])
def test_fp8_piece_plan_extremes(shape):
    """The piece plan's extremes over e4m3 pools (the one-byte kernel takes
    32 keys per stage): 2,048 short sequences, one of 131,072 keys, and both
    mixed with empty and one-key sequences; every sequence against the
    oracle."""
    g = torch.Generator().manual_seed(93)
    if shape == "many_short":
        lens = torch.randint(1, 400, (2048,), generator=g).tolist()
    elif shape == "one_long":
        lens = [131072]
    else:
        lens = torch.randint(1, 300, (500,), generator=g).tolist() + [65536, 257, 4096, 0, 1]
    case = wl.decode_case(lens, Hq=32, Hkv=8, d=128, seed=94)
    k8, v8 = (t.to(DEV) for t in _fp8_case(case))
    q, bt, cl = case.q.to(DEV), case.block_table.to(DEV), case.context_lens.to(DEV)
    err = _err()
    out = tl.tl_paged_attn_decode(q, k8, v8, bt, cl, case.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isfinite(out).all()
    assert_decode_all(out, q, k8, v8, bt, cl, case.scale, chunk=256, what=f"fp8 piece plan {shape}")


def test_fp8_decode_reports_a_query_beyond_fp16():
    """The query is rounded to fp16 for the e4m3 MMAs: a finite element beyond
    65504 is reported (TL_DEVERR_VALUE_RANGE), not silently made infinite;
    an in-range query on the same pools reports nothing."""
    case = wl.decode_case([40, 100], Hq=8, Hkv=2, d=128, seed=73)
    k8, v8 = _fp8_case(case)
    dev = lambda t: t.to(DEV)
    for big, want in [(60000.0, 0), (1e5, tl.TL_DEVERR_VALUE_RANGE)]:
        q = case.q.clone()
        q[1, 3, 17] = big
        err = _err()
        tl.tl_paged_attn_decode(dev(q), dev(k8), dev(v8), dev(case.block_table),
                                dev(case.context_lens), case.scale, error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == want


def test_fp8_decode_over_rings():
    case = wl.swa_ring_decode(seed=1, B=32)
    ring = case.extra["ring_pages"]
    k8, v8 = _fp8_case(case)
    rows = list(range(case.B))
    out, ref = _decode_fp8(case, k8, v8, rows, ring=ring)
    assert_close(out, ref, "fp8 ring decode")


@pytest.mark.parametrize("q_len,hq,window", [(4, 32, 0), (2, 32, 0), (2, 16, 0), (3, 16, 0),
                                             (2, 16, 300), (3, 8, 0)])
def test_fp8_multi_token_decode(q_len, hq, window):
    """q_len tokens x the group's heads as the kernel's rows: 16 (two row
    groups), 8, 4 (the low parts of P in columns 4-7), 6 and 3 (unused
    columns); with and without a window."""
    lengths = wl.llama8b_lengths(seed=9, B=12)
    p0 = [L - q_len for L in lengths]
    case = wl.prefill_case([0] * len(lengths), p0, T=q_len, Hq=hq, Hkv=8, d=128, seed=73,
                           window=window)
    k8 = case.k_cache.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    v8 = case.v_cache.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    oracle.kv_cache_write_fp8(case.k_new, case.v_new, k8, v8, case.slot_mapping)
    k8t = torch.from_numpy(k8).view(torch.float8_e4m3fn)
    v8t = torch.from_numpy(v8).view(torch.float8_e4m3fn)
    cl = torch.tensor(lengths, dtype=torch.int32)
    err = _err()
    out = tl.tl_paged_attn_decode_multi(case.q.to(DEV), k8t.to(DEV), v8t.to(DEV),
                                        case.block_table.to(DEV), cl.to(DEV), case.scale,
                                        window=window, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for row in range(case.B):
        ref = oracle.paged_prefill(case.q[row:row + 1], k8, v8, case.block_table[row:row + 1],
                                   case.positions[row:row + 1], case.scale, window=window)
        assert_close(out[row], ref, f"fp8 multi-token row {row}")


def _fp8_prefill_case(case):
    k8 = case.k_cache.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    v8 = case.v_cache.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    kn, vn = case.k_new.view(-1, case.Hkv, case.d), case.v_new.view(-1, case.Hkv, case.d)
    oracle.kv_cache_write_fp8(kn, vn, k8, v8, case.slot_mapping)
    return k8, v8


@pytest.mark.parametrize("window", [0, 300])
def test_fp8_prefill_matches_the_oracle(window):
    case = wl.prefill_case([0, 40, 500], [100, 3000, 0], T=512, Hq=32, Hkv=8, d=128, seed=74,
                           window=window)
    k8, v8 = _fp8_prefill_case(case)
    k8t = torch.from_numpy(k8).view(torch.float8_e4m3fn).to(DEV)
    v8t = torch.from_numpy(v8).view(torch.float8_e4m3fn).to(DEV)
    err = _err()
    out = tl.tl_paged_attn_prefill(case.q.to(DEV), k8t, v8t, case.block_table.to(DEV),
                                   case.positions.to(DEV), case.scale, window=window,
                                   error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rng = np.random.default_rng(75)
    for row in range(case.B):
        ts = sorted({0, case.T - 1, case.pads[row]} | set(rng.integers(0, case.T, 10).tolist()))
        ts = [t for t in ts if t < case.T]
        ref = oracle.paged_prefill(case.q[row:row + 1], k8, v8, case.block_table[row:row + 1],
                                   case.positions[row:row + 1], case.scale, window=window,
                                   tokens=np.asarray(ts, np.int64))
        assert_close(out[row, ts], ref, f"fp8 prefill row {row}")


def test_fp8_prefill_full_size_sampled():
    case = wl.batched_prefill(seed=0)
    k8, v8 = _fp8_prefill_case(case)
    out = tl.tl_paged_attn_prefill(case.q.to(DEV), torch.from_numpy(k8).view(torch.float8_e4m3fn).to(DEV),
                                   torch.from_numpy(v8).view(torch.float8_e4m3fn).to(DEV),
                                   case.block_table.to(DEV), case.positions.to(DEV), case.scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(76)
    for row in (0, 4, 7):
        ts = sorted(set(rng.integers(case.pads[row], case.T, 8).tolist()) | {case.T - 1})
        ref = oracle.paged_prefill(case.q[row:row + 1], k8, v8, case.block_table[row:row + 1],
                                   case.positions[row:row + 1], case.scale,
                                   tokens=np.asarray(ts, np.int64), threads=0)
        assert_close(out[row, ts], ref, f"fp8 prefill (full size) row {row}")
