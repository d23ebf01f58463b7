"""Batched right-aligned prefill on the GPU against the oracle's blockwise fold:
the full-size batch (every token), the sliding-window mix's outlier values,
edge cases, batched == solo bit for bit, page-placement invariance."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import workloads as wl
from tests.gpu_util import (assert_prefill_rows, gpu_prefill, gpu_write, on_gpu,
                            oracle_prefill_tokens, permuted_pool)
from tests.parity import assert_close

pytestmark = pytest.mark.gpu


def test_full_size_batch_every_token():
    """The B=8 x 2,048 batch: the chunk's K/V written by the GPU, then the
    call; the oracle writes the same rows into its own copies of the pools as
    they were before, then folds every token of every row."""
    case = wl.batched_prefill(seed=0, device="cuda")
    g = on_gpu(case)
    k0, v0 = g.k_cache.clone(), g.v_cache.clone()
    gpu_write(g)
    out = gpu_prefill(g)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    hkv, d = case.Hkv, case.d
    assert_prefill_rows(out, g, range(case.B), pools=(k0, v0),
                        new_rows=(g.k_new.reshape(-1, hkv, d), g.v_new.reshape(-1, hkv, d),
                                  g.slot_mapping), what="full batch")


@pytest.mark.parametrize("window", [0, 4096])
def test_outliers_every_token(window):
    """Prefill on the sliding-window mix's value distribution (1% of Q, K and V
    values x8), full and window 4,096: rows of 1,024 tokens with prior context,
    every token against the oracle."""
    case = wl.prefill_case([0, 300, 700, 37], [6144, 3000, 0, 5000], T=1024, Hq=40, Hkv=8,
                           d=128, seed=61, window=window, outlier_p=0.01, device="cuda")
    g = on_gpu(case)
    k0, v0 = g.k_cache.clone(), g.v_cache.clone()
    gpu_write(g)
    out = gpu_prefill(g)
    torch.cuda.synchronize()
    assert_prefill_rows(out, g, range(case.B), pools=(k0, v0),
                        new_rows=(g.k_new, g.v_new, g.slot_mapping), what=f"outliers w{window}")


def test_batched_equals_solo_bit_for_bit():
    case = wl.prefill_case([100, 0, 700], [3000, 0, 5000], T=1024, Hq=16, Hkv=4, d=128, seed=5)
    g = on_gpu(case)
    gpu_write(g)
    both = gpu_prefill(g)
    for row in range(case.B):
        solo = tl.tl_paged_attn_prefill(g.q[row:row + 1].contiguous(), g.k_cache, g.v_cache,
                                        g.block_table[row:row + 1].contiguous(),
                                        g.positions[row:row + 1].contiguous(), g.scale)
        torch.cuda.synchronize()
        assert torch.equal(solo[0], both[row]), f"row {row}"


def test_page_placement_invariance():
    case = wl.prefill_case([10, 300], [2100, 0], T=512, Hq=8, Hkv=2, d=128, seed=6)
    g = on_gpu(case)
    gpu_write(g)
    a = gpu_prefill(g)
    kc, vc, bt = permuted_pool(g)
    b = tl.tl_paged_attn_prefill(g.q, kc, vc, bt, g.positions, g.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("window", [0, 1, 100, 2048, 2049])
def test_block_edges_and_windows(window):
    """Rows ending at and one past a 2,048-key block boundary, length 1, a row
    with no live token, a window start crossing a block boundary, and a T that
    is not a multiple of the tile."""
    T = 130
    pads = [0, 0, T - 1, T, 5, 60]
    p0 = [2048 - T, 2049 - T, 0, 0, 4000, 2000]
    case = wl.prefill_case(pads, p0, T=T, Hq=8, Hkv=2, d=128, window=window, seed=8,
                           nan_unused=True)
    g = on_gpu(case)
    gpu_write(g)
    out = gpu_prefill(g)
    torch.cuda.synchronize()
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    # the oracle reads the pool after the oracle's own write of the chunk
    oracle.kv_cache_write(case.k_new, case.v_new, kc, vc, case.slot_mapping)
    ref = oracle.paged_prefill(case.q, kc, vc, case.block_table, case.positions, case.scale,
                               window=window)
    assert_close(out.reshape(ref.shape), ref, f"edges window={window}")
    assert torch.all(out[3] == 0)  # the row with no live token


def test_group_shapes():
    for hq, hkv in ((8, 8), (32, 8), (16, 1)):
        case = wl.prefill_case([7, 0], [100, 1500], T=200, Hq=hq, Hkv=hkv, d=128, seed=9)
        g = on_gpu(case)
        gpu_write(g)
        out = gpu_prefill(g)
        torch.cuda.synchronize()
        kc, vc = case.k_cache.clone(), case.v_cache.clone()
        oracle.kv_cache_write(case.k_new, case.v_new, kc, vc, case.slot_mapping)
        ref = oracle.paged_prefill(case.q, kc, vc, case.block_table, case.positions, case.scale)
        assert_close(out.reshape(ref.shape), ref, f"hq={hq} hkv={hkv}")


def test_bad_page_is_reported_not_faulted():
    case = wl.prefill_case([0], [500], T=64, Hq=8, Hkv=2, d=128, seed=10)
    case.pool.block_table[0, 3] = case.num_pages + 100
    g = on_gpu(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_prefill(g, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & tl.TL_DEVERR_PAGE_RANGE
    assert torch.isfinite(out).all()


def test_v_beyond_fp16_range_is_reported():
    """P.V runs in fp16: a finite V entry beyond +-65504 in the keys a call
    reads is reported (65280, the largest bf16 below fp16's overflow, is not)."""
    case = wl.prefill_case([0], [500], T=64, Hq=8, Hkv=2, d=128, seed=11)
    g = on_gpu(case)
    gpu_write(g)
    slot = case.pool.slot(0, 100)  # prior context every token sees
    for val, flagged in ((65280.0, False), (-65536.0, True)):
        vc = g.v_cache.clone()
        vc.view(-1, case.Hkv, case.d)[slot, 1, 5] = val
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        tl.tl_paged_attn_prefill(g.q, g.k_cache, vc, g.block_table, g.positions, g.scale,
                                 error_word=err)
        torch.cuda.synchronize()
        assert bool(int(err.item()) & tl.TL_DEVERR_VALUE_RANGE) == flagged, (val, int(err.item()))


def test_small_workspace_is_refused():
    case = wl.prefill_case([0], [100], T=32, Hq=8, Hkv=2, d=128, seed=12)
    g = on_gpu(case)
    need = tl.tl_paged_attn_prefill_workspace_size(1, 32, 8, 2, 128, g.block_table.shape[1],
                                                   case.page_size)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(tl.TLError) as e:
        tl.tl_paged_attn_prefill(g.q, g.k_cache, g.v_cache, g.block_table, g.positions, g.scale,
                                 workspace=ws)
    assert e.value.status == tl.TL_ERR_WORKSPACE


@pytest.mark.parametrize("kind", ["bf16", "e4m3", "int8"])
def test_workspace_sized_by_the_rows_keys(kind):
    """A table of 131,072 positions per row (8,192 pages of 16) with rows that
    read at most ~3,300 keys: a workspace sized by the rows' keys (independent
    of the table's width) gives the same bits as one as wide as the table."""
    case = wl.prefill_case([0, 100, 900], [3000, 0, 1200], T=300, Hq=16, Hkv=4, d=128, seed=13,
                           max_pages_per_seq=8192, device="cuda")
    g = on_gpu(case)
    gpu_write(g)
    B, T, hq, hkv, d = case.B, case.T, case.Hq, case.Hkv, case.d
    if kind == "int8":
        pools = [t.to("cuda") for t in wl.int8_pools(case, 14)]
        dt = tl.TL_INT8
    elif kind == "e4m3":
        pools = [g.k_cache.float().to(torch.float8_e4m3fn), g.v_cache.float().to(torch.float8_e4m3fn)]
        dt = tl.TL_FP8_E4M3
    else:
        pools = [g.k_cache, g.v_cache]
        dt = tl.TL_BF16
    wide = tl.tl_paged_attn_prefill_workspace_size_ex(B, T, hq, hkv, d, 8192, 16, 0, dt)
    narrow = tl.tl_paged_attn_prefill_workspace_size_keys(B, T, hq, hkv, d, 3300, dt)
    assert narrow * 20 < wide
    outs = []
    for nbytes in (wide, narrow):
        ws = tl.alloc_workspace(nbytes, "cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if kind == "int8":
            o = tl.tl_paged_attn_prefill_int8(g.q, *pools, g.block_table, g.positions, g.scale,
                                              workspace=ws, error_word=err)
        else:
            o = tl.tl_paged_attn_prefill(g.q, *pools, g.block_table, g.positions, g.scale,
                                         workspace=ws, error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append(o)
    assert torch.equal(outs[0], outs[1])
    # a workspace too small for a row's keys: reported, nothing outside it touched
    ws = tl.alloc_workspace(tl.tl_paged_attn_prefill_workspace_size_keys(B, T, hq, hkv, d, 1000,
                                                                         dt), "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if kind == "int8":
        tl.tl_paged_attn_prefill_int8(g.q, *pools, g.block_table, g.positions, g.scale,
                                      workspace=ws, error_word=err)
    else:
        tl.tl_paged_attn_prefill(g.q, *pools, g.block_table, g.positions, g.scale, workspace=ws,
                                 error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & tl.TL_DEVERR_CONTEXT_RANGE
