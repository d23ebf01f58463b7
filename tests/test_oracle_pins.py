"""Pins of the CPU oracle against facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a worked
figure the pages print (tests/golden), dense attention over a contiguous
history computed with library routines, a closed form, or an invariant the
pages state.  The negative controls plant a mistake in the oracle's inputs (on
the CPU) and check that the same comparison then fails.
"""
from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import oracle
from tests.dense_history import dense_reference, history_case, round_to

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _queries(case, n, seed):
    rng = np.random.default_rng(seed)
    q_st, q_vals = round_to(rng.standard_normal((n, case.Hq, case.d)), case.dtype)
    return q_st, q_vals


# ------------------------------------------------------------- the write --

def test_write_matches_fancy_index_and_skips_pads():
    rng = np.random.default_rng(1)
    P, ps, hkv, d = 6, 4, 2, 8
    kc = rng.standard_normal((P, ps, hkv, d)).astype(np.float32)
    vc = rng.standard_normal((P, ps, hkv, d)).astype(np.float32)
    slots = np.array([5, -1, 17, 0, -1, 23], dtype=np.int64)
    kn = rng.standard_normal((6, hkv, d)).astype(np.float32)
    vn = rng.standard_normal((6, hkv, d)).astype(np.float32)
    k_ref, v_ref = kc.copy(), vc.copy()
    live = slots >= 0
    k_ref.reshape(P * ps, hkv, d)[slots[live]] = kn[live]
    v_ref.reshape(P * ps, hkv, d)[slots[live]] = vn[live]
    k_o, v_o = kc.copy(), vc.copy()
    oracle.kv_cache_write(kn, vn, k_o, v_o, slots)
    assert k_o.tobytes() == k_ref.tobytes() and v_o.tobytes() == v_ref.tobytes()
    # every byte outside the live slots is unchanged
    untouched = np.ones(P * ps, dtype=bool)
    untouched[slots[live]] = False
    assert np.array_equal(k_o.reshape(P * ps, -1)[untouched], kc.reshape(P * ps, -1)[untouched])
    # negative control: a pad that writes its KV changes the pool
    bad = slots.copy()
    bad[1] = 9
    k_b, v_b = kc.copy(), vc.copy()
    oracle.kv_cache_write(kn, vn, k_b, v_b, bad)
    assert k_b.tobytes() != k_ref.tobytes()


def test_write_bf16_is_a_byte_copy():
    case = history_case([5, 9], 2, 1, 16, 4, torch.bfloat16, seed=2)
    rng = np.random.default_rng(3)
    kn, _ = round_to(rng.standard_normal((3, 1, 16)), torch.bfloat16)
    vn, _ = round_to(rng.standard_normal((3, 1, 16)), torch.bfloat16)
    slots = np.array([case.pages_of[0][1] * 4 + 0, -1, case.pages_of[1][2] * 4 + 0], np.int64)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.kv_cache_write(kn, vn, kc, vc, slots)
    flat = kc.reshape(-1, 16)
    assert np.array_equal(flat[slots[0]], kn[0, 0]) and np.array_equal(flat[slots[2]], kn[2, 0])


# ------------------------------------------ attention vs a dense history --

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_equals_dense_attention_over_the_history(dtype):
    lengths = [37, 100, 1, 16, 17]
    case = history_case(lengths, Hq=4, Hkv=2, d=64, page_size=16, dtype=dtype, seed=4)
    q_st, q_vals = _queries(case, len(lengths), 5)
    out = oracle.paged_decode(q_st, case.k_cache, case.v_cache, case.block_table, lengths,
                              case.scale)
    for b, L in enumerate(lengths):
        ref = dense_reference(case, q_vals[b], b, L - 1)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("window", [1, 5, 16, 17, 40])
def test_decode_window_equals_dense_over_last_w_keys(window):
    lengths = [37, 100, 3]
    case = history_case(lengths, Hq=6, Hkv=3, d=32, page_size=8, seed=6)
    q_st, q_vals = _queries(case, 3, 7)
    out = oracle.paged_decode(q_st, case.k_cache, case.v_cache, case.block_table, lengths,
                              case.scale, window=window)
    for b, L in enumerate(lengths):
        ref = dense_reference(case, q_vals[b], b, L - 1, window)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_prefill_equals_dense_attention_per_token():
    # two rows, right-aligned: pads (position -1) first, then live tokens
    lengths = [40, 23]
    case = history_case(lengths, Hq=4, Hkv=1, d=16, page_size=4, seed=8)
    T = 12
    positions = np.full((2, T), -1, np.int32)
    positions[0, 2:] = np.arange(30, 40)  # 2 pads, prior context 30
    positions[1, 5:] = np.arange(16, 23)  # 5 pads, prior context 16
    q_st, q_vals = _queries(case, 2 * T, 9)
    q4 = q_st.reshape(2, T, 4, 16)
    for blockwise, kb in ((False, 2048), (True, 2048), (True, 8), (True, 3)):
        out = oracle.paged_prefill(q4, case.k_cache, case.v_cache, case.block_table, positions,
                                   case.scale, blockwise=blockwise, key_block=kb)
        for b in range(2):
            for t in range(T):
                ref = dense_reference(case, q_vals[b * T + t], b, int(positions[b, t]))
                np.testing.assert_allclose(out[b * T + t], ref, rtol=1e-12, atol=1e-13)


def test_negative_control_wrong_head_mapping_is_caught():
    """If query head h read KV head h % H_kv instead of h / group, the dense
    comparison would fail: emulate that by permuting the KV heads."""
    lengths = [20]
    case = history_case(lengths, Hq=4, Hkv=2, d=16, page_size=4, seed=10)
    q_st, q_vals = _queries(case, 1, 11)
    # heads (0,1,2,3) -> kv (0,0,1,1); the mistake maps them to (0,1,0,1):
    # swap q heads 1 and 2 so the oracle's correct mapping plays the mistake
    q_bad = q_st[:, [0, 2, 1, 3], :]
    out = oracle.paged_decode(q_bad, case.k_cache, case.v_cache, case.block_table, lengths,
                              case.scale)[0][[0, 2, 1, 3]]
    ref = dense_reference(case, q_vals[0], 0, 19)
    assert np.abs(out - ref).max() > 1e-3


def test_negative_control_off_by_one_length_is_caught():
    lengths = [21]
    case = history_case(lengths, Hq=2, Hkv=1, d=16, page_size=4, seed=12)
    q_st, q_vals = _queries(case, 1, 13)
    out_short = oracle.paged_decode(q_st, case.k_cache, case.v_cache, case.block_table, [20],
                                    case.scale)
    ref = dense_reference(case, q_vals[0], 0, 20)
    assert np.abs(out_short[0] - ref).max() > 1e-3


# ------------------------------------------------------------ closed forms --

def test_length_one_returns_v0_exactly():
    case = history_case([1, 1], Hq=4, Hkv=2, d=32, page_size=16, seed=14)
    q_st, _ = _queries(case, 2, 15)
    out = oracle.paged_decode(q_st, case.k_cache, case.v_cache, case.block_table, [1, 1],
                              case.scale)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(out[b, h], case.hist_v[b][0, h // 2])


def test_length_zero_returns_zero():
    case = history_case([0, 5], Hq=2, Hkv=1, d=16, page_size=4, seed=16)
    q_st, _ = _queries(case, 2, 17)
    out = oracle.paged_decode(q_st, case.k_cache, case.v_cache, case.block_table, [0, 5],
                              case.scale)
    assert np.all(out[0] == 0.0)
    assert np.all(np.isfinite(out[1]))


def test_constant_values_give_that_constant():
    case = history_case([50], Hq=2, Hkv=1, d=16, page_size=8, seed=18)
    vc = case.v_cache.copy()
    vc[...] = -0.5
    q_st, _ = _queries(case, 1, 19)
    out = oracle.paged_decode(q_st, case.k_cache, vc, case.block_table, [50], case.scale)
    assert np.all(out == -0.5)


def test_equal_keys_give_the_mean_of_live_values():
    case = history_case([45], Hq=2, Hkv=1, d=16, page_size=8, seed=20)
    kc = case.k_cache.copy()
    kc[...] = 0.25
    q_st, _ = _queries(case, 1, 21)
    for window in (0, 7):
        out = oracle.paged_decode(q_st, kc, case.v_cache, case.block_table, [45], case.scale,
                                  window=window)
        lo = 0 if window == 0 else 45 - window
        mean = case.hist_v[0][lo:45, 0, :].mean(axis=0)
        np.testing.assert_allclose(out[0, 0], mean, rtol=1e-13, atol=1e-14)


def test_one_dominant_key_returns_its_value():
    case = history_case([30], Hq=1, Hkv=1, d=16, page_size=8, seed=22)
    q = np.zeros((1, 1, 16), np.float32)
    q[0, 0, 3] = 1.0
    kc = case.k_cache.copy()
    kc[..., 3] = 0.0
    star = 13
    pg = case.pages_of[0][star // 8]
    kc[pg, star % 8, 0, 3] = 4000.0  # score gap 1000 with scale 1/4: exp(-1000) = 0
    out = oracle.paged_decode(q, kc, case.v_cache, case.block_table, [30], case.scale)
    assert np.array_equal(out[0, 0], case.hist_v[0][star, 0])


# -------------------------------------------------------------- invariants --

def test_window_at_least_length_equals_full():
    lengths = [33, 64]
    case = history_case(lengths, Hq=2, Hkv=1, d=16, page_size=16, seed=24)
    q_st, _ = _queries(case, 2, 25)
    full = oracle.paged_decode(q_st, case.k_cache, case.v_cache, case.block_table, lengths,
                               case.scale)
    for w in (64, 65, 10_000):
        wo = oracle.paged_decode(q_st, case.k_cache, case.v_cache, case.block_table, lengths,
                                 case.scale, window=w)
        assert np.array_equal(full, wo)


def test_page_placement_does_not_change_the_result():
    lengths = [37, 100]
    a = history_case(lengths, Hq=4, Hkv=2, d=32, page_size=16, seed=26)
    # same histories, a different shuffle of the pool: rebuild the pool by
    # moving every page and rewriting the table
    rng = np.random.default_rng(27)
    P = a.k_cache.shape[0]
    new_of_old = rng.permutation(P)
    kc = np.empty_like(a.k_cache)
    vc = np.empty_like(a.v_cache)
    kc[new_of_old] = a.k_cache
    vc[new_of_old] = a.v_cache
    bt = np.where(a.block_table >= 0, new_of_old[np.maximum(a.block_table, 0)], -1).astype(np.int32)
    q_st, _ = _queries(a, 2, 28)
    o1 = oracle.paged_decode(q_st, a.k_cache, a.v_cache, a.block_table, lengths, a.scale)
    o2 = oracle.paged_decode(q_st, kc, vc, bt, lengths, a.scale)
    assert np.array_equal(o1, o2)


def _edge_prefill(key_block, window):
    """Rows at the pages' edge cases for the blockwise fold: lengths at and one
    past a block boundary, 0 and 1, a row with no live token, and (with a
    window) a window start crossing a block boundary."""
    kb = key_block
    lengths = [kb, kb + 1, 1, 3 * kb + 5, 2 * kb + 2, 0]
    case = history_case(lengths, Hq=2, Hkv=1, d=8, page_size=4, seed=30 + kb + window)
    T = 4
    pos = np.full((len(lengths), T), -1, np.int32)
    for b, L in enumerate(lengths):
        n = min(T, L)
        if n:
            pos[b, T - n:] = np.arange(L - n, L)
    return case, pos


@pytest.mark.parametrize("key_block,window", [(8, 0), (8, 5), (8, 9), (16, 0), (16, 20), (2048, 0)])
def test_blockwise_equals_one_pass_at_the_edges(key_block, window):
    case, pos = _edge_prefill(key_block, window)
    B, T = pos.shape
    q_st, q_vals = _queries(case, B * T, 31)
    q4 = q_st.reshape(B, T, case.Hq, case.d)
    one = oracle.paged_prefill(q4, case.k_cache, case.v_cache, case.block_table, pos, case.scale,
                               window=window, blockwise=False)
    blk = oracle.paged_prefill(q4, case.k_cache, case.v_cache, case.block_table, pos, case.scale,
                               window=window, blockwise=True, key_block=key_block)
    np.testing.assert_allclose(blk, one, rtol=0, atol=1e-12)
    for b in range(B):
        for t in range(T):
            ref = dense_reference(case, q_vals[b * T + t], b, int(pos[b, t]), window)
            np.testing.assert_allclose(blk[b * T + t], ref, rtol=0, atol=1e-12)
    # padding rows and the no-live row come out exactly 0
    assert np.all(blk[pos.reshape(-1) < 0] == 0.0)


def test_call_with_no_live_position_is_all_zero():
    case = history_case([10], Hq=2, Hkv=1, d=8, page_size=4, seed=40)
    pos = np.full((1, 5), -1, np.int32)
    q_st, _ = _queries(case, 5, 41)
    out = oracle.paged_prefill(q_st.reshape(1, 5, 2, 8), case.k_cache, case.v_cache,
                               case.block_table, pos, case.scale, blockwise=True, key_block=4)
    assert np.all(out == 0.0)


def test_batched_row_equals_the_row_alone():
    """A row prefilled together with others gives what it gives alone, bit for
    bit ("How serving works in Tlaloc", section 1, BatchedPrefillTest)."""
    lengths = [30, 19, 44]
    case = history_case(lengths, Hq=4, Hkv=2, d=16, page_size=4, seed=42)
    T = 10
    pos = np.full((3, T), -1, np.int32)
    pos[0, 3:] = np.arange(23, 30)
    pos[1, 0:] = np.arange(9, 19)
    pos[2, 6:] = np.arange(40, 44)
    q_st, _ = _queries(case, 3 * T, 43)
    q4 = q_st.reshape(3, T, 4, 16)
    both = oracle.paged_prefill(q4, case.k_cache, case.v_cache, case.block_table, pos,
                                case.scale, key_block=8)
    for b in range(3):
        alone = oracle.paged_prefill(q4[b:b + 1], case.k_cache, case.v_cache,
                                     case.block_table[b:b + 1], pos[b:b + 1], case.scale,
                                     key_block=8)
        assert np.array_equal(alone, both[b * T:(b + 1) * T])


def test_padding_that_writes_its_kv_changes_the_result():
    """Negative control from the same passage: a pad whose K/V lands in the
    pool changes what live tokens read."""
    lengths = [12]
    case = history_case(lengths, Hq=1, Hkv=1, d=8, page_size=4, seed=44)
    q_st, _ = _queries(case, 1, 45)
    good = oracle.paged_decode(q_st, case.k_cache, case.v_cache, case.block_table, lengths,
                               case.scale)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    rng = np.random.default_rng(46)
    kn = rng.standard_normal((1, 1, 8)).astype(np.float32)
    slot_of_pos5 = case.pages_of[0][1] * 4 + 1
    oracle.kv_cache_write(kn, kn, kc, vc, np.array([slot_of_pos5], np.int64))
    bad = oracle.paged_decode(q_st, kc, vc, case.block_table, lengths, case.scale)
    assert np.abs(bad - good).max() > 1e-6
    oracle.kv_cache_write(kn, kn, kc := case.k_cache.copy(), vc := case.v_cache.copy(),
                          np.array([-1], np.int64))
    same = oracle.paged_decode(q_st, kc, vc, case.block_table, lengths, case.scale)
    assert np.array_equal(same, good)


def test_oracle_is_deterministic_across_thread_counts():
    case = history_case([300, 77], Hq=4, Hkv=2, d=32, page_size=16, seed=47)
    q_st, _ = _queries(case, 2, 48)
    a = oracle.paged_decode(q_st, case.k_cache, case.v_cache, case.block_table, [300, 77],
                            case.scale, threads=1)
    b = oracle.paged_decode(q_st, case.k_cache, case.v_cache, case.block_table, [300, 77],
                            case.scale, threads=4)
    assert np.array_equal(a, b)


def test_out_of_range_page_is_refused():
    case = history_case([10], Hq=1, Hkv=1, d=8, page_size=4, seed=49)
    bt = case.block_table.copy()
    bt[0, 1] = 10_000
    q_st, _ = _queries(case, 1, 50)
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(q_st, case.k_cache, case.v_cache, bt, [10], case.scale)


# ------------------------------------------------------------------ sizing --

def _golden():
    with open(os.path.join(GOLDEN, "kv_sizing.json")) as f:
        return json.load(f)


def test_kv_bytes_per_token_matches_the_pages():
    g = _golden()
    for e in g["per_token"]:
        got = oracle.kv_bytes_per_token(e["layers"], e["h_kv"], e["d_head"], e["bytes"])
        assert got * e["positions"] == e["expected_bytes"], e["source"]
    for e in g["per_page"]:
        got = oracle.kv_bytes_per_token(e["layers"], e["h_kv"], e["d_head"], e["bytes"])
        assert got * e["page_size"] == e["expected_bytes"], e["source"]
    for e in g["full_history_per_sequence"]:
        got = oracle.kv_bytes_per_token(e["layers"], e["h_kv"], e["d_head"], e["bytes"])
        assert got * e["positions"] == e["expected_mib"] * 2 ** 20, e["source"]
    for e in g["gqa_ratio"]:
        mha = oracle.kv_bytes_per_token(32, e["h_q"], 128, 2)
        gqa = oracle.kv_bytes_per_token(32, e["h_kv"], 128, 2)
        assert mha // gqa == e["expected_ratio"] and mha % gqa == 0, e["source"]


# -------------------------------------------------------------------- ring --
# A sliding layer whose table is a ring reads only the ring ("How serving works
# in Tlaloc", section 2, the bullet on sliding layers; section 3, the windowed
# KV pool).  The ring layout below is built by the test from the contiguous
# histories (position j on ring page (j // ps) % R at offset j % ps, later
# positions overwriting earlier ones) and checked against dense attention
# over the histories: independent of the oracle's page arithmetic.

def _ring_layout(case, ring_pages, seed=0):
    """(k_ring, v_ring, ring_table) holding the last ring_pages * ps positions
    of every history, stored like the case's pool; the table is as wide as the
    full one (entry k holds the ring page of block k)."""
    rng = np.random.default_rng(seed)
    B, ps = len(case.lengths), case.page_size
    n_slots = ring_pages * ps
    perm = rng.permutation(B * ring_pages).reshape(B, ring_pages)
    width = max(case.block_table.shape[1], ring_pages)
    table = np.stack([perm[b][np.arange(width) % ring_pages] for b in range(B)]).astype(np.int32)
    kr = np.zeros((B * ring_pages, ps) + case.k_cache.shape[2:], dtype=case.k_cache.dtype)
    vr = np.zeros_like(kr)
    for b, L in enumerate(case.lengths):
        for j in range(max(0, L - n_slots), L):  # the positions still in the ring
            src_pg, dst_pg = case.pages_of[b][j // ps], perm[b][(j // ps) % ring_pages]
            kr[dst_pg, j % ps] = case.k_cache[src_pg, j % ps]
            vr[dst_pg, j % ps] = case.v_cache[src_pg, j % ps]
    return kr, vr, table


@pytest.mark.parametrize("window,ring_pages", [(20, 3), (20, 4), (32, 4), (7, 1), (40, 6)])
def test_ring_decode_equals_dense_over_the_window(window, ring_pages):
    lengths = [100, 37, 8, 1, 61]  # several wraps of the ring, and no wrap at all
    case = history_case(lengths, Hq=4, Hkv=2, d=16, page_size=8, seed=21)
    assert ring_pages * case.page_size >= window
    kr, vr, table = _ring_layout(case, ring_pages)
    q_st, q_vals = _queries(case, len(lengths), 22)
    out = oracle.paged_decode(q_st, kr, vr, table, lengths, case.scale, window=window,
                              ring_pages=ring_pages)
    for b, L in enumerate(lengths):
        ref = dense_reference(case, q_vals[b], b, L - 1, window)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_ring_one_page_short_changes_the_result():
    # negative control: a ring that cannot hold the window has overwritten
    # the window's oldest positions
    lengths = [100, 61, 12]
    window, ring_pages = 20, 2  # 16 slots < 20
    case = history_case(lengths, Hq=4, Hkv=2, d=16, page_size=8, seed=23)
    kr, vr, table = _ring_layout(case, ring_pages)
    q_st, q_vals = _queries(case, len(lengths), 24)
    out = oracle.paged_decode(q_st, kr, vr, table, lengths, case.scale, window=window,
                              ring_pages=ring_pages)
    for b, L in enumerate(lengths):
        ref = dense_reference(case, q_vals[b], b, L - 1, window)
        if L > ring_pages * case.page_size:
            assert np.abs(out[b] - ref).max() > 1e-3
        else:
            np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_ring_prefill_chunk_equals_dense_and_needs_its_pages():
    # a call of n tokens at p0 needs min(p0, W - 1) + n positions of ring
    window, n, ps = 24, 10, 8
    p0 = [50, 5]  # the second row has not filled a window yet
    lengths = [p + n for p in p0]
    case = history_case(lengths, Hq=2, Hkv=1, d=16, page_size=ps, seed=25)
    T = n
    positions = np.array([[p + t for t in range(T)] for p in p0], dtype=np.int32)
    rng = np.random.default_rng(26)
    q_st, q_vals = round_to(rng.standard_normal((len(p0), T, case.Hq, case.d)), case.dtype)
    need = oracle.ring_pages(window, n, ps)
    assert need == -(-(window - 1 + n) // ps)
    for ring_pages, ok in ((need, True), (need - 1, False)):
        kr, vr, table = _ring_layout(case, ring_pages)
        out = oracle.paged_prefill(q_st, kr, vr, table, positions, case.scale, window=window,
                                   ring_pages=ring_pages).reshape(len(p0), T, case.Hq, case.d)
        worst = 0.0
        for b in range(len(p0)):
            for t in range(T):
                ref = dense_reference(case, q_vals[b, t], b, int(positions[b, t]), window)
                worst = max(worst, float(np.abs(out[b, t] - ref).max()))
        if ok:
            assert worst <= 1e-12
        else:
            assert worst > 1e-3  # the first row's oldest window positions are gone


def test_ring_sizes_match_the_pages():
    with open(os.path.join(GOLDEN, "ring_sizing.json")) as f:
        g = json.load(f)
    for e in g["rings"]:
        got = oracle.ring_pages(e["window"], e["chunk"], e["page_size"])
        assert got == e["expected_pages"], e["source"]
        if "default_pages" in e:
            assert got + 1 == e["default_pages"], e["source"]


# --------------------------------------------------------------------- fp8 --
# The fp8 KV cache ("How serving works in Tlaloc", the FP8 KV cache paragraph
# of its quantisation section): e4m3fn codes with no scale, the write clamps
# to +-448 and rounds to nearest (ties to even); attention widens the codes.
# torch's float8_e4m3fn conversions are an independent implementation of the
# same format (they give NaN instead of clamping out-of-range values).

def _torch_codes(x):
    return torch.tensor(np.asarray(x, np.float64)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_values(codes):
    return torch.tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_fp8_code_values_match_torch_and_the_format():
    vals = np.array([oracle.fp8_value(c) for c in range(256)])
    ref = _torch_values(np.arange(256))
    assert np.all((vals == ref) | (np.isnan(vals) & np.isnan(ref)))
    # anchors of the format: smallest subnormal 2^-9, smallest normal 2^-6, 1, max 448, NaN
    assert oracle.fp8_value(0x01) == 2.0 ** -9 and oracle.fp8_value(0x08) == 2.0 ** -6
    assert oracle.fp8_value(0x38) == 1.0 and oracle.fp8_value(0x7E) == 448.0
    assert oracle.fp8_value(0xB8) == -1.0 and np.isnan(oracle.fp8_value(0x7F))


def test_fp8_rounding_is_nearest_with_ties_to_even():
    finite = [c for c in range(0x7F)]  # 0 .. 448, increasing
    v = _torch_values(finite)
    mids = (v[:-1] + v[1:]) / 2  # exact midpoints (ties)
    rng = np.random.default_rng(61)
    xs = np.concatenate([v, mids, -mids, rng.standard_normal(5000) * 10.0 ** rng.uniform(-4, 2.6, 5000)])
    xs = xs[np.abs(xs) < 448]
    mine = np.array([oracle.fp8_code(x) for x in xs])
    assert np.array_equal(mine, _torch_codes(xs))
    # a tie goes to the even mantissa: 1 + 1/16 lies between 1 (0x38) and 1.125 (0x39)
    assert oracle.fp8_code(1.0625) == 0x38 and oracle.fp8_code(1.1875) == 0x3A


def test_fp8_write_clamps_to_448_and_keeps_nan():
    for x, code in ((448.0, 0x7E), (460.0, 0x7E), (464.0, 0x7E), (1e9, 0x7E), (float("inf"), 0x7E),
                    (-1e9, 0xFE), (float("-inf"), 0xFE), (-448.0, 0xFE)):
        assert oracle.fp8_code(x) == code, x
    assert oracle.fp8_code(float("nan")) == 0x7F
    assert oracle.fp8_code(0.0) == 0x00 and oracle.fp8_code(-0.0) == 0x80


def test_fp8_cache_write_converts_and_skips_pads():
    rng = np.random.default_rng(62)
    P, ps, hkv, d = 5, 4, 2, 16
    kc = rng.integers(0, 256, (P, ps, hkv, d)).astype(np.uint8)
    vc = rng.integers(0, 256, (P, ps, hkv, d)).astype(np.uint8)
    before_k, before_v = kc.copy(), vc.copy()
    slots = np.array([3, -1, 17, 0, -1], dtype=np.int64)
    kn = (rng.standard_normal((5, hkv, d)) * 50).astype(np.float32)
    vn = (rng.standard_normal((5, hkv, d)) * 50).astype(np.float32)
    kn[0, 0, 0], vn[2, 1, 3] = 1000.0, -700.0  # past the range: clamped
    oracle.kv_cache_write_fp8(kn, vn, kc, vc, slots)
    exp_k, exp_v = before_k.copy(), before_v.copy()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        exp_k[s // ps, s % ps] = _torch_codes(np.clip(kn[t].astype(np.float64), -448, 448))
        exp_v[s // ps, s % ps] = _torch_codes(np.clip(vn[t].astype(np.float64), -448, 448))
    assert np.array_equal(kc, exp_k) and np.array_equal(vc, exp_v)


@pytest.mark.parametrize("window", [0, 9])
def test_fp8_decode_equals_dense_attention_over_the_codes_values(window):
    # fp8 pools (codes from torch), bf16 queries: the oracle against dense
    # attention over the codes' exact values, with library matrix products
    rng = np.random.default_rng(63)
    lengths, ps, hq, hkv, d = [30, 5, 64], 8, 4, 2, 16
    need = [(L + ps - 1) // ps for L in lengths]
    P = sum(need)
    perm = rng.permutation(P)
    bt = np.full((len(lengths), max(need)), -1, np.int32)
    kc = np.zeros((P, ps, hkv, d), np.uint8)
    vc = np.zeros_like(kc)
    hist = []
    off = 0
    for b, L in enumerate(lengths):
        pages = perm[off:off + need[b]]
        off += need[b]
        bt[b, :need[b]] = pages
        kcode = _torch_codes(rng.standard_normal((L, hkv, d)) * 3)
        vcode = _torch_codes(rng.standard_normal((L, hkv, d)) * 3)
        for j in range(L):
            kc[pages[j // ps], j % ps] = kcode[j]
            vc[pages[j // ps], j % ps] = vcode[j]
        hist.append((_torch_values(kcode), _torch_values(vcode)))
    q_st, q_vals = round_to(rng.standard_normal((len(lengths), hq, d)), torch.bfloat16)
    scale = 0.25
    out = oracle.paged_decode(q_st, kc, vc, bt, lengths, scale, window=window)
    import scipy.special
    for b, L in enumerate(lengths):
        lo = 0 if window <= 0 else max(0, L - window)
        kv, vv = hist[b]
        for h in range(hq):
            g = h // (hq // hkv)
            w = scipy.special.softmax(scale * (kv[lo:L, g] @ q_vals[b, h]))
            np.testing.assert_allclose(out[b, h], w @ vv[lo:L, g], rtol=1e-12, atol=1e-12)
