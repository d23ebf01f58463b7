"""Pins of the oracle's int8 KV pools against facts that do not depend on it.

Format (the pages name int8 KV pools without a format; it is read from the
"Int8 weights (opt-in)" paragraph of "How serving works in Tlaloc": one f32
scale per row, max |x| / 127, codes rounded half to even): each (token, KV
head) row of d values gets s = max |x| / 127 and the codes rint(x / s); a
value reads back as code x s.  Scales sit at [num_pages][H_kv][page_size].
"""
from __future__ import annotations

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from tests.dense_history import round_to


def _pools(P, ps, hkv, d, fill_code=7, fill_scale=-1.0):
    kc = np.full((P, ps, hkv, d), fill_code, np.int8)
    ks = np.full((P, hkv, ps), fill_scale, np.float32)
    return kc, kc.copy(), ks, ks.copy()


def test_int8_write_closed_forms():
    # one token, one head, d = 8; slot 0
    rows = {
        # max 127 -> scale 1: codes are the values rounded half to even
        "unit": ([127, -63.5, 2.5, 3.5, -0.5, 0.49, -127, 0], 1.0,
                 [127, -64, 2, 4, 0, 0, -127, 0]),
        # max 254 -> scale 2: 5 / 2 = 2.5 -> 2, 7 / 2 = 3.5 -> 4, 1 / 2 -> 0
        "two": ([254, 5, 7, -1, -254, 3, 0, 100], 2.0, [127, 2, 4, 0, -127, 2, 0, 50]),
        # max 12.7 -> scale ~0.1 (a binary32 quotient): values well clear of a
        # tie, -6.33 / 0.1 = -63.3 -> -63, 1.0 / 0.1 = 10
        "tenth": ([12.7, -6.33, 1.0, 0.0, 0.0, 0.0, 0.0, 0.0],
                  np.float32(12.7) / np.float32(127), [127, -63, 10, 0, 0, 0, 0, 0]),
    }
    for name, (vals, sc, codes) in rows.items():
        x = np.array(vals, np.float32).reshape(1, 1, 8)
        kc, vc, ks, vs = _pools(1, 1, 1, 8)
        assert oracle.kv_cache_write_int8(x, -x, kc, vc, ks, vs, np.array([0])) == 0
        assert ks[0, 0, 0] == np.float32(sc), name
        assert kc.ravel().tolist() == codes, (name, kc.ravel().tolist())
        assert vc.ravel().tolist() == [-c for c in codes], name
        assert vs[0, 0, 0] == np.float32(sc)


def test_int8_write_zero_row_non_finite_and_pads():
    P, ps, hkv, d = 3, 4, 2, 8
    kc, vc, ks, vs = _pools(P, ps, hkv, d)
    kn = np.zeros((3, hkv, d), np.float32)
    vn = np.zeros((3, hkv, d), np.float32)
    kn[0, 1] = [1, 2, 3, np.nan, np.inf, -np.inf, -4, 0.5]  # finite max 4
    vn[0, 0] = 0.0  # all zeros: scale 0, codes 0
    vn[0, 1] = 1e-45  # the smallest subnormal: 1e-45 / 127 underflows to 0
    kn[2] = 5.0
    slots = np.array([1 * ps + 3, -1, 2 * ps + 0], np.int64)  # page 1 offset 3; pad; page 2
    bad = oracle.kv_cache_write_int8(kn, vn, kc, vc, ks, vs, slots)
    assert bad == 3  # nan, +inf, -inf
    assert ks[1, 1, 3] == np.float32(4) / np.float32(127)
    assert kc[1, 3, 1].tolist() == [32, 64, 95, 0, 0, 0, -127, 16]
    assert vs[1, 0, 3] == 0 and np.all(vc[1, 3, 0] == 0)
    assert vs[1, 1, 3] == 0 and np.all(vc[1, 3, 1] == 0)
    # head-major scale layout: token (page 2, offset 0) heads 0 and 1
    assert ks[2, 0, 0] == np.float32(5) / np.float32(127) and ks[2, 1, 0] == ks[2, 0, 0]
    assert np.all(kc[2, 0] == 127)
    # everything else untouched (the pad wrote nothing)
    touched = np.zeros((P, ps), bool)
    touched[1, 3] = touched[2, 0] = True
    assert np.all(kc[~touched] == 7) and np.all(vc[~touched] == 7)
    st = np.zeros((P, hkv, ps), bool)
    st[1, :, 3] = st[2, :, 0] = True
    assert np.all(ks[~st] == -1) and np.all(vs[~st] == -1)


def test_int8_write_properties_on_random_rows():
    # every finite value reads back within half a step, the largest magnitude
    # of each row maps to +-127, and bf16 sources are widened exactly first
    rng = np.random.default_rng(71)
    P, ps, hkv, d = 6, 16, 4, 128
    n = 40
    for src in (torch.float32, torch.bfloat16):
        raw = rng.standard_normal((n, hkv, d)) * 10.0 ** rng.uniform(-3, 3, (n, hkv, 1))
        st, vals = round_to(raw, src)
        kc, vc, ks, vs = _pools(P, ps, hkv, d)
        slots = rng.permutation(P * ps)[:n].astype(np.int64)
        assert oracle.kv_cache_write_int8(st, st, kc, vc, ks, vs, slots) == 0
        for t, s in enumerate(slots):
            page, off = divmod(int(s), ps)
            for g in range(hkv):
                x = vals[t, g]
                sc = float(ks[page, g, off])
                code = kc[page, off, g].astype(np.float64)
                # half a step, plus the binary32 rounding of x / s (|x / s| <= 127)
                assert np.max(np.abs(code * sc - x)) <= sc * (0.5 + 127 * 2.0 ** -24)
                assert np.max(np.abs(kc[page, off, g].astype(np.int32))) == 127
                m = np.max(np.abs(x))
                assert abs(sc - m / 127) <= m / 127 * 2.0 ** -23


def _int8_case(lengths, ps, hkv, d, seed, unit_scales=False):
    rng = np.random.default_rng(seed)
    need = [(L + ps - 1) // ps for L in lengths]
    P = sum(need) + 2
    perm = rng.permutation(P)
    bt = np.full((len(lengths), max(need)), -1, np.int32)
    kc = rng.integers(-127, 128, (P, ps, hkv, d)).astype(np.int8)
    vc = rng.integers(-127, 128, (P, ps, hkv, d)).astype(np.int8)
    if unit_scales:
        ks = np.ones((P, hkv, ps), np.float32)
        vs = np.ones((P, hkv, ps), np.float32)
    else:
        ks = (rng.uniform(0.002, 0.05, (P, hkv, ps))).astype(np.float32)
        vs = (rng.uniform(0.002, 0.05, (P, hkv, ps))).astype(np.float32)
    hist = []
    off = 0
    for b, L in enumerate(lengths):
        pages = perm[off:off + need[b]]
        off += need[b]
        bt[b, :need[b]] = pages
        # the history of sequence b, by position, read with the head-major scales
        kh = np.stack([kc[pages[j // ps], j % ps].astype(np.float64) *
                       ks[pages[j // ps], :, j % ps][:, None].astype(np.float64) for j in range(L)])
        vh = np.stack([vc[pages[j // ps], j % ps].astype(np.float64) *
                       vs[pages[j // ps], :, j % ps][:, None].astype(np.float64) for j in range(L)])
        hist.append((kh, vh))
    return kc, vc, ks, vs, bt, hist


@pytest.mark.parametrize("window", [0, 7])
def test_int8_decode_equals_dense_attention_over_code_times_scale(window):
    lengths, ps, hq, hkv, d = [30, 5, 64, 1], 16, 4, 2, 16
    kc, vc, ks, vs, bt, hist = _int8_case(lengths, ps, hkv, d, 72)
    rng = np.random.default_rng(73)
    q_st, q_vals = round_to(rng.standard_normal((len(lengths), hq, d)), torch.bfloat16)
    scale = 0.25
    out = oracle.paged_decode_int8(q_st, kc, vc, ks, vs, bt, lengths, scale, window=window)
    for b, L in enumerate(lengths):
        lo = 0 if window <= 0 else max(0, L - window)
        kh, vh = hist[b]
        for h in range(hq):
            g = h // (hq // hkv)
            w = scipy.special.softmax(scale * (kh[lo:L, g] @ q_vals[b, h]))
            np.testing.assert_allclose(out[b, h], w @ vh[lo:L, g], rtol=1e-12, atol=1e-12)


def test_int8_decode_with_unit_scales_equals_the_f32_oracle():
    # scales of 1: the int8 pools hold the same numbers as f32 pools of the
    # codes' values, read by the separately pinned f32 path
    lengths, ps, hq, hkv, d = [17, 40, 3], 8, 6, 3, 32
    kc, vc, ks, vs, bt, _ = _int8_case(lengths, ps, hkv, d, 74, unit_scales=True)
    rng = np.random.default_rng(75)
    q_st, q_vals = round_to(rng.standard_normal((len(lengths), hq, d)), torch.bfloat16)
    out = oracle.paged_decode_int8(q_st, kc, vc, ks, vs, bt, lengths, 0.1)
    ref = oracle.paged_decode(q_vals.astype(np.float32), kc.astype(np.float32),
                              vc.astype(np.float32), bt, lengths, 0.1)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)


def test_int8_negative_control_token_major_scales_are_caught():
    # reading the scales as [num_pages][page_size][H_kv] instead gives another
    # result: the layout is pinned by the dense comparison above
    lengths, ps, hq, hkv, d = [24], 8, 2, 2, 16
    kc, vc, ks, vs, bt, hist = _int8_case(lengths, ps, hkv, d, 76)
    rng = np.random.default_rng(77)
    q_st, _ = round_to(rng.standard_normal((1, hq, d)), torch.bfloat16)
    good = oracle.paged_decode_int8(q_st, kc, vc, ks, vs, bt, lengths, 0.3)
    swapped = np.ascontiguousarray(ks.reshape(ks.shape[0], ps, hkv).transpose(0, 2, 1))
    bad = oracle.paged_decode_int8(q_st, kc, vc, swapped, vs, bt, lengths, 0.3)
    assert np.max(np.abs(good - bad)) > 1e-3


def _int8_prefill_inputs(lengths, n_live, pads, hq, d, seed):
    """Right-aligned prefill rows at the end of each history: row b holds
    pads[b] padding tokens (position -1) then the positions
    L_b - n_live[b] .. L_b - 1; queries bf16."""
    rng = np.random.default_rng(seed)
    B, T = len(lengths), max(n + p for n, p in zip(n_live, pads))
    pos = np.full((B, T), -1, np.int32)
    for b, (L, n) in enumerate(zip(lengths, n_live)):
        pos[b, T - n:] = np.arange(L - n, L)
    q_st, q_vals = round_to(rng.standard_normal((B, T, hq, d)), torch.bfloat16)
    return q_st, q_vals, pos


@pytest.mark.parametrize("window", [0, 9])
def test_int8_prefill_equals_dense_attention_over_code_times_scale(window):
    lengths, ps, hq, hkv, d = [30, 12, 64, 1], 8, 4, 2, 16
    kc, vc, ks, vs, bt, hist = _int8_case(lengths, ps, hkv, d, 81)
    q_st, q_vals, pos = _int8_prefill_inputs(lengths, [7, 12, 5, 1], [1, 0, 4, 6], hq, d, 82)
    scale = 0.3
    B, T = pos.shape
    out = oracle.paged_prefill_int8(q_st, kc, vc, ks, vs, bt, pos, scale, window=window)
    out = out.reshape(B, T, hq, d)
    for b in range(B):
        kh, vh = hist[b]
        for t in range(T):
            p = pos[b, t]
            if p < 0:
                assert np.all(out[b, t] == 0)
                continue
            lo = 0 if window <= 0 else max(0, p - window + 1)
            for h in range(hq):
                g = h // (hq // hkv)
                w = scipy.special.softmax(scale * (kh[lo:p + 1, g] @ q_vals[b, t, h]))
                np.testing.assert_allclose(out[b, t, h], w @ vh[lo:p + 1, g], rtol=1e-12,
                                           atol=1e-12)


def test_int8_prefill_with_unit_scales_equals_the_f32_oracle():
    lengths, ps, hq, hkv, d = [17, 40, 3], 8, 6, 3, 32
    kc, vc, ks, vs, bt, _ = _int8_case(lengths, ps, hkv, d, 83, unit_scales=True)
    q_st, q_vals, pos = _int8_prefill_inputs(lengths, [9, 40, 3], [2, 0, 5], hq, d, 84)
    out = oracle.paged_prefill_int8(q_st, kc, vc, ks, vs, bt, pos, 0.1)
    ref = oracle.paged_prefill(q_vals.astype(np.float32), kc.astype(np.float32),
                               vc.astype(np.float32), bt, pos, 0.1)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)


def test_int8_prefill_blockwise_equals_one_pass_and_batched_equals_solo():
    # key blocks of 8 keys: every row folds several blocks, some fully masked
    lengths, ps, hq, hkv, d = [45, 20, 33], 8, 4, 2, 16
    kc, vc, ks, vs, bt, _ = _int8_case(lengths, ps, hkv, d, 85)
    q_st, _, pos = _int8_prefill_inputs(lengths, [30, 20, 3], [0, 10, 27], hq, d, 86)
    blockwise = oracle.paged_prefill_int8(q_st, kc, vc, ks, vs, bt, pos, 0.25, key_block=8)
    one_pass = oracle.paged_prefill_int8(q_st, kc, vc, ks, vs, bt, pos, 0.25, blockwise=False)
    assert np.max(np.abs(blockwise - one_pass)) <= 1e-12
    B, T = pos.shape
    for b in range(B):
        solo = oracle.paged_prefill_int8(q_st[b:b + 1], kc, vc, ks, vs, bt[b:b + 1],
                                         pos[b:b + 1], 0.25, blockwise=False)
        assert np.array_equal(solo, one_pass.reshape(B, T, hq, d)[b].reshape(solo.shape))
