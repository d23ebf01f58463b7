"""int8 KV pools on the GPU against the oracle.  "How serving works in
Tlaloc" names int8 KV pools as a next step without a format; the format is
read from its "Int8 weights (opt-in)" paragraph: one f32 scale per (token, KV
head) row, max |x| / 127, codes x / scale rounded half to even.  The write is
compared bit for bit (codes and scale bits); decode within the attention
tolerance, the pools coming from the seeded generator on the host."""
import pytest
import torch

import oracle
import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import workloads as wl
from tests.gpu_util import assert_decode_all, sample_rows
from tests.parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("src", [torch.float32, torch.bfloat16])
def test_int8_write_matches_the_oracle_bit_for_bit(src):
    g = torch.Generator().manual_seed(91)
    P, ps, hkv, d, n = 40, 16, 8, 128, 300
    mag = torch.exp(torch.randn((n, hkv, 1), generator=g) * 2)
    kn = (torch.randn((n, hkv, d), generator=g) * mag).to(src)
    vn = torch.randn((n, hkv, d), generator=g).to(src)
    kn[5, 3, 7] = float("nan")
    vn[9, 0, 0] = float("inf")
    vn[11, 2] = 0.0  # a zero row: scale 0, codes 0
    slots = torch.randperm(P * ps, generator=g)[:n].to(torch.int64)
    slots[::17] = -1  # pads
    slots[3] = P * ps + 2  # out of range: reported, not written
    kc = torch.full((P, ps, hkv, d), 0x55, dtype=torch.int8)
    ks = torch.full((P, hkv, ps), 12345.0, dtype=torch.float32)
    vc, vs = kc.clone(), ks.clone()
    dev = [t.to(DEV) for t in (kc, vc, ks, vs)]
    err = _err()
    tl.tl_kv_cache_write_int8(kn.to(DEV), vn.to(DEV), *dev, slots.to(DEV), error_word=err)
    torch.cuda.synchronize()
    ok = slots.clone()
    ok[3] = -1  # the oracle refuses an out-of-range slot; the kernel skips it
    n_bad = oracle.kv_cache_write_int8(kn, vn, kc, vc, ks, vs, ok)
    assert n_bad > 0
    e = int(err.item())
    assert e & tl.TL_DEVERR_SLOT_RANGE and e & tl.TL_DEVERR_VALUE_RANGE
    assert torch.equal(dev[0].cpu(), kc) and torch.equal(dev[1].cpu(), vc)
    assert torch.equal(dev[2].cpu().view(torch.int32), ks.view(torch.int32))
    assert torch.equal(dev[3].cpu().view(torch.int32), vs.view(torch.int32))


def _sub_pool(case, pools, rows):
    """Host copies of the pages the rows use, tables renumbered to the copy."""
    ps = case.page_size
    lens = case.context_lens.tolist()
    pages, tables = [], []
    for b in rows:
        n = (max(lens[b], 0) + ps - 1) // ps
        ids = case.block_table[b, :n].tolist()
        tables.append(list(range(len(pages), len(pages) + n)))
        pages += ids
    idx = torch.tensor(pages or [0], dtype=torch.long)
    sub = [t.index_select(0, idx) for t in pools]
    bt = torch.full((len(rows), max(1, max(len(t) for t in tables))), -1, dtype=torch.int32)
    for i, t in enumerate(tables):
        if t:
            bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    return sub, bt


def _check(case, pools, window, rows=None, what=""):
    kc, vc, ks, vs = (t.to(DEV) for t in pools)
    err = _err()
    out = tl.tl_paged_attn_decode_int8(case.q.to(DEV), kc, vc, ks, vs,
                                       case.block_table.to(DEV), case.context_lens.to(DEV),
                                       case.scale, window=window, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, int(err.item())
    out = out.cpu()
    if rows is None:
        ref = oracle.paged_decode_int8(case.q, *pools, case.block_table, case.context_lens,
                                       case.scale, window=window)
        assert_close(out, ref, what)
    else:
        sub, bt = _sub_pool(case, pools, rows)
        ref = oracle.paged_decode_int8(case.q[rows], *sub, bt, case.context_lens[rows],
                                       case.scale, window=window)
        assert_close(out[rows], ref, what)
    return out


@pytest.mark.parametrize("window", [0, 37])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (32, 8), (32, 2), (40, 8), (64, 8), (8, 8)])
# groups 4, 4, 16, 5, 8 and 1
def test_int8_decode_matches_the_oracle(hq, hkv, window):
    case = wl.decode_case([0, 1, 15, 16, 17, 33, 300, 1000], Hq=hq, Hkv=hkv, d=128, seed=92,
                          window=window)
    _check(case, wl.int8_pools(case, 93), window, what=f"int8 {hq}/{hkv} w{window}")


@pytest.mark.parametrize("ps", [32, 64])
def test_int8_decode_page_sizes(ps):
    case = wl.decode_case([3, 64, 65, 500, 2049], Hq=16, Hkv=4, d=128, page_size=ps, seed=94)
    _check(case, wl.int8_pools(case, 95), 0, what=f"int8 page {ps}")


def test_int8_decode_ignores_the_garbage_of_unread_slots():
    # slots no position maps to hold code -128 and NaN scales; keys past a
    # sequence's end share a chunk (and a scale copy) with its live keys
    case = wl.decode_case([1, 17, 31, 100, 257], Hq=8, Hkv=2, d=128, seed=96, extra_pages=3)
    out = _check(case, wl.int8_pools(case, 97, nan_unused=True), 0, what="int8 nan unused")
    assert torch.isfinite(out).all()


def test_int8_decode_llama8b_shape_every_sequence():
    case = wl.llama8b_decode(seed=5, device=DEV)
    pools = [t.to(DEV) for t in wl.int8_pools(case, 98)]
    err = _err()
    out = tl.tl_paged_attn_decode_int8(case.q, *pools, case.block_table.to(DEV),
                                       case.context_lens.to(DEV), case.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_decode_all(out, case.q, pools[0], pools[1], case.block_table, case.context_lens,
                      case.scale, k_scales=pools[2], v_scales=pools[3], what="int8 llama8b B=64")


@pytest.mark.parametrize("shape", ["many_short", "one_long"])
def test_int8_piece_plan_extremes(shape):
    """The piece plan's extremes over int8 pools: 2,048 short sequences (with
    empty and one-key ones) and one of 131,072 keys; every sequence."""
    g = torch.Generator().manual_seed(95)
    if shape == "many_short":
        lens = torch.randint(1, 400, (2046,), generator=g).tolist() + [0, 1]
    else:
        lens = [131072]
    case = wl.decode_case(lens, Hq=32, Hkv=8, d=128, seed=96)
    pools = [t.to(DEV) for t in wl.int8_pools(case, 97)]
    err = _err()
    out = tl.tl_paged_attn_decode_int8(case.q.to(DEV), *pools, case.block_table.to(DEV),
                                       case.context_lens.to(DEV), case.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isfinite(out).all()
    assert_decode_all(out, case.q, pools[0], pools[1], case.block_table, case.context_lens,
                      case.scale, k_scales=pools[2], v_scales=pools[3], chunk=256,
                      what=f"int8 piece plan {shape}")


def test_int8_decode_reports_a_query_beyond_fp16():
    case = wl.decode_case([40, 70], Hq=8, Hkv=2, d=128, seed=99)
    pools = [t.to(DEV) for t in wl.int8_pools(case, 100)]
    q = case.q.clone()
    q[1, 3, 5] = 1e6
    err = _err()
    tl.tl_paged_attn_decode_int8(q.to(DEV), *pools, case.block_table.to(DEV),
                                 case.context_lens.to(DEV), case.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & tl.TL_DEVERR_VALUE_RANGE


@pytest.mark.parametrize("src", [torch.bfloat16, torch.float32])
def test_int8_fused_write_equals_the_two_calls(src):
    # tl_paged_attn_decode_write_int8 == tl_kv_cache_write_int8, then
    # tl_paged_attn_decode_int8: output, pools and error bits, bit for bit
    case = wl.decode_case([5, 17, 100, 1000, 2049], Hq=16, Hkv=4, d=128, seed=101, n_pad=3)
    pools = wl.int8_pools(case, 102)
    slots = case.slot_mapping.clone()
    live = (slots >= 0).nonzero().flatten()
    slots[live[0]] = case.num_pages * case.page_size + 9  # reported, not written
    kn, vn = case.k_new.to(src).to(DEV), case.v_new.to(src).to(DEV)
    args = (case.block_table.to(DEV), case.context_lens.to(DEV), case.scale)
    res = []
    for fused in (False, True):
        kc, vc, ks, vs = (t.to(DEV) for t in pools)
        err = _err()
        if fused:
            out = tl.tl_paged_attn_decode_write_int8(case.q.to(DEV), kn, vn, slots.to(DEV), kc,
                                                     vc, ks, vs, *args, error_word=err)
        else:
            tl.tl_kv_cache_write_int8(kn, vn, kc, vc, ks, vs, slots.to(DEV), error_word=err)
            out = tl.tl_paged_attn_decode_int8(case.q.to(DEV), kc, vc, ks, vs, *args,
                                               error_word=err)
        torch.cuda.synchronize()
        res.append((out.cpu(), kc.cpu(), vc.cpu(), ks.cpu(), vs.cpu(), int(err.item())))
    (o1, *p1, e1), (o2, *p2, e2) = res
    assert e1 == e2 and e1 & tl.TL_DEVERR_SLOT_RANGE
    assert all(torch.equal(a.view(torch.uint8), b.view(torch.uint8)) for a, b in zip(p1, p2))
    assert torch.equal(o1, o2)
    # and against the oracle: its write on the host pools, then its decode
    kc, vc, ks, vs = (t.clone() for t in pools)
    ok = slots.clone()
    ok[live[0]] = -1
    oracle.kv_cache_write_int8(case.k_new.to(src), case.v_new.to(src), kc, vc, ks, vs, ok)
    assert torch.equal(p2[0], kc) and torch.equal(p2[2].view(torch.int32), ks.view(torch.int32))
    ref = oracle.paged_decode_int8(case.q, kc, vc, ks, vs, case.block_table, case.context_lens,
                                   case.scale)
    assert_close(o2, ref, f"fused int8 from {src}")


# ----------------------------------------------------------------- prefill --

def _prefill_int8(case, pools, window=0, error_word=None):
    kc, vc, ks, vs = (t.to(DEV) for t in pools)
    err = _err() if error_word is None else error_word
    out = tl.tl_paged_attn_prefill_int8(case.q.to(DEV), kc, vc, ks, vs, case.block_table.to(DEV),
                                        case.positions.to(DEV), case.scale, window=window,
                                        error_word=err)
    torch.cuda.synchronize()
    if error_word is None:
        assert int(err.item()) == 0, int(err.item())
    return out


def _oracle_prefill_int8(case, pools, window=0, rows=None):
    rows = range(case.B) if rows is None else rows
    outs = []
    for b in rows:
        outs.append(oracle.paged_prefill_int8(case.q[b:b + 1], *pools, case.block_table[b:b + 1],
                                              case.positions[b:b + 1], case.scale,
                                              window=window))
    return outs


def test_int8_prefill_full_batch_every_token():
    """The B=8 x 2,048 batch (pads 0-1,500, prior context 0-6,144, H_q=32,
    H_kv=8) over seeded int8 pools: every token of every row."""
    case = wl.batched_prefill(seed=0)
    pools = wl.int8_pools(case, 110)
    out = _prefill_int8(case, pools).cpu()
    for b, ref in enumerate(_oracle_prefill_int8(case, pools)):
        assert_close(out[b], ref, f"int8 prefill row {b}")
    assert torch.all(out[0, :case.pads[0]] == 0)


@pytest.mark.parametrize("window", [0, 100, 2049])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (32, 8), (16, 1)])
def test_int8_prefill_windows_and_groups(hq, hkv, window):
    T = 300
    case = wl.prefill_case([0, 17, T - 1, T], [2000, 0, 4000, 10], T=T, Hq=hq, Hkv=hkv, d=128,
                           seed=111, window=window)
    pools = wl.int8_pools(case, 112, nan_unused=True)  # unread slots: code -128, scale NaN
    out = _prefill_int8(case, pools, window).cpu()
    for b, ref in enumerate(_oracle_prefill_int8(case, pools, window)):
        assert_close(out[b], ref, f"int8 prefill {hq}/{hkv} w{window} row {b}")
    assert torch.all(out[3] == 0)  # the row with no live token


def test_int8_prefill_with_values_above_8_takes_the_split_path():
    """Scales up to 0.1 make |code x scale| reach 12.7: those rows take P as
    two fp16 parts; a row whose values stay below 8 does not (same bar)."""
    case = wl.prefill_case([0, 40], [1500, 3000], T=512, Hq=32, Hkv=8, d=128, seed=113)
    pools = list(wl.int8_pools(case, 114, scale_range=(0.02, 0.1)))
    out = _prefill_int8(case, pools).cpu()
    for b, ref in enumerate(_oracle_prefill_int8(case, pools)):
        assert_close(out[b], ref, f"int8 prefill split row {b}")


def test_int8_prefill_small_values_take_the_scaled_copy():
    """The B=8 x 2,048 batch over int8 pools whose values stay small (scales
    0.004-0.012, |v| <= 1.5, an RMS near 0.5): no tile is flagged, every V
    tile is copied as fp16(code x scale) and P goes into P.V as one fp16
    value, as for 16-bit pools; every token against the oracle."""
    case = wl.batched_prefill(seed=3)
    pools = wl.int8_pools(case, 117, scale_range=(0.004, 0.012))
    out = _prefill_int8(case, pools).cpu()
    for b, ref in enumerate(_oracle_prefill_int8(case, pools)):
        assert_close(out[b], ref, f"int8 prefill small values row {b}")


@pytest.mark.parametrize("window", [0, 700])
def test_int8_prefill_mixed_tiles(window):
    """Small values with 0.2% of the scales x40 (|v| up to ~19): the tiles
    holding one are flagged and keep their codes, the others are copied
    scaled; flagged rows take P as two fp16 parts over both kinds of tile."""
    case = wl.prefill_case([0, 40, 300], [1500, 3000, 200], T=1024, Hq=32, Hkv=8, d=128,
                           seed=118, window=window)
    pools = wl.int8_pools(case, 119, scale_range=(0.004, 0.012), boost_p=0.002, boost=40.0)
    out = _prefill_int8(case, pools, window).cpu()
    for b, ref in enumerate(_oracle_prefill_int8(case, pools, window)):
        assert_close(out[b], ref, f"int8 prefill mixed tiles w{window} row {b}")


def test_int8_prefill_batched_equals_solo_bit_for_bit():
    case = wl.prefill_case([100, 0, 700], [3000, 0, 5000], T=1024, Hq=16, Hkv=4, d=128, seed=115)
    pools = wl.int8_pools(case, 116)
    both = _prefill_int8(case, pools)
    g = [t.to(DEV) for t in pools]
    for b in range(case.B):
        solo = tl.tl_paged_attn_prefill_int8(case.q[b:b + 1].to(DEV), *g,
                                             case.block_table[b:b + 1].to(DEV),
                                             case.positions[b:b + 1].to(DEV), case.scale)
        torch.cuda.synchronize()
        assert torch.equal(solo[0], both[b]), f"row {b}"


@pytest.mark.parametrize("q_len,hq,hkv", [(4, 32, 8), (2, 32, 8), (3, 16, 8), (2, 8, 8)])
def test_int8_multi_token_decode(q_len, hq, hkv):
    """q_len tokens at the end of each sequence over int8 pools (16, 8, 6 and
    2 rows per KV head: both row layouts), every token against the oracle."""
    lengths = wl.llama8b_lengths(seed=11, B=10)
    p0 = [L - q_len for L in lengths]
    case = wl.prefill_case([0] * len(lengths), p0, T=q_len, Hq=hq, Hkv=hkv, d=128, seed=120)
    pools = [t.clone() for t in wl.int8_pools(case, 121)]
    oracle.kv_cache_write_int8(case.k_new, case.v_new, *pools, case.slot_mapping)
    err = _err()
    out = tl.tl_paged_attn_decode_multi_int8(case.q.to(DEV), *(t.to(DEV) for t in pools),
                                             case.block_table.to(DEV),
                                             torch.tensor(lengths, dtype=torch.int32, device=DEV),
                                             case.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.paged_prefill_int8(case.q, *pools, case.block_table, case.positions, case.scale)
    assert_close(out.cpu().reshape(ref.shape), ref, f"int8 multi-token q_len={q_len} hq={hq}")
