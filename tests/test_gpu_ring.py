"""Sliding-window attention over a ring (the windowed KV pool of "How serving
works in Tlaloc", sections 2-3) on the GPU, through the C ABI: a ring gives the
same bits as a full-history table, agrees with the oracle's ring form, and a
ring that cannot hold the call is refused (decode) or reported (prefill)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import workloads as wl
from tests.gpu_util import assert_decode_all, gpu_write, on_gpu
from tests.parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _ring_case(lengths, **kw):
    c = wl.ring_case(lengths, device=DEV, **kw)
    c.full_table, c.ring_table = c.full_table.to(DEV), c.ring_table.to(DEV)
    c.context_lens = c.context_lens.to(DEV)
    return c


def _write_new_tokens(c):
    """Clear each sequence's last position in both layouts and write it back
    through the cache write (the ring's slot follows the ring rule)."""
    hkv, d = c.Hkv, c.d
    for k, v, slots in ((c.full_k, c.full_v, c.full_slots), (c.ring_k, c.ring_v, c.ring_slots)):
        s = slots.to(DEV)
        live = s >= 0
        k.view(-1, hkv, d)[s[live]] = 0
        v.view(-1, hkv, d)[s[live]] = 0
        err = _err()
        tl.tl_kv_cache_write(c.k_new.contiguous(), c.v_new.contiguous(), k, v, s, error_word=err)
        assert int(err.item()) == 0


@pytest.mark.parametrize("dtype,hq,hkv,d,ps,window,ring", [
    (torch.bfloat16, 40, 8, 128, 16, 300, 20),
    (torch.bfloat16, 32, 8, 128, 16, 256, 16),
    (torch.bfloat16, 8, 2, 64, 8, 40, 6),
    (torch.float32, 4, 2, 64, 16, 50, 4),
])
def test_decode_ring_equals_full_history_bit_for_bit(dtype, hq, hkv, d, ps, window, ring):
    lengths = [1, 37, 300, 301, 1000, 2047, 5000]
    c = _ring_case(lengths, window=window, ring_pages=ring, Hq=hq, Hkv=hkv, d=d, page_size=ps,
                   dtype=dtype, seed=31)
    _write_new_tokens(c)
    e1, e2 = _err(), _err()
    full = tl.tl_paged_attn_decode(c.q, c.full_k, c.full_v, c.full_table, c.context_lens,
                                   c.scale, window=window, error_word=e1)
    ring_out = tl.tl_paged_attn_decode_ring(c.q, c.ring_k, c.ring_v, c.ring_table,
                                            c.context_lens, c.scale, window, ring, error_word=e2)
    torch.cuda.synchronize()
    assert int(e1.item()) == 0 and int(e2.item()) == 0
    assert torch.equal(full, ring_out)
    ref = oracle.paged_decode(c.q.cpu(), c.ring_k.cpu(), c.ring_v.cpu(), c.ring_table.cpu(),
                              c.context_lens.cpu(), c.scale, window=window, ring_pages=ring)
    assert_close(ring_out, ref, "ring decode vs oracle")


def test_decode_ring_that_cannot_hold_the_window_is_refused():
    c = _ring_case([100, 400], window=64, ring_pages=4, Hq=8, Hkv=2, d=128, page_size=16,
                   dtype=torch.bfloat16, seed=32)
    for window, ring in ((65, 4), (64, 0), (0, 4), (64, c.ring_table.shape[1] + 1)):
        with pytest.raises(tl.TLError) as e:
            tl.tl_paged_attn_decode_ring(c.q, c.ring_k, c.ring_v, c.ring_table, c.context_lens,
                                         c.scale, window, ring)
        assert e.value.status == tl.TL_ERR_INVALID_ARG


def _prefill_inputs(c, p0, n, pads, seed, outlier_p=0.0):
    B, T = len(p0), n + max(pads)
    positions = torch.full((B, T), -1, dtype=torch.int32)
    for b in range(B):
        positions[b, T - n:] = torch.arange(p0[b], p0[b] + n, dtype=torch.int32)
    g = torch.Generator(device=DEV).manual_seed(seed)
    q = torch.randn((B, T, c.Hq, c.d), generator=g, device=DEV)
    if outlier_p > 0:  # that share of the values x8, as in the sliding-window mix
        q = torch.where(torch.rand(q.shape, generator=g, device=DEV) < outlier_p, q * 8, q)
    return q.to(c.dtype), positions.to(DEV)


def test_prefill_chunk_through_a_ring_equals_full_history_bit_for_bit():
    # a call of n tokens at p0 needs min(p0, W - 1) + n positions of ring
    window, n, ps = 300, 200, 16
    p0 = [0, 50, 700, 3000]
    ring = oracle.ring_pages(window, n, ps)
    c = _ring_case([p + n for p in p0], window=window, ring_pages=ring, Hq=32, Hkv=8, d=128,
                   page_size=ps, dtype=torch.bfloat16, seed=33)
    q, positions = _prefill_inputs(c, p0, n, pads=[0, 7, 0, 3], seed=34)
    e1, e2 = _err(), _err()
    full = tl.tl_paged_attn_prefill(q, c.full_k, c.full_v, c.full_table, positions, c.scale,
                                    window=window, error_word=e1)
    ring_out = tl.tl_paged_attn_prefill_ring(q, c.ring_k, c.ring_v, c.ring_table, positions,
                                             c.scale, window, ring, error_word=e2)
    torch.cuda.synchronize()
    assert int(e1.item()) == 0 and int(e2.item()) == 0
    assert torch.equal(full, ring_out)
    T = positions.shape[1]
    rng = np.random.default_rng(35)
    for b in range(len(p0)):
        ts = sorted({0, T - 1, T - n} | set(rng.integers(0, T, 12).tolist()))
        ref = oracle.paged_prefill(q[b:b + 1].cpu(), c.ring_k.cpu(), c.ring_v.cpu(),
                                   c.ring_table[b:b + 1].cpu(), positions[b:b + 1].cpu(),
                                   c.scale, window=window, ring_pages=ring,
                                   tokens=np.asarray(ts, np.int64))
        assert_close(ring_out[b, ts], ref, f"ring prefill row {b}")


def test_prefill_ring_with_outliers_every_token():
    """A sliding layer's prefill chunk (window 4,096) through rings, on the
    sliding-window mix's value distribution (1% of Q, K and V values x8):
    every token against the oracle's ring form."""
    window, n, ps = 4096, 512, 16
    p0 = [0, 3000, 9000, 20000]
    ring = oracle.ring_pages(window, n, ps)
    c = _ring_case([p + n for p in p0], window=window, ring_pages=ring, Hq=40, Hkv=8, d=128,
                   page_size=ps, dtype=torch.bfloat16, seed=38, outlier_p=0.01)
    q, positions = _prefill_inputs(c, p0, n, pads=[0, 5, 0, 9], seed=39, outlier_p=0.01)
    err = _err()
    out = tl.tl_paged_attn_prefill_ring(q, c.ring_k, c.ring_v, c.ring_table, positions, c.scale,
                                        window, ring, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.paged_prefill(q.cpu(), c.ring_k.cpu(), c.ring_v.cpu(), c.ring_table.cpu(),
                               positions.cpu(), c.scale, window=window, ring_pages=ring)
    assert_close(out.reshape(ref.shape), ref, "ring prefill with outliers")


def test_prefill_ring_one_page_short_is_reported():
    window, n, ps = 300, 200, 16
    p0 = [3000]  # the call spans W - 1 + n = 499 positions > (32 - 1) * 16
    ring = oracle.ring_pages(window, n, ps) - 1
    c = _ring_case([p + n for p in p0], window=window, ring_pages=ring, Hq=32, Hkv=8, d=128,
                   page_size=ps, dtype=torch.bfloat16, seed=36)
    q, positions = _prefill_inputs(c, p0, n, pads=[0], seed=37)
    err = _err()
    tl.tl_paged_attn_prefill_ring(q, c.ring_k, c.ring_v, c.ring_table, positions, c.scale,
                                  window, ring, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & tl.TL_DEVERR_CONTEXT_RANGE


def test_full_size_sliding_layer_over_rings_every_sequence():
    """The sliding layer of the mix (B=128, window 4,096) over rings of 257
    pages, the step's new rows written first: every sequence against the
    oracle's ring form (the oracle writes the rows into its own copies of
    the rings as they were before the step)."""
    case = wl.swa_ring_decode(seed=0, device=DEV)
    ring = case.extra["ring_pages"]
    g = on_gpu(case)
    k0, v0 = g.k_cache.clone(), g.v_cache.clone()
    gpu_write(g)
    err = _err()
    out = tl.tl_paged_attn_decode_ring(g.q, g.k_cache, g.v_cache, g.block_table, g.context_lens,
                                       g.scale, g.window, ring, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_decode_all(out, g.q, k0, v0, g.block_table, g.context_lens, g.scale,
                      window=g.window, ring_pages=ring,
                      new_rows=(g.k_new, g.v_new, g.slot_mapping), what="sliding layer over rings")


def _int8_layouts(c):
    """Int8 pools of both layouts of a ring case: every slot's row quantised by
    the oracle's int8 write (zero rows get scale 0 and codes 0), so a ring's
    slots hold the same codes and scales as the full history's."""
    out = []
    for k, v in ((c.full_k, c.full_v), (c.ring_k, c.ring_v)):
        P, ps, hkv, d = k.shape
        kc = torch.zeros((P, ps, hkv, d), dtype=torch.int8)
        vc = torch.zeros_like(kc)
        ks = torch.zeros((P, hkv, ps), dtype=torch.float32)
        vs = torch.zeros_like(ks)
        slots = torch.arange(P * ps, dtype=torch.int64)
        oracle.kv_cache_write_int8(k.cpu().view(-1, hkv, d), v.cpu().view(-1, hkv, d), kc, vc, ks,
                                   vs, slots)
        out.append([t.to(DEV) for t in (kc, vc, ks, vs)])
    return out


@pytest.mark.parametrize("hq,hkv,window,ring", [(40, 8, 300, 20), (32, 8, 256, 16),
                                                (16, 4, 100, 8), (64, 8, 4096, 257)])
def test_decode_ring_int8_equals_full_history_bit_for_bit(hq, hkv, window, ring):
    lengths = [1, 37, 300, 301, 1000, 2047, 5000]
    c = _ring_case(lengths, window=window, ring_pages=ring, Hq=hq, Hkv=hkv, d=128, page_size=16,
                   dtype=torch.bfloat16, seed=41)
    full, rg = _int8_layouts(c)
    e1, e2 = _err(), _err()
    full_out = tl.tl_paged_attn_decode_int8(c.q, *full, c.full_table, c.context_lens, c.scale,
                                            window=window, error_word=e1)
    ring_out = tl.tl_paged_attn_decode_ring_int8(c.q, *rg, c.ring_table, c.context_lens, c.scale,
                                                 window, ring, error_word=e2)
    torch.cuda.synchronize()
    assert int(e1.item()) == 0 and int(e2.item()) == 0
    assert torch.equal(full_out, ring_out)
    ref = oracle.paged_decode_int8(c.q.cpu(), *(t.cpu() for t in rg), c.ring_table.cpu(),
                                   c.context_lens.cpu(), c.scale, window=window, ring_pages=ring)
    assert_close(ring_out, ref, "int8 ring decode vs oracle")


def test_decode_ring_int8_that_cannot_hold_the_window_is_refused():
    c = _ring_case([100, 400], window=64, ring_pages=4, Hq=8, Hkv=2, d=128, page_size=16,
                   dtype=torch.bfloat16, seed=42)
    _, rg = _int8_layouts(c)
    for window, ring in ((65, 4), (64, 0), (0, 4)):
        with pytest.raises(tl.TLError) as e:
            tl.tl_paged_attn_decode_ring_int8(c.q, *rg, c.ring_table, c.context_lens, c.scale,
                                              window, ring)
        assert e.value.status == tl.TL_ERR_INVALID_ARG


@pytest.mark.parametrize("outlier_p", [0.0, 0.01])
def test_prefill_ring_int8_equals_full_history_bit_for_bit(outlier_p):
    """A chunk through rings of int8 pools: the same bits as the full history
    (values of N(0,1) scale: every V tile copied scaled; with 1% of the
    values x8: flagged tiles keep their codes), and every token against the
    oracle's ring form."""
    window, n, ps = 300, 200, 16
    p0 = [0, 50, 700, 3000]
    ring = oracle.ring_pages(window, n, ps)
    c = _ring_case([p + n for p in p0], window=window, ring_pages=ring, Hq=32, Hkv=8, d=128,
                   page_size=ps, dtype=torch.bfloat16, seed=43, outlier_p=outlier_p)
    q, positions = _prefill_inputs(c, p0, n, pads=[0, 7, 0, 3], seed=44, outlier_p=outlier_p)
    full, rg = _int8_layouts(c)
    e1, e2 = _err(), _err()
    full_out = tl.tl_paged_attn_prefill_int8(q, *full, c.full_table, positions, c.scale,
                                             window=window, error_word=e1)
    ring_out = tl.tl_paged_attn_prefill_ring_int8(q, *rg, c.ring_table, positions, c.scale,
                                                  window, ring, error_word=e2)
    torch.cuda.synchronize()
    assert int(e1.item()) == 0 and int(e2.item()) == 0
    assert torch.equal(full_out, ring_out)
    ref = oracle.paged_prefill_int8(q.cpu(), *(t.cpu() for t in rg), c.ring_table.cpu(),
                                    positions.cpu(), c.scale, window=window, ring_pages=ring)
    assert_close(ring_out.reshape(ref.shape), ref, f"int8 ring prefill outliers {outlier_p}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float8_e4m3fn])
def test_fused_write_and_ring_decode_equal_the_two_calls(dtype):
    """tl_paged_attn_decode_write_ring: the step's rows written at their ring
    slots and the ring decode in one call give the pools and the outputs of
    the cache write followed by tl_paged_attn_decode_ring, bit for bit."""
    window, ring = 300, 20
    c = _ring_case([1, 37, 300, 301, 1000, 2047, 5000], window=window, ring_pages=ring, Hq=40,
                   Hkv=8, d=128, page_size=16, dtype=torch.bfloat16, seed=45)
    hkv, d = c.Hkv, c.d
    s = c.ring_slots.to(DEV)
    kn, vn = c.k_new.contiguous(), c.v_new.contiguous()
    pools = []
    for _ in range(2):
        k, v = c.ring_k.clone(), c.ring_v.clone()
        live = s >= 0
        k.view(-1, hkv, d)[s[live]] = 0
        v.view(-1, hkv, d)[s[live]] = 0
        if dtype == torch.float8_e4m3fn:
            k, v = k.float().to(dtype), v.float().to(dtype)
        pools.append((k, v))
    e1, e2 = _err(), _err()
    (k1, v1), (k2, v2) = pools
    fused = tl.tl_paged_attn_decode_write_ring(c.q, kn, vn, s, k1, v1, c.ring_table,
                                               c.context_lens, c.scale, window, ring,
                                               error_word=e1)
    if dtype == torch.float8_e4m3fn:
        tl.tl_kv_cache_write_fp8(kn, vn, k2, v2, s, error_word=e2)
    else:
        tl.tl_kv_cache_write(kn, vn, k2, v2, s, error_word=e2)
    two = tl.tl_paged_attn_decode_ring(c.q, k2, v2, c.ring_table, c.context_lens, c.scale, window,
                                       ring, error_word=e2)
    torch.cuda.synchronize()
    assert int(e1.item()) == 0 and int(e2.item()) == 0
    assert torch.equal(k1.view(torch.uint8), k2.view(torch.uint8))
    assert torch.equal(v1.view(torch.uint8), v2.view(torch.uint8))
    assert torch.equal(fused, two)
    for window, ring in ((301, 18), (0, ring)):  # too short a ring; no window
        with pytest.raises(tl.TLError) as e:
            tl.tl_paged_attn_decode_write_ring(c.q, kn, vn, s, k1, v1, c.ring_table,
                                               c.context_lens, c.scale, window, ring)
        assert e.value.status == tl.TL_ERR_INVALID_ARG
