"""The decode call that writes its own new rows (tl_paged_attn_decode_write):
its result, the pools afterwards and its error bits equal those of the
separate write (tl_kv_cache_write, or tl_kv_cache_write_fp8 for e4m3 pools)
followed by tl_paged_attn_decode on the same inputs, bit for bit ("How
serving works in Tlaloc", section 1: each step writes its tokens' K/V, then
attends); and it matches the oracle."""
import pytest
import torch

import oracle
import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import workloads as wl
from tests.gpu_util import assert_decode_all, on_gpu
from tests.parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _both(g, k_cache, v_cache, k_new, v_new, slots, window=0):
    """(output, pools, error word) of the separate calls and of the fused call,
    each on its own copy of the pools."""
    res = []
    for fused in (False, True):
        kc, vc = k_cache.clone(), v_cache.clone()
        err = _err()
        if fused:
            out = tl.tl_paged_attn_decode_write(g.q, k_new, v_new, slots, kc, vc, g.block_table,
                                                g.context_lens, g.scale, window=window,
                                                error_word=err)
        else:
            if kc.dtype == torch.float8_e4m3fn:
                tl.tl_kv_cache_write_fp8(k_new, v_new, kc, vc, slots, error_word=err)
            else:
                tl.tl_kv_cache_write(k_new, v_new, kc, vc, slots, error_word=err)
            out = tl.tl_paged_attn_decode(g.q, kc, vc, g.block_table, g.context_lens, g.scale,
                                          window=window, error_word=err)
        torch.cuda.synchronize()
        res.append((out, kc, vc, int(err.item())))
    return res


def _same(res):
    (o1, k1, v1, e1), (o2, k2, v2, e2) = res
    assert e1 == e2
    assert torch.equal(k1.view(torch.uint8), k2.view(torch.uint8))
    assert torch.equal(v1.view(torch.uint8), v2.view(torch.uint8))
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("maker", [lambda: wl.llama8b_decode(seed=3),
                                   lambda: wl.tiny_decode(seed=0),
                                   lambda: wl.decode_case([0, 1, 16, 17, 300], Hq=8, Hkv=2,
                                                          d=128, seed=81, n_pad=3)])
def test_fused_equals_write_then_decode(maker):
    case = maker()
    g = on_gpu(case)
    res = _both(g, g.k_cache, g.v_cache, g.k_new, g.v_new, g.slot_mapping, g.window)
    _same(res)
    assert res[1][3] == 0


def test_fused_matches_the_oracle():
    case = wl.decode_case([5, 100, 1000, 2049], Hq=16, Hkv=4, d=128, seed=82, n_pad=2)
    g = on_gpu(case)
    (_, _, _, _), (out, kc, vc, e) = _both(g, g.k_cache, g.v_cache, g.k_new, g.v_new,
                                          g.slot_mapping)
    assert e == 0
    kr, vr = case.k_cache.clone(), case.v_cache.clone()
    oracle.kv_cache_write(case.k_new, case.v_new, kr, vr, case.slot_mapping)
    assert torch.equal(kc.cpu().view(torch.int16), kr.view(torch.int16))
    ref = oracle.paged_decode(case.q, kr, vr, case.block_table, case.context_lens, case.scale)
    assert_close(out, ref, "fused write + decode")


@pytest.mark.parametrize("src", [torch.bfloat16, torch.float32])
def test_fused_over_e4m3_pools(src):
    case = wl.llama8b_decode(seed=4, B=16)
    g = on_gpu(case)
    k8 = g.k_cache.float().to(torch.float8_e4m3fn)
    v8 = g.v_cache.float().to(torch.float8_e4m3fn)
    res = _both(g, k8, v8, g.k_new.to(src), g.v_new.to(src), g.slot_mapping)
    _same(res)
    # every sequence: the oracle converts the same new rows into its own
    # copies of the pools as they were before the call, then attends
    assert_decode_all(res[1][0], g.q, k8, v8, g.block_table, g.context_lens, g.scale,
                      new_rows=(g.k_new.to(src), g.v_new.to(src), g.slot_mapping),
                      what=f"fused e4m3 from {src}")


def test_fused_reports_a_bad_slot_and_skips_pads():
    case = wl.decode_case([40, 70], Hq=8, Hkv=2, d=128, seed=83, n_pad=2)
    g = on_gpu(case)
    slots = g.slot_mapping.clone()
    live = (slots >= 0).nonzero().flatten()
    slots[live[0]] = g.k_cache.shape[0] * g.k_cache.shape[1] + 5  # past the pools
    res = _both(g, g.k_cache, g.v_cache, g.k_new, g.v_new, slots)
    _same(res)
    assert res[1][3] & tl.TL_DEVERR_SLOT_RANGE
    # pads and the bad row wrote nothing: only the other live rows differ from before
    kc = res[1][1]
    changed = (kc != g.k_cache).flatten(2).any(-1).flatten().nonzero().flatten().tolist()
    assert sorted(changed) == sorted(int(s) for s in slots[live[1:]].tolist())
