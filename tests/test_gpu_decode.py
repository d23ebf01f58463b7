"""PAGED_ATTENTION decode on the GPU against the oracle: the five workloads at
full size (every sequence), edge cases, invariants, device-side checks."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import workloads as wl
from tests.gpu_util import assert_decode_all, gpu_decode, gpu_write, on_gpu, permuted_pool
from tests.parity import assert_close

pytestmark = pytest.mark.gpu


def _write_then_decode(case):
    g = on_gpu(case)
    gpu_write(g)
    out = gpu_decode(g)
    torch.cuda.synchronize()
    return g, out


def test_tiny_f32_all_outputs():
    case = wl.tiny_decode(seed=0)
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    g, out = _write_then_decode(case)
    oracle.kv_cache_write(case.k_new, case.v_new, kc, vc, case.slot_mapping)
    ref = oracle.paged_decode(case.q, kc, vc, case.block_table, case.context_lens, case.scale)
    assert_close(out, ref, "tiny f32")


def _step_every_sequence(case, what):
    """The step (write of the new rows, then decode) on the GPU; the oracle
    writes the same rows into its own copies of the pools as they were before
    the step, then attends; every sequence compared."""
    g = on_gpu(case)
    k0, v0 = g.k_cache.clone(), g.v_cache.clone()
    gpu_write(g)
    out = gpu_decode(g)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert_decode_all(out, g.q, k0, v0, g.block_table, g.context_lens, g.scale,
                      window=case.window, new_rows=(g.k_new, g.v_new, g.slot_mapping), what=what)


@pytest.mark.parametrize("maker", [wl.llama8b_decode, wl.longctx_decode])
def test_full_size_workloads_every_sequence(maker):
    _step_every_sequence(maker(seed=0, device="cuda"), maker.__name__)


@pytest.mark.parametrize("layer", [0, 1])
def test_sliding_window_mix_every_sequence(layer):
    """Both layers of the sliding-window mix (separate pools, window 4,096 then
    full attention, 1% of Q, K and V values x8), every sequence."""
    case = wl.swa_decode(seed=0, device="cuda", layer=layer)
    assert case.window == (4096 if layer == 0 else 0)
    _step_every_sequence(case, f"swa layer {layer}")


EDGE_LENGTHS = [0, 1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 2047, 2048, 2049, 5000]


@pytest.mark.parametrize("window", [0, 1, 16, 17, 100, 2048])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_edge_lengths_and_windows(window, dtype):
    case = wl.decode_case(EDGE_LENGTHS, Hq=8, Hkv=2, d=128, dtype=dtype, window=window, seed=7,
                          nan_unused=True)
    g = on_gpu(case)
    out = gpu_decode(g)
    torch.cuda.synchronize()
    ref = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_table,
                              case.context_lens, case.scale, window=window)
    assert_close(out, ref, f"edges w={window} {dtype}")
    assert torch.all(out[0] == 0)  # length 0 gives 0


@pytest.mark.parametrize("hq,hkv", [(16, 16), (16, 1), (40, 8), (64, 8), (32, 2)])
@pytest.mark.parametrize("d", [64, 128])
def test_head_groupings(hq, hkv, d):
    lens = [1, 40, 300, 1234]
    case = wl.decode_case(lens, Hq=hq, Hkv=hkv, d=d, seed=11, nan_unused=True)
    g = on_gpu(case)
    out = gpu_decode(g)
    torch.cuda.synchronize()
    ref = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_table,
                              case.context_lens, case.scale)
    assert_close(out, ref, f"hq={hq} hkv={hkv} d={d}")


@pytest.mark.parametrize("page_size,dtype", [(8, torch.bfloat16), (16, torch.bfloat16),
                                             (24, torch.bfloat16), (32, torch.bfloat16),
                                             (256, torch.bfloat16), (1, torch.float32),
                                             (7, torch.float32)])
def test_page_sizes(page_size, dtype):
    lens = [1, 5, 100, 513, 1500]
    case = wl.decode_case(lens, Hq=8, Hkv=2, d=128, page_size=page_size, window=300, seed=13,
                          nan_unused=True, dtype=dtype)
    g = on_gpu(case)
    out = gpu_decode(g)
    torch.cuda.synchronize()
    ref = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_table,
                              case.context_lens, case.scale, window=300)
    assert_close(out, ref, f"page_size={page_size}")


def test_bf16_page_size_not_multiple_of_8_is_refused():
    case = wl.decode_case([40], Hq=4, Hkv=2, d=128, page_size=7, seed=14)
    g = on_gpu(case)
    with pytest.raises(tl.TLError) as e:
        tl.tl_paged_attn_decode(g.q, g.k_cache, g.v_cache, g.block_table, g.context_lens,
                                g.scale)
    assert e.value.status == tl.TL_ERR_UNSUPPORTED


def test_page_placement_and_repeat_are_bit_identical():
    case = wl.llama8b_decode(seed=3, device="cuda", B=16)
    g = on_gpu(case)
    a = gpu_decode(g)
    b = gpu_decode(g)
    kc, vc, bt = permuted_pool(g)
    c = tl.tl_paged_attn_decode(g.q, kc, vc, bt, g.context_lens, g.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(a, c)


def test_bad_block_table_entry_is_reported_not_faulted():
    case = wl.decode_case([40, 100], Hq=4, Hkv=2, d=128, seed=17)
    case.pool.block_table[1, 2] = case.num_pages + 5  # a page the pool does not have
    case.pool.block_table[0, 0] = -3
    g = on_gpu(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(g, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & tl.TL_DEVERR_PAGE_RANGE
    assert torch.isfinite(out).all()


def test_context_past_the_table_is_reported():
    case = wl.decode_case([40, 100], Hq=4, Hkv=2, d=128, seed=19)
    g = on_gpu(case)
    g.context_lens = torch.tensor([40, 100 + 16 * 10], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(g, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & tl.TL_DEVERR_CONTEXT_RANGE
    assert torch.all(out[1] == 0)


def test_workspace_is_reused_across_calls_of_different_shapes():
    ws = tl.alloc_workspace(tl.tl_paged_attn_decode_workspace_size(64, 64, 8, 128), "cuda")
    for seed, lens in ((0, [3000, 10, 70000]), (1, [5] * 64)):
        case = wl.decode_case(lens, Hq=64, Hkv=8, d=128, seed=seed)
        g = on_gpu(case)
        out = gpu_decode(g, workspace=ws)
        torch.cuda.synchronize()
        ref = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_table,
                                  case.context_lens, case.scale)
        assert_close(out, ref, f"workspace reuse {seed}")


@pytest.mark.parametrize("shape", ["many_short", "one_long", "mixed"])
def test_piece_plan_extremes(shape):
    """The decode plan cuts each sequence into bulk pieces and a last round of
    small pieces (the last ~15% of every sequence longer than 256 keys), all
    within ceil(6144 / H_kv) + 2B pieces.  Batches at the ends of that range
    (thousands of short sequences, one very long one, both mixed) against the
    oracle on every sequence, every output finite and no device error."""
    g = torch.Generator().manual_seed(91)
    if shape == "many_short":
        lens = torch.randint(1, 400, (2048,), generator=g).tolist()
    elif shape == "one_long":
        lens = [131072]
    else:
        lens = torch.randint(1, 300, (500,), generator=g).tolist() + [65536, 257, 4096, 0, 1]
    case = wl.decode_case(lens, Hq=32, Hkv=8, d=128, seed=92, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g_ = on_gpu(case)
    out = gpu_decode(g_, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isfinite(out).all()
    assert_decode_all(out, g_.q, g_.k_cache, g_.v_cache, g_.block_table, g_.context_lens,
                      g_.scale, chunk=256, what=f"piece plan {shape}")


@pytest.mark.parametrize("B", [1, 3, 17, 32, 33, 127, 128, 129])
@pytest.mark.parametrize("kind", ["bf16", "e4m3", "int8"])
def test_plan_paths_and_combine_groups(B, kind):
    """Batch sizes on both sides of the plan's one-warp path (up to 128
    sequences) and the block-wide one, and across the combine's group counts
    (16 groups at B = 1 down to one from B = 33 with 8 KV heads): every
    sequence against the oracle, with lengths that give every sequence several
    pieces."""
    g = torch.Generator().manual_seed(300 + B)
    lens = torch.randint(1, 2400 if B > 32 else 9000, (B,), generator=g).tolist()
    case = wl.decode_case(lens, Hq=32, Hkv=8, d=128, seed=301 + B)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g_ = on_gpu(case)
    if kind == "int8":
        pools = wl.int8_pools(case, 302 + B)
        kc, vc, ks, vs = (t.to("cuda") for t in pools)
        out = tl.tl_paged_attn_decode_int8(g_.q, kc, vc, ks, vs, g_.block_table, g_.context_lens,
                                           case.scale, error_word=err)
        torch.cuda.synchronize()
        ref = oracle.paged_decode_int8(case.q, *pools, case.block_table, case.context_lens,
                                       case.scale)
        assert int(err.item()) == 0
        assert_close(out.cpu(), ref, f"int8 B={B}")
        return
    kc, vc = g_.k_cache, g_.v_cache
    if kind == "e4m3":
        kc, vc = kc.float().to(torch.float8_e4m3fn), vc.float().to(torch.float8_e4m3fn)
    out = tl.tl_paged_attn_decode(g_.q, kc, vc, g_.block_table, g_.context_lens, case.scale,
                                  error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isfinite(out).all()
    assert_decode_all(out, g_.q, kc, vc, g_.block_table, g_.context_lens, g_.scale,
                      chunk=64, what=f"{kind} B={B}")
