"""The allocation-free decode entry point against the regular one.

tl_paged_attn_decode_noalloc serves callers that cannot allocate device
memory on their attention path (a framework that owns all device memory
through its own pool, a latency-bound loop): its scratch is a fixed array in
the library.  Its output must equal tl_paged_attn_decode's on the same inputs
bit for bit (the same kernels and plan; only the scratch's address differs),
on two calls in a row, with a call of another shape (other lengths, batch,
window and dtype) in between, so the second compared call finds that call's
leftovers in the shared array.  Small cases are also compared with the
oracle.  This file is collected last on purpose.
"""
import pytest
import torch

import oracle
import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import build, workloads as wl
from tests.parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()


def _noalloc(case, out):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tl.tl_paged_attn_decode_noalloc(case.q, case.k_cache, case.v_cache, case.block_table,
                                    case.context_lens, case.scale, out, window=case.window,
                                    error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


def _e4m3(case):
    """The case's bf16 pools as e4m3 pools (the converting write, every slot)."""
    P, ps, hkv, d = case.k_cache.shape
    k8 = torch.empty((P, ps, hkv, d), dtype=torch.float8_e4m3fn, device="cuda")
    v8 = torch.empty_like(k8)
    every = torch.arange(P * ps, dtype=torch.int64, device="cuda")
    tl.tl_kv_cache_write_fp8(case.k_cache.view(-1, hkv, d), case.v_cache.view(-1, hkv, d), k8,
                             v8, every)
    case.k_cache, case.v_cache = k8, v8
    return case


CASES = {
    "llama8b_bf16": lambda: wl.to_device(wl.llama8b_decode(seed=5, device="cuda"), "cuda"),
    "tiny_f32": lambda: wl.to_device(wl.tiny_decode(seed=2), "cuda"),
    "window4096_bf16": lambda: wl.to_device(
        wl.decode_case([5000, 4096, 4097, 1, 9000], Hq=40, Hkv=8, d=128, window=4096, seed=7,
                       outlier_p=0.01), "cuda"),
    "e4m3": lambda: _e4m3(wl.to_device(wl.decode_case([70, 3000, 513], Hq=32, Hkv=8, d=128,
                                                       seed=8), "cuda")),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_equals_the_regular_entry_point_twice(name):
    case = CASES[name]()
    B, hq, d = case.q.shape
    assert tl.tl_paged_attn_decode_workspace_size(B, hq, case.Hkv, d) <= \
        tl.TL_DECODE_NOALLOC_SCRATCH_BYTES
    ref = tl.tl_paged_attn_decode(case.q, case.k_cache, case.v_cache, case.block_table,
                                  case.context_lens, case.scale, window=case.window)
    torch.cuda.synchronize()
    # another shape in between: its plan leaves other offsets, descriptors and
    # partials in the shared array
    other = CASES["tiny_f32" if name != "tiny_f32" else "window4096_bf16"]()
    for call in range(2):
        out = _noalloc(case, torch.full_like(ref, float("nan")))
        assert torch.equal(out, ref), f"{name}: no-alloc call {call} differs"
        _noalloc(other, torch.empty((other.B, other.Hq, other.d), dtype=torch.float32,
                                    device="cuda"))
    if B * max(case.context_lens.tolist()) <= 20000:  # small enough for the oracle here
        ref_o = oracle.paged_decode(case.q.cpu(), case.k_cache.cpu(), case.v_cache.cpu(),
                                    case.block_table.cpu(), case.context_lens.cpu(), case.scale,
                                    window=case.window)
        assert_close(out, ref_o, f"{name} against the oracle")


def test_noalloc_refuses_sizes_beyond_its_scratch():
    case = wl.to_device(wl.decode_case([40, 90], Hq=64, Hkv=8, d=128, seed=6), "cuda")
    B = 4096  # needs far more scratch than the fixed array holds
    assert tl.tl_paged_attn_decode_workspace_size(B, 64, 8, 128) > tl.TL_DECODE_NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B, 64, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((B, case.block_table.shape[1]), dtype=torch.int32, device="cuda")
    cl = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.zeros((B, 64, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(tl.TLError) as e:
        tl.tl_paged_attn_decode_noalloc(q, case.k_cache, case.v_cache, bt, cl, case.scale, out)
    assert e.value.status == tl.TL_ERR_WORKSPACE


def test_noalloc_refuses_a_missing_or_misshapen_output():
    case = wl.to_device(wl.decode_case([40, 90], Hq=8, Hkv=2, d=128, seed=9), "cuda")
    with pytest.raises(ValueError):
        tl.tl_paged_attn_decode_noalloc(case.q, case.k_cache, case.v_cache, case.block_table,
                                        case.context_lens, case.scale, None)
    small = torch.zeros((1, 8, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        tl.tl_paged_attn_decode_noalloc(case.q, case.k_cache, case.v_cache, case.block_table,
                                        case.context_lens, case.scale, small)
    with pytest.raises(ValueError):  # a block table shorter than the batch
        tl.tl_paged_attn_decode_noalloc(case.q, case.k_cache, case.v_cache,
                                        case.block_table[:1].contiguous(), case.context_lens,
                                        case.scale, torch.empty_like(small.expand(2, 8, 128)))
