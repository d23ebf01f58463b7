"""The allocation-free decode entry point against the regular one.

tl_paged_attn_decode_noalloc serves callers that cannot allocate device
memory on their attention path (a framework that owns all device memory
through its own pool, a latency-bound loop): its scratch is a fixed array in
the library.  Its output must match tl_paged_attn_decode's on the same inputs,
on two calls in a row (the second call finds the first call's leftovers in the
shared array).  This file is collected last on purpose.
"""
import pytest
import torch

import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import build, workloads as wl
from tests.parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()


def test_noalloc_matches_the_regular_entry_point_twice():
    case = wl.to_device(wl.llama8b_decode(seed=5, device="cuda"), "cuda")
    assert tl.tl_paged_attn_decode_workspace_size(64, 32, 8, 128) <= tl.TL_DECODE_NOALLOC_SCRATCH_BYTES
    ref = tl.tl_paged_attn_decode(case.q, case.k_cache, case.v_cache, case.block_table,
                                  case.context_lens, case.scale)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        tl.tl_paged_attn_decode_noalloc(case.q, case.k_cache, case.v_cache, case.block_table,
                                        case.context_lens, case.scale, out, error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out, ref.double().cpu().numpy(), f"no-alloc call {call}")


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
