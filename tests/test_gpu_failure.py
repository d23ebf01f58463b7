"""Failure paths on the GPU, made without a fault: a decode kernel whose wait
runs out returns with TL_DEVERR_TIMEOUT set, and the context stays usable.

The library bounds every in-kernel wait (about a second); after a wait gives
up, the kernel drains its own copies in flight (also bounded) and returns.
To make one wait run out, this test builds a separate copy of the decode
library in which the first stage of one warp expects 16 bytes that no copy
delivers (every copy it does issue lands) and the wait bound is about 16 ms.
The product library has neither setting."""
import ctypes
import time

import pytest
import torch

import oracle
import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import _lib, build, workloads as wl
from tests.gpu_util import gpu_decode, on_gpu
from tests.parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def stall_lib():
    path = build.build_variant("stall_first_stage", ["api.cu", "paged_decode.cu"],
                               ["TL_TEST_STALL_FIRST_STAGE=1", "TL_WAIT_CYCLES=(1ll<<25)"])
    lib = ctypes.CDLL(path)
    for name in ("tl_paged_attn_decode", "tl_get_device_error"):
        args, res = _lib.SIGNATURES[name]
        getattr(lib, name).argtypes = args
        getattr(lib, name).restype = res
    return lib


def test_a_wait_that_runs_out_sets_the_timeout_bit_and_returns(stall_lib):
    case = wl.decode_case([300, 40, 1000, 17], Hq=8, Hkv=2, d=128, seed=31)
    g = on_gpu(case)
    B, hq, d = case.B, case.Hq, case.d
    out = torch.zeros((B, hq, d), dtype=torch.float32, device="cuda")
    ws = tl.alloc_workspace(tl.tl_paged_attn_decode_workspace_size(B, hq, case.Hkv, d), "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    st = stall_lib.tl_paged_attn_decode(
        g.q.data_ptr(), g.k_cache.data_ptr(), g.v_cache.data_ptr(), g.block_table.data_ptr(),
        g.block_table.shape[1], g.context_lens.data_ptr(), out.data_ptr(), B, hq, case.Hkv, d,
        case.num_pages, case.page_size, 0, case.scale, tl.TL_BF16, ws.data_ptr(), ws.numel(),
        err.data_ptr(), stream)
    assert st == tl.TL_OK
    bits = ctypes.c_uint32(0)
    st = stall_lib.tl_get_device_error(err.data_ptr(), ctypes.byref(bits), 0, stream)
    elapsed = time.time() - t0
    assert st == tl.TL_ERR_DEVICE_TIMEOUT
    assert bits.value & tl.TL_DEVERR_TIMEOUT
    assert elapsed < 30.0  # the bounded waits ended the kernel
    # the context is still usable: the product library gives the oracle's result
    res = gpu_decode(g)
    torch.cuda.synchronize()
    ref = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_table,
                              case.context_lens, case.scale)
    assert_close(res, ref, "decode after a timed-out call")
