"""KV_CACHE_WRITE on the GPU: bit-exact against the oracle's byte copy; slot -1
writes nothing; a slot out of range is skipped and reported."""
import pytest
import torch

import oracle
from paged_kv_attention_cache_gb300 import workloads as wl
from tests.gpu_util import gpu_write, on_gpu
from tests.parity import same_bytes

pytestmark = pytest.mark.gpu


def _check_write(case):
    # host snapshot of the pool before the GPU writes it in place
    kc, vc = case.k_cache.cpu().clone(), case.v_cache.cpu().clone()
    before_k = kc.clone()
    hkv, d = kc.shape[2], kc.shape[3]
    kn = case.k_new.reshape(-1, hkv, d).cpu()
    vn = case.v_new.reshape(-1, hkv, d).cpu()
    slots = case.slot_mapping.cpu()
    g = on_gpu(case)
    gpu_write(g)
    torch.cuda.synchronize()
    oracle.kv_cache_write(kn, vn, kc, vc, slots)
    assert same_bytes(g.k_cache, kc) and same_bytes(g.v_cache, vc)
    assert not same_bytes(before_k, kc) or (slots >= 0).sum() == 0
    return g


def test_write_tiny_f32_with_pad():
    case = wl.tiny_decode(seed=0)
    assert (case.slot_mapping == -1).sum() == 1
    _check_write(case)


def test_write_llama8b_decode_tokens():
    _check_write(wl.llama8b_decode(seed=0, device="cuda"))


def test_write_prefill_chunk_16k_rows():
    case = wl.batched_prefill(seed=0, device="cuda")
    assert (case.slot_mapping == -1).sum() > 0
    _check_write(case)


def test_write_preserves_nan_payloads():
    case = wl.decode_case([20, 33], Hq=4, Hkv=2, d=64, dtype=torch.bfloat16, seed=3, n_pad=2)
    case.k_new.view(torch.int16)[0, 0, :4] = torch.tensor([0x7FC1, -1, 0x7F80, 0x0001],
                                                          dtype=torch.int16)
    _check_write(case)


def test_all_padding_writes_nothing():
    case = wl.decode_case([20, 33], Hq=4, Hkv=2, d=64, dtype=torch.bfloat16, seed=4)
    case.slot_mapping[:] = -1
    g = on_gpu(case)
    gpu_write(g)
    torch.cuda.synchronize()
    assert same_bytes(g.k_cache, case.k_cache) and same_bytes(g.v_cache, case.v_cache)


@pytest.mark.parametrize("hkv,d,dtype", [(2, 64, torch.bfloat16),   # rows of 16 vectors
                                         (8, 128, torch.bfloat16),  # 128: the vectorised path
                                         (8, 128, torch.float32),   # 256
                                         (2, 64, torch.float32)])   # 32
def test_out_of_range_slot_is_skipped_and_reported(hkv, d, dtype):
    case = wl.decode_case([20, 33, 5, 70, 1], Hq=2 * hkv, Hkv=hkv, d=d, dtype=dtype, seed=5,
                          n_pad=2)
    n_slots = case.num_pages * case.page_size
    bad = case.slot_mapping.clone()
    bad[0] = n_slots  # one past the end
    bad[1] = -7       # negative but not the padding marker
    case.slot_mapping = bad
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    g = on_gpu(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_write(g, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    live = bad.clone()
    live[(bad < 0) | (bad >= n_slots)] = -1
    oracle.kv_cache_write(case.k_new, case.v_new, kc, vc, live)
    assert same_bytes(g.k_cache, kc) and same_bytes(g.v_cache, vc)


def test_device_error_query_reads_and_clears_the_word():
    """tl_get_device_error after a write with an out-of-range slot: the slot
    bit, status TL_ERR_DEVICE_BOUNDS through the C ABI, and a cleared word."""
    import ctypes

    import paged_kv_attention_cache_gb300 as tl
    from paged_kv_attention_cache_gb300 import _lib

    case = wl.decode_case([20, 33], Hq=4, Hkv=2, d=64, dtype=torch.bfloat16, seed=6)
    case.slot_mapping[0] = case.num_pages * case.page_size + 3
    g = on_gpu(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_write(g, error_word=err)
    lib = _lib.load()
    bits = ctypes.c_uint32(0)
    st = lib.tl_get_device_error(err.data_ptr(), ctypes.byref(bits), 1,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == tl.TL_ERR_DEVICE_BOUNDS and bits.value == tl.TL_DEVERR_SLOT_RANGE
    assert int(err.item()) == 0  # cleared
    st = lib.tl_get_device_error(err.data_ptr(), ctypes.byref(bits), 0, None)
    assert st == tl.TL_OK and bits.value == 0
    assert tl.tl_get_device_error(err) == 0
