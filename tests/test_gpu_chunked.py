"""Chunked prefill and multi-token decode through the prefill entry point
("How serving works in Tlaloc", section 4: a runtime prefills a long prompt in
several calls, and chunked prefill gives whole-context results bit for bit;
a call of q tokens at the end of a sequence is the speculative-verify shape)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import workloads as wl
from tests.gpu_util import (assert_prefill_rows, gpu_prefill, gpu_write, on_gpu,
                            oracle_prefill_tokens)
from tests.parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _slice_call(g, t0, t1):
    """The same rows restricted to tokens [t0, t1) (positions and queries)."""
    import copy
    c = copy.copy(g)
    c.q = g.q[:, t0:t1].contiguous()
    c.positions = g.positions[:, t0:t1].contiguous()
    c.T = t1 - t0
    return c


@pytest.mark.parametrize("chunk", [512, 300, 64])
def test_chunked_prefill_equals_whole_context_bit_for_bit(chunk):
    # rows with prior context; the whole chunk's K/V is written first, then
    # the tokens are attended in one call or in consecutive calls of `chunk`
    case = wl.prefill_case([0, 40, 500], [100, 3000, 0], T=1024, Hq=32, Hkv=8, d=128, seed=41)
    g = on_gpu(case)
    gpu_write(g)
    whole = gpu_prefill(g)
    parts = [gpu_prefill(_slice_call(g, t0, min(t0 + chunk, case.T)))
             for t0 in range(0, case.T, chunk)]
    torch.cuda.synchronize()
    assert torch.equal(whole, torch.cat(parts, dim=1))


@pytest.mark.parametrize("q_len", [2, 4, 8])
def test_multi_token_decode_shape_matches_the_oracle(q_len):
    # B sequences of Llama-3-8B shape, each verifying q_len new tokens at the
    # end of its context: positions L - q_len .. L - 1
    lengths = wl.llama8b_lengths(seed=3, B=16)
    p0 = [L - q_len for L in lengths]
    case = wl.prefill_case([0] * len(lengths), p0, T=q_len, Hq=32, Hkv=8, d=128, seed=42)
    g = on_gpu(case)
    gpu_write(g)
    out = gpu_prefill(g)
    torch.cuda.synchronize()
    for row in (0, 5, 15):
        ref = oracle_prefill_tokens(g, row, list(range(q_len)))
        assert_close(out[row], ref, f"verify row {row}")
    # the last token of each row is a plain decode query of length L
    dec = tl.tl_paged_attn_decode(g.q[:, -1].contiguous(), g.k_cache, g.v_cache, g.block_table,
                                  torch.tensor(lengths, dtype=torch.int32, device=DEV), g.scale)
    torch.cuda.synchronize()
    ref_last = oracle.paged_decode(g.q[:, -1].cpu(), g.k_cache.cpu(), g.v_cache.cpu(),
                                   g.block_table.cpu(), torch.tensor(lengths, dtype=torch.int32),
                                   g.scale, seqs=[0, 5, 15])
    assert_close(dec[[0, 5, 15]], ref_last, "decode of the last verify token")
    assert_close(out[[0, 5, 15], -1], ref_last, "verify vs decode")


@pytest.mark.parametrize("q_len,hq,hkv,d,window", [(2, 32, 8, 128, 0), (4, 32, 8, 128, 0),
                                                    (8, 16, 8, 128, 0), (3, 40, 8, 128, 0),
                                                    (4, 32, 8, 128, 700), (6, 8, 4, 64, 0),
                                                    (16, 8, 8, 128, 0)])
def test_multi_token_decode_kernel(q_len, hq, hkv, d, window):
    # the decode kernel with q_len tokens per sequence: against the oracle, and
    # against the prefill entry point on the same tokens
    lengths = wl.llama8b_lengths(seed=5, B=24)
    lengths[0], lengths[1] = q_len, q_len + 3  # sequences hardly longer than the call
    p0 = [L - q_len for L in lengths]
    case = wl.prefill_case([0] * len(lengths), p0, T=q_len, Hq=hq, Hkv=hkv, d=d, seed=43,
                           window=window)
    g = on_gpu(case)
    gpu_write(g)
    cl = torch.tensor(lengths, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tl.tl_paged_attn_decode_multi(g.q, g.k_cache, g.v_cache, g.block_table, cl, g.scale,
                                        window=window, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for row in (0, 1, 7, 23):
        ref = oracle_prefill_tokens(g, row, list(range(q_len)))
        assert_close(out[row], ref, f"multi-token decode row {row}")
    if d == 128:
        pf = gpu_prefill(g)
        torch.cuda.synchronize()
        assert_close(out.cpu(), pf.double().cpu().numpy(), "decode_multi vs prefill")


@pytest.mark.parametrize("window", [0, 4096])
def test_multi_token_decode_outliers_every_token(window):
    """The multi-token decode on the sliding-window mix's shape and values
    (H_q=40, H_kv=8, lengths U[1024, 32768], 1% of Q, K and V values x8), 3
    tokens per sequence: every token against the oracle."""
    q_len = 3
    lengths = wl.swa_lengths(seed=2, B=16)
    p0 = [L - q_len for L in lengths]
    case = wl.prefill_case([0] * len(lengths), p0, T=q_len, Hq=40, Hkv=8, d=128, seed=45,
                           window=window, outlier_p=0.01, device=DEV)
    g = on_gpu(case)
    k0, v0 = g.k_cache.clone(), g.v_cache.clone()
    gpu_write(g)
    cl = torch.tensor(lengths, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tl.tl_paged_attn_decode_multi(g.q, g.k_cache, g.v_cache, g.block_table, cl, g.scale,
                                        window=window, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_prefill_rows(out, g, range(case.B), pools=(k0, v0),
                        new_rows=(g.k_new, g.v_new, g.slot_mapping),
                        what=f"multi-token outliers w{window}")


def test_multi_token_decode_refuses_too_many_rows():
    case = wl.prefill_case([0], [100], T=5, Hq=32, Hkv=8, d=128, seed=44)
    g = on_gpu(case)
    with pytest.raises(tl.TLError) as e:
        tl.tl_paged_attn_decode_multi(g.q, g.k_cache, g.v_cache, g.block_table,
                                      torch.tensor([105], dtype=torch.int32, device=DEV), g.scale)
    assert e.value.status == tl.TL_ERR_UNSUPPORTED
