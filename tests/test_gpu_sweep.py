"""Seeded sweeps of decode and prefill shapes over bf16, e4m3 and int8
pools: random head groupings (1-16 query heads per KV head), page sizes,
windows, batch sizes and lengths (with the edge lengths 0, 1, 15, 16, 17
mixed in), 2-4 query tokens per sequence for the multi-token calls, and
padded prefill chunks of any length; every output against the oracle.  It reaches the layouts the kernels switch between (rows-as-rows
and keys-as-rows, duplicated columns or not, one or two row groups) in
combinations no hand-written case lists."""
import random

import pytest
import torch

import oracle
import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import workloads as wl
from tests.parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _draw(rng: random.Random, kind: str):
    hkv = rng.choice([1, 2, 4, 8])
    group = rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 16])
    ps = rng.choice([16, 32, 64] if kind == "int8" else [8, 16, 24, 32, 64])
    B = rng.randint(1, 10)
    lens = [rng.choice([0, 1, 15, 16, 17, rng.randint(2, 3000)]) for _ in range(B)]
    window = rng.choice([0, 0, rng.randint(1, 2000)])
    return hkv, group, ps, lens, window


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("kind", ["bf16", "e4m3", "int8"])
@pytest.mark.parametrize("draw", range(24))
def test_decode_sweep(kind, draw):
    rng = random.Random(1000 * draw + {"bf16": 1, "e4m3": 2, "int8": 3}[kind])
    hkv, group, ps, lens, window = _draw(rng, kind)
    case = wl.decode_case(lens, Hq=hkv * group, Hkv=hkv, d=128, page_size=ps, window=window,
                          seed=rng.randint(0, 10**6))
    what = f"{kind} hkv={hkv} group={group} ps={ps} window={window} lens={lens}"
    err = _err()
    if kind == "int8":
        pools = wl.int8_pools(case, rng.randint(0, 10**6))
        kc, vc, ks, vs = (t.to(DEV) for t in pools)
        out = tl.tl_paged_attn_decode_int8(case.q.to(DEV), kc, vc, ks, vs,
                                           case.block_table.to(DEV), case.context_lens.to(DEV),
                                           case.scale, window=window, error_word=err)
        ref = oracle.paged_decode_int8(case.q, *pools, case.block_table, case.context_lens,
                                       case.scale, window=window)
    else:
        kc, vc = case.k_cache, case.v_cache
        if kind == "e4m3":
            kc, vc = kc.float().to(torch.float8_e4m3fn), vc.float().to(torch.float8_e4m3fn)
        out = tl.tl_paged_attn_decode(case.q.to(DEV), kc.to(DEV), vc.to(DEV),
                                      case.block_table.to(DEV), case.context_lens.to(DEV),
                                      case.scale, window=window, error_word=err)
        ref = oracle.paged_decode(case.q, kc, vc, case.block_table, case.context_lens, case.scale,
                                  window=window)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, what
    assert_close(out.cpu(), ref, what)


@pytest.mark.parametrize("kind", ["bf16", "e4m3", "int8"])
@pytest.mark.parametrize("draw", range(16))
def test_multi_token_sweep(kind, draw):
    rng = random.Random(5000 + 1000 * draw + {"bf16": 0, "e4m3": 1, "int8": 2}[kind])
    hkv = rng.choice([1, 2, 4, 8])
    q_len = rng.randint(2, 4)
    group = rng.choice([g for g in (1, 2, 3, 4, 5, 8) if g * q_len <= 16])
    ps = rng.choice([16, 32])
    window = rng.choice([0, rng.randint(1, 1500)])
    B = rng.randint(1, 6)
    lengths = [rng.randint(q_len, 2500) for _ in range(B)]
    p0 = [L - q_len for L in lengths]
    case = wl.prefill_case([0] * B, p0, T=q_len, Hq=hkv * group, Hkv=hkv, d=128, page_size=ps,
                           window=window, seed=rng.randint(0, 10**6))
    what = f"{kind} multi q_len={q_len} hkv={hkv} group={group} ps={ps} window={window}"
    if kind == "int8":
        pools = [t.clone() for t in wl.int8_pools(case, rng.randint(0, 10**6))]
        oracle.kv_cache_write_int8(case.k_new.view(-1, hkv, 128), case.v_new.view(-1, hkv, 128),
                                   *pools, case.slot_mapping)
        err = _err()
        out = tl.tl_paged_attn_decode_multi_int8(
            case.q.to(DEV), *(t.to(DEV) for t in pools), case.block_table.to(DEV),
            torch.tensor(lengths, dtype=torch.int32, device=DEV), case.scale, window=window,
            error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, what
        ref = oracle.paged_prefill_int8(case.q, *pools, case.block_table, case.positions,
                                        case.scale, window=window)
        assert_close(out.cpu().reshape(ref.shape), ref, what)
        return
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    if kind == "e4m3":
        k8 = kc.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
        v8 = vc.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
        oracle.kv_cache_write_fp8(case.k_new, case.v_new, k8, v8, case.slot_mapping)
        kc = torch.from_numpy(k8).view(torch.float8_e4m3fn)
        vc = torch.from_numpy(v8).view(torch.float8_e4m3fn)
    else:
        oracle.kv_cache_write(case.k_new.view(-1, hkv, 128), case.v_new.view(-1, hkv, 128), kc, vc,
                              case.slot_mapping)
    err = _err()
    out = tl.tl_paged_attn_decode_multi(case.q.to(DEV), kc.to(DEV), vc.to(DEV),
                                        case.block_table.to(DEV),
                                        torch.tensor(lengths, dtype=torch.int32, device=DEV),
                                        case.scale, window=window, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, what
    ref = oracle.paged_prefill(case.q, kc, vc, case.block_table, case.positions, case.scale,
                               window=window)
    assert_close(out.cpu().reshape(ref.shape), ref, what)


@pytest.mark.parametrize("kind", ["bf16", "e4m3", "int8"])
@pytest.mark.parametrize("draw", range(12))
def test_prefill_sweep(kind, draw):
    """Right-aligned prefill calls of random shape: 1-4 rows, chunks of 1-160
    tokens (not a multiple of the tile), any padding, prior context 0-1,500,
    1-16 query heads per KV head, windows; the chunk's rows are written into
    host copies of the pools by the oracle, and both sides read those."""
    rng = random.Random(9000 + 1000 * draw + {"bf16": 1, "e4m3": 2, "int8": 3}[kind])
    hkv = rng.choice([1, 2, 4, 8])
    group = rng.choice([g for g in (1, 2, 3, 4, 5, 8, 16) if g * hkv <= 32])
    B = rng.randint(1, 4)
    T = rng.randint(1, 160)
    pads = [rng.choice([0, rng.randint(0, T)]) for _ in range(B)]
    p0 = [rng.choice([0, rng.randint(0, 1500)]) for _ in range(B)]
    window = rng.choice([0, 0, rng.randint(1, 600)])
    ps = rng.choice([16, 32])
    case = wl.prefill_case(pads, p0, T=T, Hq=hkv * group, Hkv=hkv, d=128, page_size=ps,
                           window=window, seed=rng.randint(0, 10**6))
    what = f"{kind} prefill B={B} T={T} hkv={hkv} group={group} ps={ps} window={window}"
    kn, vn = case.k_new.view(-1, hkv, 128), case.v_new.view(-1, hkv, 128)
    err = _err()
    if kind == "int8":
        pools = [t.clone() for t in wl.int8_pools(case, rng.randint(0, 10**6))]
        oracle.kv_cache_write_int8(kn, vn, *pools, case.slot_mapping)
        out = tl.tl_paged_attn_prefill_int8(case.q.to(DEV), *(t.to(DEV) for t in pools),
                                            case.block_table.to(DEV), case.positions.to(DEV),
                                            case.scale, window=window, error_word=err)
        ref = oracle.paged_prefill_int8(case.q, *pools, case.block_table, case.positions,
                                        case.scale, window=window)
    else:
        if kind == "e4m3":
            k8 = case.k_cache.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
            v8 = case.v_cache.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
            oracle.kv_cache_write_fp8(kn, vn, k8, v8, case.slot_mapping)
            kc = torch.from_numpy(k8).view(torch.float8_e4m3fn)
            vc = torch.from_numpy(v8).view(torch.float8_e4m3fn)
        else:
            kc, vc = case.k_cache.clone(), case.v_cache.clone()
            oracle.kv_cache_write(kn, vn, kc, vc, case.slot_mapping)
        out = tl.tl_paged_attn_prefill(case.q.to(DEV), kc.to(DEV), vc.to(DEV),
                                       case.block_table.to(DEV), case.positions.to(DEV),
                                       case.scale, window=window, error_word=err)
        ref = oracle.paged_prefill(case.q, kc, vc, case.block_table, case.positions, case.scale,
                                   window=window)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, what
    assert_close(out.cpu().reshape(ref.shape), ref, what)
