"""Helpers for the GPU parity tests: run a case through the C ABI, and compute
the oracle on host copies of the same bytes (for large cases on a sample of
sequences / tokens, after copying only the pages those sequences use)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import workloads as wl

DEV = "cuda"


def gpu_write(g, error_word=None):
    hkv, d = g.k_cache.shape[2], g.k_cache.shape[3]
    err = torch.zeros(1, dtype=torch.int32, device=DEV) if error_word is None else error_word
    tl.tl_kv_cache_write(g.k_new.reshape(-1, hkv, d), g.v_new.reshape(-1, hkv, d), g.k_cache,
                         g.v_cache, g.slot_mapping, error_word=err)
    if error_word is None:
        assert int(err.item()) == 0, f"device error word {int(err.item())}"


def _clean_error_word():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def gpu_decode(g, window=None, error_word=None, out=None, workspace=None):
    """Decode through the C ABI; without a caller error word, checks that the
    device-side checks reported nothing (no range error, no timed-out wait)."""
    err = _clean_error_word() if error_word is None else error_word
    out = tl.tl_paged_attn_decode(g.q, g.k_cache, g.v_cache, g.block_table, g.context_lens,
                                  g.scale, window=g.window if window is None else window,
                                  error_word=err, out=out, workspace=workspace)
    if error_word is None:
        assert int(err.item()) == 0, f"device error word {int(err.item())}"
    return out


def gpu_prefill(g, window=None, error_word=None):
    err = _clean_error_word() if error_word is None else error_word
    out = tl.tl_paged_attn_prefill(g.q, g.k_cache, g.v_cache, g.block_table, g.positions,
                                   g.scale, window=g.window if window is None else window,
                                   error_word=err)
    if error_word is None:
        assert int(err.item()) == 0, f"device error word {int(err.item())}"
    return out


def sub_pool(k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor, rows,
             n_pages_of_row):
    """Host copies of only the pages the given rows use, with the rows' block
    tables renumbered to the copy.  Pure data movement (torch index_select)."""
    bt = block_table.cpu()
    pages, tables = [], []
    for b, n in zip(rows, n_pages_of_row):
        ids = bt[b, :n].tolist()
        tables.append(list(range(len(pages), len(pages) + n)))
        pages += ids
    if not pages:
        pages = [0]
    idx = torch.tensor(pages, dtype=torch.long, device=k_cache.device)
    kc = k_cache.index_select(0, idx).cpu()
    vc = v_cache.index_select(0, idx).cpu()
    width = max(1, max((len(t) for t in tables), default=1))
    new_bt = torch.full((len(rows), width), -1, dtype=torch.int32)
    for i, t in enumerate(tables):
        if t:
            new_bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    return kc, vc, new_bt


def oracle_decode_rows(g, rows, window=None, threads=0):
    """Oracle output [len(rows), Hq, d] for sequences `rows` of a GPU case
    (read from the GPU pool after the write)."""
    ps = g.k_cache.shape[1]
    lens = g.context_lens.cpu().tolist()
    n_pages = [(max(lens[b], 0) + ps - 1) // ps for b in rows]
    kc, vc, bt = sub_pool(g.k_cache, g.v_cache, g.block_table, rows, n_pages)
    q = g.q[list(rows)].cpu()
    cl = torch.tensor([lens[b] for b in rows], dtype=torch.int32)
    w = g.window if window is None else window
    return oracle.paged_decode(q, kc, vc, bt, cl, g.scale, window=w, threads=threads)


def oracle_prefill_tokens(g, row, ts, window=None, threads=0):
    """Oracle output [len(ts), Hq, d] for tokens ts of prefill row `row`."""
    ps = g.k_cache.shape[1]
    pos = g.positions[row].cpu()
    last = int(pos.max().item())
    kc, vc, bt = sub_pool(g.k_cache, g.v_cache, g.block_table, [row], [(last + ps) // ps])
    q = g.q[row:row + 1].cpu()
    w = g.window if window is None else window
    return oracle.paged_prefill(q, kc, vc, bt, pos.view(1, -1), g.scale, window=w,
                                tokens=np.asarray(ts, np.int64), threads=threads)


def sample_rows(lengths, n, seed=0):
    """A spread of rows: the shortest, the longest, and random others."""
    L = np.asarray(lengths)
    rng = np.random.default_rng(seed)
    pick = {int(L.argmin()), int(L.argmax())}
    others = rng.permutation(len(L))
    for b in others:
        if len(pick) >= n:
            break
        pick.add(int(b))
    return sorted(pick)


def permuted_pool(g, seed=123):
    """The same contents at other physical pages: pool'[perm[i]] = pool[i] and
    block_table' = perm[block_table]."""
    P = g.k_cache.shape[0]
    gen = torch.Generator(device="cpu").manual_seed(seed)
    perm = torch.randperm(P, generator=gen).to(g.k_cache.device)
    kc = torch.empty_like(g.k_cache)
    vc = torch.empty_like(g.v_cache)
    kc[perm] = g.k_cache
    vc[perm] = g.v_cache
    bt = g.block_table.long()
    nbt = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).to(torch.int32)
    return kc, vc, nbt


def on_gpu(case):
    return wl.to_device(case, DEV)


def assert_decode_all(out, q, k_cache, v_cache, block_table, context_lens, scale, window=0,
                      ring_pages=0, k_scales=None, v_scales=None, chunk=16, what="decode",
                      new_rows=None):
    """Every sequence's output against the oracle, `chunk` sequences at a
    time (host copies of only their pages, their tables renumbered; int8
    pools bring their scale pages along).  With new_rows = (k_new, v_new,
    slot_mapping), the pools are those before the step's write and the
    oracle applies its own write of those rows to its copies first, so no
    oracle input comes from a GPU kernel.  Returns the worst (abs, rel)."""
    from tests.parity import assert_close

    if new_rows is not None:
        kn_all, vn_all, sm_all = (t.cpu() for t in new_rows)
        sm_list = sm_all.tolist()

    B = q.shape[0]
    ps = k_cache.shape[1]
    lens = context_lens.cpu().tolist()
    bt = block_table.cpu()
    worst = (0.0, 0.0)
    view8 = k_cache.dtype == torch.float8_e4m3fn
    for r0 in range(0, B, chunk):
        rows = list(range(r0, min(B, r0 + chunk)))
        n_pages = [ring_pages if ring_pages else (max(lens[b], 0) + ps - 1) // ps for b in rows]
        pages, tables = [], []
        for b, n in zip(rows, n_pages):
            tables.append(list(range(len(pages), len(pages) + n)))
            pages += bt[b, :n].tolist()
        idx = torch.tensor(pages or [0], dtype=torch.long, device=k_cache.device)
        kc = k_cache.index_select(0, idx).cpu()
        vc = v_cache.index_select(0, idx).cpu()
        if view8:
            kc, vc = kc.view(torch.uint8).numpy(), vc.view(torch.uint8).numpy()
        sub_bt = torch.full((len(rows), max(1, max(len(t) for t in tables))), -1,
                            dtype=torch.int32)
        for i, t in enumerate(tables):
            if t:
                sub_bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
        qs = q[rows].cpu()
        cl = torch.tensor([lens[b] for b in rows], dtype=torch.int32)
        if k_scales is not None:
            ks = k_scales.index_select(0, idx.to(k_scales.device)).cpu()
            vs = v_scales.index_select(0, idx.to(v_scales.device)).cpu()
        if new_rows is not None:
            # the step's rows that land on this chunk's pages, renumbered
            where = {pg: i for i, pg in enumerate(pages)}
            sub_sm = torch.tensor([where[s // ps] * ps + s % ps if s >= 0 and s // ps in where
                                   else -1 for s in sm_list], dtype=torch.int64)
            if k_scales is not None:
                oracle.kv_cache_write_int8(kn_all, vn_all, kc, vc, ks, vs, sub_sm)
            elif view8:
                oracle.kv_cache_write_fp8(kn_all, vn_all, kc, vc, sub_sm)
            else:
                oracle.kv_cache_write(kn_all, vn_all, kc, vc, sub_sm)
        if k_scales is not None:
            ref = oracle.paged_decode_int8(qs, kc, vc, ks, vs, sub_bt, cl, scale, window=window,
                                           ring_pages=ring_pages)
        else:
            ref = oracle.paged_decode(qs, kc, vc, sub_bt, cl, scale, window=window,
                                      ring_pages=ring_pages)
        e, r = assert_close(out[rows], ref, f"{what}, sequences {rows[0]}..{rows[-1]}")
        worst = (max(worst[0], e), max(worst[1], r))
    return worst


def assert_prefill_rows(out, g, rows, window=None, ring_pages=0, what="prefill", pools=None,
                        new_rows=None):
    """Every token of the given prefill rows against the oracle's blockwise
    fold (pads: exactly 0).  pools = (k_cache, v_cache) before the call's
    write (default: g's), and new_rows = (k_new, v_new, slot_mapping) the
    rows the oracle writes into its own copies first."""
    from tests.parity import assert_close

    k_src, v_src = (g.k_cache, g.v_cache) if pools is None else pools
    ps = k_src.shape[1]
    w = g.window if window is None else window
    if new_rows is not None:
        kn_all, vn_all, sm_all = (t.cpu() for t in new_rows)
        sm_list = sm_all.tolist()
    for row in rows:
        pos = g.positions[row].cpu()
        last = int(pos.max().item())
        n = ring_pages if ring_pages else max((last + ps) // ps, 1)
        kc, vc, bt = sub_pool(k_src, v_src, g.block_table, [row], [n])
        if new_rows is not None:
            pages = g.block_table[row, :n].cpu().tolist()
            where = {pg: i for i, pg in enumerate(pages)}
            sub_sm = torch.tensor([where[s // ps] * ps + s % ps if s >= 0 and s // ps in where
                                   else -1 for s in sm_list], dtype=torch.int64)
            if kc.dtype == torch.float8_e4m3fn:
                k8, v8 = kc.view(torch.uint8).numpy(), vc.view(torch.uint8).numpy()
                oracle.kv_cache_write_fp8(kn_all, vn_all, k8, v8, sub_sm)
            else:
                oracle.kv_cache_write(kn_all, vn_all, kc, vc, sub_sm)
        if kc.dtype == torch.float8_e4m3fn:
            kc, vc = kc.view(torch.uint8).numpy(), vc.view(torch.uint8).numpy()
        ref = oracle.paged_prefill(g.q[row:row + 1].cpu(), kc, vc, bt, pos.view(1, -1), g.scale,
                                   window=w, ring_pages=ring_pages)
        assert_close(out[row], ref, f"{what}, row {row}")
        dead = (pos < 0).nonzero().flatten().tolist()
        if dead:
            assert torch.all(out[row, dead] == 0), f"{what}, row {row}: pads not 0"
