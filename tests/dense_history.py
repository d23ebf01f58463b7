"""Small cases built from contiguous per-sequence K/V histories.

Each sequence's keys and values are first drawn as one contiguous array over
its positions; the paged pool is then filled by placing position j of sequence
b at its page's slot.  Attention over the contiguous history with library
routines (matrix products and scipy's softmax) is then an independent check of
anything that reads the paged pool: it shares neither the page arithmetic nor
the loops.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List

import numpy as np
import scipy.special
import torch


def round_to(x: np.ndarray, dtype: torch.dtype):
    """(stored bits or float32 array, exact float64 values) of x rounded to dtype."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dtype)
    vals = t.double().numpy()
    if dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16), vals
    return t.numpy(), vals


@dataclass
class HistoryCase:
    lengths: List[int]
    Hq: int
    Hkv: int
    d: int
    page_size: int
    dtype: torch.dtype
    scale: float
    hist_k: List[np.ndarray]  # exact float64 values, [L, Hkv, d]
    hist_v: List[np.ndarray]
    k_cache: np.ndarray  # stored form, [P, ps, Hkv, d]
    v_cache: np.ndarray
    block_table: np.ndarray  # [B, max_pages] int32
    pages_of: List[List[int]]


def history_case(lengths, Hq, Hkv, d, page_size, dtype=torch.float32, seed=0, extra_pages=3,
                 garbage=1.0) -> HistoryCase:
    rng = np.random.default_rng(seed)
    B = len(lengths)
    need = [(L + page_size - 1) // page_size for L in lengths]
    P = sum(need) + extra_pages
    perm = rng.permutation(P).tolist()
    width = max(max(need), 1)
    bt = np.full((B, width), -1, dtype=np.int32)
    pages_of, off = [], 0
    for b, n in enumerate(need):
        pages_of.append(perm[off:off + n])
        bt[b, :n] = pages_of[-1]
        off += n
    # garbage everywhere first (finite), then the histories on their slots
    kc_f = garbage * rng.standard_normal((P, page_size, Hkv, d))
    vc_f = garbage * rng.standard_normal((P, page_size, Hkv, d))
    hist_k, hist_v = [], []
    for b, L in enumerate(lengths):
        hk = rng.standard_normal((L, Hkv, d))
        hv = rng.standard_normal((L, Hkv, d))
        for j in range(L):
            pg = pages_of[b][j // page_size]
            kc_f[pg, j % page_size] = hk[j]
            vc_f[pg, j % page_size] = hv[j]
        hist_k.append(hk)
        hist_v.append(hv)
    kc, kc_vals = round_to(kc_f, dtype)
    vc, vc_vals = round_to(vc_f, dtype)
    # exact values of the histories after rounding, read back from the rounded pool
    hk_r, hv_r = [], []
    for b, L in enumerate(lengths):
        hk_r.append(np.stack([kc_vals[pages_of[b][j // page_size], j % page_size]
                              for j in range(L)]) if L else np.zeros((0, Hkv, d)))
        hv_r.append(np.stack([vc_vals[pages_of[b][j // page_size], j % page_size]
                              for j in range(L)]) if L else np.zeros((0, Hkv, d)))
    return HistoryCase(list(lengths), Hq, Hkv, d, page_size, dtype, 1.0 / math.sqrt(d), hk_r,
                       hv_r, kc, vc, bt, pages_of)


def dense_attention(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float):
    """softmax(scale * keys @ q) @ values over a contiguous key list (float64)."""
    if keys.shape[0] == 0:
        return np.zeros(values.shape[-1])
    s = scale * (keys @ q)
    return scipy.special.softmax(s) @ values


def dense_reference(case: HistoryCase, q_vals: np.ndarray, b: int, p: int, window: int = 0):
    """[Hq, d] output of a query of sequence b at position p (q_vals [Hq, d])."""
    group = case.Hq // case.Hkv
    lo = 0 if window <= 0 else max(0, p - window + 1)
    out = np.zeros((case.Hq, case.d))
    if p < 0:
        return out
    for h in range(case.Hq):
        g = h // group
        out[h] = dense_attention(q_vals[h], case.hist_k[b][lo:p + 1, g, :],
                                 case.hist_v[b][lo:p + 1, g, :], case.scale)
    return out
