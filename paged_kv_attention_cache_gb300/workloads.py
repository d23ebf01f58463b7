"""Seeded synthetic inputs for the paged-attention path.

This module only draws inputs: sequence lengths, a shuffled page pool, block
tables, slot mappings, positions and N(0,1) values rounded once to the storage
dtype.  It holds none of the attention arithmetic, and both the CUDA path and
the CPU oracle consume the very same bytes it produces.

The shapes stand in for the pages' workloads (Llama-3-8B-shaped layers,
"Serving Models", "The 1 GiB example"; right-aligned prefill chunks with left
padding, "How serving works in Tlaloc", section 1; a sliding-window / full
layer mix, section 3), which in the pages are a real model's KV and need
weights.  Random values of the same shape, length mix and layout replace them.

Layout conventions (the library's):
  cache       [num_pages, page_size, H_kv, d]
  block_table [B, max_pages_per_seq] int32, unused entries -1
  slot        page * page_size + offset (int64), -1 = padding token
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

NAN_BF16_BITS = 0x7FC0

_CHUNK = 1 << 24


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn_into(out: torch.Tensor, g: torch.Generator, outlier_p: float = 0.0,
                outlier_scale: float = 8.0) -> torch.Tensor:
    """Fill `out` (any float dtype) with N(0,1) drawn in f32 and rounded once."""
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = torch.randn(e - s, generator=g, device=out.device, dtype=torch.float32)
        if outlier_p > 0:
            hit = torch.rand(e - s, generator=g, device=out.device) < outlier_p
            x = torch.where(hit, x * outlier_scale, x)
        flat[s:e].copy_(x)
    return out


def _randn(shape, dtype, g, device, outlier_p=0.0) -> torch.Tensor:
    return _randn_into(torch.empty(shape, dtype=dtype, device=device), g, outlier_p)


def _pages_for(length: int, page_size: int) -> int:
    return (int(length) + page_size - 1) // page_size


@dataclass
class PagedPool:
    """A shuffled page pool shared by B sequences, and their block tables."""
    num_pages: int
    page_size: int
    block_table: torch.Tensor  # [B, max_pages] int32, -1 unused
    pages_of: List[List[int]]  # physical pages of each sequence, in logical order

    def slot(self, b: int, position: int) -> int:
        return self.pages_of[b][position // self.page_size] * self.page_size + position % self.page_size


def make_pool(lengths: List[int], page_size: int, g: torch.Generator, extra_pages: int = 0,
              max_pages_per_seq: Optional[int] = None) -> PagedPool:
    """Pages for sequences of the given lengths, drawn from a seeded permutation."""
    need = [_pages_for(L, page_size) for L in lengths]
    total = sum(need) + extra_pages
    total = max(total, 1)
    perm = torch.randperm(total, generator=g, device=g.device).cpu().tolist()
    width = max(max(need) if need else 1, 1) if max_pages_per_seq is None else max_pages_per_seq
    bt = torch.full((len(lengths), width), -1, dtype=torch.int32)
    pages_of, off = [], 0
    for b, n in enumerate(need):
        pg = perm[off:off + n]
        off += n
        pages_of.append(pg)
        if n:
            bt[b, :n] = torch.tensor(pg, dtype=torch.int32)
    return PagedPool(total, page_size, bt, pages_of)


@dataclass
class DecodeCase:
    """One decode step: write one new K/V row per sequence (plus pads), then
    attend with one query per sequence of causal length context_lens[b]."""
    B: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    dtype: torch.dtype
    window: int
    scale: float
    context_lens: torch.Tensor  # [B] int32
    pool: PagedPool
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    q: torch.Tensor  # [B, Hq, d]
    k_new: torch.Tensor  # [N, Hkv, d]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor  # [N] int64
    extra: Dict = field(default_factory=dict)

    @property
    def block_table(self) -> torch.Tensor:
        return self.pool.block_table

    @property
    def num_pages(self) -> int:
        return self.pool.num_pages


def decode_case(lengths, *, Hq, Hkv, d, page_size=16, dtype=torch.bfloat16, window=0,
                seed=0, device="cpu", n_pad=0, extra_pages=0, outlier_p=0.0,
                nan_unused=False, scale=None, max_pages_per_seq=None) -> DecodeCase:
    g = _gen(seed, device)
    lengths = [int(x) for x in lengths]
    B = len(lengths)
    pool = make_pool(lengths, page_size, g, extra_pages, max_pages_per_seq)
    shape = (pool.num_pages, page_size, Hkv, d)
    k_cache = _randn(shape, dtype, g, device, outlier_p)
    v_cache = _randn(shape, dtype, g, device, outlier_p)
    q = _randn((B, Hq, d), dtype, g, device, outlier_p)
    # the new token of sequence b sits at position L_b - 1 (causal length L_b)
    live = [b for b in range(B) if lengths[b] > 0]
    slots = [pool.slot(b, lengths[b] - 1) for b in live] + [-1] * n_pad
    # interleave the pads among the live rows (deterministically)
    order = torch.randperm(len(slots), generator=g, device=g.device).cpu().tolist()
    slots = [slots[i] for i in order]
    N = len(slots)
    k_new = _randn((N, Hkv, d), dtype, g, device, outlier_p)
    v_new = _randn((N, Hkv, d), dtype, g, device, outlier_p)
    if nan_unused:
        _poison_unused(k_cache, v_cache, pool, lengths)
    return DecodeCase(B, Hq, Hkv, d, page_size, dtype, window,
                      1.0 / math.sqrt(d) if scale is None else scale,
                      torch.tensor(lengths, dtype=torch.int32), pool, k_cache, v_cache, q,
                      k_new, v_new, torch.tensor(slots, dtype=torch.int64))


def _poison_unused(k_cache, v_cache, pool: PagedPool, lengths) -> None:
    """Fill every slot no sequence position maps to with NaN."""
    used = torch.zeros(pool.num_pages * pool.page_size, dtype=torch.bool)
    for b, L in enumerate(lengths):
        for i, pg in enumerate(pool.pages_of[b]):
            n = min(pool.page_size, L - i * pool.page_size)
            used[pg * pool.page_size: pg * pool.page_size + n] = True
    idx = (~used).nonzero().view(-1).to(k_cache.device)
    for c in (k_cache, v_cache):
        flat = c.view(pool.num_pages * pool.page_size, -1)
        flat[idx] = float("nan")


def int8_pools(case, seed: int = 0, nan_unused: bool = False, scale_range=(0.005, 0.05),
               boost_p: float = 0.0, boost: float = 1.0):
    """Seeded int8 pools of a decode or prefill case's pool shape: codes
    uniform in [-127, 127] (int8 [P, page_size, H_kv, d]) and per-(slot, KV
    head) scales uniform in scale_range (float32 [P, H_kv, page_size]), as
    (k_codes, v_codes, k_scales, v_scales) on the CPU; each scale is then
    multiplied by `boost` with probability boost_p.  With nan_unused, every
    slot no sequence position maps to holds code -128 and scale NaN."""
    g = _gen(seed, "cpu")
    P, ps, hkv, d = case.pool.num_pages, case.page_size, case.Hkv, case.d
    codes = [torch.randint(-127, 128, (P, ps, hkv, d), generator=g, dtype=torch.int8)
             for _ in range(2)]
    lo, hi = scale_range
    scales = [torch.rand((P, hkv, ps), generator=g) * (hi - lo) + lo for _ in range(2)]
    if boost_p > 0.0:
        for sc in scales:
            sc[torch.rand(sc.shape, generator=g) < boost_p] *= boost
    if nan_unused:
        if isinstance(case, PrefillCase):
            lengths = [p0 + max(case.T - pad, 0) for p0, pad in zip(case.p0, case.pads)]
        else:
            lengths = case.context_lens.tolist()
        used = torch.zeros(P * ps, dtype=torch.bool)
        for b, L in enumerate(lengths):
            for i, pg in enumerate(case.pool.pages_of[b]):
                n = min(ps, L - i * ps)
                used[pg * ps: pg * ps + max(n, 0)] = True
        unused = (~used).view(P, ps)
        for c, sc in zip(codes, scales):
            c[unused] = -128
            sc.permute(0, 2, 1)[unused] = float("nan")
    return codes[0], codes[1], scales[0].contiguous(), scales[1].contiguous()


@dataclass
class PrefillCase:
    """One right-aligned batched prefill call: row b holds pad_b padding tokens
    (position -1, slot -1) and then n_b live tokens at positions p0_b ..
    p0_b + n_b - 1; positions below p0_b are prior context already in the pool."""
    B: int
    T: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    dtype: torch.dtype
    window: int
    scale: float
    pads: List[int]
    p0: List[int]
    positions: torch.Tensor  # [B, T] int32
    pool: PagedPool
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    q: torch.Tensor  # [B, T, Hq, d]
    k_new: torch.Tensor  # [B*T, Hkv, d]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor  # [B*T] int64

    @property
    def block_table(self) -> torch.Tensor:
        return self.pool.block_table

    @property
    def num_pages(self) -> int:
        return self.pool.num_pages


def prefill_case(pads, p0, *, T, Hq, Hkv, d, page_size=16, dtype=torch.bfloat16, window=0,
                 seed=0, device="cpu", extra_pages=0, nan_unused=False, scale=None,
                 max_pages_per_seq=None, outlier_p=0.0) -> PrefillCase:
    g = _gen(seed, device)
    pads = [int(x) for x in pads]
    p0 = [int(x) for x in p0]
    B = len(pads)
    lengths = [p0[b] + (T - pads[b]) if T - pads[b] > 0 else p0[b] for b in range(B)]
    pool = make_pool(lengths, page_size, g, extra_pages, max_pages_per_seq)
    shape = (pool.num_pages, page_size, Hkv, d)
    k_cache = _randn(shape, dtype, g, device, outlier_p)
    v_cache = _randn(shape, dtype, g, device, outlier_p)
    q = _randn((B, T, Hq, d), dtype, g, device, outlier_p)
    k_new = _randn((B * T, Hkv, d), dtype, g, device, outlier_p)
    v_new = _randn((B * T, Hkv, d), dtype, g, device, outlier_p)
    positions = torch.full((B, T), -1, dtype=torch.int32)
    slots = torch.full((B * T,), -1, dtype=torch.int64)
    for b in range(B):
        for t in range(pads[b], T):
            p = p0[b] + t - pads[b]
            positions[b, t] = p
            slots[b * T + t] = pool.slot(b, p)
    if nan_unused:
        _poison_unused(k_cache, v_cache, pool, lengths)
    return PrefillCase(B, T, Hq, Hkv, d, page_size, dtype, window,
                       1.0 / math.sqrt(d) if scale is None else scale, pads, p0, positions,
                       pool, k_cache, v_cache, q, k_new, v_new, slots)


@dataclass
class RingCase:
    """The same K/V history of B sequences in two layouts: a full-history pool
    (every position 0..L-1 on its own slot) and a ring pool of ring_pages pages
    per sequence, where logical block k sits on ring page k % ring_pages, so a
    later position overwrites the one ring_pages * page_size behind it.  The
    ring table is as wide as the full one: entry k holds the ring page of
    block k.  ring_slots / full_slots: where each sequence's last position
    (the new token) lives in each layout."""
    B: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    dtype: torch.dtype
    window: int
    ring_pages: int
    scale: float
    context_lens: torch.Tensor  # [B] int32
    q: torch.Tensor  # [B, Hq, d]
    full_k: torch.Tensor
    full_v: torch.Tensor
    full_table: torch.Tensor  # [B, width] int32
    ring_k: torch.Tensor
    ring_v: torch.Tensor
    ring_table: torch.Tensor  # [B, width] int32
    full_slots: torch.Tensor  # [B] int64
    ring_slots: torch.Tensor  # [B] int64
    k_new: torch.Tensor  # [B, Hkv, d]: the last position's K and V
    v_new: torch.Tensor


def ring_case(lengths, *, window, ring_pages, Hq, Hkv, d, page_size=16,
              dtype=torch.bfloat16, seed=0, device="cpu", outlier_p=0.0) -> RingCase:
    """Seeded histories in both layouts (see RingCase)."""
    g = _gen(seed, device)
    lengths = [int(x) for x in lengths]
    B = len(lengths)
    pool = make_pool(lengths, page_size, g)
    width = pool.block_table.shape[1]
    if ring_pages > width:
        raise ValueError("ring_pages is wider than the full table")
    full_k = torch.zeros((pool.num_pages, page_size, Hkv, d), dtype=dtype, device=device)
    full_v = torch.zeros_like(full_k)
    n_ring = B * ring_pages
    ring_k = torch.zeros((n_ring, page_size, Hkv, d), dtype=dtype, device=device)
    ring_v = torch.zeros_like(ring_k)
    perm = torch.randperm(n_ring, generator=g, device=g.device).cpu()
    ring_of = perm.view(B, ring_pages)
    ring_table = torch.empty((B, width), dtype=torch.int32)
    for k in range(width):
        ring_table[:, k] = ring_of[:, k % ring_pages].to(torch.int32)
    n_slots = ring_pages * page_size
    full_slots, ring_slots, k_last, v_last = [], [], [], []
    for b, L in enumerate(lengths):
        hk = _randn((L, Hkv, d), dtype, g, device, outlier_p)
        hv = _randn((L, Hkv, d), dtype, g, device, outlier_p)
        pos = torch.arange(L)
        fs = torch.tensor(pool.pages_of[b], dtype=torch.int64)[pos // page_size] * page_size + \
            pos % page_size
        full_k.view(-1, Hkv, d)[fs.to(device)] = hk
        full_v.view(-1, Hkv, d)[fs.to(device)] = hv
        # the ring keeps the last n_slots positions (older ones were overwritten)
        keep = pos[max(0, L - n_slots):]
        rs = ring_of[b][(keep // page_size) % ring_pages].to(torch.int64) * page_size + \
            keep % page_size
        ring_k.view(-1, Hkv, d)[rs.to(device)] = hk[keep.to(device)]
        ring_v.view(-1, Hkv, d)[rs.to(device)] = hv[keep.to(device)]
        full_slots.append(int(fs[-1]) if L else -1)
        ring_slots.append(int(rs[-1]) if L else -1)
        k_last.append(hk[-1] if L else torch.zeros((Hkv, d), dtype=dtype, device=device))
        v_last.append(hv[-1] if L else torch.zeros((Hkv, d), dtype=dtype, device=device))
    q = _randn((B, Hq, d), dtype, g, device, outlier_p)
    return RingCase(B, Hq, Hkv, d, page_size, dtype, window, ring_pages, 1.0 / math.sqrt(d),
                    torch.tensor(lengths, dtype=torch.int32), q, full_k, full_v,
                    pool.block_table.clone(), ring_k, ring_v, ring_table,
                    torch.tensor(full_slots, dtype=torch.int64),
                    torch.tensor(ring_slots, dtype=torch.int64),
                    torch.stack(k_last), torch.stack(v_last))


# ----------------------------------------------------------------- presets --

def tiny_decode(seed=0, device="cpu") -> DecodeCase:
    """B=2, Hq=4, Hkv=2, d=64, pages of 16, lengths {37, 100}, a pool of 16
    shuffled pages, f32; one new token per sequence plus one padding token."""
    return decode_case([37, 100], Hq=4, Hkv=2, d=64, page_size=16, dtype=torch.float32,
                       seed=seed, device=device, n_pad=1, extra_pages=16 - 10,
                       scale=1.0 / math.sqrt(64))


def llama8b_lengths(seed=0, B=64):
    g = _gen(seed + 1000, "cpu")
    return torch.randint(512, 8193, (B,), generator=g).tolist()


def llama8b_decode(seed=0, device="cpu", B=64) -> DecodeCase:
    """Llama-3-8B-shaped layer: Hq=32, Hkv=8, d=128, bf16, lengths U[512, 8192]."""
    return decode_case(llama8b_lengths(seed, B), Hq=32, Hkv=8, d=128, page_size=16,
                       dtype=torch.bfloat16, seed=seed, device=device)


def prefill_rows(seed=0, B=8, T=2048, max_pad=1500, max_p0=6144):
    g = _gen(seed + 2000, "cpu")
    pads = torch.randint(0, max_pad + 1, (B,), generator=g).tolist()
    p0 = torch.randint(0, max_p0 + 1, (B,), generator=g).tolist()
    return pads, p0


def batched_prefill(seed=0, device="cpu", B=8, T=2048, outlier_p=0.0) -> PrefillCase:
    """B=8 rows of 2,048 tokens, 0-1,500 left pads, prior context 0-6,144,
    Hq=32, Hkv=8, d=128, bf16, pages of 16 (outlier_p: that share of Q, K and
    V values multiplied by 8, as in the sliding-window mix)."""
    pads, p0 = prefill_rows(seed, B, T)
    return prefill_case(pads, p0, T=T, Hq=32, Hkv=8, d=128, page_size=16,
                        dtype=torch.bfloat16, seed=seed, device=device, outlier_p=outlier_p)


def swa_lengths(seed=0, B=128):
    g = _gen(seed + 3000, "cpu")
    return torch.randint(1024, 32769, (B,), generator=g).tolist()


def swa_decode(seed=0, device="cpu", B=128, layer=0) -> DecodeCase:
    """Sliding-window mix: Hq=40, Hkv=8, d=128, bf16, lengths U[1024, 32768];
    layer 0 has window 4,096, layer 1 full attention; 1% of values x8."""
    return decode_case(swa_lengths(seed, B), Hq=40, Hkv=8, d=128, page_size=16,
                       dtype=torch.bfloat16, window=4096 if layer == 0 else 0,
                       seed=seed + 17 * layer, device=device, outlier_p=0.01)


def swa_ring_decode(seed=0, device="cpu", B=128, window=4096, ring_pages=None) -> DecodeCase:
    """The sliding-window layer of the mix over a windowed pool: each sequence
    holds a ring of ring_pages pages (default ceil(window / 16) + 1, the
    pages' default of one spare page) with random contents, lengths
    U[1024, 32768] (most rings have wrapped), Hq=40, Hkv=8, d=128, bf16, 1%
    of values x8.  The table is ring_pages wide; the new token of sequence b
    goes to the ring slot of position L_b - 1 (logical block k on ring page
    k % ring_pages).  extra["ring_pages"] holds the ring size."""
    ps, hkv, d, hq = 16, 8, 128, 40
    ring = ring_pages or (window + ps - 1) // ps + 1
    g = _gen(seed + 4000, device)
    lengths = swa_lengths(seed, B)
    n_pages = B * ring
    perm = torch.randperm(n_pages, generator=g, device=g.device).cpu()
    table = perm.view(B, ring).to(torch.int32).contiguous()
    pages_of = [table[b].tolist() for b in range(B)]
    pool = PagedPool(n_pages, ps, table, pages_of)
    shape = (n_pages, ps, hkv, d)
    k_cache = _randn(shape, torch.bfloat16, g, device, 0.01)
    v_cache = _randn(shape, torch.bfloat16, g, device, 0.01)
    q = _randn((B, hq, d), torch.bfloat16, g, device, 0.01)
    slots = [pages_of[b][((L - 1) // ps) % ring] * ps + (L - 1) % ps for b, L in enumerate(lengths)]
    k_new = _randn((B, hkv, d), torch.bfloat16, g, device, 0.01)
    v_new = _randn((B, hkv, d), torch.bfloat16, g, device, 0.01)
    return DecodeCase(B, hq, hkv, d, ps, torch.bfloat16, window, 1.0 / math.sqrt(d),
                      torch.tensor(lengths, dtype=torch.int32), pool, k_cache, v_cache, q,
                      k_new, v_new, torch.tensor(slots, dtype=torch.int64),
                      extra={"ring_pages": ring})


def longctx_lengths(seed=0, B=256):
    g = _gen(seed + 4000, "cpu")
    z = torch.randn(B, generator=g, dtype=torch.float64)
    L = torch.exp(math.log(2048.0) + 1.0 * z).round().clamp(64, 131072)
    return [int(x) for x in L.tolist()]


def longctx_decode(seed=0, device="cpu", B=256) -> DecodeCase:
    """Long-context batch: Hq=64, Hkv=8 (8:1), d=128, bf16, lengths lognormal
    (median 2,048, sigma 1) clipped to [64, 131072]."""
    return decode_case(longctx_lengths(seed, B), Hq=64, Hkv=8, d=128, page_size=16,
                       dtype=torch.bfloat16, seed=seed, device=device)


def to_device(case, device):
    """A copy of a case with every tensor moved to `device` (tables stay int32/int64)."""
    import copy
    c = copy.copy(case)
    for name, val in vars(case).items():
        if isinstance(val, torch.Tensor):
            setattr(c, name, val.to(device))
    pool = copy.copy(case.pool)
    pool.block_table = case.pool.block_table.to(device)
    c.pool = pool
    return c
