"""The decode plan's piece arithmetic, restated on the host: every sequence's
chunk range [0, n) is tiled exactly by its bulk pieces and then its small
pieces, and a batch never gets more pieces than the workspace holds,
ceil(6144 / H_kv) + 2B (the plan kernel also refuses such a batch on the
device, with TL_DEVERR_PLAN_CAPACITY).  The constants are the build's
defaults: a target of 6,144 work items, a tail of 15% of every sequence of at
least 16 chunks in small pieces of 4 chunks, bulk pieces of at least 8."""
import numpy as np
import pytest

K_TARGET, K_MIN_SPLIT, K_SMALL, K_TAIL_PCT = 6144, 8, 4, 15


def cdiv(a, b):
    return -(-a // b)


def tail(n):
    return 0 if n < 2 * K_MIN_SPLIT else min(n, (K_TAIL_PCT * n + 99) // 100)


def plan(ns, h_kv):
    """(pieces of each sequence as (first chunk, end chunk) lists, split, small)."""
    target = cdiv(K_TARGET, h_kv)
    B, C, T = len(ns), sum(ns), sum(tail(n) for n in ns)
    half = max(target // 2, 1)
    small = max(K_SMALL, cdiv(T + B, half))
    TP = sum(cdiv(tail(n), small) for n in ns)
    budget = target + B - TP
    assert budget > 0
    split = max(K_MIN_SPLIT, cdiv(C - T, budget))
    out = []
    for n in ns:
        t = tail(n)
        bulk = [(k * split, min(n - t, (k + 1) * split)) for k in range(cdiv(n - t, split))]
        smalls = [(n - t + k * small, min(n, n - t + (k + 1) * small)) for k in range(cdiv(t, small))]
        out.append(bulk + smalls)
    return out, split, small


def check(ns, h_kv):
    pieces, _, _ = plan(ns, h_kv)
    for n, ps in zip(ns, pieces):
        x = 0
        for a, e in ps:
            assert a == x and e > a, (n, ps)
            x = e
        assert x == n
    total = sum(len(ps) for ps in pieces)
    assert total <= cdiv(K_TARGET, h_kv) + 2 * len(ns), (total, len(ns), h_kv)
    return total


def test_plan_tiles_and_bound_on_a_seeded_sweep():
    rng = np.random.default_rng(1)
    for _ in range(3000):
        B = int(rng.choice([1, 2, 7, 64, 128, 129, 256, 1024, 4096]))
        h_kv = int(rng.choice([1, 2, 4, 8, 16]))
        mx = int(rng.choice([1, 8, 40, 600, 8192, 131072 // 16]))
        check(rng.integers(0, mx + 1, B).tolist(), h_kv)


@pytest.mark.parametrize("ns", [[0] * 5, [1], [131072 // 16], [15, 16, 17], [8192] * 64,
                                [1] * 20000, [131072 // 16] * 3 + [0] * 500])
def test_plan_extremes(ns):
    for h_kv in (1, 8):
        check(ns, h_kv)


def test_llama_layer_plan():
    """The bench's Llama-3-8B layer (B=64, lengths 512-8192, 8 KV heads): bulk
    pieces of 38 chunks, a last round of 8-chunk pieces (the small-piece count
    is held to half the target plus B), 857 pieces = 6,856 work items."""
    from paged_kv_attention_cache_gb300 import workloads as wl
    ns = [(L - 1) // 16 + 1 for L in wl.llama8b_lengths(seed=0, B=64)]
    pieces, split, small = plan(ns, 8)
    assert (split, small, sum(len(p) for p in pieces)) == (38, 8, 857)
