"""tcgen05.mma issue cost by shape on this GPU: cycles of the tensor pipe per
K16 MMA issued back to back from one thread (csrc/probe_mma.cu, built as its
own library beside the default one).  Prints one JSON line: per form, the
marginal cycles per MMA, (t(160) - t(32)) / 128 (patterns of three groups:
(t(192) - t(48)) / 144) with the best of three runs of each, and the multiply-adds per cycle that implies.

    python -m paged_kv_attention_cache_gb300.probe_mma
"""
from __future__ import annotations

import ctypes
import json

from . import build

FORMS = [  # (name, M, N)
    ("SS N=128 bf16", 128, 128), ("TS N=128 fp16", 128, 128), ("SS N=256 bf16", 128, 256),
    ("TS N=256 fp16", 128, 256), ("SS N=128, two accumulators", 128, 128),
    ("SS N=64", 128, 64), ("SS N=192", 128, 192), ("SS M=64 N=128", 64, 128),
    ("SS N=32", 128, 32),
    ("attention order: PV0, S0, PV1, S1 in groups of 8", 128, 128),
    ("attention order, TMEM loads by 3 warps meanwhile", 128, 128),
    ("order PV0, PV1, S0, S1 in groups of 8", 128, 128),
    ("attention order, no column shared", 128, 128),
    ("SS bf16 / SS fp16 groups alternating", 128, 128),
    ("TS bf16 / SS bf16 groups alternating", 128, 128),
    ("TS fp16 / TS bf16 groups alternating", 128, 128),
    ("groups TS, SS, SS in turn", 128, 128),
    ("groups TS, TS, SS in turn", 128, 128),
    ("one tile, Q in TMEM: S and P.V both TS", 128, 128),
    ("SS: A and D alternating (S0, S1)", 128, 128),
    ("TS: A and D alternating (PV0, PV1)", 128, 128),
    ("TS: A fixed, D alternating", 128, 128),
    ("TS: A alternating, D fixed", 128, 128),
    ("TS: D alternating, fresh accumulator per group", 128, 128),
    ("TS: A alternating, D fixed, fresh accumulator per group", 128, 128),
    ("one tile all TS, P and Q in columns no MMA writes", 128, 128),
    ("the same, fp16, S's B K-major", 128, 128),
    ("the same, S in bf16", 128, 128),
    ("all-TS fp16, every group a fresh accumulator", 128, 128),
    ("all-TS fp16, every group accumulating", 128, 128),
    ("TS, three accumulators in turn", 128, 128),
    ("TS, four accumulators in turn", 128, 128),
    ("TS, A alternating 384 / 448", 128, 128),
    ("TS, A alternating 256 / 384", 128, 128),
    ("TS, A alternating 0 / 64", 128, 128),
    ("TS, (A, D) pairs alternating, one S buffer", 128, 128),
    ("TS, (A, D) pairs, two S buffers in turn", 128, 128),
    ("the same, both B K-major, one descriptor", 128, 128),
    ("the same, P from the other S buffer", 128, 128),
    ("TS N=64 alone", 128, 64),
    ("two tiles, Q in TMEM, 64-key S, all TS", 128, 96),
    ("attention order, P.V from shared memory too (all SS)", 128, 128),
]


def probe_library() -> ctypes.CDLL:
    lib = ctypes.CDLL(build.build_variant("probe_mma", ["probe_mma.cu"], []))
    lib.tl_probe_mma_cycles.argtypes = [ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_longlong)]
    lib.tl_probe_mma_cycles.restype = ctypes.c_int
    return lib


def timed(lib, form: int, n: int, reps: int = 3):
    """(cycles, ns) of n back-to-back MMAs of `form`, the run with the fewest
    cycles of `reps`."""
    best = None
    for _ in range(reps):
        t = (ctypes.c_longlong * 2)()
        st = lib.tl_probe_mma_cycles(form, n, t)
        if st != 0 or t[0] < 0:
            raise RuntimeError(f"probe form {form} n={n}: status {st}, cycles {t[0]}")
        if best is None or t[0] < best[0]:
            best = (t[0], t[1])
    return best


def cycles(lib, form: int, n: int, reps: int = 3) -> int:
    return timed(lib, form, n, reps)[0]


def warm_up(seconds: float = 2.0) -> None:
    """Keep the GPU busy for a while first: from idle, the part reaches its
    working clocks only under sustained load, and single-CTA probes alone do
    not provide it (measured: ~25% more cycles per MMA from a cold start)."""
    import time

    import torch
    a = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    t_end = time.time() + seconds
    while time.time() < t_end:
        for _ in range(10):
            a = (a @ a).clamp_(-1.0, 1.0)
        torch.cuda.synchronize()


def main() -> None:
    lib = probe_library()
    warm_up()
    res = []
    for f, (name, M, N) in enumerate(FORMS):
        lo, hi = (48, 192) if f in (16, 17) else (32, 160)
        c0, n0 = timed(lib, f, lo)
        c1, n1 = timed(lib, f, hi)
        per = (c1 - c0) / float(hi - lo)
        res.append({"form": name, "M": M, "N": N, "K": 16, "cycles_per_mma": round(per, 1),
                    "ns_per_mma": round((n1 - n0) / float(hi - lo), 2),
                    "sm_mhz": round(c1 / n1 * 1e3) if n1 > 0 else None,
                    "fma_per_cycle": round(M * N * 16 / per, 1)})
    print(json.dumps(res))


if __name__ == "__main__":
    main()
