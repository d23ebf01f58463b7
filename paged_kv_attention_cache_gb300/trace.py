"""Decode timeline: where a decode call's time goes between its launches.

Builds the library with -DTL_DECODE_TRACE=1 (a variant beside the default
build, _build/variants/decode_trace/libtlpa.so), loads it in place of the
default one, runs decode calls over a synthetic Llama-3-8B-shaped layer
(H_q=32, H_kv=8, d=128, pages of 16) and prints one JSON line: the median over
the calls of each phase stamp, in microseconds from the plan kernel's first
instruction (the header's TL_TRACE_* slots), and the spans between them.

    python -m paged_kv_attention_cache_gb300.trace --batch 64
    python -m paged_kv_attention_cache_gb300.trace --batch 4 --length 32768 --dtype e4m3

The stamps are %globaltimer reads on the GPU; the traced build adds a few
stores and atomics and one barrier per plan and combine CTA, nothing else, so
its times run a little above the default build's.

With --prefill it builds the library with -DTL_PREFILL_TRACE=1 instead (and
with --all-ts also -DTL_PREFILL_ALL_TS=1, the all-TS attention kernel) and
runs prefill calls over the B=8 x 2,048-token batch (0-1,500 left pads, prior
context 0-6,144, Llama-3-8B heads; the cache write of the chunk first), then
prints, over the attention CTAs, the cycles per 128-key step (both query
tiles' S and P.V over one key tile) and the share of the MMA issuer's cycles
spent waiting for the softmax's P and for the producer's K / V tiles.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import statistics

import torch

from . import _lib, build

PHASES = ("plan_start", "plan_placed", "plan_end", "attn_released", "attn_first_stage",
          "attn_end", "combine_start", "combine_end")


def build_trace_library(force: bool = False) -> str:
    return build.build_variant("decode_trace", build.SOURCES, ["TL_DECODE_TRACE=1"], force=force)


def read_stamps(lib) -> list:
    buf = (ctypes.c_uint64 * len(PHASES))()
    st = lib.tl_decode_trace_read(buf, len(PHASES))
    if st != 0:
        raise RuntimeError(f"tl_decode_trace_read: {lib.tl_status_string(st).decode()}")
    return [int(x) for x in buf]


def timeline(stamps: list) -> dict:
    """Phase times in us from the plan's start (None where a phase left no
    stamp: the pieces-placed stamp of the block-wide plan, or a call that
    launched no combine), and the spans between them."""
    t0 = stamps[0]
    out = {}
    for name, t in zip(PHASES, stamps):
        out[name] = None if t in (0, 2**64 - 1) or t < t0 else (t - t0) / 1e3
    spans = {"plan": ("plan_start", "plan_end"), "release_gap": ("plan_end", "attn_released"),
             "first_stage_latency": ("attn_released", "attn_first_stage"),
             "attention": ("attn_released", "attn_end"),
             "combine_gap": ("attn_end", "combine_start"),
             "combine": ("combine_start", "combine_end")}
    for name, (a, b) in spans.items():
        out[name] = None if out[a] is None or out[b] is None else out[b] - out[a]
    return out


def trace_calls(call, lib, calls: int, warmup: int = 2) -> dict:
    """Median timeline over `calls` traced calls of call() (after `warmup`)."""
    rows = []
    for i in range(warmup + calls):
        if lib.tl_decode_trace_reset() != 0:
            raise RuntimeError("tl_decode_trace_reset failed")
        call()
        if i >= warmup:
            rows.append(timeline(read_stamps(lib)))
    med = {}
    for k in rows[0]:
        vals = [r[k] for r in rows if r[k] is not None]
        med[k] = round(statistics.median(vals), 3) if vals else None
    return med


def build_prefill_trace_library(force: bool = False, all_ts: bool = False) -> str:
    """The prefill trace build; all_ts: with the all-TS attention kernel
    (-DTL_PREFILL_ALL_TS=1) in place of the paired SS/TS one."""
    if all_ts:
        return build.build_variant("prefill_trace_all_ts", build.SOURCES,
                                   ["TL_PREFILL_TRACE=1", "TL_PREFILL_ALL_TS=1"], force=force)
    return build.build_variant("prefill_trace", build.SOURCES, ["TL_PREFILL_TRACE=1"],
                               force=force)


PTRACE_FIELDS = ("cycles", "steps", "items", "wait_p", "wait_kv", "sm_wait_s", "sm_busy")


def prefill_step_summary(rows: list) -> dict:
    """Per-CTA rows of the prefill trace (CTAs that ran no item skipped) as
    the median and spread of the cycles per step and the waits' shares."""
    live = [r for r in rows if r[1] > 0]
    per_step = sorted(r[0] / r[1] for r in live)
    tot = sum(r[0] for r in live)
    steps = sum(r[1] for r in live)
    return {"ctas": len(live), "steps": steps,
            "items": sum(r[2] for r in live),
            "cycles_per_step_median": round(statistics.median(per_step), 1),
            "cycles_per_step_min": round(per_step[0], 1),
            "cycles_per_step_max": round(per_step[-1], 1),
            "wait_p_share": round(sum(r[3] for r in live) / tot, 4),
            "wait_kv_share": round(sum(r[4] for r in live) / tot, 4),
            # per query tile and step: the softmax's wait for S and its work
            # from S's arrival to P's release
            "softmax_wait_s_per_tile": round(sum(r[5] for r in live) / (2 * steps), 1),
            "softmax_busy_per_tile": round(sum(r[6] for r in live) / (2 * steps), 1)}


def trace_prefill(args) -> dict:
    lib = _lib.load(path=build_prefill_trace_library(all_ts=args.all_ts))
    from . import api
    from . import workloads as wl

    dev = torch.device("cuda")
    case = wl.batched_prefill(seed=args.seed, device=dev)
    g = wl.to_device(case, dev)
    ws = api.alloc_workspace(api.tl_paged_attn_prefill_workspace_size(
        case.B, case.T, case.Hq, case.Hkv, case.d, case.block_table.shape[1], case.page_size), dev)
    out = torch.empty((case.B, case.T, case.Hq, case.d), dtype=torch.float32, device=dev)
    api.tl_kv_cache_write(g.k_new.view(-1, case.Hkv, case.d), g.v_new.view(-1, case.Hkv, case.d),
                          g.k_cache, g.v_cache, g.slot_mapping)
    n_ctas = torch.cuda.get_device_properties(dev).multi_processor_count
    res = []
    for i in range(2 + args.calls):
        if lib.tl_prefill_trace_reset() != 0:
            raise RuntimeError("tl_prefill_trace_reset failed")
        api.tl_paged_attn_prefill(g.q, g.k_cache, g.v_cache, g.block_table, g.positions,
                                  case.scale, out=out, workspace=ws)
        buf = (ctypes.c_uint64 * (len(PTRACE_FIELDS) * n_ctas))()
        st = lib.tl_prefill_trace_read(buf, n_ctas)
        if st != 0:
            raise RuntimeError(f"tl_prefill_trace_read: {lib.tl_status_string(st).decode()}")
        if i >= 2:
            rows = [list(buf[k * len(PTRACE_FIELDS):(k + 1) * len(PTRACE_FIELDS)])
                    for k in range(n_ctas)]
            res.append(prefill_step_summary(rows))
    med = {k: statistics.median(r[k] for r in res) for k in res[0]}
    med.update(workload="B=8 x T=2048 prefill batch, Hq=32, Hkv=8, d=128, bf16", calls=args.calls,
               kernel="all-TS (one query tile: steps are tile-steps)" if args.all_ts
               else "paired SS/TS (steps cover both query tiles)")
    return med


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--prefill", action="store_true",
                    help="the prefill step trace instead of the decode timeline")
    ap.add_argument("--all-ts", action="store_true",
                    help="with --prefill: trace the all-TS attention kernel (a build option)")
    ap.add_argument("--batch", type=int, default=64)
    ap.add_argument("--length", type=int, default=0,
                    help="every sequence this long (default: the Llama-3-8B step's mix)")
    ap.add_argument("--dtype", choices=("bf16", "e4m3", "int8"), default="bf16")
    ap.add_argument("--calls", type=int, default=10)
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args(argv)
    if args.prefill:
        print(json.dumps(trace_prefill(args)))
        return

    lib = _lib.load(path=build_trace_library())
    from . import api
    from . import workloads as wl

    dev = torch.device("cuda")
    lens = [args.length] * args.batch if args.length else wl.llama8b_lengths(args.seed, args.batch)
    case = wl.to_device(wl.decode_case(lens, Hq=32, Hkv=8, d=128, seed=args.seed + 3,
                                       device=dev), dev)
    B, hq, hkv, d = args.batch, 32, 8, 128
    ws = api.alloc_workspace(api.tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    out = torch.empty((B, hq, d), dtype=torch.float32, device=dev)
    if args.dtype == "int8":
        kc, vc, ks, vs = (t.to(dev) for t in wl.int8_pools(case, args.seed))

        def call():
            api.tl_paged_attn_decode_int8(case.q, kc, vc, ks, vs, case.block_table,
                                          case.context_lens, case.scale, out=out, workspace=ws)
    else:
        kc, vc = case.k_cache, case.v_cache
        if args.dtype == "e4m3":
            kc, vc = kc.float().to(torch.float8_e4m3fn), vc.float().to(torch.float8_e4m3fn)

        def call():
            api.tl_paged_attn_decode(case.q, kc, vc, case.block_table, case.context_lens,
                                     case.scale, out=out, workspace=ws)
    res = trace_calls(call, lib, args.calls)
    per_key = {"bf16": 2 * d, "e4m3": d, "int8": d + 4}[args.dtype]  # K or V, one KV head
    kv_bytes = sum(lens) * hkv * per_key * 2
    res.update(batch=B, dtype=args.dtype, kv_bytes=kv_bytes, unit="us",
               lengths="llama8b mix" if not args.length else args.length)
    print(json.dumps(res))


if __name__ == "__main__":
    main()
