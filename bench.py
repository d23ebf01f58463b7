"""Benchmark: paged decode KV-read GB/s (and prefill TFLOP/s) on GB300.

One step = one pass of the decode hot path over one batch: KV_CACHE_WRITE of
the batch's new tokens, then paged-attention decode (plan + split-K kernel +
combine), on the Llama-3-8B-shaped layer (B=64, H_q=32, H_kv=8, d=128, bf16,
pages of 16, context lengths U[512, 8192], shuffled pool), through
tl_paged_attn_decode_write (the write runs inside the decode call's first
launch).  value = KV bytes the decode must read (sum over sequences of
L * 2 * H_kv * d * 2 bytes) per second.  The same step as the two separate
calls is reported too ("separate_step"), and the roofline is the decode call
timed on its own.  The batched-prefill workload (B=8 rows of 2,048 tokens) is timed
after it and reported under "prefill" in TFLOP/s.

--impl reference times the CPU oracle (the plain C double-precision
definition) on the same workload and metric on the host cores.

Multi-GPU (torchrun, one process per GPU): replicas only, every rank runs its
own batch (weak scaling); the only collective is the max of the timings.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0
METRIC = "paged decode KV-read GB/s (% of HBM peak); prefill TFLOP/s (% TC peak)"
WORKLOAD = "Llama-3-8B-shaped decode layer: B=64, Hq=32, Hkv=8, d=128, bf16, page 16, L~U[512,8192]"
# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu capture of
# these default workloads (the summaries under profiles/ give the command); they hold
# only for the kernels as they were captured and for these workloads.
DECODE_TRAFFIC = (1264400640 + 2854912, "profiles/decode_bf16_llama8b_b64.md")
PREFILL_TRAFFIC = (326684160 + 206615296, "profiles/prefill_tc_batched_b8.md")
WRITE_TRAFFIC = (40167168 + 2732032, "profiles/kv_cache_write_prefill_chunk_16k.md")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except Exception:
        return HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_over_ranks(elapsed_ms: float, units: float, device="cpu"):
    """(max elapsed over ranks, sum of units over ranks); identity on one process."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(elapsed_ms), float(units)
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def kv_bytes(lengths, window, hkv, d, elem):
    tot = 0
    for L in lengths:
        n = min(L, window) if window > 0 else L
        tot += max(n, 0) * 2 * hkv * d * elem
    return tot


def prefill_flops(positions, hq, d, window=0):
    import torch
    p = positions.to(torch.int64)
    live = p >= 0
    n = p + 1
    if window > 0:
        n = torch.clamp(n, max=window)
    return int((4 * hq * d * n[live]).sum().item())


# ------------------------------------------------------------------ ours --

def run_ours(args):
    import torch
    import torch.distributed as dist

    import paged_kv_attention_cache_gb300 as tl
    from paged_kv_attention_cache_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tl.build_library()
    stream = torch.cuda.current_stream()

    # ---- decode workload, resident in HBM
    case = wl.llama8b_decode(seed=args.seed + rank, device=dev, B=args.batch)
    g = wl.to_device(case, dev)
    B, hq, hkv, d = case.B, case.Hq, case.Hkv, case.d
    lengths = case.context_lens.tolist()
    kvb = kv_bytes(lengths, case.window, hkv, d, 2)
    q_bytes = B * hq * d * 2
    bt_bytes = sum((L + 15) // 16 for L in lengths) * 4
    ws = tl.alloc_workspace(tl.tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    out = torch.empty((B, hq, d), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        """One decode step through the fused call: the write of the 64 new
        rows and the decode, tl_paged_attn_decode_write (three kernels)."""
        tl.tl_paged_attn_decode_write(g.q, g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache,
                                      g.block_table, g.context_lens, case.scale, out=out,
                                      workspace=ws, error_word=err)

    def write():
        tl.tl_kv_cache_write(g.k_new, g.v_new, g.k_cache, g.v_cache, g.slot_mapping,
                             error_word=err)

    def decode():
        tl.tl_paged_attn_decode(g.q, g.k_cache, g.v_cache, g.block_table, g.context_lens,
                                case.scale, out=out, workspace=ws, error_word=err)

    for _ in range(args.warmup):
        step()
        write()
        decode()
    torch.cuda.synchronize()
    dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_start, s_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # keep the same load running around the timed region so the sampler
        # (100 ms period) has readings under it
        t_end = time.time() + args.soak_seconds
        while time.time() < t_end:
            for _ in range(20):
                step()
            torch.cuda.synchronize()
        # the timed region: args.steps fused steps
        start.record(stream)
        for _ in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
        # the same steps as the two separate calls, the decode call timed on
        # its own (the roofline's kernel)
        s_start.record(stream)
        for i in range(args.steps):
            write()
            dec_ev[i][0].record(stream)
            decode()
            dec_ev[i][1].record(stream)
        s_stop.record(stream)
        torch.cuda.synchronize()
        t_end = time.time() + (0.5 if args.soak_seconds > 0 else 0.0)
        while time.time() < t_end:
            for _ in range(20):
                step()
            torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during the timed decode steps")
    elapsed_ms = start.elapsed_time(stop)
    sep_ms = s_start.elapsed_time(s_stop) / args.steps
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in dec_ev)
    elapsed_ms, total_kvb = reduce_over_ranks(elapsed_ms, kvb, dev)
    ms_per_step = elapsed_ms / args.steps
    value = total_kvb / (ms_per_step * 1e-3) / 1e9

    e2e = None
    # ---- end to end through the public API, inputs from pinned host memory.
    # A step's inputs travel as one staged buffer (one host->device copy per
    # step) into one of two device slots: step k+1's copy runs on a copy
    # stream while step k computes, and step k's output is read back on the
    # copy stream once step k is done.  Every step's copies are inside the
    # timed region.
    if args.only in ("all", "decode-e2e"):
        names = ("q", "k_new", "v_new", "slot_mapping", "context_lens", "block_table")
        src_t = {n: getattr(case, n).cpu().contiguous() for n in names}
        offs, total = {}, 0
        for n in names:
            offs[n] = total
            total += (src_t[n].numel() * src_t[n].element_size() + 255) // 256 * 256
        host_buf = torch.zeros(total, dtype=torch.uint8).pin_memory()
        for n in names:
            nb = src_t[n].numel() * src_t[n].element_size()
            host_buf[offs[n]:offs[n] + nb].copy_(src_t[n].view(-1).view(torch.uint8))
        dev_buf = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]

        def view(slot, n):
            t = src_t[n]
            nb = t.numel() * t.element_size()
            return dev_buf[slot][offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)

        dev_in = [{n: view(slot, n) for n in names} for slot in range(2)]
        outs = [torch.empty((B, hq, d), dtype=torch.float32, device=dev) for _ in range(2)]
        out_host = [torch.empty((B, hq, d), dtype=torch.float32).pin_memory() for _ in range(2)]
        h2d = sum(src_t[n].numel() * src_t[n].element_size() for n in names)
        d2h = out_host[0].numel() * 4
        cstream = torch.cuda.Stream(device=dev)
        landed = [torch.cuda.Event() for _ in range(2)]    # slot's inputs are on the device
        consumed = [torch.cuda.Event() for _ in range(2)]  # slot's step is done with them
        read = [torch.cuda.Event() for _ in range(2)]      # slot's output is back on the host

        def copy_in(k):
            slot = k % 2
            cstream.wait_event(consumed[slot])
            with torch.cuda.stream(cstream):
                dev_buf[slot].copy_(host_buf, non_blocking=True)
            landed[slot].record(cstream)

        def e2e_step(k):
            slot = k % 2
            x = dev_in[slot]
            stream.wait_event(landed[slot])
            stream.wait_event(read[slot])  # the slot's previous output has been read
            tl.tl_paged_attn_decode_write(x["q"], x["k_new"], x["v_new"], x["slot_mapping"],
                                          g.k_cache, g.v_cache, x["block_table"],
                                          x["context_lens"], case.scale, out=outs[slot],
                                          workspace=ws)
            consumed[slot].record(stream)
            cstream.wait_event(consumed[slot])
            with torch.cuda.stream(cstream):
                out_host[slot].copy_(outs[slot], non_blocking=True)
            read[slot].record(cstream)

        def e2e_run(n):
            copy_in(0)
            for k in range(n):
                if k + 1 < n:
                    copy_in(k + 1)
                e2e_step(k)
            stream.wait_stream(cstream)  # the last output read ends the run

        e2e_run(args.warmup)
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        e2e_run(args.steps)
        e2.record(stream)
        torch.cuda.synchronize()
        assert torch.equal(out_host[(args.steps - 1) % 2], outs[(args.steps - 1) % 2].cpu())
        e2e_ms, _ = reduce_over_ranks(s2.elapsed_time(e2) / args.steps, 0, dev)
        e2e = {"value": round(total_kvb / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "pipeline": "one staged host->device copy per step, step k+1's copy and step "
                           "k's output read on a second stream while the next step computes"}

    hbm, bf16, bf16_sus, src = peaks()
    dec_alg = kvb + q_bytes + bt_bytes + B * hq * d * 4
    achieved = dec_alg / (dec_ms * 1e-3) / 1e9
    prefill_line, write_line, ring_line = None, None, None
    if args.only in ("all", "prefill"):
        prefill_line, write_line = run_prefill(args, rank, dev, stream, hbm, bf16, bf16_sus, src)
    if args.only in ("all", "ring"):
        ring_line = run_ring(args, dev, stream, hbm)
    verify_line = None
    if args.only in ("all", "verify"):
        verify_line = run_verify(args, dev, stream, hbm, bf16)
    fp8_line = None
    if args.only in ("all", "fp8"):
        fp8_line = run_fp8(args, dev, stream, hbm)
    int8_line = None
    if args.only in ("all", "int8"):
        int8_line = run_int8(args, dev, stream, hbm)
    swa_line = run_decode_config(args, dev, stream, hbm, "swa") \
        if args.only in ("all", "swa") else None
    longctx_line = run_decode_config(args, dev, stream, hbm, "longctx") \
        if args.only in ("all", "longctx") else None
    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    cpu = cpu_baseline(case, g, args) if (args.only == "all" and not args.no_cpu_baseline) else None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) values, shuffled page pool)",
        "config": {"workload": WORKLOAD if B == 64 else WORKLOAD.replace("B=64", f"B={B}"),
                   "batch": B, "Hq": hq, "Hkv": hkv, "d_head": d,
                   "page_size": 16, "kv_bytes_per_step": kvb,
                   "l2": "inputs larger than L2 (KV pool %.2f GB vs 129 MB L2)" % (
                       g.k_cache.numel() * 4 / 1e9),
                   "parallelism": f"replicas x{world}"},
        "frac_of_hbm_peak": round(value / world / hbm, 4),
        "roofline": {"bound": "hbm", "kernel": "decode (plan + split-K bf16 kernel + combine)",
                     "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "traffic": DECODE_TRAFFIC[0] if B == 64 else None,
                     "traffic_source": DECODE_TRAFFIC[1] + " (decode_bf16_kernel alone)",
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured"
                     else "fallback", "algorithmic_bytes_per_launch": dec_alg,
                     "ms_per_launch": round(dec_ms, 5)},
        "prefill": prefill_line,
        "kv_cache_write": write_line,
        "ring_decode": ring_line,
        "verify_decode": verify_line,
        "fp8_decode": fp8_line,
        "int8_decode": int8_line,
        "swa_decode": swa_line,
        "longctx_decode": longctx_line,
        "e2e": e2e,
        "separate_step": {"calls": "tl_kv_cache_write, then tl_paged_attn_decode (four kernels)",
                          "ms_per_step": round(sep_ms, 5),
                          "gbs": round(kvb / (sep_ms * 1e-3) / 1e9, 1),
                          "frac": round(kvb / (sep_ms * 1e-3) / 1e9 / hbm, 4)},
        "cpu_baseline": cpu,
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def l2_flush_buffer(dev):
    """A buffer twice the size of L2 (129 MB); writing it evicts what earlier
    reps left in L2."""
    import torch
    return torch.empty(256 << 20, dtype=torch.uint8, device=dev)


def run_decode_config(args, dev, stream, hbm, which):
    """A decode workload through the plain tl_paged_attn_decode call: the
    sliding-window mix (two layers, separate pools: window 4,096 then full)
    or the long-context lognormal batch.  GB/s of the K/V the call must read
    (window-clipped) plus Q, the tables and the output, per call."""
    import torch

    import paged_kv_attention_cache_gb300 as tl
    from paged_kv_attention_cache_gb300 import workloads as wl

    if which == "swa":
        cases = [wl.swa_decode(seed=args.seed, device=dev, layer=layer) for layer in (0, 1)]
        name = ("sliding-window mix: B=128, Hq=40, Hkv=8, d=128, bf16, page 16, "
                "L~U[1024,32768], 1% of values x8; layer 0 window 4096, layer 1 full, "
                "separate pools")
    else:
        cases = [wl.longctx_decode(seed=args.seed, device=dev)]
        name = ("long-context batch: B=256, Hq=64, Hkv=8, d=128, bf16, page 16, "
                "L lognormal median 2048 sigma 1 clipped to [64,131072]")
    layers = []
    for case in cases:
        g = wl.to_device(case, dev)
        B, hq, hkv, d = case.B, case.Hq, case.Hkv, case.d
        lens = case.context_lens.tolist()
        keys = sum(min(L, case.window) if case.window > 0 else L for L in lens)
        kvb = keys * 2 * hkv * d * 2
        alg = kvb + B * hq * d * 2 + B * hq * d * 4 + sum((L + 15) // 16 for L in lens) * 4
        out = torch.empty((B, hq, d), dtype=torch.float32, device=dev)
        ws = tl.alloc_workspace(tl.tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)

        def call():
            tl.tl_paged_attn_decode(g.q, g.k_cache, g.v_cache, g.block_table, g.context_lens,
                                    case.scale, window=case.window, out=out, workspace=ws,
                                    error_word=err)

        for _ in range(max(3, args.warmup)):
            call()
        torch.cuda.synchronize()
        n = 30
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"device error word {int(err.item())} in the {which} decode")
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        gbs = alg / (ms * 1e-3) / 1e9
        layers.append({"window": case.window, "kv_bytes_per_call": kvb,
                       "algorithmic_bytes_per_call": alg, "ms_per_call": round(ms, 4),
                       "gbs": round(gbs, 1), "frac": round(gbs / hbm, 4),
                       "l2": "pool %.2f GB vs 129 MB L2" % (g.k_cache.numel() * 4 / 1e9)})
        del g, out, ws
        torch.cuda.empty_cache()
    return {"workload": name, "call": "tl_paged_attn_decode", "layers": layers}


def run_ring(args, dev, stream, hbm):
    """The sliding-window layer (window 4,096) over a windowed pool of rings
    (257 pages per sequence): GB/s of the window's K/V the decode reads."""
    import torch

    import paged_kv_attention_cache_gb300 as tl
    from paged_kv_attention_cache_gb300 import workloads as wl

    case = wl.swa_ring_decode(seed=args.seed, device=dev)
    ring = case.extra["ring_pages"]
    g = wl.to_device(case, dev)
    B, hq, hkv, d = case.B, case.Hq, case.Hkv, case.d
    tl.tl_kv_cache_write(g.k_new, g.v_new, g.k_cache, g.v_cache, g.slot_mapping)
    out = torch.empty((B, hq, d), dtype=torch.float32, device=dev)
    ws = tl.alloc_workspace(tl.tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    keys = sum(min(int(L), case.window) for L in case.context_lens.tolist())
    kvb = keys * 2 * hkv * d * 2
    alg = kvb + B * hq * d * 2 + B * hq * d * 4 + B * ring * 4

    def call():
        tl.tl_paged_attn_decode_ring(g.q, g.k_cache, g.v_cache, g.block_table, g.context_lens,
                                     case.scale, case.window, ring, out=out, workspace=ws)

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    n = 50
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(n):
        call()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / n
    return {"workload": "sliding-window layer over rings: B=128, Hq=40, Hkv=8, d=128, bf16, "
                        f"window 4096, rings of {ring} pages of 16, L~U[1024,32768]",
            "kv_bytes_per_call": kvb, "ms_per_call": round(ms, 4),
            "gbs": round(alg / (ms * 1e-3) / 1e9, 1), "frac": round(alg / (ms * 1e-3) / 1e9 / hbm, 4),
            "l2": "ring pool %.2f GB vs 129 MB L2" % (g.k_cache.numel() * 4 / 1e9)}


def run_int8(args, dev, stream, hbm):
    """Decode of the Llama-3-8B-shaped batch (B=64) over int8 pools (codes and
    one f32 scale per slot and KV head): the pools are the bf16 pools written
    through tl_kv_cache_write_int8 (every slot); the step is the int8 write of
    the 64 new rows and the decode in one call (tl_paged_attn_decode_write_int8),
    with the two separate calls timed beside it."""
    import torch

    import paged_kv_attention_cache_gb300 as tl
    from paged_kv_attention_cache_gb300 import workloads as wl

    case = wl.llama8b_decode(seed=args.seed, device=dev)
    g = wl.to_device(case, dev)
    P, ps, hkv, d = g.k_cache.shape
    B, hq = case.B, case.Hq
    kc = torch.empty((P, ps, hkv, d), dtype=torch.int8, device=dev)
    vc = torch.empty_like(kc)
    ks = torch.empty((P, hkv, ps), dtype=torch.float32, device=dev)
    vs = torch.empty_like(ks)
    every = torch.arange(P * ps, dtype=torch.int64, device=dev)
    tl.tl_kv_cache_write_int8(g.k_cache.view(-1, hkv, d), g.v_cache.view(-1, hkv, d), kc, vc, ks,
                              vs, every)
    del g.k_cache, g.v_cache
    out = torch.empty((B, hq, d), dtype=torch.float32, device=dev)
    ws = tl.alloc_workspace(tl.tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    keys = int(case.context_lens.sum().item())
    kvb = keys * 2 * hkv * (d + 4)  # codes, and one f32 scale per key, K and V

    def step():  # the int8 write of the new rows and the decode, one call
        tl.tl_paged_attn_decode_write_int8(g.q, g.k_new, g.v_new, g.slot_mapping, kc, vc, ks, vs,
                                           g.block_table, g.context_lens, case.scale, out=out,
                                           workspace=ws)

    def two_calls():
        tl.tl_kv_cache_write_int8(g.k_new, g.v_new, kc, vc, ks, vs, g.slot_mapping)
        tl.tl_paged_attn_decode_int8(g.q, kc, vc, ks, vs, g.block_table, g.context_lens,
                                     case.scale, out=out, workspace=ws)

    def timed(fn, n=100):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(n):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        return s.elapsed_time(e) / n

    ms = timed(step)
    sep_ms = timed(two_calls)
    return {"workload": "Llama-3-8B-shaped decode layer over int8 pools: B=64, Hq=32, Hkv=8, "
                        "d=128, page 16, L~U[512,8192] (int8 write of 64 rows + decode)",
            "kv_bytes_per_step": kvb, "ms_per_step": round(ms, 4),
            "two_calls_ms_per_step": round(sep_ms, 4),
            "kv_gbs": round(kvb / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm": round(kvb / (ms * 1e-3) / 1e9 / hbm, 4),
            "tokens_per_s": round(B / (ms * 1e-3), 1)}


def run_fp8(args, dev, stream, hbm):
    """Decode of the Llama-3-8B-shaped batch (B=64) over e4m3 pools: the pools
    are the bf16 pools written through tl_kv_cache_write_fp8 (every slot), the
    step is the write of the 64 new rows plus the decode in one call
    (tl_paged_attn_decode_write), as for bf16."""
    import torch

    import paged_kv_attention_cache_gb300 as tl
    from paged_kv_attention_cache_gb300 import workloads as wl

    case = wl.llama8b_decode(seed=args.seed, device=dev)
    g = wl.to_device(case, dev)
    P, ps, hkv, d = g.k_cache.shape
    B, hq = case.B, case.Hq
    k8 = torch.empty((P, ps, hkv, d), dtype=torch.float8_e4m3fn, device=dev)
    v8 = torch.empty_like(k8)
    every = torch.arange(P * ps, dtype=torch.int64, device=dev)
    tl.tl_kv_cache_write_fp8(g.k_cache.view(-1, hkv, d), g.v_cache.view(-1, hkv, d), k8, v8, every)
    del g.k_cache, g.v_cache
    out = torch.empty((B, hq, d), dtype=torch.float32, device=dev)
    ws = tl.alloc_workspace(tl.tl_paged_attn_decode_workspace_size(B, hq, hkv, d), dev)
    kvb = int(case.context_lens.sum().item()) * 2 * hkv * d  # one byte per element

    def step():  # the write of the new rows (converted to e4m3) and the decode, one call
        tl.tl_paged_attn_decode_write(g.q, g.k_new, g.v_new, g.slot_mapping, k8, v8,
                                      g.block_table, g.context_lens, case.scale, out=out,
                                      workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    n = 100
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(n):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / n
    return {"workload": "Llama-3-8B-shaped decode layer over e4m3 pools: B=64, Hq=32, Hkv=8, "
                        "d=128, page 16, L~U[512,8192] (write of 64 rows + decode)",
            "kv_bytes_per_step": kvb, "ms_per_step": round(ms, 4),
            "kv_gbs": round(kvb / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm": round(kvb / (ms * 1e-3) / 1e9 / hbm, 4),
            "tokens_per_s": round(B / (ms * 1e-3), 1)}


def run_verify(args, dev, stream, hbm, bf16, q_len=4):
    """Multi-token decode (the speculative-verify shape) through
    tl_paged_attn_decode_multi: the Llama-3-8B-shaped batch (B=64) with q_len
    new tokens per sequence at positions L - q_len .. L - 1."""
    import torch

    import paged_kv_attention_cache_gb300 as tl
    from paged_kv_attention_cache_gb300 import workloads as wl

    lengths = wl.llama8b_lengths(seed=args.seed, B=64)
    case = wl.prefill_case([0] * 64, [L - q_len for L in lengths], T=q_len, Hq=32, Hkv=8, d=128,
                           seed=args.seed + 7, device=dev)
    g = wl.to_device(case, dev)
    tl.tl_kv_cache_write(g.k_new, g.v_new, g.k_cache, g.v_cache, g.slot_mapping)
    out = torch.empty((64, q_len, 32, 128), dtype=torch.float32, device=dev)
    ws = tl.alloc_workspace(tl.tl_paged_attn_decode_multi_workspace_size(64, q_len, 32, 8, 128),
                            dev)
    cl = torch.tensor(lengths, dtype=torch.int32, device=dev)
    kvb = sum(lengths) * 2 * 8 * 128 * 2
    flops = prefill_flops(case.positions, 32, 128)

    def call():
        tl.tl_paged_attn_decode_multi(g.q, g.k_cache, g.v_cache, g.block_table, cl, case.scale,
                                      out=out, workspace=ws)

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    n = 50
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(n):
        call()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / n
    return {"workload": f"Llama-3-8B-shaped batch B=64, {q_len} query tokens per sequence at its "
                        "end (speculative verify), L~U[512,8192], through tl_paged_attn_decode_multi",
            "kv_bytes_per_call": kvb, "ms_per_call": round(ms, 4),
            "kv_gbs": round(kvb / (ms * 1e-3) / 1e9, 1),
            "kv_frac_of_hbm": round(kvb / (ms * 1e-3) / 1e9 / hbm, 4),
            "tflops": round(flops / (ms * 1e-3) / 1e12, 2)}


def run_prefill(args, rank, dev, stream, hbm, bf16, bf16_sus, src):
    """Batched-prefill workload: TFLOP/s of the attention call, and the
    16K-row chunk write's GB/s."""
    import torch

    import paged_kv_attention_cache_gb300 as tl
    from paged_kv_attention_cache_gb300 import workloads as wl

    pcase = wl.batched_prefill(seed=args.seed + rank, device=dev)
    pg = wl.to_device(pcase, dev)
    flops = prefill_flops(pcase.positions, pcase.Hq, pcase.d)
    pout = torch.empty((pcase.B, pcase.T, pcase.Hq, pcase.d), dtype=torch.float32, device=dev)
    pws = tl.alloc_workspace(tl.tl_paged_attn_prefill_workspace_size(
        pcase.B, pcase.T, pcase.Hq, pcase.Hkv, pcase.d, pcase.block_table.shape[1],
        pcase.page_size), dev)
    kn = pg.k_new.view(-1, pcase.Hkv, pcase.d)
    vn = pg.v_new.view(-1, pcase.Hkv, pcase.d)
    tl.tl_kv_cache_write(kn, vn, pg.k_cache, pg.v_cache, pg.slot_mapping)

    def pf():
        tl.tl_paged_attn_prefill(pg.q, pg.k_cache, pg.v_cache, pg.block_table, pg.positions,
                                 pcase.scale, out=pout, workspace=pws)

    for _ in range(max(3, args.warmup)):
        pf()
    torch.cuda.synchronize()
    pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.prefill_steps)]
    with ClockSampler(dev.index or 0) as pclk:
        t_end = time.time() + args.soak_seconds
        while time.time() < t_end:  # the same load around the timed calls, for the sampler
            for _ in range(10):
                pf()
            torch.cuda.synchronize()
        for a, b in pev:
            a.record(stream)
            pf()
            b.record(stream)
        torch.cuda.synchronize()
    pf_ms = statistics.mean(a.elapsed_time(b) for a, b in pev)
    # the chunk write on its own (16K rows), for the write kernel's GB/s.
    # Its 80 MB fit in L2, so the writes rotate over four chunks (this one and
    # three more of other seeds, each with its own pool): a write never finds
    # its rows in L2, and the dirty rows of earlier writes are written back
    # during later ones, as in a serving loop.  Timed two ways: each call
    # alone between CUDA events (a sleep kernel first, so the host has
    # enqueued the call before the GPU reaches the first event), and sixteen
    # calls back to back in a CUDA graph (per call: the graph's time / 16).
    chunks = [pg] + [wl.to_device(wl.batched_prefill(seed=args.seed + rank + 100 + i, device=dev),
                                  dev) for i in range(3)]

    def write_chunk(c):
        tl.tl_kv_cache_write(c.k_new.view(-1, c.Hkv, c.d), c.v_new.view(-1, c.Hkv, c.d),
                             c.k_cache, c.v_cache, c.slot_mapping)

    for c in chunks:
        write_chunk(c)
    torch.cuda.synchronize()
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(40)]
    for i, (a, b) in enumerate(wev):
        torch.cuda._sleep(200000)
        a.record(stream)
        write_chunk(chunks[i % 4])
        b.record(stream)
    torch.cuda.synchronize()
    w_ms_call = statistics.mean(a.elapsed_time(b) for a, b in wev)
    gstream = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(gstream):
        with torch.cuda.graph(graph, stream=gstream):
            for i in range(16):
                write_chunk(chunks[i % 4])
    torch.cuda.synchronize()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ga.record(stream)
    for _ in range(10):
        graph.replay()
    gb.record(stream)
    torch.cuda.synchronize()
    w_ms = ga.elapsed_time(gb) / 160
    n_live_all = [int((c.slot_mapping >= 0).sum().item()) for c in chunks]
    del graph, chunks
    n_live = sum(n_live_all) / len(n_live_all)  # live rows per chunk (mean of the four)
    w_bytes = int(n_live * pcase.Hkv * pcase.d * 2 * 2 * 2 + pcase.slot_mapping.numel() * 8)
    pf_tflops = flops / (pf_ms * 1e-3) / 1e12
    prefill_line = {
        "workload": "B=8 x T=2048 right-aligned, pads U{0..1500}, prior U{0..6144}, "
                    "Hq=32, Hkv=8, d=128, bf16",
        "tflops": round(pf_tflops, 2), "ms_per_call": round(pf_ms, 4), "flops_per_call": flops,
        "roofline": {"bound": "tensor", "achieved": round(pf_tflops, 2), "peak": bf16,
                     "unit": "TFLOP/s", "frac": round(pf_tflops / bf16, 4),
                     "traffic": PREFILL_TRAFFIC[0],
                     "traffic_source": PREFILL_TRAFFIC[1] + " (prefill_tc_kernel alone)",
                     "peak_source": f"{src} bf16_tflops (burst)",
                     "frac_of_sustained": round(pf_tflops / bf16_sus, 4)},
        "clocks": pclk.summary()}
    write_line = {"workload": "the prefill chunk's K/V rows: 16,384 tokens (pads at slot -1), "
                              "Hkv=8, d=128, bf16, into the shuffled pool; four chunks in turn",
                  "rows": round(n_live, 1), "algorithmic_bytes": w_bytes,
                  "ms": round(w_ms, 5), "gbs": round(w_bytes / (w_ms * 1e-3) / 1e9, 1),
                  "frac": round(w_bytes / (w_ms * 1e-3) / 1e9 / hbm, 4),
                  "timing": "16 calls back to back in a CUDA graph, 10 replays; per call = "
                            "time / 160",
                  "ms_per_call_alone": round(w_ms_call, 5),
                  "frac_per_call_alone": round(w_bytes / (w_ms_call * 1e-3) / 1e9 / hbm, 4),
                  "l2": "four chunks in turn (256 MB of new rows, 160 MB of destination rows): "
                        "no call finds its rows in L2",
                  "traffic": WRITE_TRAFFIC[0],
                  "traffic_source": WRITE_TRAFFIC[1] + " (one write, cold; its 40 MB of row "
                                    "writes land in L2 and drain during later work)"}
    if rank == 0 and not args.no_cpu_baseline and args.only == "all":
        prefill_line["cpu_baseline"] = prefill_cpu_baseline(pcase, pg, args)
    # the same call over e4m3 pools (the bf16 pools written through the
    # converting write): the pre-pass widens K to bf16 and V to fp16 copies
    P_, ps_, hkv_, d_ = pg.k_cache.shape
    k8 = torch.empty((P_, ps_, hkv_, d_), dtype=torch.float8_e4m3fn, device=dev)
    v8 = torch.empty_like(k8)
    every = torch.arange(P_ * ps_, dtype=torch.int64, device=dev)
    tl.tl_kv_cache_write_fp8(pg.k_cache.view(-1, hkv_, d_), pg.v_cache.view(-1, hkv_, d_), k8, v8,
                             every)
    pws8 = tl.alloc_workspace(tl.tl_paged_attn_prefill_workspace_size_ex(
        pcase.B, pcase.T, pcase.Hq, pcase.Hkv, pcase.d, pcase.block_table.shape[1],
        pcase.page_size, 0, tl.TL_FP8_E4M3), dev)

    def pf8():
        tl.tl_paged_attn_prefill(pg.q, k8, v8, pg.block_table, pg.positions, pcase.scale,
                                 out=pout, workspace=pws8)

    for _ in range(max(3, args.warmup)):
        pf8()
    torch.cuda.synchronize()
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.prefill_steps)]
    for a, b in fev:
        a.record(stream)
        pf8()
        b.record(stream)
    torch.cuda.synchronize()
    f_ms = statistics.mean(a.elapsed_time(b) for a, b in fev)
    f_tflops = flops / (f_ms * 1e-3) / 1e12
    prefill_line["fp8_pools"] = {"ms_per_call": round(f_ms, 4), "tflops": round(f_tflops, 2),
                                 "frac": round(f_tflops / bf16, 4)}
    del k8, v8, pws8
    # and over int8 pools (the bf16 pools through the int8 write: one scale per
    # slot and KV head): the pre-pass widens the codes and gathers the scales
    kc8 = torch.empty((P_, ps_, hkv_, d_), dtype=torch.int8, device=dev)
    vc8 = torch.empty_like(kc8)
    ks8 = torch.empty((P_, hkv_, ps_), dtype=torch.float32, device=dev)
    vs8 = torch.empty_like(ks8)
    tl.tl_kv_cache_write_int8(pg.k_cache.view(-1, hkv_, d_), pg.v_cache.view(-1, hkv_, d_), kc8,
                              vc8, ks8, vs8, every)
    pws_i8 = tl.alloc_workspace(tl.tl_paged_attn_prefill_workspace_size_ex(
        pcase.B, pcase.T, pcase.Hq, pcase.Hkv, pcase.d, pcase.block_table.shape[1],
        pcase.page_size, 0, tl.TL_INT8), dev)

    def pf_i8():
        tl.tl_paged_attn_prefill_int8(pg.q, kc8, vc8, ks8, vs8, pg.block_table, pg.positions,
                                      pcase.scale, out=pout, workspace=pws_i8)

    for _ in range(max(3, args.warmup)):
        pf_i8()
    torch.cuda.synchronize()
    iev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.prefill_steps)]
    for a, b in iev:
        a.record(stream)
        pf_i8()
        b.record(stream)
    torch.cuda.synchronize()
    i_ms = statistics.mean(a.elapsed_time(b) for a, b in iev)
    i_tflops = flops / (i_ms * 1e-3) / 1e12
    prefill_line["int8_pools"] = {"ms_per_call": round(i_ms, 4), "tflops": round(i_tflops, 2),
                                  "frac": round(i_tflops / bf16, 4)}
    del kc8, vc8, ks8, vs8, pws_i8
    # the same shape on the sliding-window mix's values (1% of Q, K and V x8):
    # every row's V holds values above 8, so every row takes P as two fp16 parts
    ocase = wl.batched_prefill(seed=args.seed + rank + 7, device=dev, outlier_p=0.01)
    og = wl.to_device(ocase, dev)
    tl.tl_kv_cache_write(og.k_new.view(-1, ocase.Hkv, ocase.d), og.v_new.view(-1, ocase.Hkv, ocase.d),
                         og.k_cache, og.v_cache, og.slot_mapping)
    oflops = prefill_flops(ocase.positions, ocase.Hq, ocase.d)
    ows = tl.alloc_workspace(tl.tl_paged_attn_prefill_workspace_size(
        ocase.B, ocase.T, ocase.Hq, ocase.Hkv, ocase.d, ocase.block_table.shape[1],
        ocase.page_size), dev)

    def pf_o():
        tl.tl_paged_attn_prefill(og.q, og.k_cache, og.v_cache, og.block_table, og.positions,
                                 ocase.scale, out=pout, workspace=ows)

    for _ in range(max(3, args.warmup)):
        pf_o()
    torch.cuda.synchronize()
    oev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.prefill_steps)]
    for a, b in oev:
        a.record(stream)
        pf_o()
        b.record(stream)
    torch.cuda.synchronize()
    o_ms = statistics.mean(a.elapsed_time(b) for a, b in oev)
    o_tflops = oflops / (o_ms * 1e-3) / 1e12
    prefill_line["outlier_values"] = {
        "workload": "the same shape, 1% of Q, K and V values x8 (every row takes P as two fp16 "
                    "parts)", "ms_per_call": round(o_ms, 4), "tflops": round(o_tflops, 2),
        "frac": round(o_tflops / bf16, 4)}
    del og, ows
    return prefill_line, write_line


def cpu_baseline(case, g, args):
    """The oracle, as it stands, on the whole decode step of the same workload
    (the write of the new rows, then attention for all sequences), all host
    cores, repeated for about args.cpu_seconds."""
    import oracle

    kc = g.k_cache.cpu()
    vc = g.v_cache.cpu()
    q, kn, vn = case.q.cpu(), case.k_new.cpu(), case.v_new.cpu()
    sm, bt, cl = case.slot_mapping.cpu(), case.block_table.cpu(), case.context_lens.cpu()
    threads = os.cpu_count() or 1
    kvb = kv_bytes(cl.tolist(), case.window, case.Hkv, case.d, 2)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.kv_cache_write(kn, vn, kc, vc, sm)
        oracle.paged_decode(q, kc, vc, bt, cl, case.scale, window=case.window, threads=threads)
        reps += 1
        if time.perf_counter() - t0 >= args.cpu_seconds:
            break
    dt = (time.perf_counter() - t0) / reps
    # one repetition on a single thread, beside the all-cores figure
    t1 = time.perf_counter()
    oracle.kv_cache_write(kn, vn, kc, vc, sm)
    oracle.paged_decode(q, kc, vc, bt, cl, case.scale, window=case.window, threads=1)
    dt1 = time.perf_counter() - t1
    return {"value": round(kvb / dt / 1e9, 3), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "sample": f"the full decode step ({case.B} sequences), "
                                        f"{reps} repetitions, {dt:.3f} s each",
            "single_thread": {"value": round(kvb / dt1 / 1e9, 3), "unit": "GB/s",
                              "sample": f"one full decode step, {dt1:.3f} s"}}


def prefill_cpu_baseline(pcase, pg, args):
    """The oracle, as it stands, on whole rows of the batched-prefill workload
    (every token of each row, blockwise fold over 2,048-key blocks), all host
    cores, rows taken in order until about args.cpu_seconds have passed; the
    rate is the rows' algorithmic flops over the time."""
    import numpy as np

    import oracle

    kc, vc = pg.k_cache.cpu(), pg.v_cache.cpu()  # after the chunk's write
    q, pos, bt = pcase.q.cpu(), pcase.positions.cpu(), pcase.block_table.cpu()
    threads = os.cpu_count() or 1
    flops, rows, t0 = 0, 0, time.perf_counter()
    for b in range(pcase.B):
        oracle.paged_prefill(q[b:b + 1], kc, vc, bt[b:b + 1], pos[b:b + 1], pcase.scale,
                             threads=threads)
        flops += prefill_flops(pos[b:b + 1], pcase.Hq, pcase.d)
        rows += 1
        if time.perf_counter() - t0 >= args.cpu_seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 5), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{rows} of {pcase.B} rows, every token ({dt:.1f} s)"}


# ------------------------------------------------------------- reference --

def run_reference(args):
    """The oracle timed on this host's cores: each step is the whole decode
    step of the benchmark workload (write + attention for all 64 sequences)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from paged_kv_attention_cache_gb300 import workloads as wl

    case = wl.llama8b_decode(seed=args.seed, device="cpu")
    threads = os.cpu_count() or 1
    kvb = kv_bytes(case.context_lens.tolist(), case.window, case.Hkv, case.d, 2)

    def step():
        oracle.kv_cache_write(case.k_new, case.v_new, case.k_cache, case.v_cache,
                              case.slot_mapping)
        oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_table,
                            case.context_lens, case.scale, threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = kvb / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) values, shuffled page pool)",
            "config": {"workload": WORKLOAD, "batch": case.B, "Hq": case.Hq, "Hkv": case.Hkv,
                       "d_head": case.d, "page_size": 16, "kv_bytes_per_step": kvb},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                             "kind": "oracle",
                             "sample": f"the full decode step ({case.B} sequences) per step"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--prefill-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-seconds", type=float, default=2.0)
    ap.add_argument("--batch", type=int, default=64, help="decode batch (64 = the workload)")
    ap.add_argument("--only", choices=["all", "decode", "decode-e2e", "prefill", "ring",
                                       "verify", "fp8", "int8", "swa", "longctx"],
                    default="all")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
