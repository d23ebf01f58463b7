"""The trace builds and the MMA probe.  The decode trace build
(-DTL_DECODE_TRACE=1): its calls give the default library's results bit for
bit, and its timeline stamps come in the order the launches run (plan,
attention kernel, combine), for the warp-planned and the block-planned batch
sizes.  The prefill trace build (-DTL_PREFILL_TRACE=1): bit for bit too, and
its per-CTA step counters add up to the call's key tiles.  The all-TS
attention kernel (a build option) matches the oracle.  The MMA probe runs and
reports positive costs."""
import ctypes
import json
import os
import subprocess
import sys

import pytest
import torch

import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import _lib, build, trace, workloads as wl

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def trace_lib():
    lib = ctypes.CDLL(trace.build_trace_library())
    for name in ("tl_paged_attn_decode", "tl_decode_trace_reset", "tl_decode_trace_read",
                 "tl_status_string"):
        args, res = _lib.SIGNATURES[name]
        getattr(lib, name).argtypes = args
        getattr(lib, name).restype = res
    return lib


def _raw_decode(lib, g, out, ws):
    return lib.tl_paged_attn_decode(
        g.q.data_ptr(), g.k_cache.data_ptr(), g.v_cache.data_ptr(), g.block_table.data_ptr(),
        g.block_table.shape[1], g.context_lens.data_ptr(), out.data_ptr(), g.B, g.Hq, g.Hkv,
        g.d, g.num_pages, g.page_size, 0, g.scale, tl.TL_BF16, ws.data_ptr(), ws.numel(),
        None, torch.cuda.current_stream().cuda_stream)


ORDER = ("plan_start", "plan_end", "attn_released", "attn_first_stage", "attn_end",
         "combine_start", "combine_end")


@pytest.mark.parametrize("lens", [[300, 4000, 17, 2500], [700] * 200])
def test_traced_calls_match_the_default_library_and_stamp_in_order(trace_lib, lens):
    g = wl.to_device(wl.decode_case(lens, Hq=8, Hkv=2, d=128, seed=5), "cuda")
    ws = tl.alloc_workspace(tl.tl_paged_attn_decode_workspace_size(g.B, 8, 2, 128), "cuda")
    out = torch.empty((g.B, 8, 128), dtype=torch.float32, device="cuda")

    def call():
        assert _raw_decode(trace_lib, g, out, ws) == tl.TL_OK

    t = trace.trace_calls(call, trace_lib, calls=3)
    ref = tl.tl_paged_attn_decode(g.q, g.k_cache, g.v_cache, g.block_table, g.context_lens,
                                  g.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    times = [t[k] for k in ORDER]
    assert all(x is not None for x in times), t
    assert times == sorted(times), t
    assert (t["plan_placed"] is not None) == (g.B <= 128)
    assert t["attn_end"] < 1e4  # microseconds: a plausible call


def test_trace_tool_prints_a_timeline():
    r = subprocess.run([sys.executable, "-m", "paged_kv_attention_cache_gb300.trace",
                        "--batch", "8", "--length", "3000", "--calls", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    t = json.loads(r.stdout.strip().splitlines()[-1])
    assert t["batch"] == 8 and t["kv_bytes"] == 8 * 3000 * 8 * 256 * 2
    for k in ("plan", "attention", "combine"):
        assert t[k] is not None and t[k] > 0, t


@pytest.fixture(scope="module")
def ptrace_lib():
    lib = ctypes.CDLL(trace.build_prefill_trace_library())
    for name in ("tl_paged_attn_prefill", "tl_prefill_trace_reset", "tl_prefill_trace_read",
                 "tl_status_string"):
        args, res = _lib.SIGNATURES[name]
        getattr(lib, name).argtypes = args
        getattr(lib, name).restype = res
    return lib


def test_prefill_trace_build_matches_and_counts_its_steps(ptrace_lib):
    case = wl.prefill_case([3, 0, 40], [100, 0, 700], T=300, Hq=8, Hkv=2, d=128, seed=9)
    g = wl.to_device(case, "cuda")
    tl.tl_kv_cache_write(g.k_new.view(-1, 2, 128), g.v_new.view(-1, 2, 128), g.k_cache,
                         g.v_cache, g.slot_mapping)
    ws = tl.alloc_workspace(tl.tl_paged_attn_prefill_workspace_size(
        case.B, case.T, 8, 2, 128, case.block_table.shape[1], case.page_size), "cuda")
    out = torch.empty((case.B, case.T, 8, 128), dtype=torch.float32, device="cuda")
    assert ptrace_lib.tl_prefill_trace_reset() == tl.TL_OK
    st = ptrace_lib.tl_paged_attn_prefill(
        g.q.data_ptr(), g.k_cache.data_ptr(), g.v_cache.data_ptr(), g.block_table.data_ptr(),
        case.block_table.shape[1], g.positions.data_ptr(), out.data_ptr(), case.B, case.T, 8, 2,
        128, g.k_cache.shape[0], case.page_size, 0, case.scale, tl.TL_BF16, ws.data_ptr(),
        ws.numel(), None, torch.cuda.current_stream().cuda_stream)
    assert st == tl.TL_OK
    n = torch.cuda.get_device_properties(0).multi_processor_count
    f = len(trace.PTRACE_FIELDS)
    buf = (ctypes.c_uint64 * (f * n))()
    assert ptrace_lib.tl_prefill_trace_read(buf, n) == tl.TL_OK
    rows = [list(buf[f * k:f * k + f]) for k in range(n)]
    ref = tl.tl_paged_attn_prefill(g.q, g.k_cache, g.v_cache, g.block_table, g.positions,
                                   case.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    # the steps: per (row, KV head, query-tile pair) the 128-key tiles the
    # pair's live tokens can see, keys 0 .. the pair's last position (no window)
    tpt = 128 // (case.Hq // case.Hkv)
    expect = 0
    pos = case.positions
    for b in range(case.B):
        for t0 in range(0, case.T, 2 * tpt):
            p = pos[b, t0:t0 + 2 * tpt]
            live = p[p >= 0]
            if live.numel():
                expect += (int(live.max()) // 128 + 1) * case.Hkv
    assert sum(r[1] for r in rows) == expect
    s = trace.prefill_step_summary(rows)
    assert s["cycles_per_step_median"] > 0
    assert 0 <= s["wait_p_share"] <= 1 and 0 <= s["wait_kv_share"] <= 1
    assert s["softmax_busy_per_tile"] > 0


def test_mma_probe_reports_positive_costs():
    from paged_kv_attention_cache_gb300 import probe_mma
    lib = probe_mma.probe_library()
    for form in range(len(probe_mma.FORMS)):
        assert probe_mma.cycles(lib, form, 32, reps=1) > 0


def test_all_ts_prefill_variant_matches_the_oracle():
    """The all-TS attention kernel (a build option) over bf16 pools: every
    output of a small batched call (pads, prior context, a ragged last query
    tile) against the oracle."""
    import oracle
    from tests.parity import assert_close
    lib = ctypes.CDLL(build.build_variant("prefill_all_ts", build.SOURCES,
                                          ["TL_PREFILL_ALL_TS=1"]))
    for name in ("tl_paged_attn_prefill", "tl_kv_cache_write"):
        args, res = _lib.SIGNATURES[name]
        getattr(lib, name).argtypes = args
        getattr(lib, name).restype = res
    case = wl.prefill_case([5, 0, 90], [300, 0, 1500], T=200, Hq=8, Hkv=2, d=128, seed=11)
    g = wl.to_device(case, "cuda")
    tl.tl_kv_cache_write(g.k_new.view(-1, 2, 128), g.v_new.view(-1, 2, 128), g.k_cache,
                         g.v_cache, g.slot_mapping)
    ws = tl.alloc_workspace(4 * tl.tl_paged_attn_prefill_workspace_size(
        case.B, case.T, 8, 2, 128, case.block_table.shape[1], case.page_size), "cuda")
    out = torch.empty((case.B, case.T, 8, 128), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = lib.tl_paged_attn_prefill(
        g.q.data_ptr(), g.k_cache.data_ptr(), g.v_cache.data_ptr(), g.block_table.data_ptr(),
        case.block_table.shape[1], g.positions.data_ptr(), out.data_ptr(), case.B, case.T, 8, 2,
        128, g.k_cache.shape[0], case.page_size, 0, case.scale, tl.TL_BF16, ws.data_ptr(),
        ws.numel(), err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == tl.TL_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    oracle.kv_cache_write(case.k_new.view(-1, 2, 128), case.v_new.view(-1, 2, 128), kc, vc,
                          case.slot_mapping)
    ref = oracle.paged_prefill(case.q, kc, vc, case.block_table, case.positions, case.scale)
    assert_close(out.cpu().reshape(ref.shape), ref, "all-TS prefill")
