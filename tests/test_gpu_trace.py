"""The decode trace build (-DTL_DECODE_TRACE=1): its calls give the default
library's results bit for bit, and its timeline stamps come in the order the
launches run (plan, attention kernel, combine), for the warp-planned and the
block-planned batch sizes."""
import ctypes
import json
import os
import subprocess
import sys

import pytest
import torch

import paged_kv_attention_cache_gb300 as tl
from paged_kv_attention_cache_gb300 import _lib, trace, workloads as wl

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
