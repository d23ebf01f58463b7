"""The library's build options compile for sm_103a (no GPU needed): the decode
timeline trace, the prefill step trace with the all-TS attention kernel, and
the MMA probe.  The GPU tests run them (tests/test_gpu_trace.py); this keeps
them from rotting in a CPU-only run."""
import concurrent.futures as cf
import os
import subprocess
import tempfile

from paged_kv_attention_cache_gb300 import build


def _compile(src, defines, out_dir):
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + "_".join(defines) + ".o")
    cmd = [build._nvcc(), *build.ARCH, *build.NVCC_FLAGS, *("-D" + d for d in defines), "-c",
           os.path.join(build.CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, defines, r.returncode, r.stderr[-2000:]


def test_build_options_compile():
    jobs = [("paged_decode.cu", ["TL_DECODE_TRACE=1"]),
            ("paged_prefill.cu", ["TL_PREFILL_TRACE=1", "TL_PREFILL_ALL_TS=1"]),
            ("probe_mma.cu", [])]
    with tempfile.TemporaryDirectory() as d, cf.ThreadPoolExecutor(len(jobs)) as ex:
        for src, defines, rc, err in ex.map(lambda j: _compile(j[0], j[1], d), jobs):
            assert rc == 0, f"{src} {defines}: {err}"
