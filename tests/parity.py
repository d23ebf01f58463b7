"""The parity bar between the CUDA path and the oracle.

Floating point: max-abs error <= 2e-3 and max-rel error <= 1e-2, with the
relative error of element i taken as |a_i - r_i| / max(|r_i|, 0.2) (for
|r_i| < 0.2 it is the absolute criterion scaled by 1/0.2 = 5, so the two bars
meet at 2e-3 / 1e-2 = 0.2).  Integer and byte work: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

ABS_TOL = 2e-3
REL_TOL = 1e-2
REL_FLOOR = 0.2


def errors(gpu, ref):
    a = gpu.detach().double().cpu().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64).reshape(a.shape)
    err = np.abs(a - r)
    rel = err / np.maximum(np.abs(r), REL_FLOOR)
    return a, float(np.max(err, initial=0.0)), float(np.max(rel, initial=0.0))


def assert_close(gpu, ref, what=""):
    a, e, r = errors(gpu, ref)
    assert np.all(np.isfinite(a)), f"{what}: non-finite output"
    assert e <= ABS_TOL and r <= REL_TOL, f"{what}: max abs {e:.3e} (<= {ABS_TOL}), max rel {r:.3e} (<= {REL_TOL})"
    return e, r


def same_bytes(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.contiguous().view(torch.uint8).cpu(), b.contiguous().view(torch.uint8).cpu())
