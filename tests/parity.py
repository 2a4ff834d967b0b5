"""Shared tolerance of the GPU-vs-oracle parity tests.

Bar: max abs error <= 2e-3 and max rel error <= 1e-2 on fp32 outputs.  An
elementwise relative error is meaningless where the exact output is near
zero, so the relative test divides by max(|ref|, 0.2): 0.2 = 2e-3 / 1e-2,
the magnitude where the two bounds meet.  Below it the absolute bound
governs; above it the relative one does.  The raw relative error is
reported too.
"""
import numpy as np

ATOL = 2e-3
RTOL = 1e-2
REL_FLOOR = ATOL / RTOL


def errors(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(gpu - ref)
    return {
        "max_abs": float(d.max(initial=0.0)),
        "max_rel_floored": float((d / np.maximum(np.abs(ref), REL_FLOOR)).max(initial=0.0)),
        "max_rel_raw": float((d / np.maximum(np.abs(ref), 1e-30)).max(initial=0.0)),
    }


def assert_parity(gpu, ref, what=""):
    gpu = np.asarray(gpu)
    assert gpu.shape == np.asarray(ref).shape, (what, gpu.shape, np.asarray(ref).shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    e = errors(gpu, ref)
    assert e["max_abs"] <= ATOL and e["max_rel_floored"] <= RTOL, f"{what}: {e}"
    return e
