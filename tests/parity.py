"""Shared tolerance of the GPU-vs-oracle parity tests.

Two bars, both required.

1. Per element: max abs error <= 2e-3 and max rel error <= 1e-2 on fp32
   outputs.  An elementwise relative error is meaningless where the exact
   output is near zero, so the relative test divides by max(|ref|, 0.2):
   0.2 = 2e-3 / 1e-2, the magnitude where the two bounds meet.  Below it the
   absolute bound governs; above it the relative one does.  The raw
   relative error is reported too.
2. Per output row (the last axis: one query head's D values): ||gpu - ref|| /
   max(||ref||, 1e-2) <= 2e-3.  The workloads' outputs are softmax averages
   of a few x 1e-2 per element, where bar 1 alone would pass errors of
   several per cent.  The decode path's rounding (f16 P', query split into
   f16 high and low parts, fp32 sums) measures 2-4e-4 of the row's norm,
   and up to 8.5e-4 where a wide window with causal limits keeps the f16
   high part alone; the prompt path's 3.6e-4.  So a regression to several
   times that fails here.  Rows whose exact output is zero (no valid cell)
   are held to an absolute norm of 2e-5.
"""
import numpy as np

ATOL = 2e-3
RTOL = 1e-2
REL_FLOOR = ATOL / RTOL
ROW_RTOL = 2e-3
ROW_FLOOR = 1e-2


def errors(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(gpu - ref)
    D = ref.shape[-1] if ref.ndim else 1
    dr = np.linalg.norm(d.reshape(-1, D), axis=1)
    rr = np.linalg.norm(ref.reshape(-1, D), axis=1)
    return {
        "max_abs": float(d.max(initial=0.0)),
        "max_rel_floored": float((d / np.maximum(np.abs(ref), REL_FLOOR)).max(initial=0.0)),
        "max_rel_raw": float((d / np.maximum(np.abs(ref), 1e-30)).max(initial=0.0)),
        "max_row_rel": float((dr / np.maximum(rr, ROW_FLOOR)).max(initial=0.0)),
    }


def assert_parity(gpu, ref, what=""):
    gpu = np.asarray(gpu)
    assert gpu.shape == np.asarray(ref).shape, (what, gpu.shape, np.asarray(ref).shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    e = errors(gpu, ref)
    assert e["max_abs"] <= ATOL and e["max_rel_floored"] <= RTOL, f"{what}: {e}"
    assert e["max_row_rel"] <= ROW_RTOL, f"{what}: per-row error {e}"
    return e
