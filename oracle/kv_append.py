"""INT8 K/V quantise-append oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU
baseline) may import this module; the product library never calls it.

What it defines.  The pages name the step ("Strata PR #2220, R9-gpu-8: one
exact launch for QSA K and V", implementation handoff: K normalisation,
rotation and the KV append follow the K/V projections of a QSA layer) and
the format it writes (INT8 K/V pools with one fp32 scale per cell, read by
the decode-attention step), but print no quantiser.  The reading taken here
is the plainest symmetric one:

* one scale per (cell, KV head) for K and one for V: ``scale = max|x| / 127``
  (fp32 division, correctly rounded);
* ``code = x / scale`` (fp32 division) rounded to the nearest integer, ties
  to even, kept in [-127, 127];
* a row of zeros gets scale 0 and zero codes;
* new cell i of sequence b goes to the pool slot of ``pos = positions[b][i]``:
  with pages of P cells (``page_cells``, 1 by default) that is
  ``page_table[b][pos // P] * P + pos % P``; a position outside the page
  table, a page entry of -1 (the cell is not resident) or a page entry
  outside the pool writes nothing and raises a status bit.

All arithmetic is float32, element by element, so a device kernel that makes
the same float32 operations reaches the same codes and scales bit for bit.
bf16 inputs are widened to float32 exactly first.  Rows must be finite.

Pinned by ``tests/test_append_oracle.py`` (hand-worked rows in
``tests/golden/append_rows.txt``, the rounding bound, the max element, zero
rows, power-of-two scaling, routing).
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

STATUS_BAD_POSITION = 0x1
STATUS_BAD_SLOT = 0x2
STATUS_NOT_RESIDENT = 0x10

_F127 = np.float32(127.0)


def quantize_row(x) -> Tuple[np.ndarray, np.float32]:
    """One row -> (int8 codes, fp32 scale)."""
    x = np.asarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("rows must be finite")
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    if amax == 0:
        return np.zeros(x.shape, np.int8), np.float32(0.0)
    scale = np.float32(amax / _F127)
    codes = np.rint(np.divide(x, scale, dtype=np.float32))
    return np.clip(codes, -127, 127).astype(np.int8), scale


def widen(rows: np.ndarray, dtype: str) -> np.ndarray:
    """The new rows as float32 (bf16 bit patterns widened exactly)."""
    if dtype == "bf16":
        return (np.asarray(rows).astype(np.uint32) << np.uint32(16)).view(np.float32)
    return np.asarray(rows, dtype=np.float32)


def kv_append(a, k_pool: np.ndarray, v_pool: np.ndarray, k_scale: np.ndarray,
              v_scale: np.ndarray) -> int:
    """Apply one append call ``a`` (an AppendProblem) to the pools in place.

    Pools ``[B][G][N_pool][D]`` int8, scales ``[B][G][N_pool]`` fp32.
    Returns the status bits the call raises."""
    k_new = widen(a.k_new, a.dtype)
    v_new = widen(a.v_new, a.dtype)
    P = int(getattr(a, "page_cells", 1))
    status = 0
    for b in range(a.n_seq):
        for i in range(a.n_new):
            pos = int(a.positions[b, i])
            if pos < 0 or pos >= a.page_table_len * P:
                status |= STATUS_BAD_POSITION
                continue
            page = int(a.page_table[b, pos // P])
            if page == -1:
                status |= STATUS_NOT_RESIDENT
                continue
            if page < 0 or page >= a.pool_cells // P:
                status |= STATUS_BAD_SLOT
                continue
            slot = page * P + pos % P
            for g in range(a.n_kv_heads):
                k_pool[b, g, slot], k_scale[b, g, slot] = quantize_row(k_new[b, i, g])
                v_pool[b, g, slot], v_scale[b, g, slot] = quantize_row(v_new[b, i, g])
    return status
