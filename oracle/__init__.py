"""fp64 CPU oracle for QSA decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline
leg and its reference arm) may import this package.  The product library
never calls it and has no CPU fallback.

The arithmetic lives in ``qsa_oracle.c`` (plain C, double precision), built
with gcc into ``oracle/_build/``.  This wrapper only marshals numpy arrays.
It widens the caller's queries to double exactly (fp32 -> double, or bf16 bit
patterns -> fp32 -> double); no other value is converted.

Every function here is pinned by ``tests/test_oracle_pins.py`` (closed forms,
invariants, a 60-digit decimal brute force and planted-mistake checks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libqsa_oracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {0: "ok", 1: "selected position outside the page table",
          2: "page-table slot outside the pool", 3: "bad argument", 4: "out of memory"}


class OracleError(RuntimeError):
    pass


def compile_library(src: str = _SRC, out: str = _LIB_PATH, extra_flags: Sequence[str] = ()) -> str:
    """Compile the C oracle into a shared library (gcc, OpenMP when available)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", *extra_flags]
    try:
        subprocess.run(base + ["-fopenmp", "-o", tmp, src, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp, src, "-lm"], check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build() -> str:
    """Build the oracle library if missing or older than its source."""
    with _lock:
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            compile_library()
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.qsa_oracle_attend_row.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, i32, dbl, P]
    lib.qsa_oracle_attend_row.restype = i32
    lib.qsa_oracle_chunk_partial.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, i32,
                                             i32, dbl, P, P, P]
    lib.qsa_oracle_chunk_partial.restype = i32
    lib.qsa_oracle_merge.argtypes = [i32, i32, P, P, P, P]
    lib.qsa_oracle_merge.restype = None
    lib.qsa_oracle_decode_attn.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, dbl, P, P,
                                           P, P, P, P, P, P, P, P, i64, P]
    lib.qsa_oracle_decode_attn.restype = i32
    lib.qsa_oracle_threads.argtypes = []
    lib.qsa_oracle_threads.restype = i32
    lib.qsa_oracle_set_threads.argtypes = [i32]
    lib.qsa_oracle_set_threads.restype = None
    return lib


def load(path: Optional[str] = None):
    """Load (building if needed) the oracle library; ``path`` loads another
    build of it, e.g. a planted-mistake variant compiled by a test."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def widen_queries(q: np.ndarray, q_dtype: str) -> np.ndarray:
    """Exact widening of the caller's queries to double."""
    if q_dtype == "bf16":
        f32 = (np.asarray(q, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
        return f32.astype(np.float64)
    return np.asarray(q, dtype=np.float32).astype(np.float64)


def _limit(limit) -> int:
    return 0x7FFFFFFF if limit is None else int(limit)


def _check(err: int):
    if err:
        raise OracleError(ERRORS.get(err, f"oracle error {err}"))


def threads() -> int:
    return load().qsa_oracle_threads()


def set_threads(n: int) -> None:
    load().qsa_oracle_set_threads(int(n))


def attend_row(q_row, k_codes, v_codes, k_scale, v_scale, page_table, sel,
               softmax_scale: float, lib=None, page_cells: int = 1,
               limit: Optional[int] = None) -> np.ndarray:
    """One query row against one (sequence, KV head): the unchunked definition.

    q_row [D] (any float dtype, used as double), k/v codes int8 [pool][D],
    scales fp32 [pool], page_table int32 [pages] (pages of page_cells cells),
    sel int32 [n] logical positions; ``limit``: the row sees only positions
    below it (None: no limit).
    """
    lib = lib or load()
    q = _c(q_row, np.float64)
    k = _c(k_codes, np.int8)
    v = _c(v_codes, np.int8)
    ks = _c(k_scale, np.float32)
    vs = _c(v_scale, np.float32)
    pt = _c(page_table, np.int32)
    sl = _c(sel, np.int32)
    D = q.shape[0]
    out = np.zeros(D, dtype=np.float64)
    _check(lib.qsa_oracle_attend_row(D, k.shape[0], pt.shape[0], int(page_cells), _limit(limit),
                                     _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(ks), _ptr(vs), _ptr(pt), _ptr(sl), sl.shape[0],
                                     float(softmax_scale), _ptr(out)))
    return out


def chunk_partial(q_row, k_codes, v_codes, k_scale, v_scale, page_table, sel, start: int,
                  count: int, softmax_scale: float, lib=None, page_cells: int = 1,
                  limit: Optional[int] = None):
    """(m, l, o) of list positions [start, start+count) for one query row."""
    lib = lib or load()
    q = _c(q_row, np.float64)
    k = _c(k_codes, np.int8)
    v = _c(v_codes, np.int8)
    ks = _c(k_scale, np.float32)
    vs = _c(v_scale, np.float32)
    pt = _c(page_table, np.int32)
    sl = _c(sel, np.int32)
    if start < 0 or count < 0 or start + count > sl.shape[0]:
        raise OracleError("chunk outside the list")
    D = q.shape[0]
    m = np.zeros(1, np.float64)
    l = np.zeros(1, np.float64)
    o = np.zeros(D, np.float64)
    _check(lib.qsa_oracle_chunk_partial(D, k.shape[0], pt.shape[0], int(page_cells), _limit(limit),
                                        _ptr(q), _ptr(k), _ptr(v),
                                        _ptr(ks), _ptr(vs), _ptr(pt), _ptr(sl), int(start),
                                        int(count), float(softmax_scale), _ptr(m), _ptr(l),
                                        _ptr(o)))
    return float(m[0]), float(l[0]), o


def merge(m, l, o, lib=None) -> np.ndarray:
    """Merge chunk partials: m, l [n_chunks], o [n_chunks][D]."""
    lib = lib or load()
    m = _c(m, np.float64)
    l = _c(l, np.float64)
    o = _c(o, np.float64)
    n, D = o.shape
    out = np.zeros(D, np.float64)
    lib.qsa_oracle_merge(D, n, _ptr(m), _ptr(l), _ptr(o), _ptr(out))
    return out


def row_partials(q_row, k_codes, v_codes, k_scale, v_scale, page_table, sel,
                 chunk_cells: int, softmax_scale: float, lib=None, page_cells: int = 1):
    """Partials of every chunk of the list for one row: arrays m, l, o."""
    n = int(np.asarray(sel).shape[0])
    n_chunks = (n + chunk_cells - 1) // chunk_cells
    D = int(np.asarray(q_row).shape[0])
    ms = np.zeros(n_chunks)
    ls = np.zeros(n_chunks)
    os_ = np.zeros((n_chunks, D))
    for c in range(n_chunks):
        start = c * chunk_cells
        cnt = min(chunk_cells, n - start)
        ms[c], ls[c], os_[c] = chunk_partial(q_row, k_codes, v_codes, k_scale, v_scale,
                                             page_table, sel, start, cnt, softmax_scale, lib,
                                             page_cells)
    return ms, ls, os_


def decode_attn(p, rows: Optional[Sequence[int]] = None, lib=None) -> np.ndarray:
    """The whole call for a problem ``p`` (attributes as drawn by the input
    generator).  Returns double [B][T][G*H][D], or [len(rows)][D] when flat row
    ids ((b*T + t)*G*H + h) are given."""
    lib = lib or load()
    q = widen_queries(p.q, p.q_dtype)
    q = np.ascontiguousarray(q)
    k = _c(p.k_pool, np.int8)
    v = _c(p.v_pool, np.int8)
    ks = _c(p.k_scale, np.float32)
    vs = _c(p.v_scale, np.float32)
    pt = _c(p.page_table, np.int32)
    sl = _c(p.sel, np.int32)
    offs = _c(p.sel_offsets, np.int64)
    lim = getattr(p, "q_limit", None)
    lim = None if lim is None else _c(lim, np.int32).reshape(p.n_seq, p.n_queries)
    GH = p.n_kv_heads * p.q_per_kv
    total = p.n_seq * p.n_queries * GH
    if rows is None:
        out = np.zeros((total, p.head_dim), np.float64)
        rows_arr = None
        n_rows = total
    else:
        rows_arr = _c(rows, np.int64)
        n_rows = rows_arr.shape[0]
        out = np.zeros((n_rows, p.head_dim), np.float64)
    _check(lib.qsa_oracle_decode_attn(
        p.n_seq, p.n_kv_heads, p.q_per_kv, p.head_dim, p.n_queries, p.pool_cells,
        p.page_table_len, int(getattr(p, "page_cells", 1)), float(p.softmax_scale), _ptr(q), _ptr(k), _ptr(v), _ptr(ks),
        _ptr(vs), _ptr(pt), _ptr(sl), _ptr(offs), _ptr(lim) if lim is not None else None,
        _ptr(rows_arr) if rows_arr is not None else None, n_rows, _ptr(out)))
    if rows is None:
        return out.reshape(p.n_seq, p.n_queries, GH, p.head_dim)
    return out


def flat_row(p, b: int, t: int, h: int) -> int:
    """Flat output-row id of (sequence b, query t, head h = g*H + j)."""
    GH = p.n_kv_heads * p.q_per_kv
    return (b * p.n_queries + t) * GH + h
