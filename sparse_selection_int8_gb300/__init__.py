"""QSA decode attention over INT8 K/V pools for GB300 (sm_103a).

A thin Python binding of the C ABI in ``include/qsa.h`` (libqsa.so, built
in-tree by :mod:`sparse_selection_int8_gb300.build`).  The functions keep the
C names and only marshal arguments: torch CUDA tensors (or raw device
addresses as ints) become pointers, and the current torch stream becomes the
launch stream.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU fallback.  Loading fails loudly when the library is
missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from .build import LIB as _LIB_PATH

QSA_OK = 0
QSA_ERR_INVALID_ARG = -1
QSA_ERR_UNSUPPORTED = -2
QSA_ERR_WORKSPACE = -3
QSA_ERR_CUDA = -4

QSA_F32 = 0
QSA_BF16 = 1

QSA_ALGO_AUTO = 0
QSA_ALGO_SIMT = 1
QSA_ALGO_TCGEN05 = 2

QSA_STATUS_BAD_POSITION = 0x1
QSA_STATUS_BAD_SLOT = 0x2
QSA_STATUS_BAD_OFFSETS = 0x4
QSA_STATUS_TIMEOUT = 0x8
QSA_STATUS_NOT_RESIDENT = 0x10
QSA_STATUS_BAD_LIMITS = 0x20
QSA_STATUS_LAUNCH = 0x40
QSA_STATUS_BAD_EXTENT = 0x80

HEAD_DIM = 256


class QsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {qsa_status_string(code)} ({code})")


class qsa_shape(ctypes.Structure):
    _fields_ = [
        ("n_kv_heads", ctypes.c_int32),
        ("q_per_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("n_queries", ctypes.c_int32),
        ("pool_cells", ctypes.c_int32),
        ("page_table_len", ctypes.c_int32),
        ("chunk_cells", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("q_dtype", ctypes.c_int32),
        ("algo", ctypes.c_int32),
        ("page_cells", ctypes.c_int32),
    ]


class qsa_select_shape(ctypes.Structure):
    _fields_ = [
        ("n_queries", ctypes.c_int32),
        ("idx_heads", ctypes.c_int32),
        ("idx_dim", ctypes.c_int32),
        ("block_cells", ctypes.c_int32),
        ("max_blocks", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
    ]


def make_shape(*, n_kv_heads: int, q_per_kv: int, n_queries: int, pool_cells: int,
               page_table_len: int, chunk_cells: int, softmax_scale: float,
               q_dtype: int = QSA_F32, algo: int = QSA_ALGO_AUTO,
               head_dim: int = HEAD_DIM, page_cells: int = 1) -> qsa_shape:
    return qsa_shape(n_kv_heads, q_per_kv, head_dim, n_queries, pool_cells, page_table_len,
                     chunk_cells, softmax_scale, q_dtype, algo, page_cells)


_lib = None

_VP = ctypes.c_void_p
_SIG = {
    "qsa_workspace_bytes": ([ctypes.POINTER(qsa_shape), ctypes.c_int32, ctypes.c_int32,
                             ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int32),
    "qsa_decode_attn_step": ([ctypes.POINTER(qsa_shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                              ctypes.c_int32, _VP, _VP, ctypes.c_size_t, _VP, _VP],
                             ctypes.c_int32),
    "qsa_decode_attn_batch": ([ctypes.POINTER(qsa_shape), ctypes.c_int32, _VP, _VP, _VP, _VP,
                               _VP, _VP, _VP, _VP, ctypes.c_int32, _VP, _VP, ctypes.c_size_t,
                               _VP, _VP], ctypes.c_int32),
    "qsa_partials_view": ([ctypes.POINTER(qsa_shape), ctypes.c_int32, ctypes.c_int32, _VP,
                           ctypes.POINTER(_VP), ctypes.POINTER(_VP), ctypes.POINTER(_VP),
                           ctypes.POINTER(ctypes.c_int32)], ctypes.c_int32),
    "qsa_status_string": ([ctypes.c_int32], ctypes.c_char_p),
    "qsa_decode_attn_step_noalloc": ([ctypes.POINTER(qsa_shape), _VP, _VP, _VP, _VP, _VP, _VP,
                                      _VP, ctypes.c_int32, _VP, _VP, _VP], ctypes.c_int32),
    "qsa_decode_attn_batch_limited": ([ctypes.POINTER(qsa_shape), ctypes.c_int32, _VP, _VP, _VP,
                                       _VP, _VP, _VP, _VP, _VP, ctypes.c_int32, _VP, _VP, _VP,
                                       ctypes.c_size_t, _VP, _VP], ctypes.c_int32),
    "qsa_kv_append": ([ctypes.POINTER(qsa_shape), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                       _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int32),
    "qsa_set_wait_limit": ([ctypes.c_int64], None),
    "qsa_select_workspace_bytes": ([ctypes.POINTER(qsa_select_shape), ctypes.c_int32,
                                    ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int32),
    "qsa_select_blocks": ([ctypes.POINTER(qsa_select_shape), ctypes.c_int32, _VP, _VP, _VP, _VP, _VP,
                           _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP, _VP], ctypes.c_int32),
}


def library_path() -> str:
    return _LIB_PATH


def load_library(path: Optional[str] = None):
    """Load libqsa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"libqsa.so not found at {p}: build it with "
            "`python -m sparse_selection_int8_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIG.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("device tensor expected")
    if not x.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str):
    if code != QSA_OK:
        raise QsaError(code, where)


def qsa_set_wait_limit(cycles: int) -> None:
    """Testing aid: bound of the kernels' device-side waits in SM clock
    cycles for later calls (0 restores the default)."""
    load_library().qsa_set_wait_limit(int(cycles))


def qsa_status_string(code: int) -> str:
    return load_library().qsa_status_string(int(code)).decode()


def qsa_workspace_bytes(shape: qsa_shape, n_seq: int, max_selected: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().qsa_workspace_bytes(ctypes.byref(shape), int(n_seq),
                                                int(max_selected), ctypes.byref(out)),
           "qsa_workspace_bytes")
    return int(out.value)


def qsa_decode_attn_step(shape: qsa_shape, q, k_pool, v_pool, k_scale, v_scale, page_table,
                         sel, n_sel: int, out, workspace, workspace_bytes: int,
                         status=None, stream=None) -> None:
    _check(load_library().qsa_decode_attn_step(
        ctypes.byref(shape), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
        _ptr(v_scale), _ptr(page_table), _ptr(sel), int(n_sel), _ptr(out), _ptr(workspace),
        int(workspace_bytes), _ptr(status), _stream(stream)), "qsa_decode_attn_step")


def qsa_decode_attn_batch(shape: qsa_shape, n_seq: int, q, k_pool, v_pool, k_scale, v_scale,
                          page_table, sel, sel_offsets, max_selected: int, out, workspace,
                          workspace_bytes: int, status=None, stream=None) -> None:
    _check(load_library().qsa_decode_attn_batch(
        ctypes.byref(shape), int(n_seq), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
        _ptr(v_scale), _ptr(page_table), _ptr(sel), _ptr(sel_offsets), int(max_selected),
        _ptr(out), _ptr(workspace), int(workspace_bytes), _ptr(status), _stream(stream)),
        "qsa_decode_attn_batch")


def qsa_decode_attn_batch_limited(shape: qsa_shape, n_seq: int, q, k_pool, v_pool, k_scale,
                                  v_scale, page_table, sel, sel_offsets, max_selected: int,
                                  q_limit, out, workspace, workspace_bytes: int, status=None,
                                  stream=None) -> None:
    _check(load_library().qsa_decode_attn_batch_limited(
        ctypes.byref(shape), int(n_seq), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
        _ptr(v_scale), _ptr(page_table), _ptr(sel), _ptr(sel_offsets), int(max_selected),
        _ptr(q_limit), _ptr(out), _ptr(workspace), int(workspace_bytes), _ptr(status),
        _stream(stream)), "qsa_decode_attn_batch_limited")


def qsa_decode_attn_step_noalloc(shape: qsa_shape, q, k_pool, v_pool, k_scale, v_scale,
                                 page_table, sel, n_sel: int, out, status=None,
                                 stream=None) -> None:
    """qsa_decode_attn_step with the library's fixed scratch array instead of
    a workspace (for callers that cannot allocate device memory)."""
    _check(load_library().qsa_decode_attn_step_noalloc(
        ctypes.byref(shape), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
        _ptr(v_scale), _ptr(page_table), _ptr(sel), int(n_sel), _ptr(out), _ptr(status),
        _stream(stream)), "qsa_decode_attn_step_noalloc")


def qsa_partials_view(shape: qsa_shape, n_seq: int, max_selected: int, workspace):
    """Device addresses (m, l, o) of the chunk partials and the chunk count."""
    m, l, o = _VP(), _VP(), _VP()
    nch = ctypes.c_int32(0)
    _check(load_library().qsa_partials_view(ctypes.byref(shape), int(n_seq), int(max_selected),
                                             _ptr(workspace), ctypes.byref(m), ctypes.byref(l),
                                             ctypes.byref(o), ctypes.byref(nch)),
           "qsa_partials_view")
    return m.value, l.value, o.value, int(nch.value)




def qsa_kv_append(shape: qsa_shape, n_seq: int, n_new: int, kv_dtype: int, k_new, v_new,
                  positions, page_table, k_pool, v_pool, k_scale, v_scale, status=None,
                  stream=None) -> None:
    """Quantise new K/V rows into the INT8 pools (see include/qsa.h)."""
    _check(load_library().qsa_kv_append(
        ctypes.byref(shape), int(n_seq), int(n_new), int(kv_dtype), _ptr(k_new), _ptr(v_new),
        _ptr(positions), _ptr(page_table), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
        _ptr(v_scale), _ptr(status), _stream(stream)), "qsa_kv_append")




def qsa_select_workspace_bytes(shape: qsa_select_shape, n_seq: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().qsa_select_workspace_bytes(ctypes.byref(shape), int(n_seq), ctypes.byref(out)),
           "qsa_select_workspace_bytes")
    return int(out.value)


def qsa_select_blocks(shape: qsa_select_shape, n_seq: int, q_idx, pooled, n_live, steps, scores, kept,
                      sel, sel_offsets, workspace, workspace_bytes: int, status=None, stream=None) -> None:
    """Block scores, top-k and the selected-cell list (see include/qsa.h)."""
    _check(load_library().qsa_select_blocks(
        ctypes.byref(shape), int(n_seq), _ptr(q_idx), _ptr(pooled), _ptr(n_live), _ptr(steps),
        _ptr(scores), _ptr(kept), _ptr(sel), _ptr(sel_offsets), _ptr(workspace), int(workspace_bytes),
        _ptr(status), _stream(stream)), "qsa_select_blocks")


from .device import DeviceAppend, DeviceProblem, DeviceSelection, run_problem, partials_of  # noqa: E402,F401
