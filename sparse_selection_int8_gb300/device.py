"""Device-resident problem: uploads host arrays with torch and calls the C ABI.

Only marshalling lives here: torch allocates device memory and copies the
host arrays; every computation is a libqsa kernel launched through
``qsa_decode_attn_step`` / ``qsa_decode_attn_batch``.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from . import (QSA_ALGO_AUTO, QSA_BF16, QSA_F32, make_shape, qsa_decode_attn_batch,
               qsa_decode_attn_batch_limited, qsa_decode_attn_step, qsa_kv_append,
               qsa_partials_view, qsa_select_blocks, qsa_select_shape, qsa_select_workspace_bytes,
               qsa_workspace_bytes)


def _to_dev(torch, a: np.ndarray, device, pin: bool = False):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if pin:
        t = t.pin_memory()
    return t.to(device, non_blocking=pin)


class DeviceProblem:
    """A problem (as drawn by the input generator) resident in device memory.

    Attributes mirror the C ABI arguments; ``out`` and ``workspace`` are
    allocated once and reused by every ``run``.
    """

    def __init__(self, p, device: str = "cuda", algo: int = QSA_ALGO_AUTO,
                 max_selected: Optional[int] = None):
        import torch
        self.p = p
        self.device = device
        if p.q_dtype == "bf16":
            self.q = _to_dev(torch, np.asarray(p.q).view(np.int16), device).view(torch.bfloat16)
        else:
            self.q = _to_dev(torch, p.q.astype(np.float32), device)
        self.k_pool = _to_dev(torch, p.k_pool, device)
        self.v_pool = _to_dev(torch, p.v_pool, device)
        self.k_scale = _to_dev(torch, p.k_scale, device)
        self.v_scale = _to_dev(torch, p.v_scale, device)
        self.page_table = _to_dev(torch, p.page_table, device)
        self.sel = _to_dev(torch, p.sel if p.sel.size else np.zeros(1, np.int32), device)
        self.sel_offsets = _to_dev(torch, p.sel_offsets, device)
        lim = getattr(p, "q_limit", None)
        self.q_limit = None if lim is None else _to_dev(torch, np.asarray(lim, np.int32), device)
        self.n_seq = p.n_seq
        self.max_selected = p.max_selected if max_selected is None else max_selected
        self.shape = make_shape(n_kv_heads=p.n_kv_heads, q_per_kv=p.q_per_kv,
                                n_queries=p.n_queries, pool_cells=p.pool_cells,
                                page_table_len=p.page_table_len, chunk_cells=p.chunk_cells,
                                softmax_scale=p.softmax_scale,
                                q_dtype=QSA_BF16 if p.q_dtype == "bf16" else QSA_F32,
                                algo=algo, head_dim=p.head_dim,
                                page_cells=getattr(p, "page_cells", 1))
        self.ws_bytes = qsa_workspace_bytes(self.shape, self.n_seq, self.max_selected)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        self.out = torch.empty((p.n_seq, p.n_queries, p.n_kv_heads * p.q_per_kv, p.head_dim),
                               dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def run(self, batch: Optional[bool] = None, stream=None, out=None):
        """One call.  ``batch=None`` uses the step entry for one sequence and
        the batch entry otherwise."""
        out = self.out if out is None else out
        if self.q_limit is not None:  # causal limits: the batch entry that takes them
            qsa_decode_attn_batch_limited(self.shape, self.n_seq, self.q, self.k_pool, self.v_pool,
                                          self.k_scale, self.v_scale, self.page_table, self.sel,
                                          self.sel_offsets, self.max_selected, self.q_limit, out,
                                          self.workspace, self.ws_bytes, self.status, stream)
            return out
        if batch is None:
            batch = self.n_seq != 1
        if batch:
            qsa_decode_attn_batch(self.shape, self.n_seq, self.q, self.k_pool, self.v_pool,
                                  self.k_scale, self.v_scale, self.page_table, self.sel,
                                  self.sel_offsets, self.max_selected, out, self.workspace,
                                  self.ws_bytes, self.status, stream)
        else:
            assert self.n_seq == 1
            qsa_decode_attn_step(self.shape, self.q, self.k_pool, self.v_pool, self.k_scale,
                                 self.v_scale, self.page_table, self.sel,
                                 int(self.p.sel.shape[0]), out, self.workspace, self.ws_bytes,
                                 self.status, stream)
        return out


class DeviceAppend:
    """An append call (as drawn by the input generator) resident in device
    memory: new rows, positions, page table, and the pools it writes."""

    def __init__(self, a, device: str = "cuda"):
        import torch
        self.a = a
        if a.dtype == "bf16":
            self.k_new = _to_dev(torch, np.asarray(a.k_new).view(np.int16), device).view(torch.bfloat16)
            self.v_new = _to_dev(torch, np.asarray(a.v_new).view(np.int16), device).view(torch.bfloat16)
        else:
            self.k_new = _to_dev(torch, a.k_new.astype(np.float32), device)
            self.v_new = _to_dev(torch, a.v_new.astype(np.float32), device)
        self.positions = _to_dev(torch, a.positions, device)
        self.page_table = _to_dev(torch, a.page_table, device)
        self.k_pool = _to_dev(torch, a.k_pool, device)
        self.v_pool = _to_dev(torch, a.v_pool, device)
        self.k_scale = _to_dev(torch, a.k_scale, device)
        self.v_scale = _to_dev(torch, a.v_scale, device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.kv_dtype = QSA_BF16 if a.dtype == "bf16" else QSA_F32
        self.shape = make_shape(n_kv_heads=a.n_kv_heads, q_per_kv=1, n_queries=1,
                                pool_cells=a.pool_cells, page_table_len=a.page_table_len,
                                chunk_cells=1, softmax_scale=1.0, head_dim=a.head_dim,
                                page_cells=getattr(a, "page_cells", 1))

    def run(self, stream=None):
        a = self.a
        qsa_kv_append(self.shape, a.n_seq, a.n_new, self.kv_dtype, self.k_new, self.v_new,
                      self.positions, self.page_table, self.k_pool, self.v_pool, self.k_scale,
                      self.v_scale, self.status, stream)


class DeviceSelection:
    """A block-selection call (as drawn by the input generator) resident in
    device memory, with its outputs: scores, kept block ids, the list and
    its offsets."""

    def __init__(self, sp, device: str = "cuda"):
        import torch
        self.sp = sp
        self.q_idx = _to_dev(torch, sp.q_idx.astype(np.float32), device)
        self.pooled = _to_dev(torch, np.asarray(sp.pooled).view(np.int16), device)
        self.n_live = _to_dev(torch, sp.n_live.astype(np.int32), device)
        self.steps = None if sp.steps is None else _to_dev(torch, sp.steps.astype(np.int32), device)
        self.shape = qsa_select_shape(sp.n_queries, sp.idx_heads, sp.idx_dim, sp.block_cells,
                                      sp.max_blocks, sp.top_k)
        B, T = sp.n_seq, sp.n_queries
        self.max_selected = min(T * sp.top_k, sp.max_blocks) * sp.block_cells
        self.scores = torch.empty((B, T, sp.max_blocks), dtype=torch.float32, device=device)
        self.kept = torch.empty((B, T, sp.top_k), dtype=torch.int32, device=device)
        self.sel = torch.empty(max(B * self.max_selected, 1), dtype=torch.int32, device=device)
        self.sel_offsets = torch.empty(B + 1, dtype=torch.int32, device=device)
        self.ws_bytes = qsa_select_workspace_bytes(self.shape, B)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def run(self, stream=None):
        qsa_select_blocks(self.shape, self.sp.n_seq, self.q_idx, self.pooled, self.n_live, self.steps,
                          self.scores, self.kept, self.sel, self.sel_offsets, self.workspace, self.ws_bytes,
                          self.status, stream)

    def result(self):
        """(scores, kept, sel, sel_offsets) copied to host."""
        off = self.sel_offsets.cpu().numpy()
        return (self.scores.cpu().numpy(), self.kept.cpu().numpy(), self.sel[:int(off[-1])].cpu().numpy(), off)


def run_problem(p, algo: int = QSA_ALGO_AUTO, batch: Optional[bool] = None) -> np.ndarray:
    """Upload, run once, and return the output as a float32 numpy array."""
    import torch
    dp = DeviceProblem(p, algo=algo)
    out = dp.run(batch=batch)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def partials_of(dp: DeviceProblem):
    """Copy the chunk partials of the last call to host: (m, l, o) with shapes
    [n_seq][G][n_chunks][R] and [n_seq][G][n_chunks][R][D]."""
    import torch
    m_ptr, l_ptr, o_ptr, n_chunks = qsa_partials_view(dp.shape, dp.n_seq, dp.max_selected,
                                                      dp.workspace)
    p = dp.p
    R = p.n_queries * p.q_per_kv
    rows = dp.n_seq * p.n_kv_heads * n_chunks * R
    base = dp.workspace.data_ptr()
    ws = dp.workspace

    def view(ptr, count):
        off = ptr - base
        return ws[off:off + count * 4].view(torch.float32).cpu().numpy()

    m = view(m_ptr, rows).reshape(dp.n_seq, p.n_kv_heads, n_chunks, R)
    l = view(l_ptr, rows).reshape(dp.n_seq, p.n_kv_heads, n_chunks, R)
    o = view(o_ptr, rows * p.head_dim).reshape(dp.n_seq, p.n_kv_heads, n_chunks, R, p.head_dim)
    return m, l, o
