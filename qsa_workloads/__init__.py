"""Seeded synthetic inputs for QSA decode attention over INT8 K/V pools.

This module only draws inputs: queries, INT8 K/V pools with per-cell fp32
scales, permuted page tables and selected-cell lists.  It holds none of the
attention arithmetic, so both the fp64 oracle (``oracle/``) and the CUDA
library (``sparse_selection_int8_gb300``) can be fed from it without sharing
any of the method's steps.

Shapes and distributions follow the workloads the Strata pages describe
("Strata PR #2220, attn_chunk_q8_v3_kernel", kernel table: synthetic INT8
pools, permuted page table, 12 query heads per KV head, head_dim 256,
600 / 2,051 selected cells, 1-4 queries) and the five named configurations
below.  Random numbers come from numpy's PCG64 bit generator seeded with the
configuration seed; every array is produced on the host.

Layouts (all C-contiguous):

* ``q``           f32 ``[B][T][G*H][D]`` (or bf16 bit patterns as uint16)
* ``k_pool``      int8 ``[B][G][N_pool][D]`` (same for ``v_pool``)
* ``k_scale``     f32 ``[B][G][N_pool]`` (same for ``v_scale``)
* ``page_table``  int32 ``[B][N_log]``; entry = pool slot, or -1 (masked)
* ``sel``         int32 ``[sum n_b]`` logical positions, CSR by ``sel_offsets``
* ``sel_offsets`` int32 ``[B+1]``

Query head ``j`` of KV head ``g`` is head index ``g*H + j``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

SEED_BASE = 0x51A5E000


@dataclass
class Problem:
    """One decode-attention call: inputs plus the shape parameters."""

    n_seq: int
    n_kv_heads: int
    q_per_kv: int
    head_dim: int
    n_queries: int
    pool_cells: int
    page_table_len: int
    chunk_cells: int
    softmax_scale: float
    q_dtype: str  # "f32" or "bf16"
    q: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    k_scale: np.ndarray
    v_scale: np.ndarray
    page_table: np.ndarray
    sel: np.ndarray
    sel_offsets: np.ndarray
    name: str = ""
    notes: dict = field(default_factory=dict)
    page_cells: int = 1  # cells per page: the page table has one entry per page
    # optional causal limits [B][T]: query t of sequence b sees positions < q_limit[b][t]
    q_limit: Optional[np.ndarray] = None

    @property
    def n_positions(self) -> int:
        """Logical positions the page table covers."""
        return self.page_table_len * self.page_cells

    @property
    def rows_per_kv(self) -> int:
        """Query rows scored per KV head: T queries x H heads."""
        return self.n_queries * self.q_per_kv

    @property
    def n_selected(self) -> np.ndarray:
        return np.diff(self.sel_offsets.astype(np.int64))

    @property
    def max_selected(self) -> int:
        return int(self.n_selected.max()) if self.n_seq else 0

    def sel_of(self, b: int) -> np.ndarray:
        return self.sel[self.sel_offsets[b]:self.sel_offsets[b + 1]]


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the 16-bit patterns as uint16.  Used to draw bf16 queries.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))
    return ((b + rounding) >> np.uint64(16)).astype(np.uint16)


def f32_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _codes(rng: np.random.Generator, shape) -> np.ndarray:
    """INT8 codes uniform in [-127, 127] (the symmetric int8 range)."""
    return rng.integers(-127, 128, size=shape, dtype=np.int8)


def _scales(rng: np.random.Generator, shape) -> np.ndarray:
    """Per-cell fp32 scales uniform in [0.005, 0.02]."""
    return rng.uniform(0.005, 0.02, size=shape).astype(np.float32)


def _page_table(rng: np.random.Generator, pool_cells: int, page_table_len: int,
                mask_fraction: float) -> np.ndarray:
    """A permuted page table: logical position -> pool slot, -1 = not resident.

    With ``page_table_len == pool_cells`` it is a random permutation of the
    pool.  A longer table maps ``pool_cells`` random positions and marks the
    rest -1.  ``mask_fraction`` additionally sets that share of the entries to
    -1 (page -1 masking).
    """
    pt = np.full(page_table_len, -1, dtype=np.int32)
    mapped = min(pool_cells, page_table_len)
    where = rng.permutation(page_table_len)[:mapped]
    pt[where] = rng.permutation(pool_cells)[:mapped].astype(np.int32)
    if mask_fraction > 0:
        n_mask = int(round(mask_fraction * page_table_len))
        pt[rng.choice(page_table_len, size=n_mask, replace=False)] = -1
    return pt


def _select_sorted(rng: np.random.Generator, page_table_len: int, n: int) -> np.ndarray:
    """n logical positions drawn without replacement, sorted ascending."""
    return np.sort(rng.choice(page_table_len, size=n, replace=False)).astype(np.int32)


def _select_clustered(rng: np.random.Generator, page_table_len: int, n: int,
                      clustered_share: float = 0.3, run_min: int = 8,
                      run_max: int = 64) -> np.ndarray:
    """Sorted selection where ``clustered_share`` of the cells lie in contiguous
    logical runs of length U[run_min, run_max]; the rest are isolated draws."""
    taken = np.zeros(page_table_len, dtype=bool)
    target = int(round(clustered_share * n))
    placed = 0
    while placed < target:
        run = int(rng.integers(run_min, run_max + 1))
        run = min(run, target - placed)
        start = int(rng.integers(0, page_table_len - run + 1))
        if taken[max(start - 1, 0):start + run + 1].any():
            continue  # keep runs separate so each stays a run of its own
        taken[start:start + run] = True
        placed += run
    free = np.flatnonzero(~taken)
    rest = rng.choice(free, size=n - placed, replace=False)
    taken[rest] = True
    return np.flatnonzero(taken).astype(np.int32)


def make_problem(*, n_seq: int = 1, n_kv_heads: int = 1, q_per_kv: int = 12,
                 head_dim: int = 256, n_queries: int = 1, pool_cells: int = 4096,
                 page_table_len: Optional[int] = None,
                 n_selected: Sequence[int] | int = 600, chunk_cells: int = 64,
                 softmax_scale: float = 1.0 / 16.0, q_dtype: str = "f32",
                 selection: str = "sorted", mask_fraction: float = 0.0,
                 seed: int = SEED_BASE, name: str = "", page_cells: int = 1) -> Problem:
    """Draw one seeded problem.

    ``selection`` is ``"sorted"`` (without replacement, ascending),
    ``"clustered"`` (30% of cells in runs of 8-64) or ``"full"`` (every
    logical position 0..N_log-1 in page-table order).  With ``page_cells``
    P > 1 the page table maps pages of P cells: ``page_table_len`` entries
    (default pool_cells / P), each a page of the pool or -1, covering
    ``page_table_len * P`` logical positions.
    """
    assert pool_cells % page_cells == 0
    if page_table_len is None:
        page_table_len = pool_cells // page_cells
    n_pos = page_table_len * page_cells
    if isinstance(n_selected, (int, np.integer)):
        n_list: List[int] = [int(n_selected)] * n_seq
    else:
        n_list = [int(v) for v in n_selected]
    assert len(n_list) == n_seq
    rng = np.random.Generator(np.random.PCG64(seed))
    G, H, D, T = n_kv_heads, q_per_kv, head_dim, n_queries

    k_pool = _codes(rng, (n_seq, G, pool_cells, D))
    v_pool = _codes(rng, (n_seq, G, pool_cells, D))
    k_scale = _scales(rng, (n_seq, G, pool_cells))
    v_scale = _scales(rng, (n_seq, G, pool_cells))
    pts, sels = [], []
    for b in range(n_seq):
        pts.append(_page_table(rng, pool_cells // page_cells, page_table_len, mask_fraction))
        n = n_list[b]
        if selection == "sorted":
            sels.append(_select_sorted(rng, n_pos, n))
        elif selection == "clustered":
            sels.append(_select_clustered(rng, n_pos, n))
        elif selection == "full":
            assert n == n_pos
            sels.append(np.arange(n_pos, dtype=np.int32))
        else:
            raise ValueError(selection)
    q32 = rng.standard_normal((n_seq, T, G * H, D), dtype=np.float64).astype(np.float32)
    q = bf16_bits_from_f32(q32) if q_dtype == "bf16" else q32
    offsets = np.zeros(n_seq + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(n_list)
    sel = np.concatenate(sels).astype(np.int32) if sels else np.zeros(0, np.int32)
    return Problem(n_seq=n_seq, n_kv_heads=G, q_per_kv=H, head_dim=D, n_queries=T,
                   pool_cells=pool_cells, page_table_len=page_table_len,
                   chunk_cells=chunk_cells, softmax_scale=float(softmax_scale),
                   q_dtype=q_dtype, q=np.ascontiguousarray(q), k_pool=k_pool,
                   v_pool=v_pool, k_scale=k_scale, v_scale=v_scale,
                   page_table=np.stack(pts).astype(np.int32), sel=sel,
                   sel_offsets=offsets, name=name, page_cells=page_cells)


# ---------------------------------------------------------------------------
# The five named workloads.  The numbering is the order they are listed in.
# ---------------------------------------------------------------------------

def tiny_decode(seed_offset: int = 0) -> Problem:
    """1 KV head x 12 query heads, D 256, 1 query, 4,096-cell pool, 600
    selected cells, chunk 64."""
    return make_problem(n_seq=1, n_kv_heads=1, n_queries=1, pool_cells=4096,
                        n_selected=600, chunk_cells=64,
                        seed=SEED_BASE + 1 + seed_offset, name="tiny_decode")


def qsa_decode(n_queries: int, seed_offset: int = 0) -> Problem:
    """The pages' kernel-table shape: 32,768-cell pool, 2,051 selected cells,
    1-4 queries (MTP verify window), chunk 128."""
    return make_problem(n_seq=1, n_kv_heads=1, n_queries=n_queries,
                        pool_cells=32768, n_selected=2051, chunk_cells=128,
                        seed=SEED_BASE + 2 + 16 * n_queries + seed_offset,
                        name=f"qsa_decode_T{n_queries}")


def batched_decode(seed_offset: int = 0) -> Problem:
    """16 sequences x 2 KV heads, 4 queries, 32,768-cell pools, per-sequence
    selections of U[600, 2051] cells, chunk 128."""
    rng = np.random.Generator(np.random.PCG64(SEED_BASE + 3 + seed_offset))
    n_sel = [int(v) for v in rng.integers(600, 2052, size=16)]
    return make_problem(n_seq=16, n_kv_heads=2, n_queries=4, pool_cells=32768,
                        n_selected=n_sel, chunk_cells=128,
                        seed=SEED_BASE + 3 + 1000 + seed_offset, name="batched_decode")


def long_context(seed_offset: int = 0) -> Problem:
    """8 sequences x 2 KV heads, 2 queries, 131,072-cell pools, 16,384 sorted
    selected cells with 30% clustered runs of 8-64, chunk 256 (64 chunks)."""
    return make_problem(n_seq=8, n_kv_heads=2, n_queries=2, pool_cells=131072,
                        n_selected=16384, chunk_cells=256, selection="clustered",
                        seed=SEED_BASE + 4 + seed_offset, name="long_context")


def long_context_paged(page_cells: int = 16, seed_offset: int = 0) -> Problem:
    """long_context with a page table of ``page_cells``-cell pages (a
    companion case: the clustered runs then sit on physically contiguous
    slots)."""
    return make_problem(n_seq=8, n_kv_heads=2, n_queries=2, pool_cells=131072,
                        n_selected=16384, chunk_cells=256, selection="clustered",
                        page_cells=page_cells, seed=SEED_BASE + 4 + seed_offset,
                        name=f"long_context_pages{page_cells}")


def prompt_shaped(seed_offset: int = 0, n_queries: int = 2048,
                  pool_cells: int = 32768, chunk_cells: int = 11008) -> Problem:
    """1 KV head x 12 query heads, 2,048 bf16 queries against all 32,768 cells
    in page-table order, no causal mask.  Chunk 11,008 cells: three split-K
    chunks (86, 86 and 84 tiles of 128 cells)."""
    return make_problem(n_seq=1, n_kv_heads=1, n_queries=n_queries,
                        pool_cells=pool_cells, n_selected=pool_cells,
                        chunk_cells=chunk_cells, q_dtype="bf16", selection="full",
                        seed=SEED_BASE + 5 + seed_offset, name="prompt_shaped")


def prompt_causal(seed_offset: int = 0) -> Problem:
    """The prompt-shaped call as a causal prefill: the 2,048 queries are the
    tokens at the pool's last 2,048 positions, each seeing the positions up
    to its own (limit 30,721 + t).  A companion case; the configuration
    itself has the causal mask off."""
    p = prompt_shaped(seed_offset)
    p.q_limit = (p.n_positions - p.n_queries + 1 + np.arange(p.n_queries, dtype=np.int32))[None, :]
    p.name = "prompt_causal"
    return p


CONFIGS = {
    "tiny_decode": tiny_decode,
    "qsa_decode": qsa_decode,
    "batched_decode": batched_decode,
    "long_context": long_context,
    "prompt_shaped": prompt_shaped,
}


# ---------------------------------------------------------------------------
# K/V append calls: new rows quantised into the INT8 pools.
# ---------------------------------------------------------------------------

@dataclass
class AppendProblem:
    """One K/V append call plus the pools it writes into.

    ``k_new``/``v_new`` ``[B][n_new][G][D]`` f32 (or bf16 bit patterns as
    uint16); ``positions`` int32 ``[B][n_new]`` logical positions; pools,
    scales and page table laid out as in :class:`Problem`."""

    n_seq: int
    n_kv_heads: int
    head_dim: int
    n_new: int
    pool_cells: int
    page_table_len: int
    dtype: str  # "f32" or "bf16"
    k_new: np.ndarray
    v_new: np.ndarray
    positions: np.ndarray
    page_table: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    k_scale: np.ndarray
    v_scale: np.ndarray
    name: str = ""
    page_cells: int = 1  # cells per page: the page table has one entry per page


def make_append(*, n_seq: int = 1, n_kv_heads: int = 1, head_dim: int = 256, n_new: int = 4,
                pool_cells: int = 4096, page_table_len: Optional[int] = None,
                dtype: str = "f32", mask_fraction: float = 0.0, seed: int = SEED_BASE,
                name: str = "", page_cells: int = 1) -> AppendProblem:
    """Draw one seeded append call.

    New rows are N(0,1) values times a per-row magnitude log-uniform in
    [0.05, 20] (projection outputs of varied size), rounded to bf16 when
    ``dtype == "bf16"``.  Each sequence appends ``n_new`` distinct logical
    positions whose pages are resident, drawn without replacement.  The pools
    start as in :func:`make_problem` (random codes and scales), so a slot the
    call must not touch keeps visibly different contents.  ``page_cells`` as
    in :func:`make_problem`."""
    assert pool_cells % page_cells == 0
    if page_table_len is None:
        page_table_len = pool_cells // page_cells
    rng = np.random.Generator(np.random.PCG64(seed))
    G, D = n_kv_heads, head_dim
    k_pool = _codes(rng, (n_seq, G, pool_cells, D))
    v_pool = _codes(rng, (n_seq, G, pool_cells, D))
    k_scale = _scales(rng, (n_seq, G, pool_cells))
    v_scale = _scales(rng, (n_seq, G, pool_cells))
    pts, poss = [], []
    for b in range(n_seq):
        pt = _page_table(rng, pool_cells // page_cells, page_table_len, mask_fraction)
        resident = np.flatnonzero(np.repeat(pt, page_cells) >= 0)  # resident positions
        assert resident.size >= n_new, "not enough resident positions"
        poss.append(rng.choice(resident, size=n_new, replace=False).astype(np.int32))
        pts.append(pt)

    def rows():
        mag = np.exp(rng.uniform(np.log(0.05), np.log(20.0), size=(n_seq, n_new, G, 1)))
        x = (rng.standard_normal((n_seq, n_new, G, D)) * mag).astype(np.float32)
        return bf16_bits_from_f32(x) if dtype == "bf16" else x

    k_new, v_new = rows(), rows()
    return AppendProblem(n_seq=n_seq, n_kv_heads=G, head_dim=D, n_new=n_new,
                         pool_cells=pool_cells, page_table_len=page_table_len, dtype=dtype,
                         k_new=k_new, v_new=v_new,
                         positions=np.stack(poss).reshape(n_seq, n_new).astype(np.int32),
                         page_table=np.stack(pts).astype(np.int32), k_pool=k_pool,
                         v_pool=v_pool, k_scale=k_scale, v_scale=v_scale, name=name,
                         page_cells=page_cells)


def decode_step_append(seed_offset: int = 0) -> AppendProblem:
    """A verify window's append for the batched shape: 16 sequences x 2 KV
    heads, 4 new cells each, into 32,768-cell pools."""
    return make_append(n_seq=16, n_kv_heads=2, n_new=4, pool_cells=32768,
                       seed=SEED_BASE + 16 + seed_offset, name="append_decode_step")


def prompt_append(seed_offset: int = 0) -> AppendProblem:
    """The prompt-shaped pool written in one call: 32,768 new cells of one
    sequence with 2 KV heads (the rows of a 32,768-token prefill)."""
    return make_append(n_seq=1, n_kv_heads=2, n_new=32768, pool_cells=32768,
                       seed=SEED_BASE + 17 + seed_offset, name="append_prompt")


# ---------------------------------------------------------------- selection

@dataclass
class SelectProblem:
    """One block-selection call (the QSA selection scorer and its top-k).

    ``q_idx``   f32 ``[B][T][idx_heads * idx_dim]``: the window's indexer queries
    ``pooled``  bf16 bit patterns ``[B][max_blocks][idx_heads * idx_dim]``: one
                pooled indexer key per block of ``block_cells`` positions
    ``n_live``  int32 ``[B]``: live positions per sequence
    ``steps``   int32 ``[B][T]``: each query's position, or None
    """

    n_seq: int
    n_queries: int
    idx_heads: int
    idx_dim: int
    block_cells: int
    max_blocks: int
    top_k: int
    q_idx: np.ndarray
    pooled: np.ndarray
    n_live: np.ndarray
    steps: Optional[np.ndarray]
    name: str = ""


def make_selection(*, n_seq: int = 1, n_queries: int = 2, idx_heads: int = 4, idx_dim: int = 64,
                   block_cells: int = 64, max_blocks: int = 256, top_k: int = 16,
                   n_live: Sequence[int] | int | None = None, with_steps: bool = True,
                   integer: bool = False, seed: int = SEED_BASE + 40, name: str = "") -> SelectProblem:
    """Draw one seeded selection problem.

    Pooled keys and queries are N(0,1) (keys rounded to bf16), or, with
    ``integer``, whole numbers in [-8, 8] (every score is then an integer
    below 2^24, exact in any summation order).  ``n_live`` defaults to the
    full capacity; the window's queries sit at the last positions
    (steps[b][t] = n_live[b] - T + t) when ``with_steps``.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    F = idx_heads * idx_dim
    cap = max_blocks * block_cells
    if n_live is None:
        lives = [cap] * n_seq
    elif isinstance(n_live, (int, np.integer)):
        lives = [int(n_live)] * n_seq
    else:
        lives = [int(v) for v in n_live]
    assert len(lives) == n_seq and all(0 <= v <= cap for v in lives)
    if integer:
        pooled_f = rng.integers(-8, 9, (n_seq, max_blocks, F)).astype(np.float32)
        q_idx = rng.integers(-8, 9, (n_seq, n_queries, F)).astype(np.float32)
    else:
        pooled_f = rng.standard_normal((n_seq, max_blocks, F)).astype(np.float32)
        q_idx = rng.standard_normal((n_seq, n_queries, F)).astype(np.float32)
    steps = None
    if with_steps:
        steps = np.array([[max(v - n_queries + t, 0) for t in range(n_queries)] for v in lives], dtype=np.int32)
    return SelectProblem(n_seq=n_seq, n_queries=n_queries, idx_heads=idx_heads, idx_dim=idx_dim,
                         block_cells=block_cells, max_blocks=max_blocks, top_k=top_k, q_idx=q_idx,
                         pooled=bf16_bits_from_f32(pooled_f), n_live=np.array(lives, dtype=np.int32),
                         steps=steps, name=name)


def long_selection(seed_offset: int = 0) -> SelectProblem:
    """Selection in front of the long-context shape: 8 sequences of 131,072
    live positions in blocks of 64 (2,048 pooled keys of 4 x 64 indexer
    values each), 2 queries, 128 blocks kept per query: 8,192-16,384 cells
    per sequence, the long-context configuration's selection size."""
    return make_selection(n_seq=8, n_queries=2, idx_heads=4, idx_dim=64, block_cells=64,
                          max_blocks=2048, top_k=128, seed=SEED_BASE + 41 + seed_offset,
                          name="long_selection")
