"""fp64 CPU oracle for QSA block selection -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` may import this
module; the product library never calls it and has no CPU fallback.

What the selection computes (the QSA selection scorer and its top-k, "Strata
issue #8, round 9: performance candidate set on v0.2.9", R9-gpu-9, with the
long-context select and TOPK_SPLIT of the "Absorbed, considered and dropped"
list): the pages name the scorer ``qsa_block_scores_rows`` over pooled keys,
a dead tail, per-query indexer vectors and steps, and the top-k that turns
the scores into the selected cells the decode attention reads.  They print no
formula; the reading here, step by step in the pages' order:

1. Blocks.  The positions of a sequence are cut into blocks of R
   (block j covers positions [jR, (j+1)R)); each block has one pooled indexer
   key of F = idx_heads * idx_dim values.  Positions at or past the sequence's
   live extent n_live are dead: a block is live while jR < n_live, and a live
   block's last cell is min((j+1)R, n_live) - 1.
2. Scores.  For query t of the window, block j scores
   s[t][j] = sum over heads h and dims d of q_idx[t][h][d] * pooled[j][h][d]
   (the indexer heads' dot products, summed), when j is live and starts at or
   before the query's position steps[t] (no step: every live block); any
   other block scores -inf and is never selected.
3. Top-k.  Each query keeps the top_k blocks of highest score among its
   candidates; equal scores go to the lower block index; with fewer
   candidates it keeps all of them.  The kept ids are listed ascending.
4. Selection.  The sequence's list is the union of its queries' kept blocks,
   expanded to their live positions in ascending order: the ``sel`` list one
   qsa_decode_attn_batch call consumes (CSR offsets over the sequences).

Scores are evaluated in double precision from the exact inputs (bf16 pooled
keys widened exactly, fp32 queries).  Every function is pinned by
``tests/test_select_oracle.py``.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import numpy as np


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact double values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def candidates(n_blocks: int, block_cells: int, n_live: int, step: Optional[int]) -> np.ndarray:
    """Step 1-2: which blocks a query may select (bool [n_blocks])."""
    starts = np.arange(n_blocks, dtype=np.int64) * block_cells
    ok = starts < n_live
    if step is not None:
        ok &= starts <= step
    return ok


def block_scores(q_idx: np.ndarray, pooled: np.ndarray, block_cells: int, n_live: int,
                 steps: Optional[Sequence[int]]) -> np.ndarray:
    """Step 2 for one sequence: q_idx [T][F] (float), pooled [n_blocks][F]
    (float values) -> scores [T][n_blocks] in double, -inf off the candidates."""
    q = np.asarray(q_idx, dtype=np.float64)
    k = np.asarray(pooled, dtype=np.float64)
    T, n_blocks = q.shape[0], k.shape[0]
    out = np.full((T, n_blocks), -np.inf)
    for t in range(T):
        ok = candidates(n_blocks, block_cells, n_live, None if steps is None else int(steps[t]))
        # the plain definition: one dot product per candidate block
        for j in np.nonzero(ok)[0]:
            out[t, j] = float(np.dot(q[t], k[j]))
    return out


def top_k(scores_row: np.ndarray, k: int) -> np.ndarray:
    """Step 3 for one query: ascending ids of the k best finite scores, equal
    scores to the lower id (a full sort by (-score, id))."""
    s = np.asarray(scores_row, dtype=np.float64)
    ids = [j for j in range(s.shape[0]) if np.isfinite(s[j])]
    ids.sort(key=lambda j: (-s[j], j))
    return np.array(sorted(ids[:k]), dtype=np.int32)


def expand(blocks: Sequence[int], block_cells: int, n_live: int) -> np.ndarray:
    """Step 4: ascending live positions of the given blocks."""
    pos: List[int] = []
    for j in sorted(set(int(b) for b in blocks)):
        pos.extend(range(j * block_cells, min((j + 1) * block_cells, n_live)))
    return np.array(pos, dtype=np.int32)


def select_sequence(q_idx, pooled, block_cells: int, n_live: int, steps, k: int
                    ) -> Tuple[np.ndarray, List[np.ndarray], np.ndarray]:
    """One sequence: (scores [T][n_blocks], kept ids per query, positions)."""
    s = block_scores(q_idx, pooled, block_cells, n_live, steps)
    kept = [top_k(s[t], k) for t in range(s.shape[0])]
    union = sorted(set(int(j) for kk in kept for j in kk))
    return s, kept, expand(union, block_cells, n_live)


def select_batch(p):
    """A whole call for a selection problem ``p`` (as drawn by the input
    generator): scores [B][T][max_blocks], kept [B][T][top_k] (-1 padded),
    sel (concatenated positions) and sel_offsets [B+1]."""
    B, T, nb, k = p.n_seq, p.n_queries, p.max_blocks, p.top_k
    pooled = widen_bf16(p.pooled)
    q = np.asarray(p.q_idx, dtype=np.float32).astype(np.float64)
    scores = np.zeros((B, T, nb))
    kept = np.full((B, T, k), -1, dtype=np.int32)
    sels, offs = [], [0]
    for b in range(B):
        steps = None if p.steps is None else p.steps[b]
        s, kk, pos = select_sequence(q[b].reshape(T, -1), pooled[b].reshape(nb, -1), p.block_cells,
                                     int(p.n_live[b]), steps, k)
        scores[b] = s
        for t in range(T):
            kept[b, t, :len(kk[t])] = kk[t]
        sels.append(pos)
        offs.append(offs[-1] + len(pos))
    sel = np.concatenate(sels) if sels else np.zeros(0, np.int32)
    return scores, kept, sel.astype(np.int32), np.array(offs, dtype=np.int32)
