"""The block-selection oracle against its pins, and the pins against planted
mistakes.  CPU only.

Pins: a hand-worked case (``tests/golden/select_blocks.txt``); scores
against an independent per-element sum over heads and dims; top-k against
a full ranking with the tie rule done another way (lexicographic keys); the
dead tail, the causal step and the partial last block on their own;
invariants (k above the candidate count keeps every candidate; the union of
the queries' sets; expansion counts).  The planted mistakes are text edits
of a copy of ``oracle/select_blocks.py`` loaded as its own module.
"""
import importlib.util
import os
import shutil
import sys
import tempfile

import numpy as np
import pytest

import oracle.select_blocks as osb
import qsa_workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "select_blocks.txt")
SRC = osb.__file__


def load_golden():
    f = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split(":", 1)
            f[k.strip()] = v.strip()
    rows = lambda s, typ: [[typ(x) for x in r.split()] for r in s.split("|")]
    return {
        "R": int(f["block_cells"]), "H": int(f["idx_heads"]), "D": int(f["idx_dim"]),
        "n_live": int(f["n_live"]), "steps": [int(x) for x in f["steps"].split()],
        "k": int(f["top_k"]), "q": np.array(rows(f["q_idx"], float)),
        "pooled": np.array(rows(f["pooled"], float)),
        "scores": np.array(rows(f["scores"], float)),
        "kept": [np.array(r, np.int32) for r in rows(f["kept"], int)],
        "sel": np.array([int(x) for x in f["sel"].split()], np.int32),
    }


# ---------------------------------------------------------------- pins

def pin_golden(m=osb):
    g = load_golden()
    s, kept, sel = m.select_sequence(g["q"], g["pooled"], g["R"], g["n_live"], g["steps"], g["k"])
    assert np.array_equal(s, g["scores"]), s
    assert all(np.array_equal(a, b) for a, b in zip(kept, g["kept"])), kept
    assert np.array_equal(sel, g["sel"]), sel


def pin_scores_by_elements(m=osb):
    """Integer inputs: every score equals the sum over (head, dim) done one
    element at a time in Python integers."""
    p = wl.make_selection(n_seq=1, n_queries=3, idx_heads=3, idx_dim=5, block_cells=4, max_blocks=9,
                          top_k=3, n_live=30, integer=True, seed=77)
    q = p.q_idx[0].astype(np.int64)
    k = m.widen_bf16(p.pooled[0]).astype(np.int64)
    s = m.block_scores(q, k, 4, 30, p.steps[0])
    for t in range(3):
        for j in range(9):
            if j * 4 < 30 and j * 4 <= p.steps[0][t]:
                want = 0
                for h in range(3):
                    for d in range(5):
                        want += int(q[t, h * 5 + d]) * int(k[j, h * 5 + d])
                assert s[t, j] == want, (t, j)
            else:
                assert s[t, j] == -np.inf


def pin_topk_ranking(m=osb):
    """Top-k equals the first k of a ranking by the key (-score, id), built
    here with numpy's lexsort, on scores with many ties."""
    rng = np.random.Generator(np.random.PCG64(5))
    for trial in range(20):
        n = int(rng.integers(1, 60))
        s = rng.integers(-3, 4, n).astype(np.float64)
        s[rng.random(n) < 0.2] = -np.inf
        k = int(rng.integers(1, 70))
        order = np.lexsort((np.arange(n), -s))   # primary -s, secondary id
        want = np.sort([j for j in order if np.isfinite(s[j])][:k]).astype(np.int32)
        assert np.array_equal(m.top_k(s, k), want), (trial, s, k)


def pin_dead_tail_and_step(m=osb):
    """Blocks at or past the live extent and blocks that start after the
    query's position are never candidates, whatever their keys."""
    F, R, nb = 4, 8, 10
    q = np.ones((2, F))
    pooled = np.ones((nb, F))
    pooled[9] = 100.0       # dead (start 72 >= n_live 70)
    pooled[5] = 50.0        # starts at 40: after query 0's position 39, visible to query 1
    s, kept, sel = m.select_sequence(q, pooled, R, 70, [39, 69], 2)
    assert s[0, 9] == -np.inf and s[1, 9] == -np.inf and s[0, 5] == -np.inf and s[1, 5] == 200.0
    assert 5 not in kept[0] and 9 not in kept[0] and 9 not in kept[1] and 5 in kept[1]
    # block 8 (positions 64..71) is partial: only 64..69 are live
    s2, kept2, sel2 = m.select_sequence(q, np.where(np.arange(nb)[:, None] == 8, 30.0, 1.0) * np.ones((nb, F)),
                                        R, 70, [69, 69], 1)
    assert np.array_equal(sel2, np.arange(64, 70, dtype=np.int32))


def pin_all_candidates_and_union(m=osb):
    """k above the candidate count keeps every candidate; the list is the
    union of the queries' sets, expanded."""
    p = wl.make_selection(n_seq=1, n_queries=3, idx_heads=2, idx_dim=4, block_cells=5, max_blocks=12,
                          top_k=4, n_live=53, integer=True, seed=91)
    q = p.q_idx[0]
    k = m.widen_bf16(p.pooled[0])
    s, kept, sel = m.select_sequence(q, k, 5, 53, None, 100)
    for t in range(3):
        assert np.array_equal(kept[t], np.arange(11, dtype=np.int32))   # blocks 0..10 are live
    assert np.array_equal(sel, np.arange(53, dtype=np.int32))
    s, kept, sel = m.select_sequence(q, k, 5, 53, p.steps[0], 4)
    union = sorted(set(int(j) for kk in kept for j in kk))
    want = [x for j in union for x in range(5 * j, min(5 * j + 5, 53))]
    assert np.array_equal(sel, np.array(want, np.int32))
    assert all(len(kk) == 4 for kk in kept)


def pin_batch_layout(m=osb):
    """A batch call is the per-sequence calls concatenated, with CSR offsets."""
    p = wl.make_selection(n_seq=3, n_queries=2, idx_heads=2, idx_dim=8, block_cells=16, max_blocks=20,
                          top_k=3, n_live=[320, 17, 0], integer=True, seed=13)
    scores, kept, sel, off = m.select_batch(p)
    assert off[0] == 0 and off[-1] == sel.shape[0]
    for b in range(3):
        s, kk, pos = m.select_sequence(p.q_idx[b], m.widen_bf16(p.pooled[b]), 16, int(p.n_live[b]),
                                       p.steps[b], 3)
        assert np.array_equal(sel[off[b]:off[b + 1]], pos)
        assert np.array_equal(scores[b], s)
        for t in range(2):
            assert np.array_equal(kept[b, t, :len(kk[t])], kk[t]) and np.all(kept[b, t, len(kk[t]):] == -1)
    assert off[3] - off[2] == 0          # no live position: nothing selected


def pin_bf16_patterns(m=osb):
    """Pooled keys are bf16 bit patterns: sign, 8 exponent bits (bias 127),
    7 mantissa bits, decoded here by hand."""
    pats = {0x3F80: 1.0, 0xC000: -2.0, 0x4100: 8.0, 0xC110: -9.0, 0x3FC1: 1.5078125, 0x0000: 0.0,
            0x3E80: 0.25}
    got = m.widen_bf16(np.array(list(pats), dtype=np.uint16))
    assert np.array_equal(got, np.array(list(pats.values()))), got


PINS = [pin_golden, pin_bf16_patterns, pin_scores_by_elements, pin_topk_ranking, pin_dead_tail_and_step,
        pin_all_candidates_and_union, pin_batch_layout]


@pytest.mark.parametrize("pin", PINS, ids=[f.__name__ for f in PINS])
def test_pin(pin):
    pin()


# (name, text in the oracle source, replacement): plausible slips
MUTANTS = [
    ("tie_to_higher_id", "ids.sort(key=lambda j: (-s[j], j))", "ids.sort(key=lambda j: (-s[j], -j))"),
    ("step_strict", "ok &= starts <= step", "ok &= starts < step"),
    ("dead_tail_ignored", "ok = starts < n_live", "ok = starts >= 0"),
    ("expansion_ignores_live", "range(j * block_cells, min((j + 1) * block_cells, n_live))",
     "range(j * block_cells, (j + 1) * block_cells)"),
    ("intersection_not_union", "union = sorted(set(int(j) for kk in kept for j in kk))",
     "union = sorted(set.intersection(*[set(int(j) for j in kk) for kk in kept]))"),
    ("first_head_only", "out[t, j] = float(np.dot(q[t], k[j]))",
     "out[t, j] = float(np.dot(q[t][:q.shape[1] // 2], k[j][:q.shape[1] // 2]))"),
    ("keeps_k_plus_one", "return np.array(sorted(ids[:k]), dtype=np.int32)",
     "return np.array(sorted(ids[:k + 1]), dtype=np.int32)"),
    ("bf16_shift_8", "b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)",
     "b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(8)"),
]


def test_mutant_anchors_unique():
    src = open(SRC).read()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, name


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new):
    src = open(SRC).read()
    tmp = tempfile.mkdtemp(prefix="select_mutant_")
    try:
        path = os.path.join(tmp, "select_blocks.py")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        spec = importlib.util.spec_from_file_location(f"select_mutant_{name}", path)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        failed = []
        for pin in PINS:
            try:
                pin(mod)
            except (AssertionError, ValueError, IndexError, TypeError):
                failed.append(pin.__name__)
        assert failed, f"no pin catches {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
