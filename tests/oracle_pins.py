"""Pins for the fp64 oracle: checks against facts that do not come from the
oracle itself.

The pages print no attention outputs, partials or scores, so the oracle is
pinned by (i) hand-worked fixtures under ``tests/golden/``, (ii) closed forms
(a single cell, equal scores, two cells, a dominant cell), (iii) a 60-digit
``decimal`` brute force that materialises the dequantised rows and applies
no max shift, and (iv) invariants of the definition (page-table relabelling,
masking equals removal, chunk-size invariance, the merge identity, list
order, duplicates, GQA head mapping).

Every pin is a function ``pin_*(lib)`` that raises ``AssertionError`` when the
oracle library ``lib`` disagrees, so the planted-mistake test can run the same
pins against deliberately broken builds of the oracle.
"""
from __future__ import annotations

import math
import os
from decimal import Decimal, localcontext
from fractions import Fraction

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------
# helpers (independent of the oracle's C code)
# --------------------------------------------------------------------------

def load_golden(name):
    fields = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            fields[key.strip()] = val.strip()

    def nums(s, typ=float):
        return [typ(x) for x in s.split()]

    def mat(s, typ):
        return np.array([[typ(x) for x in row.split()] for row in s.split("|")])

    return {
        "D": int(fields["head_dim"]),
        "scale": float(fields["softmax_scale"]),
        "q": np.array(nums(fields["q"]), dtype=np.float64) if "q" in fields else None,
        "q_bf16_bits": (np.array([int(x, 16) for x in fields["q_bf16_bits"].split()], dtype=np.uint16)
                        if "q_bf16_bits" in fields else None),
        "page_table": np.array(nums(fields["page_table"], int), dtype=np.int32),
        "sel": np.array(nums(fields["sel"], int), dtype=np.int32),
        "k_codes": mat(fields["k_codes"], int).astype(np.int8),
        "k_scale": np.array(nums(fields["k_scale"]), dtype=np.float32),
        "v_codes": mat(fields["v_codes"], int).astype(np.int8),
        "v_scale": np.array(nums(fields["v_scale"]), dtype=np.float32),
        "expected": np.array([float(Fraction(x)) for x in fields["expected"].split()]),
        "tol": float(fields["tolerance"]),
        "page_cells": int(fields.get("page_cells", "1")),
        "fields": fields,
    }


def small_case(seed, n_pool=16, n_sel=6, D=8, mask=0, q_scale=1.0):
    """A small random problem for one (sequence, KV head) and one query row."""
    rng = np.random.Generator(np.random.PCG64(seed))
    k = rng.integers(-127, 128, (n_pool, D), dtype=np.int8)
    v = rng.integers(-127, 128, (n_pool, D), dtype=np.int8)
    ks = rng.uniform(0.005, 0.02, n_pool).astype(np.float32)
    vs = rng.uniform(0.005, 0.02, n_pool).astype(np.float32)
    pt = rng.permutation(n_pool).astype(np.int32)
    if mask:
        pt[rng.choice(n_pool, mask, replace=False)] = -1
    sel = np.sort(rng.choice(n_pool, n_sel, replace=False)).astype(np.int32)
    q = (rng.standard_normal(D) * q_scale).astype(np.float32).astype(np.float64)
    return q, k, v, ks, vs, pt, sel


def dequant(codes, scales):
    return codes.astype(np.float64) * scales.astype(np.float64)[:, None]


def decimal_brute_force(q, k, v, ks, vs, pt, sel, scale, digits=60):
    """Softmax attention evaluated in ``digits``-digit decimal arithmetic
    straight from its definition: out = sum e^{s_i} v_i / sum e^{s_i}, with no
    max shift; masked cells (page entry -1) are left out."""
    with localcontext() as ctx:
        ctx.prec = digits
        valid = [int(pt[p]) for p in sel if int(pt[p]) != -1]
        D = len(q)
        if not valid:
            return np.zeros(D)
        qd = [Decimal(float(x)) for x in q]
        sc = Decimal(float(scale))
        num = [Decimal(0)] * D
        den = Decimal(0)
        for c in valid:
            kh = [Decimal(float(ks[c])) * Decimal(int(k[c, d])) for d in range(D)]
            s = sc * sum(qd[d] * kh[d] for d in range(D))
            e = s.exp()
            den += e
            for d in range(D):
                num[d] += e * Decimal(float(vs[c])) * Decimal(int(v[c, d]))
        return np.array([float(num[d] / den) for d in range(D)])


def rel_close(a, b, rtol):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = max(np.abs(b).max(initial=0.0), 1e-300)
    return np.abs(a - b).max(initial=0.0) <= rtol * scale


# --------------------------------------------------------------------------
# pins
# --------------------------------------------------------------------------

def pin_golden_masked_mean(lib):
    g = load_golden("masked_mean.txt")
    out = oracle.attend_row(g["q"], g["k_codes"], g["v_codes"], g["k_scale"], g["v_scale"],
                            g["page_table"], g["sel"], g["scale"], lib=lib)
    assert np.abs(out - g["expected"]).max() <= g["tol"] + 1e-15, (out, g["expected"])


def pin_golden_dominant_cell(lib):
    g = load_golden("dominant_cell.txt")
    out = oracle.attend_row(g["q"], g["k_codes"], g["v_codes"], g["k_scale"], g["v_scale"],
                            g["page_table"], g["sel"], g["scale"], lib=lib)
    assert np.array_equal(out, g["expected"]), (out, g["expected"])


def pin_golden_paged_mean(lib):
    g = load_golden("paged_mean.txt")
    out = oracle.attend_row(g["q"], g["k_codes"], g["v_codes"], g["k_scale"], g["v_scale"],
                            g["page_table"], g["sel"], g["scale"], lib=lib, page_cells=g["page_cells"])
    assert np.abs(out - g["expected"]).max() <= g["tol"] + 1e-15, (out, g["expected"])


def pin_golden_bf16_queries(lib, ora=oracle):
    """bf16 query bit patterns go through the whole-call driver, whose
    widening turns them into the exact values the hand-worked case uses.
    ``ora`` is the oracle module (a test passes altered copies of it)."""
    from types import SimpleNamespace
    g = load_golden("bf16_queries.txt")
    n_pool, D = g["k_codes"].shape
    p = SimpleNamespace(
        n_seq=1, n_kv_heads=1, q_per_kv=1, head_dim=D, n_queries=1, pool_cells=n_pool,
        page_table_len=g["page_table"].shape[0], page_cells=1, softmax_scale=g["scale"],
        q_dtype="bf16", q=g["q_bf16_bits"].reshape(1, 1, 1, D),
        k_pool=g["k_codes"].reshape(1, 1, n_pool, D), v_pool=g["v_codes"].reshape(1, 1, n_pool, D),
        k_scale=g["k_scale"].reshape(1, 1, n_pool), v_scale=g["v_scale"].reshape(1, 1, n_pool),
        page_table=g["page_table"].reshape(1, -1), sel=g["sel"],
        sel_offsets=np.array([0, g["sel"].shape[0]], np.int64), q_limit=None)
    out = ora.decode_attn(p, lib=lib).reshape(D)
    assert np.abs(out - g["expected"]).max() <= g["tol"] + 1e-15, (out, g["expected"])


def pin_page_relabelling(lib):
    """Moving whole pages of the pool (rows and scales) and rewriting the page
    table to match changes no output: bit for bit in fp64."""
    P, n_pages, D = 4, 8, 8
    rng = np.random.Generator(np.random.PCG64(1300))
    k = rng.integers(-127, 128, (P * n_pages, D), dtype=np.int8)
    v = rng.integers(-127, 128, (P * n_pages, D), dtype=np.int8)
    ks = rng.uniform(0.005, 0.02, P * n_pages).astype(np.float32)
    vs = rng.uniform(0.005, 0.02, P * n_pages).astype(np.float32)
    pt = rng.permutation(n_pages).astype(np.int32)
    pt[3] = -1
    sel = np.sort(rng.choice(P * n_pages, 20, replace=False)).astype(np.int32)
    q = rng.standard_normal(D)
    ref = oracle.attend_row(q, k, v, ks, vs, pt, sel, 0.4, lib=lib, page_cells=P)
    perm = rng.permutation(n_pages)  # new page of old page i: perm[i]
    rows = np.empty(P * n_pages, np.int64)
    for i in range(n_pages):
        rows[perm[i] * P:(perm[i] + 1) * P] = np.arange(i * P, (i + 1) * P)
    pt2 = np.where(pt >= 0, perm[np.maximum(pt, 0)], -1).astype(np.int32)
    out = oracle.attend_row(q, k[rows], v[rows], ks[rows], vs[rows], pt2, sel, 0.4, lib=lib,
                            page_cells=P)
    assert np.array_equal(out, ref)
    assert not np.array_equal(out, oracle.attend_row(q, k[rows], v[rows], ks[rows], vs[rows], pt,
                                                     sel, 0.4, lib=lib, page_cells=P))


def pin_one_page_is_the_pool(lib):
    """A single page holding the whole pool: the offset alone places each
    position, so the result is that of one-cell pages in pool order."""
    q, k, v, ks, vs, _, sel = small_case(1400, n_pool=16, n_sel=7)
    one = oracle.attend_row(q, k, v, ks, vs, np.array([0], np.int32), sel, 0.3, lib=lib, page_cells=16)
    ident = oracle.attend_row(q, k, v, ks, vs, np.arange(16, dtype=np.int32), sel, 0.3, lib=lib)
    assert np.array_equal(one, ident)


def pin_golden_causal_window(lib):
    g = load_golden("causal_window.txt")
    for t in (0, 1):
        limit = int(g["fields"][f"limit_{t}"])
        expected = np.array([float(Fraction(x)) for x in g["fields"][f"expected_{t}"].split()])
        out = oracle.attend_row(g["q"], g["k_codes"], g["v_codes"], g["k_scale"], g["v_scale"],
                                g["page_table"], g["sel"], g["scale"], lib=lib, limit=limit)
        assert np.abs(out - expected).max() <= g["tol"] + 1e-15, (t, out, expected)


def pin_limit_equals_removal(lib):
    """A causal limit L gives, bit for bit, the result of the list without its
    positions >= L (in list order), for partials as well."""
    q, k, v, ks, vs, pt, sel = small_case(1500, n_pool=64, n_sel=30, mask=5)
    rng = np.random.default_rng(1501)
    sel = rng.permutation(sel).astype(np.int32)
    for L in (0, 1, 17, 40, 64, 1000):
        kept = sel[sel < L]
        a = oracle.attend_row(q, k, v, ks, vs, pt, sel, 0.5, lib=lib, limit=L)
        b = oracle.attend_row(q, k, v, ks, vs, pt, kept, 0.5, lib=lib)
        assert np.array_equal(a, b), L
        m, l, o = oracle.chunk_partial(q, k, v, ks, vs, pt, sel, 0, 30, 0.5, lib=lib, limit=L)
        m2, l2, o2 = oracle.chunk_partial(q, k, v, ks, vs, pt, kept, 0, len(kept), 0.5, lib=lib)
        assert (m, l) == (m2, l2) and np.array_equal(o, o2), L


def pin_limits_in_whole_call(lib):
    """The whole-call driver applies limits[b][t] to query t of sequence b."""
    import qsa_workloads as wl
    p = wl.make_problem(n_seq=2, n_kv_heads=2, q_per_kv=3, n_queries=3, head_dim=16,
                        pool_cells=256, n_selected=[40, 25], chunk_cells=8, seed=1600)
    p.q_limit = np.array([[60, 120, 200], [30, 31, 256]], np.int32)
    out = oracle.decode_attn(p, lib=lib)
    q = oracle.widen_queries(p.q, p.q_dtype)
    for b in range(2):
        for t in range(3):
            for h in range(6):
                g = h // 3
                ref = oracle.attend_row(q[b, t, h], p.k_pool[b, g], p.v_pool[b, g], p.k_scale[b, g],
                                        p.v_scale[b, g], p.page_table[b], p.sel_of(b), p.softmax_scale,
                                        lib=lib, limit=int(p.q_limit[b, t]))
                assert np.array_equal(out[b, t, h], ref), (b, t, h)


def pin_single_cell_is_its_v(lib):
    """One valid cell: weight 1, normaliser 1, output = its dequantised V row."""
    for seed in range(4):
        q, k, v, ks, vs, pt, _ = small_case(100 + seed, D=256, n_pool=32)
        pos = seed * 7 % 32
        out = oracle.attend_row(q, k, v, ks, vs, pt, np.array([pos], np.int32), 1 / 16, lib=lib)
        slot = pt[pos]
        expect = float(vs[slot]) * v[slot].astype(np.float64)
        assert np.array_equal(out, expect), seed
        # the same cell with masked neighbours around it
        pt2 = pt.copy()
        others = [p for p in range(32) if p != pos][:5]
        pt2[others] = -1
        sel = np.array(sorted(others + [pos]), np.int32)
        out2 = oracle.attend_row(q, k, v, ks, vs, pt2, sel, 1 / 16, lib=lib)
        assert np.array_equal(out2, expect), seed


def pin_equal_scores_give_mean(lib):
    """q = 0, or softmax scale 0, or identical K rows: equal weights, so the
    output is the mean of the selected dequantised V rows."""
    q, k, v, ks, vs, pt, sel = small_case(7, n_pool=512, n_sel=300, D=256)
    slots = pt[sel]
    mean = dequant(v[slots], vs[slots]).mean(axis=0)
    out0 = oracle.attend_row(np.zeros_like(q), k, v, ks, vs, pt, sel, 1 / 16, lib=lib)
    assert rel_close(out0, mean, 1e-13)
    out1 = oracle.attend_row(q, k, v, ks, vs, pt, sel, 0.0, lib=lib)
    assert rel_close(out1, mean, 1e-13)
    k_same = np.repeat(k[:1], k.shape[0], axis=0)
    ks_same = np.full_like(ks, ks[0])
    out2 = oracle.attend_row(q, k_same, v, ks_same, vs, pt, sel, 1 / 16, lib=lib)
    assert rel_close(out2, mean, 1e-12)


def pin_two_cells_sigmoid(lib):
    """Two cells: weights sigma(s1 - s2) and sigma(s2 - s1)."""
    for seed in range(6):
        q, k, v, ks, vs, pt, _ = small_case(200 + seed, n_pool=16, D=64, q_scale=3.0)
        sel = np.array([3, 11], np.int32)
        a, b = pt[3], pt[11]
        ka = dequant(k[[a]], ks[[a]])[0]
        kb = dequant(k[[b]], ks[[b]])[0]
        sa = 0.25 * math.fsum(q * ka)
        sb = 0.25 * math.fsum(q * kb)
        wa = 1.0 / (1.0 + math.exp(sb - sa))
        wb = 1.0 / (1.0 + math.exp(sa - sb))
        expect = wa * dequant(v[[a]], vs[[a]])[0] + wb * dequant(v[[b]], vs[[b]])[0]
        out = oracle.attend_row(q, k, v, ks, vs, pt, sel, 0.25, lib=lib)
        assert rel_close(out, expect, 1e-13), seed


def pin_dominant_cell_no_overflow(lib):
    """A query parallel to one cell's K row with a huge softmax scale: that
    cell takes all the weight; scores near 1e5 must not overflow."""
    q, k, v, ks, vs, pt, sel = small_case(9, n_pool=64, n_sel=20, D=256)
    target = int(sel[13])
    slot = pt[target]
    qd = dequant(k[[slot]], ks[[slot]])[0]
    out = oracle.attend_row(qd, k, v, ks, vs, pt, sel, 1e3, lib=lib)
    expect = dequant(v[[slot]], vs[[slot]])[0]
    assert np.all(np.isfinite(out))
    assert rel_close(out, expect, 1e-12)


def pin_empty_and_all_masked(lib):
    q, k, v, ks, vs, pt, sel = small_case(11, n_pool=16, n_sel=5, D=16)
    out = oracle.attend_row(q, k, v, ks, vs, pt, np.zeros(0, np.int32), 1.0, lib=lib)
    assert np.array_equal(out, np.zeros(16))
    pt_all = np.full_like(pt, -1)
    out = oracle.attend_row(q, k, v, ks, vs, pt_all, sel, 1.0, lib=lib)
    assert np.array_equal(out, np.zeros(16))
    m, l, o = oracle.chunk_partial(q, k, v, ks, vs, pt_all, sel, 0, 5, 1.0, lib=lib)
    assert m == -math.inf and l == 0.0 and not o.any()


def pin_decimal_brute_force(lib):
    """Tiny random cases against a 60-digit decimal evaluation."""
    cases = [(300 + s, 12, 1 + s % 8, 8, s % 3) for s in range(10)]
    cases += [(400, 8, 3, 256, 0), (401, 40, 9, 256, 2)]
    for seed, n_pool, n_sel, D, mask in cases:
        q, k, v, ks, vs, pt, sel = small_case(seed, n_pool, n_sel, D, mask, q_scale=2.0)
        out = oracle.attend_row(q, k, v, ks, vs, pt, sel, 0.7, lib=lib)
        ref = decimal_brute_force(q, k, v, ks, vs, pt, sel, 0.7)
        assert rel_close(out, ref, 1e-13), (seed, np.abs(out - ref).max())


def pin_partials_against_decimal(lib):
    """Chunk partials (m, l, o) against their decimal definitions."""
    q, k, v, ks, vs, pt, sel = small_case(500, n_pool=32, n_sel=10, D=16, mask=4)
    for start, cnt in [(0, 4), (4, 6), (2, 1), (0, 10)]:
        m, l, o = oracle.chunk_partial(q, k, v, ks, vs, pt, sel, start, cnt, 0.5, lib=lib)
        valid = [int(pt[p]) for p in sel[start:start + cnt] if int(pt[p]) != -1]
        if not valid:
            assert m == -math.inf and l == 0.0
            continue
        with localcontext() as ctx:
            ctx.prec = 60
            s = []
            for c in valid:
                s.append(Decimal(0.5) * sum(Decimal(float(q[d])) * Decimal(float(ks[c]))
                                            * Decimal(int(k[c, d])) for d in range(16)))
            mm = max(s)
            ll = sum((x - mm).exp() for x in s)
            oo = [sum((x - mm).exp() * Decimal(float(vs[c])) * Decimal(int(v[c, d]))
                      for x, c in zip(s, valid)) for d in range(16)]
        assert abs(m - float(mm)) <= 1e-14 * max(1.0, abs(float(mm)))
        assert abs(l - float(ll)) <= 1e-14 * float(ll)
        assert rel_close(o, [float(x) for x in oo], 1e-13)


def pin_page_table_relabelling(lib):
    """Permuting the pool rows (and scales) and rewriting the page table to
    match leaves the output unchanged, bit for bit."""
    q, k, v, ks, vs, pt, sel = small_case(600, n_pool=128, n_sel=40, D=256, mask=10)
    out = oracle.attend_row(q, k, v, ks, vs, pt, sel, 1 / 16, lib=lib)
    rng = np.random.Generator(np.random.PCG64(601))
    perm = rng.permutation(128)          # new slot of old slot s is perm[s]
    inv = np.argsort(perm)
    k2, v2, ks2, vs2 = k[inv], v[inv], ks[inv], vs[inv]
    pt2 = np.where(pt >= 0, perm[np.maximum(pt, 0)], -1).astype(np.int32)
    out2 = oracle.attend_row(q, k2, v2, ks2, vs2, pt2, sel, 1 / 16, lib=lib)
    assert np.array_equal(out, out2)


def pin_masking_equals_removal(lib):
    q, k, v, ks, vs, pt, sel = small_case(700, n_pool=128, n_sel=50, D=256)
    drop = sel[::3]
    pt_m = pt.copy()
    pt_m[drop] = -1
    out_masked = oracle.attend_row(q, k, v, ks, vs, pt_m, sel, 1 / 16, lib=lib)
    kept = np.array([p for p in sel if p not in set(drop.tolist())], np.int32)
    out_removed = oracle.attend_row(q, k, v, ks, vs, pt, kept, 1 / 16, lib=lib)
    assert np.array_equal(out_masked, out_removed)
    ref = decimal_brute_force(q, k, v, ks, vs, pt, kept, 1 / 16, digits=40)
    assert rel_close(out_masked, ref, 1e-13)


def pin_chunk_size_invariance(lib):
    """Chunked partials merged in order equal the unchunked result for any
    chunk size, including 1, non-divisors, the list length and beyond."""
    q, k, v, ks, vs, pt, sel = small_case(800, n_pool=256, n_sel=130, D=256, mask=20,
                                          q_scale=2.0)
    ref = oracle.attend_row(q, k, v, ks, vs, pt, sel, 1 / 16, lib=lib)
    for C in (1, 7, 63, 64, 65, 129, 130, 131, 1000):
        m, l, o = oracle.row_partials(q, k, v, ks, vs, pt, sel, C, 1 / 16, lib=lib)
        out = oracle.merge(m, l, o, lib=lib)
        assert rel_close(out, ref, 1e-13), C


def pin_merge_identity(lib):
    """merge(partial(A), partial(B)) equals partial(A u B) normalised, and the
    partial of A u B equals the pairwise LSE combination of the two."""
    q, k, v, ks, vs, pt, sel = small_case(900, n_pool=64, n_sel=30, D=32, q_scale=3.0)
    mA, lA, oA = oracle.chunk_partial(q, k, v, ks, vs, pt, sel, 0, 11, 0.5, lib=lib)
    mB, lB, oB = oracle.chunk_partial(q, k, v, ks, vs, pt, sel, 11, 19, 0.5, lib=lib)
    mU, lU, oU = oracle.chunk_partial(q, k, v, ks, vs, pt, sel, 0, 30, 0.5, lib=lib)
    M = max(mA, mB)
    assert mU == M
    assert abs(lU - (lA * math.exp(mA - M) + lB * math.exp(mB - M))) <= 1e-13 * lU
    assert rel_close(oU, oA * math.exp(mA - M) + oB * math.exp(mB - M), 1e-13)
    out = oracle.merge([mA, mB], [lA, lB], np.stack([oA, oB]), lib=lib)
    assert rel_close(out, oU / lU, 1e-13)
    # an empty chunk between them changes nothing
    out3 = oracle.merge([mA, -math.inf, mB], [lA, 0.0, lB], np.stack([oA, 0 * oA, oB]), lib=lib)
    assert rel_close(out3, out, 1e-15)


def pin_order_and_duplicates(lib):
    """List order does not matter; a duplicated entry counts twice."""
    q, k, v, ks, vs, pt, sel = small_case(1000, n_pool=64, n_sel=25, D=64, q_scale=2.0)
    ref = oracle.attend_row(q, k, v, ks, vs, pt, sel, 0.3, lib=lib)
    rng = np.random.Generator(np.random.PCG64(1001))
    shuf = rng.permutation(sel).astype(np.int32)
    assert rel_close(oracle.attend_row(q, k, v, ks, vs, pt, shuf, 0.3, lib=lib), ref, 1e-13)
    a, b = int(sel[0]), int(sel[1])
    sa_, sb_ = pt[a], pt[b]
    dup = oracle.attend_row(q, k, v, ks, vs, pt, np.array([a, a, b], np.int32), 0.3, lib=lib)
    s_a = 0.3 * math.fsum(q * dequant(k[[sa_]], ks[[sa_]])[0])
    s_b = 0.3 * math.fsum(q * dequant(k[[sb_]], ks[[sb_]])[0])
    wa = 2 * math.exp(s_a) / (2 * math.exp(s_a) + math.exp(s_b))
    expect = wa * dequant(v[[sa_]], vs[[sa_]])[0] + (1 - wa) * dequant(v[[sb_]], vs[[sb_]])[0]
    assert rel_close(dup, expect, 1e-13)


def pin_call_layout(lib):
    """Whole-call indexing: head h = g*H + j reads KV head g of its sequence,
    and query row (b, t, h) is the one that is scored.

    Each (sequence, KV head) pool holds V rows that are constant and equal to
    a code naming (b, g): the output of any row must be that code times the
    scale, whatever the weights.  Then each query row is aimed at one cell
    whose V row encodes (t, h)."""
    from qsa_workloads import make_problem
    p = make_problem(n_seq=2, n_kv_heads=2, q_per_kv=3, head_dim=32, n_queries=2,
                     pool_cells=64, n_selected=[20, 33], chunk_cells=8, seed=1234)
    B, G, H, T, D = 2, 2, 3, 2, 32
    p.v_scale[:] = 0.25
    for b in range(B):
        for g in range(G):
            p.v_pool[b, g] = 10 * b + 3 * g + 1
    out = oracle.decode_attn(p, lib=lib)
    for b in range(B):
        for t in range(T):
            for h in range(G * H):
                g = h // H
                assert np.allclose(out[b, t, h], 0.25 * (10 * b + 3 * g + 1), rtol=0,
                                   atol=1e-13), (b, t, h)
    # aim every query row at its own cell: the K rows of the aimed cells are
    # one-hot on distinct dimensions, every other K row is zero
    p2 = make_problem(n_seq=2, n_kv_heads=2, q_per_kv=3, head_dim=32, n_queries=2,
                      pool_cells=64, n_selected=[24, 24], chunk_cells=8, seed=99)
    p2.k_pool[:] = 0
    p2.q[:] = 0
    for b in range(B):
        sel_b = p2.sel_of(b)
        for t in range(T):
            for h in range(G * H):
                g = h // H
                i = t * G * H + h
                slot = p2.page_table[b, int(sel_b[i % len(sel_b)])]
                p2.k_pool[b, g, slot, i] = 127
                p2.q[b, t, h, i] = 2000.0
    rows = [oracle.flat_row(p2, b, t, h) for b in range(B) for t in range(T)
            for h in range(G * H)]
    part = oracle.decode_attn(p2, rows=rows, lib=lib)
    full = oracle.decode_attn(p2, lib=lib)
    i = 0
    for b in range(B):
        sel_b = p2.sel_of(b)
        for t in range(T):
            for h in range(G * H):
                g = h // H
                slot = p2.page_table[b, int(sel_b[(t * G * H + h) % len(sel_b)])]
                expect = p2.v_pool[b, g, slot].astype(np.float64) * p2.v_scale[b, g, slot]
                assert np.allclose(full[b, t, h], expect, rtol=1e-6, atol=1e-6), (b, t, h)
                assert np.array_equal(part[i], full[b, t, h])
                i += 1


def pin_rejects_bad_indices(lib):
    q, k, v, ks, vs, pt, sel = small_case(1100, n_pool=16, n_sel=4, D=8)
    for bad_sel in ([0, 16], [-1, 2]):
        try:
            oracle.attend_row(q, k, v, ks, vs, pt, np.array(bad_sel, np.int32), 1.0, lib=lib)
        except oracle.OracleError:
            pass
        else:
            raise AssertionError(f"position {bad_sel} accepted")
    pt_bad = pt.copy()
    pt_bad[3] = 16
    try:
        oracle.attend_row(q, k, v, ks, vs, pt_bad, np.array([3], np.int32), 1.0, lib=lib)
    except oracle.OracleError:
        pass
    else:
        raise AssertionError("slot 16 of a 16-cell pool accepted")


PINS = [
    pin_golden_masked_mean,
    pin_golden_dominant_cell,
    pin_golden_paged_mean,
    pin_golden_bf16_queries,
    pin_page_relabelling,
    pin_one_page_is_the_pool,
    pin_golden_causal_window,
    pin_limit_equals_removal,
    pin_limits_in_whole_call,
    pin_single_cell_is_its_v,
    pin_equal_scores_give_mean,
    pin_two_cells_sigmoid,
    pin_dominant_cell_no_overflow,
    pin_empty_and_all_masked,
    pin_decimal_brute_force,
    pin_partials_against_decimal,
    pin_page_table_relabelling,
    pin_masking_equals_removal,
    pin_chunk_size_invariance,
    pin_merge_identity,
    pin_order_and_duplicates,
    pin_call_layout,
    pin_rejects_bad_indices,
]
