"""Pins for the K/V append oracle (``oracle/kv_append.py``), CPU only.

The pages print no quantiser and no appended values, so the oracle is pinned
by hand-worked rows (``tests/golden/append_rows.txt``: max |x| = 127 x 2^k, so
every quotient is exact and the expected codes are plain round-half-even),
the rounding bound of the definition, the max element, zero rows,
power-of-two scaling, bf16 inputs, and a hand-worked routing example.  The
planted-mistake test runs the same pins against altered copies of the
oracle's source and requires each alteration to fail at least one.
"""
import os
import types

import numpy as np
import pytest

import qsa_workloads as wl
from oracle import kv_append as ka

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "append_rows.txt")


def golden_rows():
    f = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split(":", 1)
            f[k.strip()] = [float(x) for x in v.split()]
    rows = []
    for tag in "abcd":
        rows.append((np.array(f[f"row_{tag}"], np.float32), np.array(f[f"codes_{tag}"]).astype(np.int8),
                     np.float32(f[f"scale_{tag}"][0])))
    return rows


def one_call(m, k_rows, v_rows, page_table, positions, pool_cells, dtype="f32"):
    """A single-sequence, single-KV-head call on pools filled with a marker."""
    n_new, D = len(positions), k_rows.shape[-1]
    a = wl.AppendProblem(n_seq=1, n_kv_heads=1, head_dim=D, n_new=n_new, pool_cells=pool_cells,
                         page_table_len=len(page_table), dtype=dtype,
                         k_new=k_rows.reshape(1, n_new, 1, D), v_new=v_rows.reshape(1, n_new, 1, D),
                         positions=np.array(positions, np.int32).reshape(1, n_new),
                         page_table=np.array(page_table, np.int32).reshape(1, -1),
                         k_pool=None, v_pool=None, k_scale=None, v_scale=None)
    kp = np.full((1, 1, pool_cells, D), 99, np.int8)
    vp = np.full((1, 1, pool_cells, D), 99, np.int8)
    ks = np.full((1, 1, pool_cells), -1.0, np.float32)
    vs = np.full((1, 1, pool_cells), -1.0, np.float32)
    st = m.kv_append(a, kp, vp, ks, vs)
    return st, kp[0, 0], vp[0, 0], ks[0, 0], vs[0, 0]


# ------------------------------------------------------------------ pins

def pin_golden_rows(m):
    for x, codes, scale in golden_rows():
        c, s = m.quantize_row(x)
        assert s == scale, (s, scale)
        assert np.array_equal(c, codes), (c, codes)


def pin_golden_through_append(m):
    """K from one hand-worked row and V from another land in their own pools."""
    (a_x, a_c, a_s), (b_x, b_c, b_s) = golden_rows()[:2]
    st, kp, vp, ks, vs = one_call(m, a_x[None], b_x[None], [2, 0, 1], [0], 3)
    assert st == 0
    assert np.array_equal(kp[2], a_c) and ks[2] == a_s
    assert np.array_equal(vp[2], b_c) and vs[2] == b_s


def pin_round_trip_bound(m):
    """|code * scale - x| <= scale * (1/2 + 2^-16): rounding to nearest of a
    correctly rounded quotient (the 2^-16 covers the quotient's rounding)."""
    rng = np.random.default_rng(5100)
    for _ in range(200):
        x = (rng.standard_normal(256) * np.exp(rng.uniform(-6, 6))).astype(np.float32)
        c, s = m.quantize_row(x)
        err = np.abs(c.astype(np.float64) * float(s) - x.astype(np.float64))
        assert np.all(err <= float(s) * (0.5 + 2.0 ** -16)), err.max() / float(s)


def pin_max_element(m):
    """The element of largest magnitude gets code +-127 with its sign, and
    127 * scale is within one fp32 rounding of it."""
    rng = np.random.default_rng(5200)
    for _ in range(200):
        x = (rng.standard_normal(256) * np.exp(rng.uniform(-6, 6))).astype(np.float32)
        c, s = m.quantize_row(x)
        i = int(np.argmax(np.abs(x)))
        assert int(c[i]) == (127 if x[i] > 0 else -127)
        assert abs(127.0 * float(s) - abs(float(x[i]))) <= abs(float(x[i])) * 2.0 ** -22


def pin_zero_row(m):
    c, s = m.quantize_row(np.zeros(256, np.float32))
    assert s == 0 and not np.any(c)


def pin_pow2_scaling(m):
    """Scaling a row by 2^k scales its scale by 2^k and keeps its codes."""
    rng = np.random.default_rng(5300)
    x = rng.standard_normal(256).astype(np.float32)
    c0, s0 = m.quantize_row(x)
    for k in (-20, -7, -1, 1, 5, 20):
        c, s = m.quantize_row(x * np.float32(2.0 ** k))
        assert np.array_equal(c, c0) and s == np.float32(s0 * np.float32(2.0 ** k))


def pin_bf16_rows(m):
    """bf16 inputs: row b of the fixture, whose values are bf16-exact except
    0.99 (bf16 0.98828125, still code 0), gives the same codes."""
    x, codes, scale = golden_rows()[1]
    bits = (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    st, kp, vp, ks, vs = one_call(m, bits[None], bits[None], [0], [0], 1, dtype="bf16")
    assert st == 0 and ks[0] == scale and np.array_equal(kp[0], codes)


def pin_routing(m):
    """Hand-worked routing: page table [3, -1, 0, 7, 1] over a 4-cell pool,
    new rows 0..5 at positions [0, 2, 1, 3, 4, 9]: row 0 (max 127, scale 1)
    -> slot 3, row 1 (max 63.5, scale 0.5) -> slot 0, row 4 (max 127) ->
    slot 1; row 2's position is not resident, row 3's page entry 7 is outside
    the pool, row 5's position is outside the page table; slot 2 keeps its
    contents."""
    x = np.array([[127.0] * 8, [63.5] * 8, [254.0] * 8, [1.0] * 8, [-127.0] * 8, [2.0] * 8],
                 np.float32)
    st, kp, vp, ks, vs = one_call(m, x, -x, [3, -1, 0, 7, 1], [0, 2, 1, 3, 4, 9], 4)
    assert st == ka.STATUS_NOT_RESIDENT | ka.STATUS_BAD_SLOT | ka.STATUS_BAD_POSITION, st
    assert ks.tolist() == [0.5, 1.0, -1.0, 1.0], ks
    assert kp[3].tolist() == [127] * 8 and kp[0].tolist() == [127] * 8
    assert kp[1].tolist() == [-127] * 8 and vp[1].tolist() == [127] * 8
    assert kp[2].tolist() == [99] * 8 and vp[2].tolist() == [99] * 8 and vs[2] == -1.0


def pin_paged_routing(m):
    """Pages of two cells, page table [1, -1, 0] over a 4-cell pool: new rows
    at positions [0, 5, 2, 4, 6] go to slots 2 (page 1, offset 0), 1 (page 0,
    offset 1), nowhere (page -1), 0 (page 0, offset 0), nowhere (position 6
    is past the 3 pages x 2 cells); slot 3 keeps its contents."""
    x = np.array([[127.0] * 8, [63.5] * 8, [1.0] * 8, [254.0] * 8, [2.0] * 8], np.float32)
    a = wl.AppendProblem(n_seq=1, n_kv_heads=1, head_dim=8, n_new=5, pool_cells=4, page_table_len=3,
                         dtype="f32", k_new=x.reshape(1, 5, 1, 8), v_new=(-x).reshape(1, 5, 1, 8),
                         positions=np.array([[0, 5, 2, 4, 6]], np.int32),
                         page_table=np.array([[1, -1, 0]], np.int32), k_pool=None, v_pool=None,
                         k_scale=None, v_scale=None, page_cells=2)
    kp = np.full((1, 1, 4, 8), 99, np.int8)
    vp = np.full((1, 1, 4, 8), 99, np.int8)
    ks = np.full((1, 1, 4), -1.0, np.float32)
    vs = np.full((1, 1, 4), -1.0, np.float32)
    st = m.kv_append(a, kp, vp, ks, vs)
    assert st == ka.STATUS_NOT_RESIDENT | ka.STATUS_BAD_POSITION, st
    assert ks[0, 0].tolist() == [2.0, 0.5, 1.0, -1.0], ks
    assert kp[0, 0, 3].tolist() == [99] * 8 and vp[0, 0, 2].tolist() == [-127] * 8


def pin_kv_heads_and_sequences(m):
    """Every (sequence, KV head) row goes to its own pool at the slot of its
    own sequence's page table; the other slots keep their contents."""
    a = wl.make_append(n_seq=3, n_kv_heads=2, n_new=5, pool_cells=64, head_dim=16, seed=5400)
    kp, vp, ks, vs = a.k_pool.copy(), a.v_pool.copy(), a.k_scale.copy(), a.v_scale.copy()
    assert m.kv_append(a, kp, vp, ks, vs) == 0
    touched = np.zeros((3, 64), bool)
    for b in range(3):
        for i in range(5):
            slot = int(a.page_table[b, a.positions[b, i]])
            touched[b, slot] = True
            for g in range(2):
                x = a.k_new[b, i, g]
                amax = float(np.max(np.abs(x)))
                assert int(kp[b, g, slot][np.argmax(np.abs(x))]) in (127, -127)
                assert abs(127.0 * float(ks[b, g, slot]) - amax) <= amax * 2.0 ** -22
    for b in range(3):
        assert np.array_equal(kp[b][:, ~touched[b]], a.k_pool[b][:, ~touched[b]])
        assert np.array_equal(vs[b][:, ~touched[b]], a.v_scale[b][:, ~touched[b]])


PINS = [pin_golden_rows, pin_golden_through_append, pin_round_trip_bound, pin_max_element,
        pin_zero_row, pin_pow2_scaling, pin_bf16_rows, pin_routing, pin_paged_routing,
        pin_kv_heads_and_sequences]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(ka)


# (name, text in the oracle source, replacement): plausible slips.
MUTANTS = [
    ("scale_over_128", "scale = np.float32(amax / _F127)", "scale = np.float32(amax / np.float32(128.0))"),
    ("truncate", "codes = np.rint(np.divide(x, scale, dtype=np.float32))",
     "codes = np.trunc(np.divide(x, scale, dtype=np.float32))"),
    ("half_away_from_zero", "codes = np.rint(np.divide(x, scale, dtype=np.float32))",
     "y = np.divide(x, scale, dtype=np.float32)\n    codes = np.sign(y) * np.floor(np.abs(y) + 0.5)"),
    ("signed_max", "amax = np.float32(np.max(np.abs(x)))", "amax = np.float32(np.max(x))"),
    ("v_from_k_rows", "v_scale[b, g, slot] = quantize_row(v_new[b, i, g])",
     "v_scale[b, g, slot] = quantize_row(k_new[b, i, g])"),
    ("slot_is_position", "slot = page * P + pos % P", "slot = pos"),
    ("page_offset_dropped", "slot = page * P + pos % P", "slot = page * P"),
    ("not_resident_to_page0", "if page == -1:\n                status |= STATUS_NOT_RESIDENT\n                continue",
     "if page == -1:\n                page = 0"),
    ("bf16_high_bits_dropped", "np.asarray(rows).astype(np.uint32) << np.uint32(16)",
     "np.asarray(rows).astype(np.uint32) << np.uint32(15)"),
    ("wrong_kv_head", "k_pool[b, g, slot], k_scale[b, g, slot] = quantize_row(k_new[b, i, g])",
     "k_pool[b, g, slot], k_scale[b, g, slot] = quantize_row(k_new[b, i, 0])"),
]


def _mutant(old, new):
    src = open(ka.__file__).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("kv_append_mutant")
    exec(compile(src.replace(old, new), "kv_append_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new):
    mod = _mutant(old, new)
    failed = []
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {name}"
