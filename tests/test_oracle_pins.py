"""The oracle against its pins, and the pins against planted mistakes.

Runs on the CPU only.  Each pin is defined in ``tests/oracle_pins.py``.  The
planted-mistake test compiles altered copies of the oracle source (in a
temporary directory, never in the tree) and requires every alteration to be
caught by at least one pin.
"""
import os
import shutil
import tempfile

import pytest

import oracle
from oracle_pins import PINS

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "qsa_oracle.c")


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


# (name, text in the oracle source, replacement).  Each is a plausible slip:
# a dropped term, a wrong sign or index, an operand taken from the wrong array.
MUTANTS = [
    ("drop_v_scale", "++d) out[d] += w * (vs * (double)v_row[d]);",
     "++d) out[d] += w * ((double)v_row[d]);"),
    ("partial_drops_v_scale", "o_out[d] += w * (vs * (double)v_row[d]);",
     "o_out[d] += w * ((double)v_row[d]);"),
    ("partial_l_off_by_max", "double w = exp(s[i] - m);\n            l += w;",
     "double w = exp(s[i] - m);\n            l += 1.0;"),
    ("drop_k_scale", "double k_hat = (double)k_scale * (double)k_row[d];",
     "double k_hat = (double)k_row[d];"),
    ("drop_softmax_scale", "return softmax_scale * dot;", "return dot;"),
    ("flip_exp_sign", "double w = exp(s[i] - m);\n            L += w;",
     "double w = exp(m - s[i]);\n            L += w;"),
    ("no_max_shift", "double w = exp(s[i] - m);\n            L += w;",
     "double w = exp(s[i]);\n            L += w;"),
    ("position_not_slot", "cell_score(D, q, k_codes + (size_t)slot * D",
     "cell_score(D, q, k_codes + (size_t)(sel[start + i] % pool_cells) * D"),
    ("k_from_v_pool", "int err = score_range(D, pool_cells, page_table_len, page_cells, limit, q, k_codes,\n                          k_scale, page_table, sel, 0, n_sel",
     "int err = score_range(D, pool_cells, page_table_len, page_cells, limit, q, v_codes,\n                          k_scale, page_table, sel, 0, n_sel"),
    ("masked_as_slot0", "if (s == -1) { *slot = -1; return ORACLE_OK; }",
     "if (s == -1) { *slot = 0; return ORACLE_OK; }"),
    ("chunk_ignores_start", "sel[start + i], &slot", "sel[i], &slot"),
    ("merge_no_rescale", "double f = exp(m[c] - M);", "double f = 1.0;"),
    ("page_offset_dropped", "*slot = s * page_cells + pos % page_cells;", "*slot = s * page_cells;"),
    ("page_entry_as_cell", "*slot = s * page_cells + pos % page_cells;", "*slot = s + pos % page_cells;"),
    ("page_index_is_position", "int32_t s = page_table[pos / page_cells];",
     "int32_t s = page_table[pos % page_table_len];"),
    ("limit_ignored", "if (sel[start + i] >= limit) slot = -1;", ""),
    ("limit_off_by_one", "if (sel[start + i] >= limit) slot = -1;", "if (sel[start + i] > limit) slot = -1;"),
    ("limit_of_first_query", "limits ? limits[(size_t)b * T + t] : INT32_MAX",
     "limits ? limits[(size_t)b * T] : INT32_MAX"),
    ("kv_head_by_modulo", "int g = h / H;", "int g = h % G;"),
    ("normaliser_dropped", "for (int d = 0; d < D; ++d) out[d] /= L;\n    }\n    free(slots);",
     "\n    }\n    free(slots);"),
    ("v_row_from_position", "const int8_t *v_row = v_codes + (size_t)slots[i] * D;\n            double vs = (double)v_scale[slots[i]];\n            for (int d = 0; d < D; ++d) out[d]",
     "const int8_t *v_row = v_codes + (size_t)(sel[i] % pool_cells) * D;\n            double vs = (double)v_scale[slots[i]];\n            for (int d = 0; d < D; ++d) out[d]"),
]


def test_mutants_are_distinct_edits():
    src = open(ORACLE_SRC).read()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, f"mutant {name}: anchor found {src.count(old)} times"


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib_path = oracle.compile_library(path, os.path.join(tmp, f"lib_{name}.so"))
        lib = oracle.load(lib_path)
        failed = []
        for pin in PINS:
            try:
                pin(lib)
            except (AssertionError, oracle.OracleError, FloatingPointError, ValueError):
                failed.append(pin.__name__)
        assert failed, f"no pin catches the planted mistake {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


# Planted mistakes in the oracle's Python wrapper: the exact widening of bf16
# query bit patterns (the prompt-shaped configuration's queries).  Each edit
# is applied to a copy of oracle/__init__.py loaded as a separate module; the
# C library stays the correct one.
ORACLE_PY = os.path.join(os.path.dirname(oracle.__file__), "__init__.py")
WIDEN_ANCHOR = "(np.asarray(q, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)"
PY_MUTANTS = [
    ("bf16_shift_by_8", WIDEN_ANCHOR,
     "(np.asarray(q, dtype=np.uint16).astype(np.uint32) << np.uint32(8)).view(np.float32)"),
    ("bf16_read_as_fp16", WIDEN_ANCHOR,
     "np.asarray(q, dtype=np.uint16).view(np.float16).astype(np.float32)"),
    ("bf16_low_mantissa_bit_dropped", WIDEN_ANCHOR,
     "((np.asarray(q, dtype=np.uint16).astype(np.uint32) & np.uint32(0xFFFE)) << np.uint32(16)).view(np.float32)"),
    ("bf16_sign_dropped", WIDEN_ANCHOR,
     "((np.asarray(q, dtype=np.uint16).astype(np.uint32) & np.uint32(0x7FFF)) << np.uint32(16)).view(np.float32)"),
]


def _load_module_from_source(src: str, name: str):
    import importlib.util
    import sys
    tmp = tempfile.mkdtemp(prefix="oracle_pymutant_")
    path = os.path.join(tmp, "__init__.py")
    with open(path, "w") as f:
        f.write(src)
    spec = importlib.util.spec_from_file_location(name, path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod
    spec.loader.exec_module(mod)
    return mod, tmp


def test_widening_anchor_is_unique():
    assert open(ORACLE_PY).read().count(WIDEN_ANCHOR) == 1


@pytest.mark.parametrize("name,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_planted_widening_mistake_is_caught(name, old, new, oracle_lib):
    from oracle_pins import pin_golden_bf16_queries
    src = open(ORACLE_PY).read()
    assert src.count(old) == 1
    mod, tmp = _load_module_from_source(src.replace(old, new), f"oracle_mutant_{name}")
    try:
        with pytest.raises(AssertionError):
            pin_golden_bf16_queries(oracle_lib, ora=mod)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
