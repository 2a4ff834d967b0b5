"""The shared parity gate (tests/parity.py) checked on the CPU against the
numpy emulation of the decode kernel's arithmetic (tests/test_error_model.py).

The emulated arithmetic (queries as f16 high and low parts, f16 P', fp32 sums
and merge) passes with room to spare.  Two planted losses of precision fail
the per-row bar although they pass the per-element one: queries rounded to
bf16, and the kernel's own error made ten times larger.
"""
import numpy as np
import pytest

import oracle
import parity
from test_error_model import PROBLEMS, emulate


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


@pytest.fixture(scope="module", params=sorted(PROBLEMS))
def case(request):
    p = PROBLEMS[request.param]()
    return request.param, p, oracle.decode_attn(p), emulate(p)


def test_kernel_arithmetic_passes_with_margin(case):
    name, p, ref, out = case
    e = parity.assert_parity(out, ref, name)
    assert e["max_row_rel"] <= parity.ROW_RTOL / 4, (name, e)


def test_queries_in_bf16_fail_the_row_bar(case):
    name, p, ref, _ = case
    e = parity.errors(emulate(p, q_round="bf16"), ref)
    assert e["max_abs"] <= parity.ATOL and e["max_rel_floored"] <= parity.RTOL, (name, e)
    assert e["max_row_rel"] > parity.ROW_RTOL, (name, e)


def test_tenfold_error_fails_the_row_bar(case):
    name, p, ref, out = case
    e = parity.errors(ref + 10.0 * (out.astype(np.float64) - ref), ref)
    assert e["max_abs"] <= parity.ATOL and e["max_rel_floored"] <= parity.RTOL, (name, e)
    assert e["max_row_rel"] > parity.ROW_RTOL, (name, e)


def test_rows_of_zeros_are_held_to_an_absolute_norm():
    ref = np.zeros((3, 256))
    assert parity.errors(ref, ref)["max_row_rel"] == 0.0
    off = ref.copy()
    off[1, 7] = 3e-5  # a norm above 2e-5 on a row whose exact value is zero
    assert parity.errors(off, ref)["max_row_rel"] > parity.ROW_RTOL
