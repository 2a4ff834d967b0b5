"""The tensor-core decode path's error against bounds derived from its
arithmetic (tests/error_model.py), on the decode configurations.

For every output element: |gpu - refq| <= B (the probabilistic bound of the
kernel's fp32/f16 arithmetic after the query rounding) and <= A (its worst
case), and |gpu - ref64| <= A + A_q, where ref64 is the fp64 oracle on the
caller's queries and refq the oracle on the queries the kernel multiplies
(f16 hi + lo; hi alone only for windows of more than 64 rows with causal
limits, which these calls do not have).  Per output row, relative to the row's norm:
||gpu - ref64|| <= ||refq - ref64|| + ||B||, the exact cost of the query
rounding plus the bound of the rest.  Whether the kernel applied the low
part shows in the mean error: the output is nearer the oracle on the
queries it was meant to multiply than the oracle on the other choice.
"""
import numpy as np
import pytest

import oracle
import qsa_workloads as wl
import error_model as em

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_selection_int8_gb300 import build
    build.build()
    oracle.build()


CONFIGS = {
    "tiny_decode": lambda: wl.tiny_decode(),
    "qsa_decode_T1": lambda: wl.qsa_decode(1),
    "qsa_decode_T2": lambda: wl.qsa_decode(2),
    "qsa_decode_T3": lambda: wl.qsa_decode(3),
    "qsa_decode_T4": lambda: wl.qsa_decode(4),
    "qsa_decode_T6": lambda: wl.make_problem(n_queries=6, pool_cells=32768, n_selected=2051, chunk_cells=128,
                                             seed=9900),
    "batched_T6": lambda: wl.make_problem(n_seq=3, n_kv_heads=2, n_queries=6, pool_cells=8192,
                                          n_selected=[2051, 700, 1300], chunk_cells=128, seed=9901),
    "batched_decode": lambda: wl.batched_decode(),
    "long_context": lambda: wl.long_context(),
    "long_context_pages16": lambda: wl.long_context_paged(16),
}


@pytest.mark.parametrize("name", list(CONFIGS))
def test_decode_error_inside_derived_bounds(name):
    import sparse_selection_int8_gb300 as qsa
    p = CONFIGS[name]()
    dp = qsa.DeviceProblem(p, algo=qsa.QSA_ALGO_TCGEN05)
    dp.out.fill_(float("nan"))
    dp.run()
    torch.cuda.synchronize()
    assert int(dp.status.item()) == 0
    gpu = dp.out.cpu().numpy().astype(np.float64)
    ref64 = oracle.decode_attn(p)
    ref16 = oracle.decode_attn(em.with_kernel_queries(p))
    A, B, Aq, emax = em.problem_bounds(p)
    assert emax < 1e-2
    d16 = np.abs(gpu - ref16)
    assert np.all(d16 <= B), f"{name}: max |gpu - ref16| / B = {float((d16 / B).max()):.3g}"
    assert np.all(d16 <= A), f"{name}: max |gpu - ref16| / A = {float((d16 / A).max()):.3g}"
    assert np.all(np.abs(gpu - ref64) <= A + Aq), name
    D = p.head_dim
    lhs = np.linalg.norm((gpu - ref64).reshape(-1, D), axis=1)
    rhs = (np.linalg.norm((ref16 - ref64).reshape(-1, D), axis=1)
           + np.linalg.norm(B.reshape(-1, D), axis=1))
    assert np.all(lhs <= rhs), f"{name}: row-norm bound"
    other = oracle.decode_attn(em.with_kernel_queries(p, split=not em.split_applies(p)))
    assert em.split_visible(gpu, ref16, other), f"{name}: the output follows the other query rounding"
    rn = np.linalg.norm(ref64.reshape(-1, D), axis=1)
    print(f"{name}: split {em.split_applies(p)}; max |gpu-refq|/B {float((d16 / B).max()):.3f}; per row, relative to the row norm: "
          f"error {float((lhs / rn).max()):.2e}, of it the query rounding {float((em.row_norm_errors(ref16, ref64)).max()):.2e}, "
          f"bound {float((rhs / rn).max()):.2e}")
