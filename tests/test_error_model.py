"""The decode path's error bounds (tests/error_model.py) checked on the CPU.

A numpy emulation of the tensor-core kernel's arithmetic (queries split into
f16 hi + lo, fp32 scores, f16 P', fp32 sums and merge) must stay inside bounds
A and B against the fp64 oracle on the kernel's queries hi + lo, and inside
A + A_q against the oracle on the caller's queries, with a partial per chunk
and with partials over runs of chunks.  Planted changes of the
arithmetic (P' rounded to bf16; queries rounded to bf16) must leave bound B:
it is not vacuous.  Queries rounded to f16 with no low part stay inside B (the
query rounding is about as large as the P' rounding), so whether the low part
is applied is told apart by the mean error against the two references.  (The a-priori
bound A_q of the query rounding is a worst case over every rounding direction
and far looser than the rounding's actual effect, which the tests take exactly
from the oracle on the kernel's queries.)
"""
import numpy as np
import pytest

import oracle
import qsa_workloads as wl
import error_model as em


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def emulate(p, p_round=np.float16, q_round="split", run_chunks=1):
    """The kernel's arithmetic in numpy: partials over runs of run_chunks
    chunks (one chunk by default) against the run's maximum with sigma = the
    run's largest V scale, merged in fp32."""
    T, G, H, D = p.n_queries, p.n_kv_heads, p.q_per_kv, p.head_dim
    out = np.zeros((p.n_seq, T, G * H, D), np.float32)
    log2e = np.float32(1.0 / np.log(2.0))
    ln2 = np.float32(np.log(2.0))
    for b in range(p.n_seq):
        for g in range(G):
            kc, vc, ks, vs = em.cells_of(p, b, g)
            rows = np.asarray(p.q, np.float32)[b, :, g * H:(g + 1) * H, :].reshape(T * H, D)
            if q_round == "split":
                hi = rows.astype(np.float16).astype(np.float32)
                lo = (rows - hi).astype(np.float16).astype(np.float32)
                q16 = None
            elif q_round is np.float16:
                q16 = rows.astype(np.float16).astype(np.float32)
            else:  # bf16: keep the high 16 bits, rounded to nearest even
                u = rows.view(np.uint32).astype(np.uint64)
                u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
                q16 = u.astype(np.uint32).view(np.float32)
            ksc = (ks.astype(np.float32) * np.float32(p.softmax_scale) * log2e).astype(np.float32)
            if q16 is None:  # K.hi + K.lo into one fp32 accumulator
                S = (hi @ kc.astype(np.float32).T + lo @ kc.astype(np.float32).T).astype(np.float32)
            else:
                S = q16 @ kc.astype(np.float32).T                # fp32 sums
            x = (S * ksc[None, :]).astype(np.float32)            # log2 units
            C = p.chunk_cells * run_chunks
            ms, ls, os_ = [], [], []
            for c0 in range(0, kc.shape[0], C):
                xc = x[:, c0:c0 + C]
                m = xc.max(axis=1, keepdims=True)
                pr = np.exp2(xc - m).astype(np.float32)
                sig = np.float32(np.abs(vs[c0:c0 + C]).max())
                pp = (pr * (vs[c0:c0 + C].astype(np.float32) / sig)[None, :]).astype(np.float32)
                pq = pp.astype(p_round).astype(np.float32) if p_round is np.float16 else \
                    ((pp.view(np.uint32).astype(np.uint64) + 0x7FFF + ((pp.view(np.uint32) >> 16) & 1))
                     >> 16 << 16).astype(np.uint32).view(np.float32)
                os_.append(sig * (pq @ vc[c0:c0 + C].astype(np.float32)))
                ls.append(pr.sum(axis=1, dtype=np.float32))
                ms.append(m[:, 0] * ln2)
            ms, ls, os_ = np.array(ms), np.array(ls), np.array(os_)
            Mx = ms.max(axis=0)
            f = np.exp(ms - Mx[None, :]).astype(np.float32)
            o = (f[:, :, None] * os_).sum(axis=0) / (f * ls).sum(axis=0)[:, None]
            out[b, :, g * H:(g + 1) * H, :] = o.reshape(T, H, D)
    return out


PROBLEMS = {
    "tiny_decode": lambda: wl.tiny_decode(),
    "qsa_decode_T4": lambda: wl.qsa_decode(4),
    "two_heads_chunk_200": lambda: wl.make_problem(n_seq=2, n_kv_heads=2, n_queries=2, pool_cells=8192,
                                                   n_selected=[1500, 333], chunk_cells=200, seed=9800),
}


@pytest.fixture(scope="module", params=sorted(PROBLEMS))
def case(request):
    p = PROBLEMS[request.param]()
    A, B, Aq, emax = em.problem_bounds(p, run_chunks=1)  # the emulation: a partial per chunk
    ref64 = oracle.decode_attn(p)
    ref16 = oracle.decode_attn(em.with_kernel_queries(p))
    return request.param, p, A, B, Aq, emax, ref64, ref16


def test_emulated_kernel_inside_bounds(case):
    name, p, A, B, Aq, emax, ref64, ref16 = case
    assert emax < 1e-2, name
    out = emulate(p)
    d16 = np.abs(out - ref16)
    assert np.all(d16 <= B), (name, float((d16 / B).max()))
    assert np.all(d16 <= A), (name, float((d16 / A).max()))
    assert np.all(np.abs(out - ref64) <= A + Aq), name
    # the query rounding alone stays inside its a-priori bound
    assert np.all(np.abs(ref16 - ref64) <= Aq), name


@pytest.mark.parametrize("run_chunks", [3, 8])
def test_emulated_runs_inside_the_default_bounds(case, run_chunks):
    """Partials over runs of up to RUN_CHUNKS chunks (as one CTA accumulates
    them) stay inside the bounds taken for such runs."""
    name, p, A, B, Aq, emax, ref64, ref16 = case
    A8, B8, Aq8, _ = em.problem_bounds(p)
    out = emulate(p, run_chunks=run_chunks)
    d16 = np.abs(out - ref16)
    assert np.all(d16 <= B8) and np.all(d16 <= A8), (name, float((d16 / B8).max()))
    assert np.all(np.abs(out - ref64) <= A8 + Aq8), name


def test_p_in_bf16_leaves_the_bounds(case):
    """P' rounded to bf16 (2^-8) instead of f16: outside bound B."""
    name, p, A, B, Aq, emax, ref64, ref16 = case
    out = emulate(p, p_round="bf16")
    assert np.any(np.abs(out - ref16) > B), name


def test_queries_in_bf16_leave_the_bounds(case):
    """Queries rounded to bf16: outside bound B around the oracle on the
    kernel's queries."""
    name, p, A, B, Aq, emax, ref64, ref16 = case
    out = emulate(p, q_round="bf16")
    assert np.any(np.abs(out - ref16) > B), name


def test_low_part_shows_in_the_mean_error(case):
    """With the split the output is nearer (on average over the elements) the
    oracle on hi + lo than the oracle on hi alone; without it, the reverse."""
    name, p, A, B, Aq, emax, ref64, ref16 = case
    r_hi = oracle.decode_attn(em.with_kernel_queries(p, split=False))
    for mode, split in (("split", True), (np.float16, False)):
        out = emulate(p, q_round=mode)
        assert em.split_visible(out, ref16, r_hi) == split, (name, mode)


def test_f16_only_model_holds_for_f16_only_arithmetic(case):
    """The bounds for hi alone (windows of more than 64 rows over several
    pairs) hold for the emulation that uses hi alone."""
    name, p, A, B, Aq, emax, ref64, ref16 = case
    A1, B1, Aq1, _ = em.problem_bounds(p, split=False, run_chunks=1)
    r1 = oracle.decode_attn(em.with_kernel_queries(p, split=False))
    out = emulate(p, q_round=np.float16)
    d = np.abs(out - r1)
    assert np.all(d <= B1) and np.all(d <= A1) and np.all(np.abs(out - ref64) <= A1 + Aq1), name


def test_row_norm_bound(case):
    """Per row: ||out - ref64|| <= ||ref16 - ref64|| + ||B|| (the exact effect
    of the query rounding plus the bound of the rest)."""
    name, p, A, B, Aq, emax, ref64, ref16 = case
    out = emulate(p)
    D = p.head_dim
    lhs = np.linalg.norm((out - ref64).reshape(-1, D), axis=1)
    rhs = np.linalg.norm((ref16 - ref64).reshape(-1, D), axis=1) + np.linalg.norm(B.reshape(-1, D), axis=1)
    assert np.all(lhs <= rhs), name


def test_run_cap_matches_the_kernel():
    """The bounds take a partial's fp32 sums over at most RUN_CHUNKS chunks:
    the decode kernel's own cap on the chunks a CTA accumulates."""
    import os
    import re
    src = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "sparse_selection_int8_gb300", "csrc", "qsa_chunk_tc.cu")
    m = re.search(r"constexpr int kRunChunks = (\d+);", open(src).read())
    assert m and int(m.group(1)) == em.RUN_CHUNKS
