"""GPU parity of the decode kernel's row split at its block boundaries.

A call on one (sequence, KV head) with few chunks splits its T*H rows into
blocks of 16 (or 32, 48, 64) rows within half the SMs; a call over several
pairs with more than 24 rows splits them into blocks of 24 with one query
image per (pair, block).  Rows just below, at and above each block size, a
last block of a single row, and chunk counts that change the block size are
checked against the fp64 oracle, and a single-pair call's step and batch
entries against each other bit for bit.
"""
import numpy as np
import pytest

import oracle
import qsa_workloads as wl
from parity import assert_parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_selection_int8_gb300 import build
    build.build()
    oracle.build()


def run(p, batch=None):
    import sparse_selection_int8_gb300 as qsa
    dp = qsa.DeviceProblem(p, algo=qsa.QSA_ALGO_TCGEN05)
    dp.workspace.fill_(0xFF)   # NaN bytes: an unwritten partial or query image shows
    dp.out.fill_(float("nan"))
    dp.run(batch=batch)
    torch.cuda.synchronize()
    assert int(dp.status.item()) == 0
    return dp.out.cpu().numpy()


# (q_per_kv, n_queries): rows 15, 16, 17, 31, 33, 48, 49 and 65 (a last block of one row)
SINGLE = [(15, 1), (16, 1), (17, 1), (31, 1), (11, 3), (12, 4), (7, 7), (13, 5)]


@pytest.mark.parametrize("H,T", SINGLE)
def test_single_pair_blocks(H, T):
    p = wl.make_problem(n_seq=1, n_kv_heads=1, q_per_kv=H, n_queries=T, pool_cells=8192,
                        n_selected=2051, chunk_cells=128, seed=9950 + H * 8 + T)
    assert_parity(run(p), oracle.decode_attn(p), f"single pair, {H * T} rows")


@pytest.mark.parametrize("chunk", [16, 64, 512])
def test_single_pair_chunk_counts_change_the_blocks(chunk):
    """2,051 cells in 129 / 33 / 5 chunks: 48 rows go unsplit, to 32-row or
    16-row blocks as the chunks leave SMs free."""
    p = wl.make_problem(n_seq=1, n_kv_heads=1, n_queries=4, pool_cells=8192, n_selected=2051,
                        chunk_cells=chunk, seed=9970 + chunk)
    assert_parity(run(p), oracle.decode_attn(p), f"single pair, chunk {chunk}")


def test_single_pair_step_equals_batch_bitwise():
    p = wl.make_problem(n_seq=1, n_kv_heads=1, n_queries=3, pool_cells=8192, n_selected=1500,
                        chunk_cells=128, seed=9980)
    a = run(p, batch=False)
    b = run(p, batch=True)
    assert np.array_equal(a, b)


# (q_per_kv, n_queries): rows 24 (no split), 25, 36, 47, 48, 49 (last block of one row), 72
MULTI = [(12, 2), (25, 1), (12, 3), (47, 1), (12, 4), (7, 7), (12, 6)]


@pytest.mark.parametrize("H,T", MULTI)
def test_multi_pair_blocks(H, T):
    p = wl.make_problem(n_seq=3, n_kv_heads=2, q_per_kv=H, n_queries=T, pool_cells=8192,
                        n_selected=[2051, 129, 700], chunk_cells=128, seed=9990 + H * 8 + T)
    assert_parity(run(p), oracle.decode_attn(p), f"3 sequences x 2 KV heads, {H * T} rows")


def test_multi_pair_with_empty_sequences():
    p = wl.make_problem(n_seq=4, n_kv_heads=2, n_queries=4, pool_cells=4096,
                        n_selected=[0, 300, 0, 1025], chunk_cells=64, seed=9999)
    assert_parity(run(p), oracle.decode_attn(p), "ragged batch with empty sequences, 48 rows")
