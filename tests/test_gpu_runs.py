"""GPU parity of the decode kernel's runs: a CTA that takes several
consecutive chunks of one (sequence, KV head) accumulates them into one
partial (at most eight chunks), and the merge combines the runs' partials.

Each layout below has more chunks than CTAs, so runs form.  The cases are:

- pairs that straddle CTA boundaries;
- runs cut at eight chunks (CTAs of more than eight items);
- row blocks with runs;
- one pair with more chunks than SMs;
- causal limits;
- pages of 16 cells;
- empty sequences among full ones.

Each is checked against the fp64 oracle.  Repeated calls into a workspace
filled with NaN bytes must give the same bits.
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


def run(p):
    import sparse_selection_int8_gb300 as qsa
    dp = qsa.DeviceProblem(p, algo=qsa.QSA_ALGO_TCGEN05)
    dp.workspace.fill_(0xFF)   # NaN bytes: a partial or run count left unwritten shows
    dp.out.fill_(float("nan"))
    dp.run()
    torch.cuda.synchronize()
    assert int(dp.status.item()) == 0
    return dp, dp.out.cpu().numpy()


def window_limits(p, rng, step):
    """Query t of sequence b sees positions below base_b + step * t, base_b
    near the middle of the sequence's selected positions."""
    lim = np.zeros((p.n_seq, p.n_queries), np.int32)
    for b in range(p.n_seq):
        s = np.sort(p.sel_of(b))
        base = int(s[len(s) // 2]) if len(s) else 0
        lim[b] = base + step * np.arange(p.n_queries) + int(rng.integers(0, 3))
    return lim


CASES = {
    # 131 chunks per KV head over 2 heads: about 2 items per CTA, pairs straddle CTAs
    "straddling": dict(n_seq=6, n_kv_heads=2, q_per_kv=12, n_queries=2, pool_cells=8192,
                       n_selected=[2051, 700, 1300, 0, 129, 4000], chunk_cells=64, seed=9601),
    # 688 chunks per KV head, 16-cell chunks: about 10 items per CTA, runs cut at 8
    "runs_cut_at_eight": dict(n_seq=2, n_kv_heads=2, q_per_kv=12, n_queries=1, pool_cells=16384,
                              n_selected=[8000, 3000], chunk_cells=16, seed=9602),
    # 48 rows in two 24-row blocks, 264 items per block
    "row_blocks": dict(n_seq=4, n_kv_heads=2, q_per_kv=12, n_queries=4, pool_cells=8192,
                       n_selected=2051, chunk_cells=64, seed=9603),
    # one (sequence, KV head) with 313 chunks: more chunks than SMs
    "one_pair_313_chunks_12_rows": dict(n_seq=1, n_kv_heads=1, q_per_kv=12, n_queries=1, pool_cells=65536,
                                        n_selected=40000, chunk_cells=128, seed=9604),
    "one_pair_313_chunks_48_rows": dict(n_seq=1, n_kv_heads=1, q_per_kv=12, n_queries=4, pool_cells=65536,
                                        n_selected=40000, chunk_cells=128, seed=9605),
    # two-tile chunks (the long-context chunk size)
    "two_tile_chunks": dict(n_seq=8, n_kv_heads=2, q_per_kv=12, n_queries=2, pool_cells=16384,
                            n_selected=[6000, 300, 5000, 2051, 0, 4097, 256, 7000], chunk_cells=256,
                            seed=9606),
    "pages_of_16": dict(n_seq=4, n_kv_heads=2, q_per_kv=12, n_queries=2, pool_cells=16384,
                        n_selected=[5000, 3000, 4500, 1000], chunk_cells=64, page_cells=16, seed=9607),
    "empty_sequences": dict(n_seq=8, n_kv_heads=2, q_per_kv=12, n_queries=2, pool_cells=8192,
                            n_selected=[0, 3000, 0, 0, 2500, 0, 1, 0], chunk_cells=32, seed=9608),
}


@pytest.mark.parametrize("name", list(CASES))
def test_runs_against_oracle(name):
    p = wl.make_problem(name=name, **CASES[name])
    _, out = run(p)
    assert_parity(out, oracle.decode_attn(p), name)


@pytest.mark.parametrize("T,H,G", [(2, 12, 2), (4, 12, 1), (3, 5, 3)])
def test_runs_with_causal_limits(T, H, G):
    rng = np.random.default_rng(9650 + 10 * T + H + G)
    p = wl.make_problem(n_seq=4, n_kv_heads=G, q_per_kv=H, n_queries=T, pool_cells=16384,
                        n_selected=[6000, 2500, 37, 4000], chunk_cells=32, mask_fraction=0.05,
                        seed=int(rng.integers(1 << 30)))
    p.q_limit = window_limits(p, rng, 53)
    _, out = run(p)
    assert_parity(out, oracle.decode_attn(p), f"runs with limits T={T} H={H} G={G}")


@pytest.mark.parametrize("name", ["straddling", "runs_cut_at_eight", "one_pair_313_chunks_48_rows"])
def test_runs_bit_identical_across_calls(name):
    p = wl.make_problem(name=name, **CASES[name])
    dp, out0 = run(p)
    for _ in range(3):
        dp.workspace.fill_(0xFF)
        dp.out.fill_(float("nan"))
        dp.run()
        torch.cuda.synchronize()
        assert int(dp.status.item()) == 0
        assert dp.out.cpu().numpy().tobytes() == out0.tobytes()
