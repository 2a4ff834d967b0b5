"""GPU parity of QSA block selection (scores, top-k, the selected list)
against the fp64 oracle, through the C ABI.

With whole-number inputs (keys and queries in [-8, 8]) every score is an
integer below 2^24, exact in fp32 whatever the order of the additions, so
the scores, the kept block ids, the list and its offsets must match the
oracle bit for bit.  With N(0,1) inputs the fp32 scores differ from the
oracle's by at most F * 2^-24 * sum |q * k| (a bound for any order of F
additions); the kept sets are then checked for validity: the right count,
and no candidate left out that scores above a kept one by more than twice
that bound.
"""
import numpy as np
import pytest

import oracle
import oracle.select_blocks as osb
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


def run(sp):
    import sparse_selection_int8_gb300 as qsa
    ds = qsa.DeviceSelection(sp)
    ds.scores.fill_(float("nan"))
    ds.kept.fill_(-7)
    ds.run()
    torch.cuda.synchronize()
    return ds, ds.result()


def check_exact(sp, what):
    ds, (s, k, sel, off) = run(sp)
    rs, rk, rsel, roff = osb.select_batch(sp)
    assert np.array_equal(s, rs.astype(np.float32)), what
    assert np.array_equal(k, rk), what
    assert np.array_equal(off, roff), what
    assert np.array_equal(sel, rsel), what
    assert int(ds.status.item()) == 0
    return ds


CASES = [
    dict(n_seq=1, n_queries=1, idx_heads=1, idx_dim=8, block_cells=1, max_blocks=7, top_k=3),
    dict(n_seq=3, n_queries=2, idx_heads=4, idx_dim=64, block_cells=64, max_blocks=300, top_k=17,
         n_live=[19200, 1000, 0]),
    dict(n_seq=2, n_queries=4, idx_heads=2, idx_dim=4, block_cells=5, max_blocks=1000, top_k=999,
         n_live=[4999, 5000]),
    dict(n_seq=4, n_queries=8, idx_heads=8, idx_dim=128, block_cells=16, max_blocks=512, top_k=64),
    dict(n_seq=1, n_queries=3, idx_heads=4, idx_dim=64, block_cells=64, max_blocks=16384, top_k=256),
    dict(n_seq=2, n_queries=2, idx_heads=16, idx_dim=64, block_cells=32, max_blocks=100, top_k=100,
         with_steps=False),
    dict(n_seq=5, n_queries=1, idx_heads=2, idx_dim=16, block_cells=7, max_blocks=33, top_k=1,
         n_live=[1, 7, 8, 230, 231]),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_integer_inputs_exact(case):
    check_exact(wl.make_selection(integer=True, seed=9300 + case, **CASES[case]), f"case {case}")


def test_many_ties_exact():
    """Keys of one value in a few places: most scores tie, the top-k
    boundary falls inside a tie, the lower ids must win."""
    sp = wl.make_selection(n_seq=2, n_queries=2, idx_heads=1, idx_dim=8, block_cells=3, max_blocks=500,
                           top_k=37, integer=True, seed=9400)
    sp.pooled[:] = wl.bf16_bits_from_f32(np.sign(wl.f32_from_bf16_bits(sp.pooled)))
    check_exact(sp, "ties")


def test_long_selection_integer_exact():
    sp = wl.long_selection()
    spi = wl.make_selection(n_seq=sp.n_seq, n_queries=sp.n_queries, idx_heads=sp.idx_heads, idx_dim=sp.idx_dim,
                            block_cells=sp.block_cells, max_blocks=sp.max_blocks, top_k=sp.top_k, integer=True,
                            seed=9401)
    check_exact(spi, "long selection, whole numbers")


def test_long_selection_float_valid():
    sp = wl.long_selection()
    ds, (s, k, sel, off) = run(sp)
    rs, rk, rsel, roff = osb.select_batch(sp)
    q = sp.q_idx.astype(np.float64)
    keys = osb.widen_bf16(sp.pooled)
    F = sp.idx_heads * sp.idx_dim
    for b in range(sp.n_seq):
        bound = F * 2.0 ** -24 * np.abs(q[b]) @ np.abs(keys[b]).T      # [T][NB]
        fin = np.isfinite(rs[b])
        assert np.array_equal(np.isfinite(s[b]), fin)
        assert np.all(np.abs(s[b][fin] - rs[b][fin]) <= bound[fin] + 1e-30)
        for t in range(sp.n_queries):
            kept = k[b, t][k[b, t] >= 0]
            assert len(kept) == min(sp.top_k, int(fin[t].sum()))
            assert np.all(np.diff(kept) > 0)
            out = np.setdiff1d(np.nonzero(fin[t])[0], kept)
            if len(out) and len(kept):
                worst_kept = (rs[b, t, kept] + bound[t, kept]).min()
                best_out = (rs[b, t, out] - bound[t, out]).max()
                assert best_out <= worst_kept + 2 * bound[t].max()
        # the list is the expansion of the union of the kept sets
        union = sorted(set(int(j) for t in range(sp.n_queries) for j in k[b, t] if j >= 0))
        assert np.array_equal(sel[off[b]:off[b + 1]], osb.expand(union, sp.block_cells, int(sp.n_live[b])))


def test_repeat_and_back_to_back():
    """Calls of two problems alternate on one stream: each result is
    bit-identical to its first call (the bitmaps start empty every call)."""
    import sparse_selection_int8_gb300 as qsa
    a = wl.make_selection(n_seq=3, n_queries=2, max_blocks=700, top_k=40, seed=9500)
    b = wl.make_selection(n_seq=3, n_queries=2, max_blocks=700, top_k=40, seed=9501)
    da, db = qsa.DeviceSelection(a), qsa.DeviceSelection(b)
    first = []
    for ds in (da, db):
        ds.run()
        torch.cuda.synchronize()
        first.append(ds.result())
    for _ in range(3):
        for ds, ref in ((da, first[0]), (db, first[1])):
            ds.run()
            torch.cuda.synchronize()
            got = ds.result()
            assert all(np.array_equal(x.view(np.uint32) if x.dtype == np.float32 else x,
                                      y.view(np.uint32) if y.dtype == np.float32 else y) for x, y in zip(got, ref))


def test_bad_extent_is_clamped_and_reported():
    import sparse_selection_int8_gb300 as qsa
    sp = wl.make_selection(n_seq=2, n_queries=1, max_blocks=10, block_cells=4, top_k=3, n_live=[40, 40],
                           integer=True, seed=9600, with_steps=False)
    ds = qsa.DeviceSelection(sp)
    ds.n_live.copy_(torch.tensor([-5, 99], dtype=torch.int32))
    ds.run()
    torch.cuda.synchronize()
    assert int(ds.status.item()) & qsa.QSA_STATUS_BAD_EXTENT
    s, k, sel, off = ds.result()
    sp.n_live[:] = [0, 40]
    rs, rk, rsel, roff = osb.select_batch(sp)
    assert np.array_equal(k, rk) and np.array_equal(sel, rsel) and np.array_equal(off, roff)


def test_selection_feeds_attention():
    """The selected list drives a qsa_decode_attn_batch call directly (device
    to device): the output matches the oracle's attention over the oracle's
    list on the same pools."""
    import sparse_selection_int8_gb300 as qsa
    sp = wl.make_selection(n_seq=2, n_queries=2, idx_heads=4, idx_dim=64, block_cells=16, max_blocks=256,
                           top_k=12, integer=True, seed=9700)
    ds = qsa.DeviceSelection(sp)
    ds.run()
    _, _, rsel, roff = osb.select_batch(sp)
    p = wl.make_problem(n_seq=2, n_kv_heads=2, n_queries=2, pool_cells=sp.max_blocks * sp.block_cells,
                        n_selected=[int(roff[1] - roff[0]), int(roff[2] - roff[1])], chunk_cells=128, seed=9701)
    p.sel = rsel.astype(np.int32)
    p.sel_offsets = roff.astype(np.int32)
    dp = qsa.DeviceProblem(p, max_selected=ds.max_selected)
    qsa.qsa_decode_attn_batch(dp.shape, 2, dp.q, dp.k_pool, dp.v_pool, dp.k_scale, dp.v_scale, dp.page_table,
                              ds.sel, ds.sel_offsets, ds.max_selected, dp.out, dp.workspace, dp.ws_bytes,
                              dp.status)
    torch.cuda.synchronize()
    assert int(dp.status.item()) == 0
    assert_parity(dp.out.cpu().numpy(), oracle.decode_attn(p), "attention over the selected list")
