"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every configuration of the workload set, the pages' edge cases (0/1/2/3/63/
64/65 selected cells, page -1 masking), chunk sizes around the tile sizes,
ragged batches, out-of-range indices, determinism of the chunk partials and
bit-exact index handling.  Tolerance: ``tests/parity.py``.
"""
import numpy as np
import pytest

import oracle
import qsa_workloads as wl
from parity import assert_parity, errors

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ALGOS = ["auto", "simt", "tcgen05"]


def algo_code(name):
    import sparse_selection_int8_gb300 as qsa
    return {"auto": qsa.QSA_ALGO_AUTO, "simt": qsa.QSA_ALGO_SIMT,
            "tcgen05": qsa.QSA_ALGO_TCGEN05}[name]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_selection_int8_gb300 import build
    build.build()
    oracle.build()


def run(p, algo="auto", batch=None, poison=True, max_selected=None):
    import sparse_selection_int8_gb300 as qsa
    dp = qsa.DeviceProblem(p, algo=algo_code(algo), max_selected=max_selected)
    if poison:
        dp.workspace.fill_(0xFF)   # NaN bytes: any read of an unwritten partial shows
        dp.out.fill_(float("nan"))
    dp.run(batch=batch)
    torch.cuda.synchronize()
    return dp, dp.out.cpu().numpy()


def check_full(p, algo, what):
    dp, out = run(p, algo)
    ref = oracle.decode_attn(p)
    e = assert_parity(out, ref, what)
    assert int(dp.status.item()) == 0
    return e


# ---------------------------------------------------------------- workloads

@pytest.mark.parametrize("algo", ALGOS)
def test_tiny_decode(algo):
    check_full(wl.tiny_decode(), algo, "tiny_decode")


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_qsa_decode(algo, T):
    check_full(wl.qsa_decode(T), algo, f"qsa_decode T={T}")


@pytest.mark.parametrize("algo", ALGOS)
def test_batched_decode(algo):
    check_full(wl.batched_decode(), algo, "batched_decode")


@pytest.mark.parametrize("algo", ["auto"])
def test_long_context(algo):
    check_full(wl.long_context(), algo, "long_context")


@pytest.mark.parametrize("algo", ["auto", "simt"])
def test_prompt_shaped_sampled_rows(algo):
    """Full size (2,048 bf16 queries x 32,768 cells); the oracle computes a
    sample of output rows one by one."""
    p = wl.prompt_shaped()
    dp, out = run(p, algo)
    rng = np.random.Generator(np.random.PCG64(5))
    GH = p.n_kv_heads * p.q_per_kv
    ts = np.concatenate([[0, p.n_queries - 1], rng.integers(0, p.n_queries, 30)])
    hs = rng.integers(0, GH, ts.shape[0])
    rows = [oracle.flat_row(p, 0, int(t), int(h)) for t, h in zip(ts, hs)]
    ref = oracle.decode_attn(p, rows=rows)
    got = np.stack([out[0, t, h] for t, h in zip(ts, hs)])
    assert_parity(got, ref, "prompt_shaped")
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("algo", ["auto"])
def test_prompt_shaped_small_full(algo):
    """A smaller prompt-shaped call (256 bf16 queries x 4,096 cells, two
    chunks with a ragged tail) checked on every output row."""
    p = wl.prompt_shaped(n_queries=256, pool_cells=4096, chunk_cells=3000)
    check_full(p, algo, "prompt_small")


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("n", [0, 1, 2, 3, 63, 64, 65, 127, 128, 129, 300])
def test_selected_counts(algo, n):
    p = wl.make_problem(n_queries=2, pool_cells=1024, n_selected=n, chunk_cells=64,
                        seed=7000 + n)
    dp, out = run(p, algo)
    ref = oracle.decode_attn(p)
    assert_parity(out, ref, f"n={n}")
    if n == 0:
        assert np.array_equal(out, np.zeros_like(out))


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("C", [1, 7, 64, 127, 128, 129, 256, 2051, 5000])
def test_chunk_sizes(algo, C):
    p = wl.make_problem(n_queries=2, pool_cells=8192, n_selected=2051, chunk_cells=C,
                        seed=7100 + C)
    check_full(p, algo, f"C={C}")


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("T", [1, 3, 5, 6, 8])
def test_query_counts_and_heads(algo, T):
    p = wl.make_problem(n_queries=T, q_per_kv=12, n_kv_heads=3, pool_cells=2048,
                        n_selected=700, chunk_cells=128, seed=7200 + T)
    check_full(p, algo, f"T={T} G=3")


@pytest.mark.parametrize("algo", ALGOS)
def test_page_minus_one_masking(algo):
    p = wl.make_problem(n_queries=4, pool_cells=4096, n_selected=1500, chunk_cells=128,
                        mask_fraction=0.4, seed=7300)
    check_full(p, algo, "masked")
    # every selected cell masked -> zeros
    p.page_table[:] = -1
    dp, out = run(p, algo)
    assert np.array_equal(out, np.zeros_like(out))


@pytest.mark.parametrize("algo", ALGOS)
def test_out_of_range_entries_are_masked_and_reported(algo):
    import sparse_selection_int8_gb300 as qsa
    p = wl.make_problem(n_queries=2, pool_cells=2048, n_selected=600, chunk_cells=64,
                        seed=7400)
    clean_sel = p.sel.copy()
    bad_pos = [5, 77, 300]
    bad_slot_pos = [10, 200]
    p.sel[bad_pos] = [-3, 2048, 99999]
    for i in bad_slot_pos:
        p.page_table[0, p.sel[i]] = 5000 if i == 10 else -7
    dp, out = run(p, algo)
    st = int(dp.status.item())
    assert st & qsa.QSA_STATUS_BAD_POSITION and st & qsa.QSA_STATUS_BAD_SLOT
    keep = np.ones(600, bool)
    keep[bad_pos + bad_slot_pos] = False
    q = wl.make_problem(n_queries=2, pool_cells=2048, n_selected=600, chunk_cells=64,
                        seed=7400)
    q.sel = clean_sel[keep]
    q.sel_offsets = np.array([0, keep.sum()], np.int32)
    ref = oracle.decode_attn(q)
    assert_parity(out, ref, "bad entries")


@pytest.mark.parametrize("algo", ALGOS)
def test_ragged_batch_with_empty_sequences(algo):
    lens = [0, 1, 65, 600, 0, 2051, 129, 3]
    p = wl.make_problem(n_seq=len(lens), n_kv_heads=2, n_queries=3, pool_cells=4096,
                        n_selected=lens, chunk_cells=128, seed=7500)
    dp, out = run(p, algo, max_selected=2100)
    assert_parity(out, oracle.decode_attn(p), "ragged")
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert np.array_equal(out[4], np.zeros_like(out[4]))


@pytest.mark.parametrize("algo", ["auto", "tcgen05"])
@pytest.mark.parametrize("H,T", [(12, 4), (16, 4), (5, 3), (10, 4), (1, 1)])
def test_many_segments_per_cta(algo, H, T):
    """Hundreds of short sequences: every CTA of the decode kernel walks
    several (sequence, KV head) segments, so query tiles are reloaded during
    the walk (both buffering modes: rows up to 48 and 64), with row counts
    that are not multiples of 8 or 16 and some masked pages."""
    rng = np.random.default_rng(7700 + 10 * H + T)
    lens = [int(v) for v in rng.integers(1, 300, size=400)]
    p = wl.make_problem(n_seq=len(lens), n_kv_heads=2, q_per_kv=H, n_queries=T, pool_cells=512,
                        n_selected=lens, chunk_cells=128, mask_fraction=0.1, seed=7700 + 10 * H + T)
    dp, out = run(p, algo, max_selected=max(lens))
    assert_parity(out, oracle.decode_attn(p), f"many segments H={H} T={T}")
    assert int(dp.status.item()) == 0


@pytest.mark.parametrize("algo", ["auto", "tcgen05"])
@pytest.mark.parametrize("H,T,G", [(12, 6, 1), (12, 6, 2), (16, 5, 1), (10, 7, 2)])
def test_wide_windows(algo, H, T, G):
    """Windows of 65-80 query rows (five to seven queries) on the cells-on-M
    decode kernel: one O buffer in tensor memory, 8-row score blocks past 64,
    the query tile converted in the kernel (one KV head) or staged (two), and
    chunks of one tile, two tiles and a partial second tile."""
    for C in (128, 256, 200):
        p = wl.make_problem(n_kv_heads=G, q_per_kv=H, n_queries=T, pool_cells=8192,
                            n_selected=2051, chunk_cells=C, mask_fraction=0.05,
                            seed=9100 + 100 * H + 10 * T + G + C)
        check_full(p, algo, f"wide window H={H} T={T} G={G} C={C}")


@pytest.mark.parametrize("H,T", [(12, 1), (12, 4), (12, 6), (16, 5)])
@pytest.mark.parametrize("G", [1, 2])
def test_decode_path_rescaling(H, T, G):
    """K scales that grow along the list make each row's running max climb by
    tens of log2 units (O is rescaled in tensor memory whenever the reference
    max moves by more than 2^8), and V scales that grow 100x make the chunk's
    V reference move (a tile's largest V scale above 16x the reference), in
    one chunk of 16 tiles.  bf16 queries convert to f16 exactly."""
    p = wl.make_problem(n_kv_heads=G, q_per_kv=H, n_queries=T, pool_cells=4096,
                        n_selected=2048, chunk_cells=2048, q_dtype="bf16",
                        seed=9300 + 10 * H + T + 1000 * G)
    pos = np.argsort(p.page_table[0]).astype(np.float64)  # list position order of each slot
    frac = pos / p.page_table_len
    p.k_scale[0, :] = (0.005 + 0.055 * frac).astype(np.float32)
    p.v_scale[0, :] = (0.0002 * 100.0 ** frac).astype(np.float32)
    check_full(p, "auto", f"decode rescaling H={H} T={T} G={G}")


def expanded_table(p):
    """The same problem with its page table written out per cell (P = 1)."""
    import copy
    P = p.page_cells
    e = copy.copy(p)
    pt = np.repeat(p.page_table, P, axis=1).astype(np.int64)
    off = np.tile(np.arange(P), p.page_table_len)[None, :]
    e.page_table = np.where(pt >= 0, pt * P + off, -1).astype(np.int32)
    e.page_table_len = p.page_table_len * P
    e.page_cells = 1
    return e


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("P", [2, 16, 64])
def test_paged_tables(algo, P):
    """Page tables of P-cell pages with masked pages, on a ragged batch and on
    one sequence: against the oracle, and bit-identical to the same calls with
    the table written out per cell (every cell must resolve to the same slot)."""
    for n_seq, lens in ((3, [700, 1500, 37]), (1, [2051])):
        p = wl.make_problem(n_seq=n_seq, n_kv_heads=2, n_queries=2, pool_cells=8192,
                            n_selected=lens, chunk_cells=128, mask_fraction=0.1,
                            page_cells=P, seed=9500 + P + n_seq)
        dp, out = run(p, algo)
        assert_parity(out, oracle.decode_attn(p), f"paged P={P} B={n_seq}")
        assert int(dp.status.item()) == 0
        _, out1 = run(expanded_table(p), algo)
        assert np.array_equal(out.view(np.uint32), out1.view(np.uint32)), f"P={P} B={n_seq}"


@pytest.mark.parametrize("algo", ["auto", "tcgen05"])
def test_paged_prompt_path(algo):
    p = wl.make_problem(n_queries=64, pool_cells=2048, n_selected=2048, chunk_cells=1024,
                        q_dtype="bf16", selection="full", page_cells=16, seed=9600)
    dp, out = run(p, algo)
    assert_parity(out, oracle.decode_attn(p), "paged prompt path")
    _, out1 = run(expanded_table(p), algo)
    assert np.array_equal(out.view(np.uint32), out1.view(np.uint32))


@pytest.mark.parametrize("algo", ALGOS)
def test_paged_bad_entries_are_masked_and_reported(algo):
    import sparse_selection_int8_gb300 as qsa
    p = wl.make_problem(n_kv_heads=1, n_queries=1, pool_cells=1024, n_selected=300,
                        chunk_cells=64, page_cells=8, seed=9700)
    p.sel[5] = p.page_table_len * 8           # one past the last position
    p.page_table[0, p.sel[40] // 8] = 1024 // 8  # one past the last pool page
    dp, out = run(p, algo)
    assert int(dp.status.item()) == qsa.QSA_STATUS_BAD_POSITION | qsa.QSA_STATUS_BAD_SLOT
    q = copy_problem_masking(p)
    assert_parity(out, oracle.decode_attn(q), "paged bad entries")


def copy_problem_masking(p):
    """The oracle's view of a call with bad entries: they count as masked."""
    import copy
    q = copy.copy(p)
    q.page_table = p.page_table.copy()
    bad_page = p.page_table[0] >= p.pool_cells // p.page_cells
    q.page_table[0, bad_page] = -1
    keep = (p.sel >= 0) & (p.sel < p.page_table_len * p.page_cells)
    q.sel = p.sel[keep]
    q.sel_offsets = np.array([0, q.sel.shape[0]], np.int32)
    return q


def window_limits(p, rng, step=1):
    """Causal limits of a verify window per sequence: query t sees positions
    below base + step * t, with base around the middle of the sequence's
    selected positions (so some selected cells lie beyond every limit)."""
    lim = np.zeros((p.n_seq, p.n_queries), np.int32)
    for b in range(p.n_seq):
        s = np.sort(p.sel_of(b))
        base = int(s[len(s) // 2]) if len(s) else 0
        lim[b] = base + step * np.arange(p.n_queries) + int(rng.integers(0, 3))
    return lim


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("T,H,G", [(1, 12, 1), (4, 12, 1), (6, 12, 2), (3, 5, 3)])
def test_causal_limits(algo, T, H, G):
    """Per-query causal limits inside the window, on ragged batches (chunks of
    one and two tiles) and with the limits spread far apart (step 97) or
    consecutive (step 1): against the oracle."""
    rng = np.random.default_rng(9800 + 10 * T + H + G)
    for C, step in ((128, 1), (256, 97)):
        p = wl.make_problem(n_seq=3, n_kv_heads=G, q_per_kv=H, n_queries=T, pool_cells=4096,
                            n_selected=[600, 1300, 37], chunk_cells=C, mask_fraction=0.05,
                            seed=int(rng.integers(1 << 30)))
        p.q_limit = window_limits(p, rng, step)
        dp, out = run(p, algo)
        assert_parity(out, oracle.decode_attn(p), f"limits T={T} H={H} G={G} C={C}")
        assert int(dp.status.item()) == 0


@pytest.mark.parametrize("algo", ALGOS)
def test_paged_tables_with_causal_limits(algo):
    """Pages of 16 cells and causal limits in one call (the decode kernel's
    page stage resolves both from the same position)."""
    rng = np.random.default_rng(9870)
    p = wl.make_problem(n_seq=3, n_kv_heads=2, n_queries=4, pool_cells=8192,
                        n_selected=[900, 2051, 300], chunk_cells=128, mask_fraction=0.1,
                        page_cells=16, seed=9871)
    p.q_limit = window_limits(p, rng, 37)
    dp, out = run(p, algo)
    assert_parity(out, oracle.decode_attn(p), "paged with limits")
    assert int(dp.status.item()) == 0


@pytest.mark.parametrize("algo", ALGOS)
def test_limits_beyond_every_position_change_nothing(algo):
    """Limits at or above every position: bit for bit the unlimited call."""
    p = wl.make_problem(n_seq=2, n_kv_heads=2, n_queries=4, pool_cells=4096,
                        n_selected=[900, 2051], chunk_cells=128, seed=9900)
    _, ref = run(p, algo)
    p.q_limit = np.full((2, 4), p.n_positions, np.int32)
    _, out = run(p, algo)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("algo", ALGOS)
def test_limits_on_a_wide_window(algo):
    """More than 80 query rows with limits (the rows-on-M kernel under auto):
    a causal prefill of 64 queries over 2,048 cells in 128-cell tiles, each
    query seeing the positions up to its own, and the same window with limits
    cutting tiles at ragged places."""
    ref = None
    for lim0, step in ((1984, 1), (700, 23)):
        p = wl.make_problem(n_queries=64, pool_cells=2048, n_selected=2048, chunk_cells=1024,
                            q_dtype="bf16", selection="full", seed=9950)
        p.q_limit = (lim0 + step * np.arange(64, dtype=np.int32))[None, :]
        dp, out = run(p, algo)
        assert_parity(out, oracle.decode_attn(p), f"limits on a wide window {lim0}+{step}t")
        assert int(dp.status.item()) == 0


def test_decreasing_limits_are_reported():
    import sparse_selection_int8_gb300 as qsa
    p = wl.make_problem(n_seq=2, n_queries=3, pool_cells=1024, n_selected=200, chunk_cells=64,
                        seed=9960)
    p.q_limit = np.array([[100, 200, 300], [500, 400, 600]], np.int32)
    dp, _ = run(p, "auto")
    assert int(dp.status.item()) == qsa.QSA_STATUS_BAD_LIMITS


@pytest.mark.parametrize("algo", ["auto", "simt"])
def test_batch_list_above_bound_is_clamped(algo):
    import sparse_selection_int8_gb300 as qsa
    p = wl.make_problem(n_seq=2, n_queries=1, pool_cells=2048, n_selected=[300, 500],
                        chunk_cells=64, seed=7600)
    dp, out = run(p, algo, max_selected=400)
    assert int(dp.status.item()) & qsa.QSA_STATUS_BAD_OFFSETS
    q = wl.make_problem(n_seq=2, n_queries=1, pool_cells=2048, n_selected=[300, 500],
                        chunk_cells=64, seed=7600)
    q.sel = np.concatenate([q.sel_of(0), q.sel_of(1)[:400]])
    q.sel_offsets = np.array([0, 300, 700], np.int32)
    assert_parity(out, oracle.decode_attn(q), "clamped")


@pytest.mark.parametrize("algo", ALGOS)
def test_output_guard_untouched(algo):
    import sparse_selection_int8_gb300 as qsa
    p = wl.make_problem(n_queries=2, pool_cells=1024, n_selected=200, chunk_cells=64,
                        seed=7700)
    dp = qsa.DeviceProblem(p, algo=algo_code(algo))
    n = dp.out.numel()
    big = torch.full((n + 2048,), 12345.0, device="cuda")
    view = big[1024:1024 + n].view_as(dp.out)
    dp.run(out=view)
    torch.cuda.synchronize()
    b = big.cpu().numpy()
    assert np.all(b[:1024] == 12345.0) and np.all(b[1024 + n:] == 12345.0)
    assert_parity(view.cpu().numpy(), oracle.decode_attn(p), "guard")


# ------------------------------------------------- determinism and indexing

@pytest.mark.parametrize("algo", ALGOS)
def test_partials_bit_identical_across_runs(algo):
    import sparse_selection_int8_gb300 as qsa
    p = wl.qsa_decode(4)
    dp = qsa.DeviceProblem(p, algo=algo_code(algo))
    dp.run()
    torch.cuda.synchronize()
    m0, l0, o0 = qsa.partials_of(dp)
    out0 = dp.out.cpu().numpy()
    side = torch.cuda.Stream()
    for i in range(10):
        dp.workspace.fill_(0xFF)
        if i % 2:
            with torch.cuda.stream(side):
                dp.run(stream=side)
            side.synchronize()
        else:
            dp.run()
            torch.cuda.synchronize()
        m, l, o = qsa.partials_of(dp)
        assert m.tobytes() == m0.tobytes() and l.tobytes() == l0.tobytes()
        assert o.tobytes() == o0.tobytes()
        assert dp.out.cpu().numpy().tobytes() == out0.tobytes()


@pytest.mark.parametrize("algo", ALGOS)
def test_partials_against_oracle(algo):
    import sparse_selection_int8_gb300 as qsa
    p = wl.make_problem(n_queries=2, pool_cells=4096, n_selected=700, chunk_cells=128,
                        mask_fraction=0.1, seed=7800)
    dp = qsa.DeviceProblem(p, algo=algo_code(algo))
    dp.run()
    torch.cuda.synchronize()
    m, l, o = qsa.partials_of(dp)
    qd = oracle.widen_queries(p.q, p.q_dtype)
    H = p.q_per_kv
    for r in range(p.n_queries * H):
        t, j = divmod(r, H)
        om, ol, oo = oracle.row_partials(qd[0, t, j], p.k_pool[0, 0], p.v_pool[0, 0],
                                         p.k_scale[0, 0], p.v_scale[0, 0], p.page_table[0],
                                         p.sel, p.chunk_cells, p.softmax_scale)
        for c in range(len(om)):
            if ol[c] == 0:
                assert l[0, 0, c, r] == 0 and m[0, 0, c, r] == -np.inf
                continue
            assert abs(m[0, 0, c, r] - om[c]) <= 2e-3, (r, c)
            # the normalised chunk output and the denominator relative to the max
            assert abs(l[0, 0, c, r] / ol[c] - 1) <= 1e-2, (r, c)
            assert_parity(o[0, 0, c, r] / l[0, 0, c, r], oo[c] / ol[c], f"chunk {c} row {r}")


@pytest.mark.parametrize("algo", ALGOS)
def test_step_and_batch_agree_bitwise(algo):
    p = wl.qsa_decode(3)
    _, a = run(p, algo, batch=False)
    _, b = run(p, algo, batch=True)
    assert a.tobytes() == b.tobytes()


@pytest.mark.parametrize("algo", ALGOS)
def test_page_table_relabelling_bit_identical(algo):
    """Permuting the pool rows and rewriting the page table consistently gives
    the same bits: the kernels see the same values in the same order."""
    p = wl.make_problem(n_queries=4, pool_cells=4096, n_selected=1000, chunk_cells=128,
                        mask_fraction=0.05, seed=7900)
    _, a = run(p, algo)
    rng = np.random.Generator(np.random.PCG64(7901))
    perm = rng.permutation(p.pool_cells)
    inv = np.argsort(perm)
    p.k_pool[0, 0] = p.k_pool[0, 0][inv]
    p.v_pool[0, 0] = p.v_pool[0, 0][inv]
    p.k_scale[0, 0] = p.k_scale[0, 0][inv]
    p.v_scale[0, 0] = p.v_scale[0, 0][inv]
    pt = p.page_table[0]
    p.page_table[0] = np.where(pt >= 0, perm[np.maximum(pt, 0)], -1)
    _, b = run(p, algo)
    assert a.tobytes() == b.tobytes()


@pytest.mark.parametrize("algo", ALGOS)
def test_single_cell_gather_is_exact(algo):
    """Each sequence selects one cell whose V row encodes its slot; with a
    power-of-two V scale the output must equal scale x code exactly."""
    n_seq, pool = 64, 512
    p = wl.make_problem(n_seq=n_seq, n_kv_heads=2, n_queries=2, pool_cells=pool,
                        n_selected=1, chunk_cells=64, seed=8000)
    d = np.arange(256)
    for s in range(pool):
        p.v_pool[:, :, s, :] = ((s * 7 + d * 13) % 255 - 127).astype(np.int8)
    p.v_scale[:] = 2.0 ** -6
    _, out = run(p, algo)
    for b in range(n_seq):
        slot = p.page_table[b, p.sel[b]]
        expect = (((slot * 7 + d * 13) % 255) - 127) * 2.0 ** -6
        for t in range(2):
            for h in range(24):
                assert np.array_equal(out[b, t, h], expect.astype(np.float32)), (b, t, h)


# ------------------------------------------------- prompt-shaped path (rows on M)

@pytest.mark.parametrize("algo", ["auto", "tcgen05"])
@pytest.mark.parametrize("q_dtype", ["bf16", "f32"])
def test_prompt_path_masked_ragged(algo, q_dtype):
    """Many query rows per KV head (the rows-on-M tensor-core path) with
    page -1 masking, a chunk that is not a multiple of 128 cells, a row count
    that is not a multiple of 128, and both query types."""
    p = wl.make_problem(n_queries=13, q_per_kv=12, pool_cells=3000, n_selected=2500,
                        chunk_cells=1000, q_dtype=q_dtype, mask_fraction=0.2, seed=8100)
    check_full(p, algo, f"prompt masked {q_dtype}")


@pytest.mark.parametrize("algo", ["auto", "tcgen05"])
def test_prompt_path_ragged_batch(algo):
    lens = [0, 700, 129, 1500]
    p = wl.make_problem(n_seq=4, n_kv_heads=2, n_queries=7, q_per_kv=12, pool_cells=2048,
                        n_selected=lens, chunk_cells=512, q_dtype="bf16", seed=8200)
    dp, out = run(p, algo, max_selected=1600)
    assert_parity(out, oracle.decode_attn(p), "prompt ragged batch")
    assert np.array_equal(out[0], np.zeros_like(out[0]))


@pytest.mark.parametrize("algo", ["auto"])
def test_prompt_path_partials_bit_identical(algo):
    import sparse_selection_int8_gb300 as qsa
    p = wl.prompt_shaped(n_queries=64, pool_cells=2048, chunk_cells=1024)
    dp = qsa.DeviceProblem(p, algo=algo_code(algo))
    dp.run()
    torch.cuda.synchronize()
    m0, l0, o0 = qsa.partials_of(dp)
    for _ in range(3):
        dp.workspace.fill_(0xFF)
        dp.run()
        torch.cuda.synchronize()
        m, l, o = qsa.partials_of(dp)
        assert m.tobytes() == m0.tobytes() and l.tobytes() == l0.tobytes() and o.tobytes() == o0.tobytes()


def test_prompt_path_growing_scores():
    """K scales that grow along the list make each row's running max climb by
    tens of log2 units across the tiles, which forces the rescaling of O in
    tensor memory (the reference moves when the max grows by more than 2^8).
    bf16 queries meet bf16 K codes exactly, so only fp32 accumulation and the
    f16 P and V_hat roundings differ from the oracle."""
    p = wl.make_problem(n_queries=16, q_per_kv=12, pool_cells=4096, n_selected=4096,
                        chunk_cells=4096, q_dtype="bf16", selection="full", seed=8300)
    ks = np.linspace(0.005, 0.1, p.pool_cells, dtype=np.float32)
    p.k_scale[0, 0] = ks[p.page_table[0].argsort()]  # cell at list position i gets ks[i]
    check_full(p, "auto", "prompt growing scores")


@pytest.mark.parametrize("cells", [256, 512, 1536])
def test_prompt_path_multi_tile_repeatable(cells):
    """Chunks of two or more 128-cell tiles on the rows-on-M path: every row
    against the oracle, and the output bit-identical over repeated calls (the
    last tiles' P.V must be complete before the partials are read)."""
    import sparse_selection_int8_gb300 as qsa
    p = wl.prompt_shaped(n_queries=11, pool_cells=cells, chunk_cells=cells)
    ref = oracle.decode_attn(p)
    first = None
    for _ in range(5):
        dp = qsa.DeviceProblem(p, algo=algo_code("tcgen05"))
        dp.out.fill_(float("nan"))
        dp.run()
        torch.cuda.synchronize()
        out = dp.out.cpu().numpy()
        assert_parity(out, ref, f"prompt {cells} cells")
        if first is None:
            first = out
        assert out.tobytes() == first.tobytes()


@pytest.mark.parametrize("batch", [False, True])
def test_back_to_back_calls_share_one_workspace(batch):
    """Calls on one stream with no synchronisation between them, alternating
    between two problems of one shape and all using the same workspace: a
    call's kernels start while the previous call's merge is still reading the
    partials this call overwrites, so every output is checked against the
    oracle (and against a lone call of the same problem, bitwise)."""
    import sparse_selection_int8_gb300 as qsa
    if batch:
        probs = [wl.make_problem(n_seq=4, n_kv_heads=2, n_queries=2, pool_cells=4096,
                                 n_selected=[700, 1500, 129, 2051], chunk_cells=128,
                                 seed=9100 + k) for k in range(2)]
    else:
        probs = [wl.qsa_decode(1, seed_offset=k) for k in range(2)]
    dps = [qsa.DeviceProblem(p) for p in probs]
    refs = [oracle.decode_attn(p) for p in probs]
    alone = []
    for dp in dps:
        dp.run(batch=batch)
        torch.cuda.synchronize()
        alone.append(dp.out.cpu().numpy())
    ws, ws_bytes = dps[0].workspace, dps[0].ws_bytes
    # outputs made ready first: nothing but the library's own kernels runs
    # between the calls
    outs = [torch.full_like(dps[i % 2].out, float("nan")) for i in range(8)]
    torch.cuda.synchronize()
    for i, out in enumerate(outs):
        dp = dps[i % 2]
        if batch:
            qsa.qsa_decode_attn_batch(dp.shape, dp.n_seq, dp.q, dp.k_pool, dp.v_pool, dp.k_scale,
                                      dp.v_scale, dp.page_table, dp.sel, dp.sel_offsets,
                                      dp.max_selected, out, ws, ws_bytes, dp.status, None)
        else:
            qsa.qsa_decode_attn_step(dp.shape, dp.q, dp.k_pool, dp.v_pool, dp.k_scale, dp.v_scale,
                                     dp.page_table, dp.sel, int(dp.p.sel.shape[0]), out, ws,
                                     ws_bytes, dp.status, None)
    torch.cuda.synchronize()
    for i, out in enumerate(outs):
        got = out.cpu().numpy()
        assert_parity(got, refs[i % 2], f"back-to-back call {i}")
        assert got.tobytes() == alone[i % 2].tobytes()
    assert all(int(dp.status.item()) == 0 for dp in dps)
