"""The seeded input generator's recipes (CPU): the structures the parity
tests and the bench rely on — page tables of pages, resident and distinct
append positions, causal windows — hold for the inputs it draws."""
import numpy as np
import pytest

import qsa_workloads as wl


@pytest.mark.parametrize("P", [1, 16, 64])
def test_paged_problem_structure(P):
    p = wl.make_problem(n_seq=3, n_kv_heads=2, pool_cells=4096, n_selected=[700, 1500, 0],
                        chunk_cells=128, mask_fraction=0.1, page_cells=P, seed=11 + P)
    pages = 4096 // P
    assert p.page_table.shape == (3, pages) and p.page_table_len == pages
    for b in range(3):
        pt = p.page_table[b]
        live = pt[pt >= 0]
        assert np.array_equal(np.sort(live), np.unique(live)) and live.max(initial=0) < pages
        assert abs((pt < 0).sum() - round(0.1 * pages)) <= 1
        s = p.sel_of(b)
        assert np.all(np.diff(s) > 0) and (s.size == 0 or (s[0] >= 0 and s[-1] < pages * P))
    # P = 1 draws what the configurations always drew (same seed, same arrays)
    if P == 1:
        q = wl.make_problem(n_seq=3, n_kv_heads=2, pool_cells=4096, n_selected=[700, 1500, 0],
                            chunk_cells=128, mask_fraction=0.1, seed=12)
        assert np.array_equal(q.page_table, p.page_table) and np.array_equal(q.sel, p.sel)


@pytest.mark.parametrize("P", [1, 4])
def test_append_positions_are_resident_and_distinct(P):
    a = wl.make_append(n_seq=4, n_kv_heads=2, n_new=50, pool_cells=1024, mask_fraction=0.3,
                       page_cells=P, seed=21)
    for b in range(4):
        pos = a.positions[b]
        assert np.unique(pos).size == pos.size
        assert np.all(a.page_table[b][pos // P] >= 0)
    assert a.k_new.shape == (4, 50, 2, 256) and a.k_new.dtype == np.float32


def test_prompt_causal_window():
    p = wl.prompt_causal()
    lim = p.q_limit[0]
    assert lim.shape == (2048,) and np.all(np.diff(lim) == 1)
    assert lim[-1] == p.n_positions and lim[0] == p.n_positions - 2047
