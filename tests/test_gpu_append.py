"""GPU parity of qsa_kv_append (the INT8 K/V append) against its oracle.

Codes and scales are integer/bit results of fp32 arithmetic that both sides
do in the same precision (correctly rounded divisions, round half to even),
so every byte of the pools and every scale must match the oracle exactly,
and slots the call must not touch must keep their contents.
"""
import numpy as np
import pytest

import qsa_workloads as wl
from oracle import kv_append as ka

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_selection_int8_gb300 import build
    build.build()


def gpu_append(a):
    import sparse_selection_int8_gb300 as qsa
    d = qsa.DeviceAppend(a)
    d.run()
    torch.cuda.synchronize()
    return (d.k_pool.cpu().numpy(), d.v_pool.cpu().numpy(), d.k_scale.cpu().numpy(),
            d.v_scale.cpu().numpy(), int(d.status.item()))


def oracle_append(a):
    kp, vp, ks, vs = a.k_pool.copy(), a.v_pool.copy(), a.k_scale.copy(), a.v_scale.copy()
    st = ka.kv_append(a, kp, vp, ks, vs)
    return kp, vp, ks, vs, st


def assert_same(a, what):
    got = gpu_append(a)
    ref = oracle_append(a)
    for name, g, r in zip(("k_pool", "v_pool", "k_scale", "v_scale"), got[:4], ref[:4]):
        if g.dtype == np.float32:
            g, r = g.view(np.uint32), r.view(np.uint32)
        bad = np.argwhere(g != r)
        assert bad.size == 0, f"{what}: {name} differs at {bad[:5].tolist()} ({bad.shape[0]} places)"
    assert got[4] == ref[4], f"{what}: status {got[4]:#x} vs oracle {ref[4]:#x}"
    return got


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_step_append(dtype):
    a = wl.make_append(n_seq=16, n_kv_heads=2, n_new=4, pool_cells=32768, dtype=dtype,
                       seed=wl.SEED_BASE + 16)
    assert_same(a, f"decode-step append {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n_seq,G,n_new", [(1, 1, 1), (3, 2, 37), (5, 3, 200), (2, 1, 1000)])
def test_append_shapes(dtype, n_seq, G, n_new):
    a = wl.make_append(n_seq=n_seq, n_kv_heads=G, n_new=n_new, pool_cells=2048,
                       page_table_len=3000, mask_fraction=0.1, dtype=dtype,
                       seed=6100 + 100 * n_seq + 10 * G + n_new)
    assert_same(a, f"append B={n_seq} G={G} n_new={n_new} {dtype}")


@pytest.mark.parametrize("P", [2, 16])
def test_paged_append(P):
    a = wl.make_append(n_seq=3, n_kv_heads=2, n_new=300, pool_cells=4096, mask_fraction=0.2,
                       page_cells=P, seed=6700 + P)
    a.positions[1, 7] = a.page_table_len * P          # past the last position
    bad = np.flatnonzero(a.page_table[2] >= 0)[0]
    a.page_table[2, bad] = 4096 // P                   # past the last pool page
    a.positions[2, 3] = bad * P + P - 1
    assert_same(a, f"paged append P={P}")


def test_prompt_sized_append():
    """A whole 32,768-cell pool of two KV heads written in one call (more
    warps than the grid, so the grid-stride loop runs several rounds)."""
    assert_same(wl.prompt_append(), "prompt-sized append")


def test_hand_worked_rows():
    """The golden rows (tiled to 256 elements: same maximum, tiled codes),
    plus rows of zeros, through the device kernel."""
    from test_append_oracle import golden_rows
    rows = golden_rows()
    a = wl.make_append(n_seq=1, n_kv_heads=1, n_new=len(rows), pool_cells=64, seed=6200)
    a.k_new[0, :, 0] = np.stack([np.tile(x, 16) for x, _, _ in rows])
    a.v_new[0, :, 0] = -a.k_new[0, :, 0]
    kp, vp, ks, vs, st = assert_same(a, "hand-worked rows")
    for i, (_, codes, scale) in enumerate(rows):
        slot = a.page_table[0, a.positions[0, i]]
        assert ks[0, 0, slot] == scale and np.array_equal(kp[0, 0, slot], np.tile(codes, 16))
        assert np.array_equal(vp[0, 0, slot], -np.tile(codes, 16).astype(np.int16))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_near_ties(dtype):
    """Elements at and one ulp either side of (k + 1/2) * scale, where the
    code depends on the last bit of the quotient x / scale: the device's
    division must round exactly as the oracle's fp32 division does."""
    from qsa_workloads import bf16_bits_from_f32, f32_from_bf16_bits
    rng = np.random.default_rng(6600 if dtype == "f32" else 6601)
    a = wl.make_append(n_seq=2, n_kv_heads=2, n_new=500, pool_cells=1024, dtype=dtype, seed=6602)
    rows = np.empty((2, 500, 2, 256), np.float32)
    for idx in np.ndindex(2, 500, 2):
        amax = np.float32(np.exp(rng.uniform(np.log(1e-3), np.log(1e3))))
        if dtype == "bf16":
            amax = f32_from_bf16_bits(bf16_bits_from_f32(np.array([amax])))[0]
        s = np.float32(amax / np.float32(127))
        k = rng.integers(0, 126, 256).astype(np.float32)
        x = ((k + np.float32(0.5)) * s).astype(np.float32)
        step = rng.integers(-1, 2, 256)
        x = np.where(step > 0, np.nextafter(x, np.float32(np.inf)),
                     np.where(step < 0, np.nextafter(x, np.float32(-np.inf)), x)).astype(np.float32)
        x *= np.where(rng.integers(0, 2, 256) > 0, np.float32(1), np.float32(-1))
        x[rng.integers(0, 256)] = amax
        rows[idx] = x
    if dtype == "bf16":
        a.k_new = bf16_bits_from_f32(rows)
        a.v_new = bf16_bits_from_f32(-rows)
    else:
        a.k_new, a.v_new = rows, -rows
    assert_same(a, f"near ties {dtype}")


def test_bad_entries_are_skipped_and_reported():
    a = wl.make_append(n_seq=2, n_kv_heads=2, n_new=8, pool_cells=256, seed=6300)
    a.positions[0, 1] = -3                    # outside the page table
    a.positions[1, 2] = a.page_table_len      # outside the page table
    a.page_table[0, a.positions[0, 3]] = -1   # not resident
    a.page_table[1, a.positions[1, 5]] = 256  # outside the pool
    kp, vp, ks, vs, st = assert_same(a, "bad entries")
    assert st == (ka.STATUS_BAD_POSITION | ka.STATUS_NOT_RESIDENT | ka.STATUS_BAD_SLOT)


def test_graph_replay_and_repeat():
    """Captured in a CUDA graph and replayed: the same pools as one eager call."""
    import sparse_selection_int8_gb300 as qsa
    a = wl.make_append(n_seq=4, n_kv_heads=2, n_new=16, pool_cells=1024, seed=6400)
    ref = oracle_append(a)
    d = qsa.DeviceAppend(a)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d.run(stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        d.run(stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(d.k_pool.cpu().numpy(), ref[0])
    assert np.array_equal(d.v_scale.cpu().numpy().view(np.uint32), ref[3].view(np.uint32))


def test_append_then_attend():
    """Cells appended by the kernel and then selected by the attention call
    give the oracle's attention over the oracle's appended pools."""
    import oracle
    import sparse_selection_int8_gb300 as qsa
    from parity import assert_parity
    oracle.build()
    p = wl.make_problem(n_kv_heads=2, n_queries=2, pool_cells=4096, n_selected=600,
                        chunk_cells=128, seed=6500)
    a = wl.make_append(n_seq=1, n_kv_heads=2, n_new=64, pool_cells=4096, seed=6501)
    a.page_table = p.page_table.copy()
    a.k_pool, a.v_pool, a.k_scale, a.v_scale = p.k_pool, p.v_pool, p.k_scale, p.v_scale
    rng = np.random.default_rng(6502)
    a.positions[0] = rng.choice(p.sel, size=64, replace=False)  # half of them selected
    # rows of the size the pools hold (scales near 0.005-0.02, |v_hat| <= ~2.5),
    # the regime the attention tolerance is stated for
    a.k_new = (rng.standard_normal(a.k_new.shape) * 0.5).astype(np.float32)
    a.v_new = (rng.standard_normal(a.v_new.shape) * 0.5).astype(np.float32)
    kp, vp, ks, vs, _ = oracle_append(a)
    d = qsa.DeviceAppend(a)
    dp = qsa.DeviceProblem(p)
    d.k_pool, d.v_pool, d.k_scale, d.v_scale = dp.k_pool, dp.v_pool, dp.k_scale, dp.v_scale
    d.run()
    dp.run()
    torch.cuda.synchronize()
    p.k_pool, p.v_pool, p.k_scale, p.v_scale = kp, vp, ks, vs
    assert_parity(dp.out.cpu().numpy(), oracle.decode_attn(p), "append then attend")
