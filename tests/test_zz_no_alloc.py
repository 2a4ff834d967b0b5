"""The workspace-free entry point, qsa_decode_attn_step_noalloc.

It serves callers that cannot allocate device memory where they run decode
attention; its chunk partials live in the library's own fixed device array.
The GPU test calls it through the C ABI twice in a row (two different
problems, so the second call runs over the first call's leftovers) and
checks each output bit for bit against qsa_decode_attn_step's on the same
inputs (the same kernels run in the same order, so a leftover of the
previous call or a wrong offset inside the fixed array would show), and
against the fp64 oracle within the parity tolerance of the other tests.
This file is collected last.
"""
import ctypes

import numpy as np
import pytest

import qsa_workloads as wl
import sparse_selection_int8_gb300 as qsa
from sparse_selection_int8_gb300 import build as qsa_build
import oracle
from parity import assert_parity

FAKE = 1 << 32  # aligned, never dereferenced: the size check rejects first


def test_oversize_request_rejected_without_launch():
    qsa_build.build()
    lib = qsa.load_library()
    s = qsa.make_shape(n_kv_heads=1, q_per_kv=12, n_queries=4, pool_cells=1 << 20,
                       page_table_len=1 << 20, chunk_cells=1, softmax_scale=1 / 16)
    # 48 rows x 258 floats per chunk of one cell: 10,000 cells need ~49 MiB
    code = lib.qsa_decode_attn_step_noalloc(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE,
                                            FAKE, FAKE, 10000, FAKE + 4096, None, None)
    assert code == qsa.QSA_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_matches_step_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qsa_build.build()
    lib = qsa.load_library()
    for p in (wl.qsa_decode(4), wl.tiny_decode()):
        dp = qsa.DeviceProblem(p)
        dp.run()  # the existing entry point, with a workspace
        torch.cuda.synchronize()
        ref = dp.out.cpu().numpy()
        out = torch.full_like(dp.out, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        code = lib.qsa_decode_attn_step_noalloc(
            ctypes.byref(dp.shape), dp.q.data_ptr(), dp.k_pool.data_ptr(), dp.v_pool.data_ptr(),
            dp.k_scale.data_ptr(), dp.v_scale.data_ptr(), dp.page_table.data_ptr(),
            dp.sel.data_ptr(), int(p.sel.shape[0]), out.data_ptr(), status.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
        assert code == qsa.QSA_OK, qsa.qsa_status_string(code)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert int(status.item()) == 0
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"noalloc vs step ({p.name})"
        assert_parity(got, oracle.decode_attn(p), f"noalloc vs oracle ({p.name})")
