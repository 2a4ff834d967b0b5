"""The device-side time-out path of the tensor-core kernels.

Every mbarrier wait of the decode and prompt-shaped kernels is bounded.  A
wait that runs out sets QSA_STATUS_TIMEOUT; the kernel then stops waiting,
lets each issuing thread drain its own tensor-core operations and copies,
frees its tensor memory and returns.  These tests make a correct call's waits
run out by setting the bound to a few SM clock cycles through the test-only
``qsa_set_wait_limit``; nothing is broken on purpose.  Each checks that the
call returns and its stream completes, that the bit is set, and that a normal
call on the same stream afterwards matches the oracle (the context and the
library are still usable).
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


def _timed_out_then_correct(p, algo, batch):
    import sparse_selection_int8_gb300 as qsa
    dp = qsa.DeviceProblem(p, algo=algo)
    qsa.qsa_set_wait_limit(16)
    try:
        dp.run(batch=batch)          # every kernel of this call sees 16-cycle waits
    finally:
        qsa.qsa_set_wait_limit(0)
    torch.cuda.synchronize()         # the call's kernels have ended
    assert int(dp.status.item()) & qsa.QSA_STATUS_TIMEOUT
    assert not int(dp.status.item()) & qsa.QSA_STATUS_LAUNCH
    # the same problem again on the same stream, default bound
    dp.status.zero_()
    dp.out.fill_(float("nan"))
    dp.run(batch=batch)
    torch.cuda.synchronize()
    assert int(dp.status.item()) == 0
    return dp.out.cpu().numpy()


@pytest.mark.parametrize("case", ["qsa_decode_T4", "batched_small", "long_small"])
def test_decode_kernel_times_out_and_recovers(case):
    import sparse_selection_int8_gb300 as qsa
    if case == "qsa_decode_T4":
        p, batch = wl.qsa_decode(4), False
    elif case == "batched_small":
        p = wl.make_problem(n_seq=5, n_kv_heads=2, n_queries=2, pool_cells=4096,
                            n_selected=[300, 900, 0, 1500, 129], chunk_cells=128, seed=9100)
        batch = True
    else:
        p = wl.make_problem(n_seq=2, n_kv_heads=2, n_queries=2, pool_cells=16384,
                            n_selected=4096, chunk_cells=256, seed=9101)
        batch = True
    out = _timed_out_then_correct(p, qsa.QSA_ALGO_TCGEN05, batch)
    assert_parity(out, oracle.decode_attn(p), f"after a time-out ({case})")


def test_prompt_kernel_times_out_and_recovers():
    import sparse_selection_int8_gb300 as qsa
    p = wl.make_problem(n_queries=32, pool_cells=2048, n_selected=2048, chunk_cells=512,
                        q_dtype="bf16", seed=9102)
    out = _timed_out_then_correct(p, qsa.QSA_ALGO_TCGEN05, False)
    assert_parity(out, oracle.decode_attn(p), "prompt kernel after a time-out")


def test_default_bound_restored_between_calls():
    """Calls after the bound is reset see no time-out, back to back."""
    import sparse_selection_int8_gb300 as qsa
    p = wl.qsa_decode(2)
    dp = qsa.DeviceProblem(p)
    for _ in range(3):
        dp.run()
    torch.cuda.synchronize()
    assert int(dp.status.item()) == 0
    assert_parity(dp.out.cpu().numpy(), oracle.decode_attn(p), "default bound")
