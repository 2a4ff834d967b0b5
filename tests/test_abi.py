"""Host-side checks of the C ABI: the library builds, loads, exports every
function ``include/qsa.h`` declares, sizes its workspace as documented and
rejects bad arguments before any CUDA call.  No kernel runs here."""
import ctypes
import os
import re

import pytest

import sparse_selection_int8_gb300 as qsa
from sparse_selection_int8_gb300 import build as qsa_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "qsa.h")


@pytest.fixture(scope="module")
def lib():
    qsa_build.build()
    return qsa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(qsa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("qsa_decode_attn_step", "qsa_decode_attn_batch", "qsa_workspace_bytes",
                     "qsa_partials_view", "qsa_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(qsa.library_path())
    for name in declared_functions():
        assert hasattr(raw, name), name


def shape(**kw):
    base = dict(n_kv_heads=1, q_per_kv=12, n_queries=1, pool_cells=4096, page_table_len=4096,
                chunk_cells=64, softmax_scale=1 / 16)
    base.update(kw)
    return qsa.make_shape(**base)


def test_workspace_bytes_layout(lib):
    s = shape(n_queries=4, chunk_cells=128)
    n_chunks = (2051 + 127) // 128
    rows = n_chunks * 48
    got = qsa.qsa_workspace_bytes(s, 1, 2051)
    assert got >= rows * 4 * 2 + rows * 256 * 4
    assert got % 256 == 0
    assert qsa.qsa_workspace_bytes(s, 1, 0) == 0
    # grows linearly with sequences
    assert qsa.qsa_workspace_bytes(s, 8, 2051) >= 8 * rows * 258 * 4


@pytest.mark.parametrize("n_seq,G,T", [(1, 1, 4), (8, 2, 2), (16, 2, 4), (3, 3, 1)])
def test_decode_workspace_holds_query_images_and_run_counts(lib, n_seq, G, T):
    """The tensor-core decode path's workspace is the partials (as the
    CUDA-core path's) plus the staged query images, (N + 48) rows of 1 KB per
    (sequence, KV head) with N the rows rounded up to 16 (1,024-byte aligned),
    plus one int32 run count per (sequence, KV head) (256-byte aligned)."""
    def align(v, a):
        return -(-v // a) * a
    tc = qsa.qsa_workspace_bytes(shape(n_queries=T, n_kv_heads=G, algo=qsa.QSA_ALGO_TCGEN05), n_seq, 2051)
    simt = qsa.qsa_workspace_bytes(shape(n_queries=T, n_kv_heads=G, algo=qsa.QSA_ALGO_SIMT), n_seq, 2051)
    N = -(-(12 * T) // 16) * 16
    assert tc - simt == align(n_seq * G * (N + 48) * 512 * 2, 1024) + align(n_seq * G * 4, 256)


def test_partials_view_offsets(lib):
    s = shape(n_queries=2, chunk_cells=256, n_kv_heads=2)
    base = 1 << 20
    m, l, o, n = qsa.qsa_partials_view(s, 8, 16384, base)
    assert n == 64
    rows = 8 * 2 * 64 * 24
    assert m == base and l >= m + rows * 4 and o >= l + rows * 4
    assert (l - base) % 256 == 0 and (o - base) % 256 == 0


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 128, qsa.QSA_ERR_UNSUPPORTED),
    ("q_per_kv", 0, qsa.QSA_ERR_INVALID_ARG),
    ("q_per_kv", 65, qsa.QSA_ERR_UNSUPPORTED),
    ("n_queries", 0, qsa.QSA_ERR_INVALID_ARG),
    ("chunk_cells", 0, qsa.QSA_ERR_INVALID_ARG),
    ("pool_cells", -1, qsa.QSA_ERR_INVALID_ARG),
    ("q_dtype", 7, qsa.QSA_ERR_INVALID_ARG),
    ("algo", 9, qsa.QSA_ERR_INVALID_ARG),
    ("softmax_scale", float("nan"), qsa.QSA_ERR_INVALID_ARG),
])
def test_bad_shape_rejected(lib, field, value, code):
    s = shape()
    setattr(s, field, value)
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_workspace_bytes(s, 1, 100)
    assert e.value.code == code


FAKE = 1 << 32  # an aligned, never-dereferenced address: every call below fails its checks


def step_args(**over):
    a = dict(q=FAKE, k_pool=FAKE, v_pool=FAKE, k_scale=FAKE, v_scale=FAKE, page_table=FAKE,
             sel=FAKE, n_sel=100, out=FAKE + 4096, workspace=FAKE, workspace_bytes=1 << 30)
    a.update(over)
    return a


def call_step(lib, s, a):
    return lib.qsa_decode_attn_step(ctypes.byref(s), a["q"], a["k_pool"], a["v_pool"],
                                    a["k_scale"], a["v_scale"], a["page_table"], a["sel"],
                                    a["n_sel"], a["out"], a["workspace"], a["workspace_bytes"],
                                    None, None)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), qsa.QSA_ERR_INVALID_ARG),
    (dict(k_pool=None), qsa.QSA_ERR_INVALID_ARG),
    (dict(out=None), qsa.QSA_ERR_INVALID_ARG),
    (dict(sel=None), qsa.QSA_ERR_INVALID_ARG),
    (dict(n_sel=-1), qsa.QSA_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), qsa.QSA_ERR_INVALID_ARG),          # misaligned queries
    (dict(k_pool=FAKE + 4), qsa.QSA_ERR_INVALID_ARG),     # misaligned pool
    (dict(workspace=FAKE + 16), qsa.QSA_ERR_INVALID_ARG), # workspace not 256-aligned
    (dict(workspace=None), qsa.QSA_ERR_INVALID_ARG),
    (dict(workspace_bytes=64), qsa.QSA_ERR_WORKSPACE),
    (dict(out=FAKE), qsa.QSA_ERR_INVALID_ARG),            # out aliases q
])
def test_step_rejects_before_launch(lib, over, code):
    assert call_step(lib, shape(), step_args(**over)) == code


def test_batch_rejects_before_launch(lib):
    s = shape()
    args = [ctypes.byref(s), 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE]
    # null offsets
    assert lib.qsa_decode_attn_batch(*args, None, 100, FAKE + 4096, FAKE, 1 << 30, None,
                                     None) == qsa.QSA_ERR_INVALID_ARG
    # zero sequences
    args0 = [ctypes.byref(s), 0] + args[2:]
    assert lib.qsa_decode_attn_batch(*args0, FAKE, 100, FAKE + 4096, FAKE, 1 << 30, None,
                                     None) == qsa.QSA_ERR_INVALID_ARG
    # negative bound
    assert lib.qsa_decode_attn_batch(*args, FAKE, -5, FAKE + 4096, FAKE, 1 << 30, None,
                                     None) == qsa.QSA_ERR_INVALID_ARG


def append_args(**over):
    mb = 1 << 20
    a = dict(n_seq=2, n_new=4, kv_dtype=qsa.QSA_F32, k_new=FAKE, v_new=FAKE + mb, positions=FAKE + 2 * mb,
             page_table=FAKE + 3 * mb, k_pool=FAKE + 4 * mb, v_pool=FAKE + 5 * mb,
             k_scale=FAKE + 6 * mb, v_scale=FAKE + 7 * mb)
    a.update(over)
    return a


def call_append(lib, s, a):
    return lib.qsa_kv_append(ctypes.byref(s), a["n_seq"], a["n_new"], a["kv_dtype"], a["k_new"],
                             a["v_new"], a["positions"], a["page_table"], a["k_pool"], a["v_pool"],
                             a["k_scale"], a["v_scale"], None, None)


@pytest.mark.parametrize("over,code", [
    (dict(k_new=None), qsa.QSA_ERR_INVALID_ARG),
    (dict(positions=None), qsa.QSA_ERR_INVALID_ARG),
    (dict(v_scale=None), qsa.QSA_ERR_INVALID_ARG),
    (dict(n_new=-1), qsa.QSA_ERR_INVALID_ARG),
    (dict(n_seq=-1), qsa.QSA_ERR_INVALID_ARG),
    (dict(kv_dtype=7), qsa.QSA_ERR_INVALID_ARG),
    (dict(k_new=FAKE + 8), qsa.QSA_ERR_INVALID_ARG),      # misaligned rows
    (dict(v_pool=FAKE + (5 << 20) + 4), qsa.QSA_ERR_INVALID_ARG),
    (dict(k_pool=FAKE), qsa.QSA_ERR_INVALID_ARG),         # pool aliases the new K rows
    (dict(v_scale=FAKE + (6 << 20)), qsa.QSA_ERR_INVALID_ARG),  # one scale array for K and V
])
def test_append_rejects_before_launch(lib, over, code):
    assert call_append(lib, shape(), append_args(**over)) == code


@pytest.mark.parametrize("page_cells,pool_cells,code", [
    (-1, 4096, qsa.QSA_ERR_INVALID_ARG),
    (3, 4096, qsa.QSA_ERR_INVALID_ARG),   # the pool is not a whole number of pages
    (16, 4096, qsa.QSA_OK),
    (0, 4096, qsa.QSA_OK),                # 0 means one cell per page
])
def test_page_size_checked(lib, page_cells, pool_cells, code):
    s = shape(pool_cells=pool_cells, page_table_len=256)
    s.page_cells = page_cells
    out = ctypes.c_size_t(0)
    assert lib.qsa_workspace_bytes(ctypes.byref(s), 1, 100, ctypes.byref(out)) == code
    if code != qsa.QSA_OK:
        assert call_append(lib, s, append_args()) == code


def test_append_checks_shape_and_skips_empty_calls(lib):
    s = shape()
    s.head_dim = 128
    assert call_append(lib, s, append_args()) == qsa.QSA_ERR_UNSUPPORTED
    s = shape()
    s.pool_cells = 0
    assert call_append(lib, s, append_args()) == qsa.QSA_ERR_INVALID_ARG
    # nothing to append: success without touching the device (none here)
    assert call_append(lib, shape(), append_args(n_new=0)) == qsa.QSA_OK
    assert call_append(lib, shape(), append_args(n_seq=0)) == qsa.QSA_OK


def test_limited_batch_rejects_before_launch(lib):
    s = shape()
    base = [ctypes.byref(s), 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 100]
    tail = [FAKE + 4096, FAKE, 1 << 30, None, None]
    assert lib.qsa_decode_attn_batch_limited(*base, None, *tail) == qsa.QSA_ERR_INVALID_ARG
    assert lib.qsa_decode_attn_batch_limited(*base, FAKE + 2, *tail) == qsa.QSA_ERR_INVALID_ARG
    base_no_offsets = base[:9] + [None, 100]
    assert lib.qsa_decode_attn_batch_limited(*base_no_offsets, FAKE, *tail) == qsa.QSA_ERR_INVALID_ARG


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4):
        assert qsa.qsa_status_string(code)
    assert qsa.qsa_status_string(12345) == "unknown status"


def test_binding_has_no_cpu_path():
    """The product package never imports the oracle."""
    pkg = os.path.dirname(qsa.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "qsa_oracle" not in text, f


def test_select_rejects_before_launch(lib):
    """qsa_select_blocks checks its shape and pointers before any launch."""
    s = qsa.qsa_select_shape(2, 4, 64, 64, 2048, 128)
    size = ctypes.c_size_t(0)
    assert lib.qsa_select_workspace_bytes(ctypes.byref(s), 8, ctypes.byref(size)) == qsa.QSA_OK
    assert size.value > 0
    args = lambda sh, n=8: [ctypes.byref(sh), n, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                            size.value, None, None]
    for field, value, code in (("n_queries", 9, qsa.QSA_ERR_UNSUPPORTED), ("n_queries", 0, qsa.QSA_ERR_INVALID_ARG),
                               ("idx_dim", 63, qsa.QSA_ERR_UNSUPPORTED), ("idx_dim", 512, qsa.QSA_ERR_UNSUPPORTED),
                               ("max_blocks", 16385, qsa.QSA_ERR_UNSUPPORTED),
                               ("top_k", 2049, qsa.QSA_ERR_UNSUPPORTED), ("block_cells", 0, qsa.QSA_ERR_INVALID_ARG)):
        bad = qsa.qsa_select_shape(2, 4, 64, 64, 2048, 128)
        setattr(bad, field, value)
        assert lib.qsa_select_blocks(*args(bad)) == code, field
    assert lib.qsa_select_blocks(*args(s, 0)) == qsa.QSA_ERR_INVALID_ARG
    small = args(s)
    small[11] = size.value - 1
    assert lib.qsa_select_blocks(*small) == qsa.QSA_ERR_WORKSPACE
    misaligned = args(s)
    misaligned[3] = FAKE + 8  # pooled keys must be 16-byte aligned
    assert lib.qsa_select_blocks(*misaligned) == qsa.QSA_ERR_INVALID_ARG
