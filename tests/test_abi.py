"""The C ABI without a GPU: the library builds and loads, exports every entry
point declared in include/qsa.h, and rejects bad arguments on the host
(returning an error status and launching nothing).  No call here reaches a
CUDA launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")


@pytest.fixture(scope="module")
def L():
    import sparse_attention_indexer_index_gb300 as qsa
    qsa.build()
    return qsa.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ["qsa_compress_keys", "qsa_index_scores", "topk_select", "qsa_expand_slots",
              "qsa_indexer_select"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    assert L.qsa_status_string(0) == b"ok"
    assert L.qsa_status_string(-2) == b"unsupported size or layout"
    assert L.qsa_version() >= 100


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: the checks fail first


def test_topk_rejects_bad_k(L):
    for k in (0, -1, 2049):
        assert L.topk_select(FAKE, 100, None, 1, 100, k, None, 0, None, 0, FAKE, None, None, 0,
                             None) == -2


def test_topk_rejects_null_output_and_slots_without_table(L):
    assert L.topk_select(FAKE, 100, None, 1, 100, 8, None, 0, None, 0, None, None, None, 0, None) == -1
    assert L.topk_select(FAKE, 100, None, 1, 100, 8, None, 0, None, 64, FAKE, FAKE, None, 0, None) == -1
    # n_max beyond the leading dimension
    assert L.topk_select(FAKE, 100, None, 1, 101, 8, None, 0, None, 0, FAKE, None, None, 0, None) == -1


def test_expand_rejects_page_size_not_multiple_of_4(L):
    assert L.qsa_expand_slots(FAKE, 512, 1, FAKE, 1, FAKE, FAKE, 10, 62, None, FAKE, None) == -2
    assert L.qsa_expand_slots(FAKE, 4096, 1, FAKE, 1, FAKE, FAKE, 10, 64, None, FAKE, None) == -2


def test_scores_reject_short_page_table_and_leading_dim(L):
    # max_len 8192 needs 128 pages of 64, table has 100
    assert L.qsa_index_scores(FAKE, FAKE, 1 << 20, 1, FAKE, 1, FAKE, 8192, 1, FAKE, 100, 64, FAKE,
                              2048, 0, None) == -1
    # ld_scores below max_len/4
    assert L.qsa_index_scores(FAKE, FAKE, 1 << 20, 1, FAKE, 1, FAKE, 8192, 1, FAKE, 128, 64, FAKE,
                              2047, 0, None) == -1
    # misaligned q
    assert L.qsa_index_scores(ctypes.c_void_p(0x1002), FAKE, 1 << 20, 1, FAKE, 1, FAKE, 8192, 1, FAKE,
                              128, 64, FAKE, 2048, 0, None) == -1


def test_indexer_select_rejects_small_workspace(L):
    need = L.qsa_indexer_select_workspace_size(6, 80000, 512)
    assert need >= 6 * 20000 * 4
    assert L.qsa_indexer_select(FAKE, FAKE, 1 << 20, 1, FAKE, 6, FAKE, 80000, 6, FAKE, 1250, 64, 512,
                                None, None, FAKE, None, 0, FAKE, need - 1, None) == -3
    assert L.qsa_indexer_select(FAKE, FAKE, 1 << 20, 1, FAKE, 6, FAKE, 80000, 6, FAKE, 1250, 64, 4096,
                                None, None, FAKE, None, 0, FAKE, need, None) == -2


def test_compress_rejects_bad_arguments(L):
    assert L.qsa_compress_keys(None, FAKE, FAKE, 4, 1, FAKE, 4, 64, 10000.0, FAKE, 16, None) == -1
    assert L.qsa_compress_keys(FAKE, FAKE, FAKE, 4, 1, FAKE, 4, 6, 10000.0, FAKE, 16, None) == -2
    assert L.qsa_compress_keys(FAKE, FAKE, FAKE, 4, 1, FAKE, 4, 64, 0.0, FAKE, 16, None) == -1
    # nothing to do is fine and touches nothing
    assert L.qsa_compress_keys(None, None, None, 0, 0, None, 0, 0, 10000.0, None, 0, None) == 0


def test_zero_rows_are_a_no_op(L):
    assert L.topk_select(None, 0, None, 0, 0, 8, None, 0, None, 0, None, None, None, 0, None) == 0
    assert L.qsa_indexer_select(None, None, 0, 0, None, 0, None, 0, 0, None, 0, 64, 512, None, None,
                                None, None, 0, None, 0, None) == 0


def test_select_blocks_rejects_bad_arguments(L):
    rrs = FAKE
    # k_blk out of range
    assert L.qsa_select_blocks(FAKE, 8, 1, rrs, 1, FAKE, 32, FAKE, 1, 64, 0, None, None, FAKE, None) == -2
    # no output slots
    assert L.qsa_select_blocks(FAKE, 8, 1, rrs, 1, FAKE, 32, FAKE, 1, 64, 4, None, None, None, None) == -1
    # leading dimension shorter than max_len / 4
    assert L.qsa_select_blocks(FAKE, 4, 1, rrs, 1, FAKE, 32, FAKE, 1, 64, 4, None, None, FAKE, None) == -1
    # page size not a multiple of 4
    assert L.qsa_select_blocks(FAKE, 8, 1, rrs, 1, FAKE, 32, FAKE, 1, 6, 4, None, None, FAKE, None) == -2


def test_indexshare_rejects_bad_arguments(L):
    f = L.qsa_indexshare_slots
    # k_blk out of range; too many drafted columns
    assert f(FAKE, FAKE, 1, FAKE, 0, 3, 1, FAKE, 1, FAKE, FAKE, 4, 64, None, FAKE, None) == -2
    assert f(FAKE, FAKE, 1, FAKE, 512, (1 << 16) + 1, 1, FAKE, 1, FAKE, FAKE, 4, 64, None, FAKE, None) == -2
    # negative drafted columns; no output slots; no request -> kept-row map
    assert f(FAKE, FAKE, 1, FAKE, 512, -1, 1, FAKE, 1, FAKE, FAKE, 4, 64, None, FAKE, None) == -1
    assert f(FAKE, FAKE, 1, FAKE, 512, 3, 1, FAKE, 1, FAKE, FAKE, 4, 64, None, None, None) == -1
    assert f(FAKE, FAKE, 1, None, 512, 3, 1, FAKE, 1, FAKE, FAKE, 4, 64, None, FAKE, None) == -1
    # kept rows announced but not given
    assert f(None, FAKE, 1, FAKE, 512, 3, 1, FAKE, 1, FAKE, FAKE, 4, 64, None, FAKE, None) == -1
    # page size not a multiple of 4
    assert f(FAKE, FAKE, 1, FAKE, 512, 3, 1, FAKE, 1, FAKE, FAKE, 4, 62, None, FAKE, None) == -2
    # no rows: nothing to do
    assert f(None, None, 0, None, 512, 3, 0, None, 0, None, None, 0, 64, None, None, None) == 0


def test_sparse_attn_rejects_bad_arguments(L):
    f = L.qsa_sparse_attn
    c = ctypes.c_float(0.0625)
    # group size 3, 32 (too many heads per KV head), head_dim 64
    assert f(FAKE, FAKE, FAKE, 100, 1, 6, 2, 128, FAKE, 8, 8, c, FAKE, None, None, 0, None) == -2
    assert f(FAKE, FAKE, FAKE, 100, 1, 32, 1, 128, FAKE, 8, 8, c, FAKE, None, None, 0, None) == -2
    assert f(FAKE, FAKE, FAKE, 100, 1, 16, 1, 256, FAKE, 8, 8, c, FAKE, None, None, 0, None) == -2
    assert f(FAKE, FAKE, FAKE, 100, 1, 8, 1, 64, FAKE, 8, 8, c, FAKE, None, None, 0, None) == -2
    # entries beyond the leading dimension; misaligned q; no output
    assert f(FAKE, FAKE, FAKE, 100, 1, 8, 1, 128, FAKE, 8, 9, c, FAKE, None, None, 0, None) == -1
    assert f(ctypes.c_void_p(0x1002), FAKE, FAKE, 100, 1, 8, 1, 128, FAKE, 8, 8, c, FAKE, None, None, 0,
             None) == -1
    assert f(FAKE, FAKE, FAKE, 100, 1, 8, 1, 128, FAKE, 8, 8, c, None, None, None, 0, None) == -1
    # a long row needs the workspace
    need = L.qsa_sparse_attn_workspace_size(1, 8, 128, 2051)
    assert need > 0 and L.qsa_sparse_attn_workspace_size(1, 8, 128, 256) == 0
    assert f(FAKE, FAKE, FAKE, 100, 1, 8, 1, 128, FAKE, 2051, 2051, c, FAKE, None, None, 0, None) == -3
    # no rows: nothing to do
    assert f(None, None, None, 0, 0, 8, 1, 128, None, 0, 0, c, None, None, None, 0, None) == 0


def test_append_keys_rejects_bad_arguments(L):
    f = L.qsa_append_keys
    # page size not a multiple of 4; no ring; bad RoPE base
    assert f(FAKE, FAKE, FAKE, 2, FAKE, FAKE, 4, 6, 10000.0, FAKE, 64, None) == -2
    assert f(FAKE, FAKE, FAKE, 2, None, FAKE, 4, 64, 10000.0, FAKE, 64, None) == -1
    assert f(FAKE, FAKE, FAKE, 2, FAKE, FAKE, 4, 64, 0.0, FAKE, 64, None) == -1
    # misaligned ring
    assert f(FAKE, FAKE, FAKE, 2, ctypes.c_void_p(0x1008), FAKE, 4, 64, 10000.0, FAKE, 64, None) == -1
    # no requests: nothing to do
    assert f(None, None, None, 0, None, None, 0, 64, 10000.0, None, 0, None) == 0


def test_cpython_entry_points_match_ctypes_on_host_checks(L):
    """The CPython entry points of the per-step calls (_fastcall.c, built
    beside the library where the Python headers are present) reach the same
    C functions as ctypes: the host-side checks give the same statuses, and
    a wrong argument count or an int32 out of range raises before any call."""
    from sparse_attention_indexer_index_gb300 import _build
    if not os.path.exists(_build.fastcall_path()):
        pytest.skip("the CPython entry points were not built (no Python headers here)")
    from sparse_attention_indexer_index_gb300 import _fastcall as fc
    X = 0x1000
    need = L.qsa_indexer_select_workspace_size(6, 80000, 512)
    a = (X, X, 1 << 20, 1, X, 6, X, 80000, 6, X, 1250, 64, 512, None, None, X, None, 0, X, need - 1, None)
    assert fc.qsa_indexer_select(*a) == L.qsa_indexer_select(*a) == -3
    a_k = a[:12] + (4096,) + a[13:19] + (need,) + a[20:]
    assert fc.qsa_indexer_select(*a_k) == L.qsa_indexer_select(*a_k) == -2
    g = a[:1] + (X,) + a[1:]  # gated: the gates after q
    assert fc.qsa_indexer_select_gated(*g) == L.qsa_indexer_select_gated(*g) == -3
    z = (None, None, 0, 0, None, 0, None, 0, 0, None, 0, 64, 512, None, None, None, None, 0, None, 0, None)
    assert fc.qsa_indexer_select(*z) == 0
    d = (X, X, X, X, 10000.0, X, X, 1 << 20, 1, X, 6, X, 80000, 6, X, 1250, 64, 4096, None, None, X, None, 0, X,
         need, None)
    assert fc.qsa_decode_step(*d) == L.qsa_decode_step(*d) == -2
    dg = d[:6] + (X,) + d[6:]
    assert fc.qsa_decode_step_gated(*dg) == L.qsa_decode_step_gated(*dg) == -2
    with pytest.raises(TypeError):
        fc.qsa_decode_step(*d[:-1])
    with pytest.raises(OverflowError):
        fc.qsa_decode_step(*(d[:10] + (1 << 40,) + d[11:]))


def test_binding_call_path_with_and_without_the_cpython_entry_points(L):
    """The binding's dispatcher reaches the same C function through the
    CPython entry points (when built) and through ctypes (when not)."""
    import sparse_attention_indexer_index_gb300 as qsa
    X = 0x1000
    need = L.qsa_indexer_select_workspace_size(6, 80000, 512)
    d = (X, X, X, X, 10000.0, X, X, 1 << 20, 1, X, 6, X, 80000, 6, X, 1250, 64, 4096, None, None, X, None, 0, X,
         need, None)
    saved = qsa._fast
    try:
        qsa._fast = None  # load the CPython entry points if they were built
        assert qsa._call("qsa_decode_step", *d) == -2
        qsa._fast = False  # ctypes only
        assert qsa._call("qsa_decode_step", *d) == -2
        assert qsa._call("qsa_indexer_select_workspace_size", 6, 80000, 512) == need
    finally:
        qsa._fast = saved


def test_cpython_entry_points_are_optional(monkeypatch, tmp_path):
    """Without the Python headers the CPython entry points are not built (and
    the binding keeps to ctypes); nothing is raised."""
    import sysconfig
    from sparse_attention_indexer_index_gb300 import _build
    real = sysconfig.get_paths

    def no_headers(*a, **k):
        paths = dict(real(*a, **k))
        paths["include"] = str(tmp_path / "no_python_headers")
        return paths

    monkeypatch.setattr(sysconfig, "get_paths", no_headers)
    assert _build.build_fastcall(force=True) is None
