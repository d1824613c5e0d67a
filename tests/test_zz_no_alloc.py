"""The allocation-free variant of the fused indexer call.

Some callers cannot allocate device memory at the moment the indexer runs: a
decode step that is being recorded into a CUDA graph, an inference engine
whose memory plan is fixed before serving starts, or a plugin hosted by
another framework that hands it no allocator.  They cannot provide the
workspace that qsa_indexer_select needs for its scores, so
qsa_indexer_select_noalloc keeps those scores in a fixed scratch array that
belongs to the library.

This test calls the new entry point through the C ABI twice in a row, on two
different workloads (so the second call runs on scratch left dirty by the
first), and checks each result against the ordinary qsa_indexer_select with a
caller workspace: the selected blocks, positions and slots must be identical
(both paths score in the same kernel, so the scores, and with them the exact
top-k, agree bit for bit).  It also checks that a call whose scores would not
fit the scratch array is refused without launching anything.

The file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
from gpu_util import bf16_dev, to_dev
from workloads import c2_verify, decode_workload

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20  # QSA_NOALLOC_SCRATCH_BYTES in include/qsa.h


@pytest.fixture(scope="module")
def lib():
    import sparse_attention_indexer_index_gb300 as qsa
    qsa.build()
    L = qsa.lib()
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f = L.qsa_indexer_select_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [p, p, i64, i32, p, i32, p, i32, i32, p, i64, i32, i32, p, p, p, p]
    return qsa, L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _device_state(w):
    import torch
    pool = np.zeros((w.pool_rows, 128), np.uint16)
    oracle.compress(w.raw_keys, w.block_req, w.block_id, w.page_table, w.page_size, w.rope_base, pool)
    return {
        "q": bf16_dev(w.q), "pool": bf16_dev(pool), "rrs": to_dev(w.req_row_start),
        "rl": to_dev(w.row_len), "pt": to_dev(w.page_table),
        "stream": ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
    }


def _noalloc(L, w, d):
    import torch
    width = 4 * w.k_blk + 3
    blocks = torch.full((w.n_rows, w.k_blk), -7, dtype=torch.int32, device="cuda")
    pos = torch.full((w.n_rows, width), -7, dtype=torch.int32, device="cuda")
    slots = torch.full((w.n_rows, width), -7, dtype=torch.int32, device="cuda")
    st = L.qsa_indexer_select_noalloc(
        _ptr(d["q"]), _ptr(d["pool"]), d["pool"].shape[0], w.n_req, _ptr(d["rrs"]), w.n_rows,
        _ptr(d["rl"]), w.max_len, w.max_rows_per_req, _ptr(d["pt"]), d["pt"].shape[1], w.page_size,
        w.k_blk, _ptr(blocks), _ptr(pos), _ptr(slots), d["stream"])
    assert st == 0, L.qsa_status_string(st)
    return blocks, pos, slots


def _with_workspace(qsa, w, d):
    out = qsa.indexer_select(d["q"], d["pool"], d["rrs"], d["rl"], d["pt"], w.page_size, w.max_len,
                             w.max_rows_per_req, k_blk=w.k_blk, want_blocks=True, want_pos=True)
    return out["blocks"], out["pos"], out["slots"]


def test_noalloc_matches_workspace_path_on_two_calls_in_a_row(lib):
    import torch
    qsa, L = lib
    wa = c2_verify(3)  # 6 rows, L = 80,000: 480 KB of scores
    wb = decode_workload(62, [[1030, 1031, 1032], [4099], [17], [2051, 2052]], page_size=16,
                         k_blk=512)
    da, db = _device_state(wa), _device_state(wb)
    got_a = _noalloc(L, wa, da)
    got_b = _noalloc(L, wb, db)  # second call in a row, on the first call's scratch
    torch.cuda.synchronize()
    want_a = _with_workspace(qsa, wa, da)
    want_b = _with_workspace(qsa, wb, db)
    torch.cuda.synchronize()
    for got, want in ((got_a, want_a), (got_b, want_b)):
        for g, e in zip(got, want):
            assert torch.equal(g, e)
    assert qsa.device_status(clear=True) == 0


def test_noalloc_refuses_calls_beyond_the_scratch_array(lib):
    _, L = lib
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the size check fails first
    max_len = 131072
    n_rows = SCRATCH_BYTES // (4 * (max_len // 4)) + 1
    st = L.qsa_indexer_select_noalloc(fake, fake, 1 << 20, 1, fake, n_rows, fake, max_len, n_rows,
                                      fake, max_len // 64, 64, 512, None, None, fake, None)
    assert st == -2  # QSA_ERR_UNSUPPORTED
    # the largest call that fits is accepted by the same check (not launched here)
    assert (n_rows - 1) * 4 * (max_len // 4) <= SCRATCH_BYTES


def test_noalloc_on_a_decode_batch_and_without_device_allocation(lib):
    """32 requests of one row each on 64-token pages (the batched decode
    shape, one-row tiles in the scorer) through the allocation-free call:
    identical to the workspace path, and a warm call changes the device's
    free memory by nothing (its outputs allocated beforehand)."""
    import torch
    qsa, L = lib
    rng = np.random.default_rng(64)
    rows = [[int(x)] for x in rng.integers(4096, 40_000, size=32)]
    w = decode_workload(64, rows, page_size=64, k_blk=512)
    d = _device_state(w)
    got = _noalloc(L, w, d)  # warm: first call on this shape
    torch.cuda.synchronize()
    want = _with_workspace(qsa, w, d)
    torch.cuda.synchronize()
    for g, e in zip(got, want):
        assert torch.equal(g, e)
    width = 4 * w.k_blk + 3
    slots = torch.full((w.n_rows, width), -7, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    st = L.qsa_indexer_select_noalloc(
        _ptr(d["q"]), _ptr(d["pool"]), d["pool"].shape[0], w.n_req, _ptr(d["rrs"]), w.n_rows,
        _ptr(d["rl"]), w.max_len, w.max_rows_per_req, _ptr(d["pt"]), d["pt"].shape[1], w.page_size,
        w.k_blk, None, None, _ptr(slots), d["stream"])
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert st == 0
    assert free1 == free0
    assert torch.equal(slots, want[2])
    assert qsa.device_status(clear=True) == 0
