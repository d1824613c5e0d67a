"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars: compressed keys within 1 BF16 ulp plus 2^-22 absolute, with more than
99% of elements bit-identical (FP32 vs FP64 normalisation and rotation), scores within 2e-5 * (1/sqrt(128)) * sum|q k| + 1e-6 of the FP64
oracle (FP32 accumulation of exact BF16 products), and selection, expansion
and slot translation bit-exact when both sides see the same FP32 scores.
"""
import numpy as np
import pytest

import oracle
from gpu_util import bf16_dev, bf16_host, key_tolerance, score_tolerance, to_dev
from workloads import (c1_decode, c2_verify, c2_batched, c3_batched, c4_dsa_topk, c5_prefill,
                       decode_workload, indexshare_mtp, normal_bf16, topk_workload, TOPK_DISTS)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qsa():
    import sparse_attention_indexer_index_gb300 as m
    m.build()
    m.lib()
    return m


@pytest.fixture(autouse=True)
def _no_device_faults(qsa):
    yield
    assert qsa.device_status(clear=True) == 0, "a device-side bounds check fired"


def oracle_pool(w):
    pool = np.zeros((w.pool_rows, 128), np.uint16)
    oracle.compress(w.raw_keys, w.block_req, w.block_id, w.page_table, w.page_size, w.rope_base, pool)
    return pool


def gpu_pool(qsa, w):
    import torch
    pool = torch.zeros((w.pool_rows, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(bf16_dev(w.raw_keys), to_dev(w.block_id), pool, block_req=to_dev(w.block_req),
                      page_table=to_dev(w.page_table), page_size=w.page_size, rope_base=w.rope_base)
    return pool


# ----------------------------------------------------------------- compress
SMALL_DECODE = [
    ("one_row_ragged_tiles", [[4 * 300 + 2]], 64),
    ("verify_rows", [[5001, 5002, 5003, 5004, 5005, 5006]], 64),
    ("multi_request", [[37, 40, 41], [9], [1030, 1031], [4096 * 4 + 3]], 16),
    ("tiny_pages", [[77, 78], [130]], 4),
    ("ten_rows", [[2000 + i for i in range(10)], [513]], 32),
    # one row per request on 16-token pages: the CUDA-core streaming scorer
    ("one_row_small_pages", [[1002], [4001], [77], [9000]], 16),
]




@pytest.mark.parametrize("name,rows,P", SMALL_DECODE)
def test_compress_parity(qsa, name, rows, P):
    w = decode_workload(21, rows, page_size=P, k_blk=64)
    want = oracle_pool(w)
    got = bf16_host(gpu_pool(qsa, w))
    a, b = oracle.bf16_to_float(got), oracle.bf16_to_float(want)
    bad = np.abs(a - b) > key_tolerance(a, b)
    assert not bad.any(), (np.argwhere(bad)[:5], a[bad][:5], b[bad][:5])
    assert (got == want).mean() > 0.99


def test_compress_parity_long_positions_sampled(qsa):
    """The c3 workload (32 requests up to 131,072 tokens): every block on the
    GPU, a random sample of 4,000 blocks on the oracle."""
    w = c3_batched(0)
    got = bf16_host(gpu_pool(qsa, w))
    rng = np.random.default_rng(5)
    for i in rng.choice(w.n_blocks, 4000, replace=False):
        r, b = int(w.block_req[i]), int(w.block_id[i])
        row = oracle.pool_row(w.page_table[r], b, w.page_size)
        want = oracle.compress_block(w.raw_keys[4 * i: 4 * i + 4], 4 * b, w.rope_base)
        a, e = oracle.bf16_to_float(got[row]), oracle.bf16_to_float(want)
        assert (np.abs(a - e) <= key_tolerance(a, e)).all(), (i, a, e)


# ----------------------------------------------------------------- scores
@pytest.mark.parametrize("name,rows,P", SMALL_DECODE)
def test_scores_parity(qsa, name, rows, P):
    import torch
    w = decode_workload(22, rows, page_size=P, k_blk=64)
    pool_h = oracle_pool(w)
    ld = w.max_len // 4 + 40
    n_fill = ld - 8
    want = oracle.index_scores(w.q, pool_h, w.req_row_start, w.row_len, w.page_table, w.page_size, ld)
    scores = torch.full((w.n_rows, ld), 7.0, device="cuda")
    qsa.index_scores(bf16_dev(w.q), bf16_dev(pool_h), to_dev(w.req_row_start), to_dev(w.row_len),
                     to_dev(w.page_table), w.page_size, w.max_len, w.max_rows_per_req, scores=scores,
                     n_fill=n_fill)
    got = scores.cpu().numpy()
    tol = score_tolerance(w.q, pool_h, w.req_row_start, w.row_len, w.page_table, w.page_size, ld)
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        err = np.abs(got[t, :nb].astype(np.float64) - want[t, :nb])
        assert (err <= tol[t, :nb]).all(), (t, err.max())
        assert np.isneginf(got[t, nb:n_fill]).all()
        assert (got[t, n_fill:] == 7.0).all()


# ----------------------------------------------------------------- top-k
def run_topk(qsa, w, k=None, with_slots=True):
    k = k or w.k
    idx, slots = qsa.topk_select(to_dev(w.scores), k, n_valid=to_dev(w.n_valid),
                                 n_max=int(w.n_valid.max()) if w.n_valid.size else 0,
                                 page_table=to_dev(w.page_table) if with_slots else None,
                                 page_size=w.page_size)
    ref_idx, ref_slots = oracle.topk(w.scores, k, n_valid=w.n_valid,
                                     page_table=w.page_table if with_slots else None,
                                     page_size=w.page_size)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    if with_slots:
        assert np.array_equal(slots.cpu().numpy(), ref_slots)


@pytest.mark.parametrize("dist", TOPK_DISTS)
@pytest.mark.parametrize("k", [1, 7, 512, 2048])
def test_topk_parity_ragged(qsa, dist, k):
    run_topk(qsa, topk_workload(31, 9, 6000, k=k, dist=dist, ragged=True), k)


@pytest.mark.parametrize("n_rows,n", [(1, 100_000), (3, 50_000), (40, 33_000), (40, 20_000), (200, 3000), (400, 3000),
                                      (5, 32_768), (2, 32_772)])
def test_topk_parity_row_lengths(qsa, n_rows, n):
    """Rows kept in shared memory (<= 32,768 scores) and rows streamed through
    the bulk-copy ring, around the boundary between the two."""
    run_topk(qsa, topk_workload(32, n_rows, n, k=2048, dist="fp16dup"))


@pytest.mark.parametrize("n", [20_000, 45_000])
def test_topk_misleading_sample_falls_back_to_exact_histogram(qsa, n):
    """The selection first estimates a lower bound for the k-th key from
    1024 evenly strided scores (positions floor(j*n/1024)).  Planting the
    largest values exactly there makes the estimate too high (fewer than k
    candidates); the exact whole-row histogram must take over."""
    rng = np.random.default_rng(n + 1)
    s = (rng.standard_normal((2, n)) * 0.01).astype(np.float32)
    pos = (np.arange(1024, dtype=np.int64) * n) // 1024
    s[0, pos] = 100.0 + rng.standard_normal(1024).astype(np.float32)
    s[1, pos] = 5.0
    nv = np.full(2, n, np.int32)
    for k in [1500, 2048]:
        idx, _ = qsa.topk_select(to_dev(s), k, n_valid=to_dev(nv), n_max=n)
        ref, _ = oracle.topk(s, k, n_valid=nv)
        assert np.array_equal(idx.cpu().numpy(), ref), k


@pytest.mark.parametrize("n", [20_000, 45_000])
def test_topk_heavy_ties_take_the_full_row_path(qsa, n):
    """So many scores share the boundary bin that the candidate list would
    overflow: the exact passes and the emission run over the whole row."""
    rng = np.random.default_rng(n)
    s = np.zeros((4, n), np.float32)
    s[0] = 1.5                                              # all equal
    s[1] = rng.integers(0, 3, size=n).astype(np.float32)    # three values
    s[2] = (rng.integers(0, 64, size=n) / 64.0 + 1.0).astype(np.float32)  # one top-bits bin
    s[3] = rng.standard_normal(n).astype(np.float32)        # ordinary row beside them
    nv = np.full(4, n, np.int32)
    for k in [512, 2048]:
        idx, _ = qsa.topk_select(to_dev(s), k, n_valid=to_dev(nv), n_max=n)
        ref, _ = oracle.topk(s, k, n_valid=nv)
        assert np.array_equal(idx.cpu().numpy(), ref), k


@pytest.mark.parametrize("n,copies", [(20_000, 5), (32_768, 5), (20_000, 19)])
def test_topk_hard_rows_many_rows(qsa, n, copies):
    """The same hard rows (all equal, three values, one top-bits bin, the
    sample planted with the largest values) in launches of 24 and 80 rows,
    which take the single-CTA selection instead of one cluster per row."""
    rng = np.random.default_rng(n + 7)
    base = np.zeros((4, n), np.float32)
    base[0] = 1.5
    base[1] = rng.integers(0, 3, size=n).astype(np.float32)
    base[2] = (rng.integers(0, 64, size=n) / 64.0 + 1.0).astype(np.float32)
    base[3] = (rng.standard_normal(n) * 0.01).astype(np.float32)
    base[3, (np.arange(1024, dtype=np.int64) * n) // 1024] = 100.0
    s = np.concatenate([base] * copies + [rng.standard_normal((4, n)).astype(np.float32)])
    nv = np.full(s.shape[0], n, np.int32)
    for k in [512, 2048]:
        idx, _ = qsa.topk_select(to_dev(s), k, n_valid=to_dev(nv), n_max=n)
        ref, _ = oracle.topk(s, k, n_valid=nv)
        assert np.array_equal(idx.cpu().numpy(), ref), k


@pytest.mark.parametrize("n", [3000, 20_000, 32_768])
def test_topk_many_rows_small_ctas(qsa, n):
    """More than two rows per SM (one small CTA per row, three per SM): ordinary
    rows, rows with every entry equal (the candidate lists overflow: whole-row
    walks), three values, one top-bits bin, and rows whose sampled entries
    (32 runs of 32) hold the largest values (too few entries above the
    sampled bound: the level-0 histogram is redone over the row)."""
    rng = np.random.default_rng(n + 3)
    rows = []
    for r in range(320):
        kind = r % 5
        if kind == 0:
            x = np.full(n, 1.5, np.float32)
        elif kind == 1:
            x = rng.integers(0, 3, size=n).astype(np.float32)
        elif kind == 2:
            x = (rng.integers(0, 64, size=n) / 64.0 + 1.0).astype(np.float32)
        elif kind == 3:
            x = (rng.standard_normal(n) * 0.01).astype(np.float32)
            for run in range(32):
                p = ((run * n) // 32) & ~3
                x[p:p + 32] = 100.0 + rng.standard_normal(min(32, n - p)).astype(np.float32)
        else:
            x = rng.standard_normal(n).astype(np.float32)
        rows.append(x)
    s = np.stack(rows)
    nv = np.full(s.shape[0], n, np.int32)
    nv[7] = 100      # fewer entries than k
    nv[11] = n - 3   # ragged tail
    for k in [512, 2048]:
        idx, _ = qsa.topk_select(to_dev(s), k, n_valid=to_dev(nv), n_max=n)
        ref, _ = oracle.topk(s, k, n_valid=nv)
        assert np.array_equal(idx.cpu().numpy(), ref), k


@pytest.mark.parametrize("dist", TOPK_DISTS)
def test_topk_parity_dsa_full_size(qsa, dist):
    """64 rows x 80,000 FP32 scores, k = 2048, with slot translation."""
    run_topk(qsa, c4_dsa_topk(0, dist))


@pytest.mark.parametrize("dist", TOPK_DISTS)
def test_topk_long_rows_1m_verify_shape(qsa, dist):
    """6 rows of 1,000,000 FP32 scores (long-context verify step), k = 2048,
    with slots: one cluster of 16 CTAs per row, slices larger than shared
    memory (the rest re-read from L2)."""
    run_topk(qsa, topk_workload(61, 6, 1_000_000, k=2048, dist=dist))


@pytest.mark.parametrize("k", [1, 777, 2048])
def test_topk_long_rows_ragged(qsa, k):
    """12 long rows of ragged valid lengths (some no longer than k, one
    empty) in one launch: clusters of 8 CTAs, empty slices in the last CTAs
    of short rows."""
    w = topk_workload(62, 12, 300_000, k=k, dist="normal")
    w.n_valid[:] = [300_000, 299_999, 33_001, 150_003, 2048, 777, 0, 5, 64_000, 131_071, 40_000, 250_001]
    run_topk(qsa, w, k)


def test_topk_long_rows_heavy_ties(qsa):
    """Long rows where the k-th key is shared by most of the row: all equal,
    three values, one top-bits bin, +-0 and NaN mixed in; the radix levels
    run to the full key and the equal entries are taken by index."""
    rng = np.random.default_rng(63)
    n = 200_000
    s = np.zeros((5, n), np.float32)
    s[0] = 1.5
    s[1] = rng.integers(0, 3, size=n).astype(np.float32)
    s[2] = (rng.integers(0, 64, size=n) / 64.0 + 1.0).astype(np.float32)
    s[3] = np.where(rng.random(n) < 0.5, np.float32(0.0), np.float32(-0.0))
    s[3, ::7] = np.nan
    s[4] = rng.standard_normal(n).astype(np.float32)
    s[4, -3000:] = np.inf
    nv = np.full(5, n, np.int32)
    for k in [512, 2048]:
        idx, _ = qsa.topk_select(to_dev(s), k, n_valid=to_dev(nv), n_max=n)
        ref, _ = oracle.topk(s, k, n_valid=nv)
        assert np.array_equal(idx.cpu().numpy(), ref), k


def test_topk_special_rows(qsa):
    import torch
    n = 5000
    s = np.zeros((6, n), np.float32)
    s[0] = 0.25                                    # all equal -> 0..k-1
    s[1] = -0.0                                    # signed zeros tie with +0
    s[1, ::3] = 0.0
    s[2] = np.nan                                  # NaN below everything
    s[2, 4000:] = -np.inf
    s[3] = np.arange(n, dtype=np.float32)          # strictly increasing
    s[4] = -np.arange(n, dtype=np.float32)
    s[5, 100] = np.inf
    nv = np.array([n, n, n, n, n, 0], np.int32)
    for k in [1, 100, 2048]:
        idx, _ = qsa.topk_select(to_dev(s), k, n_valid=to_dev(nv), n_max=n)
        ref, _ = oracle.topk(s, k, n_valid=nv)
        assert np.array_equal(idx.cpu().numpy(), ref), k


# ----------------------------------------------------------------- expand
@pytest.mark.parametrize("P", [4, 16, 64])
def test_expand_parity(qsa, P):
    rng = np.random.default_rng(P)
    lens = [[int(x) for x in rng.integers(0, 9000, size=4)] + [1, 2, 3, 4, 5]]
    w = decode_workload(41, lens, page_size=P, k_blk=512)
    k = 512
    sel = np.full((w.n_rows, k), -1, np.int32)
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        c = np.sort(rng.permutation(nb)[:k])
        sel[t, :c.size] = c
    pos, slots = qsa.expand_slots(to_dev(sel), to_dev(w.req_row_start), to_dev(w.row_len),
                                  to_dev(w.page_table), w.page_size)
    rpos, rslots = oracle.expand(sel, w.req_row_start, w.row_len, w.page_table, w.page_size)
    assert np.array_equal(pos.cpu().numpy(), rpos)
    assert np.array_equal(slots.cpu().numpy(), rslots)


# ----------------------------------------------------------------- fused path
def check_fused(qsa, w, sample_rows=None, select_rows=None):
    import torch
    pool_h = oracle_pool(w) if w.n_blocks < 200_000 else None
    if pool_h is None:
        pool = gpu_pool(qsa, w)
        pool_h = bf16_host(pool)
    else:
        pool = bf16_dev(pool_h)
    ld = (w.max_len // 4 + 3) // 4 * 4
    scores = torch.full((w.n_rows, ld), float("nan"), device="cuda")
    out = qsa.indexer_select(bf16_dev(w.q), pool, to_dev(w.req_row_start), to_dev(w.row_len),
                             to_dev(w.page_table), w.page_size, w.max_len, w.max_rows_per_req,
                             k_blk=w.k_blk, want_blocks=True, want_pos=True, scores_out=scores)
    s = scores.cpu().numpy()
    rows = np.arange(w.n_rows) if sample_rows is None else sample_rows
    # scores against the oracle (on the same keys)
    rr = w.row_req()
    for t in rows:
        r = int(rr[t])
        nb = int(w.row_len[t]) // 4
        sub_rrs = np.array([0, 1], np.int32)
        want = oracle.index_scores(w.q[t:t + 1], pool_h, sub_rrs, w.row_len[t:t + 1],
                                   w.page_table[r:r + 1], w.page_size, max(1, nb))
        tol = score_tolerance(w.q[t:t + 1], pool_h, sub_rrs, w.row_len[t:t + 1],
                              w.page_table[r:r + 1], w.page_size, max(1, nb))
        err = np.abs(s[t, :nb].astype(np.float64) - want[0, :nb])
        assert (err <= tol[0, :nb]).all(), (t, float(err.max()))
    # selection / expansion / slots bit-exact on the GPU's own scores
    if select_rows is None:
        sel_ref, _ = oracle.topk(s, w.k_blk, n_valid=w.row_len // 4)
        pos_ref, slots_ref = oracle.expand(sel_ref, w.req_row_start, w.row_len, w.page_table, w.page_size)
        assert np.array_equal(out["blocks"].cpu().numpy(), sel_ref)
        assert np.array_equal(out["pos"].cpu().numpy(), pos_ref)
        assert np.array_equal(out["slots"].cpu().numpy(), slots_ref)
    else:
        blocks, pos, slots = (out[k].cpu().numpy() for k in ("blocks", "pos", "slots"))
        for t in select_rows:
            r = int(rr[t])
            nb = int(w.row_len[t]) // 4
            sel = oracle.topk_row(s[t, :nb], w.k_blk)
            p_ref, s_ref = oracle.expand_row(sel, int(w.row_len[t]), w.page_table[r], w.page_size)
            assert np.array_equal(blocks[t], sel), t
            assert np.array_equal(pos[t], p_ref), t
            assert np.array_equal(slots[t], s_ref), t
    return out


@pytest.mark.parametrize("name,rows,P", SMALL_DECODE)
def test_fused_parity_small(qsa, name, rows, P):
    check_fused(qsa, decode_workload(51, rows, page_size=P, k_blk=64))


def test_fused_parity_padding_and_pending(qsa):
    """Rows with fewer visible blocks than k (padding), L mod 4 = 0..3, L < 4."""
    w = decode_workload(52, [[1, 2, 3, 4, 5, 6, 7], [2047, 2048, 2049, 2050, 2051]], page_size=64,
                        k_blk=512)
    out = check_fused(qsa, w)
    slots = out["slots"].cpu().numpy()
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        n_out = 4 * min(nb, 512) + int(w.row_len[t]) % 4
        assert (slots[t, n_out:] == -1).all() and (slots[t, :n_out] >= 0).all()


def test_fused_parity_c1_decode(qsa):
    check_fused(qsa, c1_decode(0))


def test_fused_parity_c2_verify(qsa):
    check_fused(qsa, c2_verify(0))


def test_fused_parity_c3_batched_sampled(qsa):
    w = c3_batched(0)
    check_fused(qsa, w, sample_rows=np.arange(0, w.n_rows, 4))


def test_fused_parity_prefill_chunk(qsa):
    """300 consecutive query rows of one request: the tensor-core scorer with
    several row tiles (the last one partial) and causal visibility per row."""
    check_fused(qsa, decode_workload(53, [[4000 + i for i in range(300)]], page_size=64, k_blk=512))


def test_fused_parity_prefill_ragged_row_tiles(qsa):
    """777 consecutive query rows: the prefill tile-height plan (more than 64
    rows per request) takes 40-row tiles on 152 SMs, so the last row tile
    holds 17 rows, and every key tile but the causal edge is fully visible to
    its row tile (the epilogue's fast path)."""
    check_fused(qsa, decode_workload(57, [[6001 + i for i in range(777)]], page_size=64, k_blk=512))


def test_fused_parity_prefill_c5_sampled(qsa):
    """The full prefill chunk (4096 rows, L = 131,072): scores checked on 24
    sampled rows, selection and slots on 64."""
    w = c5_prefill(0)
    rng = np.random.default_rng(7)
    check_fused(qsa, w, sample_rows=np.sort(rng.choice(w.n_rows, 24, replace=False)),
                select_rows=np.sort(rng.choice(w.n_rows, 64, replace=False)))


def test_fused_parity_verify_batched_sampled(qsa):
    """32 verify requests of 6 rows at L = 80,000 (tensor-core scorer, one key
    tile per CTA): scores on every 8th row, selection on all rows."""
    w = c2_batched(0)
    check_fused(qsa, w, sample_rows=np.arange(0, w.n_rows, 8))


def test_fused_workspace_path_matches_scores_out_path(qsa):
    """Scores kept in the caller's workspace give the same slots."""
    w = c2_verify(1)
    pool = gpu_pool(qsa, w)
    args = (bf16_dev(w.q), pool, to_dev(w.req_row_start), to_dev(w.row_len), to_dev(w.page_table),
            w.page_size, w.max_len, w.max_rows_per_req)
    import torch
    ld = (w.max_len // 4 + 3) // 4 * 4
    a = qsa.indexer_select(*args, k_blk=512, scores_out=torch.empty((w.n_rows, ld), device="cuda"))
    b = qsa.indexer_select(*args, k_blk=512)
    assert torch.equal(a["slots"], b["slots"])


@pytest.mark.parametrize("case", ["ragged_small", "c2_verify"])
def test_select_blocks_parity(qsa, case):
    """The selection half alone (scores given): bit-exact against the
    oracle's top-k and expansion on the same FP32 scores, including rows with
    fewer visible blocks than k and every pending-token count."""
    if case == "ragged_small":
        w = decode_workload(54, [[1, 5, 9], [2051, 4096, 7001, 20_002]], page_size=64, k_blk=512)
    else:
        w = c2_verify(0)
    rng = np.random.default_rng(11)
    ld = (w.max_len // 4 + 3) // 4 * 4
    s = rng.standard_normal((w.n_rows, ld)).astype(np.float32)
    out = qsa.select_blocks(to_dev(s), to_dev(w.req_row_start), to_dev(w.row_len), to_dev(w.page_table),
                            w.page_size, w.max_len, k_blk=w.k_blk, want_blocks=True, want_pos=True)
    sel_ref, _ = oracle.topk(s, w.k_blk, n_valid=w.row_len // 4)
    pos_ref, slots_ref = oracle.expand(sel_ref, w.req_row_start, w.row_len, w.page_table, w.page_size)
    assert np.array_equal(out["blocks"].cpu().numpy(), sel_ref)
    assert np.array_equal(out["pos"].cpu().numpy(), pos_ref)
    assert np.array_equal(out["slots"].cpu().numpy(), slots_ref)


# ----------------------------------------------------------------- IndexShare
def _dev_fault_bits(flags):
    """Oracle flags -> device fault bits (1: cut at the width -> bit 4;
    2: kept block incomplete at the capture, 4: kept row out of range -> bit 0)."""
    return (16 if flags & 1 else 0) | (1 if flags & 6 else 0)


@pytest.mark.parametrize("P", [4, 16, 64])
def test_indexshare_parity_kept_selections(qsa, P):
    """Draft rows reading kept selections: rows before, at and after the
    capture, every cap_len mod 4, kept rows with fewer blocks than k, kept
    rows shared by several requests, several rows per request."""
    rng = np.random.default_rng(100 + P)
    k, n_extra = 512, 5
    cap_len = np.array([0, 3, 4, 9, 2050, 2051, 2052, 2053, 7001, 20_000], np.int32)
    cap = np.full((cap_len.size, k), -1, np.int32)
    for c, L0 in enumerate(cap_len):
        nb0 = int(L0) // 4
        if nb0:
            cap[c] = oracle.topk_row(rng.standard_normal(nb0).astype(np.float32), k)
    cap_row = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 9, 4], np.int32)
    rows = []
    for r, c in enumerate(cap_row):
        L0 = int(cap_len[c])
        rows.append([max(0, L0 - 3), L0, L0 + 1, L0 + 3, L0 + n_extra] if r % 2 == 0 else [L0 + 2])
    row_len = np.array([x for rr in rows for x in rr], np.int32)
    rrs = np.concatenate([[0], np.cumsum([len(rr) for rr in rows])]).astype(np.int32)
    ctx = max(int(row_len.max()), 1)
    pt = np.stack([rng.permutation(ctx // P + 8) for _ in rows]).astype(np.int32)
    pos, slots = qsa.indexshare_slots(to_dev(cap), to_dev(cap_len), to_dev(cap_row), n_extra, to_dev(rrs),
                                      to_dev(row_len), to_dev(pt), P)
    rpos, rslots, flags = oracle.indexshare(cap, cap_len, cap_row, n_extra, rrs, row_len, pt, P)
    assert flags == 0
    assert np.array_equal(pos.cpu().numpy(), rpos)
    assert np.array_equal(slots.cpu().numpy(), rslots)


def test_indexshare_parity_faults(qsa):
    """Rows whose list does not fit, kept blocks incomplete at the capture
    and a kept row out of range: the same output as the oracle, and the
    device fault bits set."""
    P, k, n_extra = 16, 8, 2
    cap = np.array([[0, 3, 5, 9, -1, -1, -1, -1], [1, 2, 40, -1, -1, -1, -1, -1]], np.int32)
    cap_len = np.array([41, 30], np.int32)
    pt = np.arange(16, dtype=np.int32)[None, :].repeat(3, 0)[:, ::-1].copy()
    for cap_row, row_len, want_flags in [
        ([0, 0, 0], [45, 60, 100], 1),       # tails of 5, 20 and 60 positions, room for 21
        ([1, 1, 1], [30, 31, 33], 2),        # block 40 was not complete at L = 30
        ([0, 2, 0], [41, 41, 41], 4),        # request 1 points past the kept rows
    ]:
        rrs = np.arange(4, dtype=np.int32)
        cr, rl = np.array(cap_row, np.int32), np.array(row_len, np.int32)
        pos, slots = qsa.indexshare_slots(to_dev(cap), to_dev(cap_len), to_dev(cr), n_extra, to_dev(rrs),
                                          to_dev(rl), to_dev(pt), P)
        rpos, rslots, flags = oracle.indexshare(cap, cap_len, cr, n_extra, rrs, rl, pt, P)
        assert flags == want_flags
        assert qsa.device_status(clear=True) == _dev_fault_bits(flags)
        assert np.array_equal(pos.cpu().numpy(), rpos)
        assert np.array_equal(slots.cpu().numpy(), rslots)


def test_indexshare_after_fused_draft_extend(qsa):
    """One MTP iteration: the fused indexer runs on each request's
    draft-extend row, its selection is kept, and the draft rows read it
    (positions up to 3 tokens past the capture, pending counts 0-3, rows with
    fewer visible blocks than k)."""
    import torch
    w = indexshare_mtp(3, n_req=6, lo=1000, hi=30_000, n_draft=3, page_size=64)
    n_draft = 3
    ext_rows = w.req_row_start[:-1]
    ext_len = w.row_len[ext_rows].copy()
    pool = gpu_pool(qsa, w)
    ext_rrs = np.arange(w.n_req + 1, dtype=np.int32)
    ld = (int(ext_len.max()) // 4 + 3) // 4 * 4
    scores = torch.empty((w.n_req, ld), device="cuda")
    ext = qsa.indexer_select(bf16_dev(w.q[ext_rows]), pool, to_dev(ext_rrs), to_dev(ext_len),
                             to_dev(w.page_table), w.page_size, int(ext_len.max()), 1, k_blk=512,
                             want_blocks=True, scores_out=scores)
    kept = ext["blocks"]
    sel_ref, _ = oracle.topk(scores.cpu().numpy(), 512, n_valid=ext_len // 4)
    assert np.array_equal(kept.cpu().numpy(), sel_ref)
    # the draft rows of this iteration: request r's rows after its first
    draft = np.concatenate([np.arange(w.req_row_start[r] + 1, w.req_row_start[r + 1]) for r in range(w.n_req)])
    d_len = w.row_len[draft]
    d_rrs = np.arange(0, w.n_req * n_draft + 1, n_draft, dtype=np.int32)
    cap_row = np.arange(w.n_req, dtype=np.int32)
    pos, slots = qsa.indexshare_slots(kept, to_dev(ext_len), to_dev(cap_row), n_draft + 1, to_dev(d_rrs),
                                      to_dev(d_len), to_dev(w.page_table), w.page_size)
    rpos, rslots, flags = oracle.indexshare(sel_ref, ext_len, cap_row, n_draft + 1, d_rrs, d_len,
                                            w.page_table, w.page_size)
    assert flags == 0
    assert np.array_equal(pos.cpu().numpy(), rpos)
    assert np.array_equal(slots.cpu().numpy(), rslots)


def test_select_blocks_long_context(qsa):
    """Block selection for rows past 131,072 tokens (more than 32,768
    blocks, up to a 1M-token context): the long-row cluster kernel in QSA
    mode, with every pending-token count and slot translation."""
    P = 64
    row_len = np.array([1_000_003, 524_289, 131_074, 400_000], np.int32)
    rrs = np.array([0, 1, 2, 4], np.int32)  # the last request has two rows
    rng = np.random.default_rng(12)
    ld_pt = (int(row_len.max()) + P - 1) // P
    page_table = rng.permutation(3 * ld_pt).astype(np.int32).reshape(3, ld_pt)
    max_len = int(row_len.max())
    ld = (max_len // 4 + 3) // 4 * 4
    s = (rng.standard_normal((row_len.size, ld)) * 0.1).astype(np.float32)
    s[1, ::5] = 0.25  # many exact ties in one row
    out = qsa.select_blocks(to_dev(s), to_dev(rrs), to_dev(row_len), to_dev(page_table), P, max_len, k_blk=512,
                            want_blocks=True, want_pos=True)
    sel_ref, _ = oracle.topk(s, 512, n_valid=row_len // 4)
    pos_ref, slots_ref = oracle.expand(sel_ref, rrs, row_len, page_table, P)
    assert np.array_equal(out["blocks"].cpu().numpy(), sel_ref)
    assert np.array_equal(out["pos"].cpu().numpy(), pos_ref)
    assert np.array_equal(out["slots"].cpu().numpy(), slots_ref)


# ----------------------------------------------------------------- sparse attention
def _attn_check(qsa, q, k, v, slots, scale, faults=0):
    import torch
    from gpu_util import attn_tolerance
    out, lse = qsa.sparse_attn(bf16_dev(q), bf16_dev(k), bf16_dev(v), to_dev(slots), scale)
    ro, rl, f = oracle.sparse_attn(q, k, v, slots, scale)
    assert qsa.device_status(clear=True) == faults
    o = out.cpu().numpy().astype(np.float64)
    tol = attn_tolerance(q, k, v, slots, scale)
    err = np.abs(o - ro)
    assert (err <= tol).all(), float((err / tol).max())
    l = lse.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    assert np.abs(l[fin] - rl[fin]).max(initial=0.0) <= 1e-5 * (1 + np.abs(rl[fin]).max(initial=0.0))
    return out


@pytest.mark.parametrize("h_q,h_kv,d", [(16, 2, 256), (8, 2, 256), (4, 4, 256), (1, 1, 256), (16, 1, 128),
                                        (8, 4, 128), (2, 1, 128)])
def test_sparse_attn_parity_shapes(qsa, h_q, h_kv, d):
    """Rows of 2051 entries (several chunks per row, merged) with masked
    entries, duplicates, a fully masked row and a single-entry row."""
    rng = np.random.default_rng(h_q * 1000 + h_kv * 10 + d)
    n_slots, rows, w = 5000, 5, 2051
    q = normal_bf16(rng, (rows, h_q, d))
    k = normal_bf16(rng, (n_slots, h_kv, d))
    v = normal_bf16(rng, (n_slots, h_kv, d))
    slots = rng.integers(0, n_slots, size=(rows, w)).astype(np.int32)
    slots[0, rng.random(w) < 0.3] = -1
    slots[1, -300:] = -1
    slots[2] = -1
    slots[3] = -1
    slots[3, 1234] = 77
    slots[4, 100:200] = slots[4, 0]
    _attn_check(qsa, q, k, v, slots, d ** -0.5)


@pytest.mark.parametrize("w", [1, 31, 64, 256, 257, 700])
def test_sparse_attn_parity_row_widths(qsa, w):
    """One chunk per row (<= 256 entries) and the split path just past it."""
    rng = np.random.default_rng(w)
    q = normal_bf16(rng, (3, 8, 128))
    k = normal_bf16(rng, (900, 1, 128))
    v = normal_bf16(rng, (900, 1, 128))
    slots = rng.integers(-1, 900, size=(3, w)).astype(np.int32)
    _attn_check(qsa, q, k, v, slots, 0.1)


def test_sparse_attn_slot_past_the_cache_is_flagged(qsa):
    rng = np.random.default_rng(5)
    q = normal_bf16(rng, (2, 8, 256))
    k = normal_bf16(rng, (100, 1, 256))
    v = normal_bf16(rng, (100, 1, 256))
    slots = rng.integers(0, 100, size=(2, 300)).astype(np.int32)
    slots[1, 7] = 100
    _attn_check(qsa, q, k, v, slots, 0.0625, faults=1)


def test_sparse_attn_after_the_fused_indexer(qsa):
    """The end-to-end decode path: slots from qsa_indexer_select (top-512
    blocks, pending tokens, -1 padding for short contexts) feed the sparse
    attention over a synthetic paged K/V cache."""
    import torch
    w = decode_workload(71, [[20_003], [1500], [9000, 9001]], page_size=64, k_blk=512)
    pool = gpu_pool(qsa, w)
    out = qsa.indexer_select(bf16_dev(w.q), pool, to_dev(w.req_row_start), to_dev(w.row_len),
                             to_dev(w.page_table), w.page_size, w.max_len, w.max_rows_per_req, k_blk=512)
    slots = out["slots"].cpu().numpy()
    rng = np.random.default_rng(72)
    n_slots = w.n_pages * w.page_size
    h_q, h_kv, d = 16, 2, 256
    qa = normal_bf16(rng, (w.n_rows, h_q, d))
    k = normal_bf16(rng, (n_slots, h_kv, d))
    v = normal_bf16(rng, (n_slots, h_kv, d))
    assert (slots[1] == -1).sum() > 0  # the short context is padded
    _attn_check(qsa, qa, k, v, slots, d ** -0.5)


# ----------------------------------------------------------------- key path (ring)
def _ring_case(seed, firsts, counts, P):
    """Requests with raw keys for positions 0 .. first+count-1, the ring and
    pool state after the first `first` positions (built by the oracle), and
    the tokens of one more call."""
    rng = np.random.default_rng(seed)
    n_req = len(firsts)
    ctx = [int(f + c) for f, c in zip(firsts, counts)]
    raw = [normal_bf16(rng, (max(L, 1), 128)) for L in ctx]
    pages = max(1, (max(ctx) + P - 1) // P)
    pt = rng.permutation(n_req * pages).astype(np.int32).reshape(n_req, pages)
    pool = np.zeros((n_req * pages * P // 4, 128), np.uint16)
    ring = np.zeros((n_req, 4, 128), np.uint16)
    for r in range(n_req):  # the context before the call, in one chunk per request
        if firsts[r] == 0:
            continue
        rts = np.zeros(n_req + 1, np.int32)
        rts[r + 1:] = firsts[r]
        oracle.append_keys(raw[r][:firsts[r]], rts, np.zeros(n_req, np.int32), ring, pt, P, 10000.0, pool)
    new = np.concatenate([raw[r][firsts[r]:firsts[r] + counts[r]] for r in range(n_req)] + [np.zeros((0, 128), np.uint16)])
    rts = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return new, rts, np.array(firsts, np.int32), ring, pool, pt


@pytest.mark.parametrize("P", [4, 16, 64])
def test_append_keys_parity(qsa, P):
    """One decode/verify call over requests with every first-position phase,
    calls completing 0, 1 or 2 blocks, a request with no tokens, and a long
    call (13 tokens, 3 blocks): the ring bit-exact, the pool within the
    compressed-key bound of the oracle."""
    import torch
    firsts = [0, 1, 2, 3, 5, 6, 7, 8, 12, 400, 4093]
    counts = [1, 6, 6, 6, 2, 6, 13, 0, 3, 6, 7]
    new, rts, fp, ring, pool, pt = _ring_case(30 + P, firsts, counts, P)
    g_ring = bf16_dev(ring).view(torch.bfloat16).reshape(ring.shape).contiguous()
    g_pool = bf16_dev(pool).view(torch.bfloat16).reshape(pool.shape).contiguous()
    qsa.append_keys(bf16_dev(new).reshape(-1, 128), to_dev(rts), to_dev(fp), g_ring, g_pool, to_dev(pt), P)
    oracle.append_keys(new, rts, fp, ring, pt, P, 10000.0, pool)
    assert np.array_equal(bf16_host(g_ring).reshape(ring.shape), ring)
    got = bf16_host(g_pool)
    a, b = oracle.bf16_to_float(got), oracle.bf16_to_float(pool)
    bad = np.abs(a - b) > key_tolerance(a, b)
    assert not bad.any(), np.argwhere(bad)[:5]
    assert (got == pool).mean() > 0.99


def test_append_keys_sequence_matches_direct_compression(qsa):
    """A request built by 40 calls of 1-9 tokens on the GPU holds the same
    pool as the compression of all its complete blocks at once."""
    import torch
    P, L = 16, 203
    rng = np.random.default_rng(44)
    raw = normal_bf16(rng, (L, 128))
    pt = rng.permutation(16).astype(np.int32)[None]
    g_pool = torch.zeros((16 * P // 4, 128), dtype=torch.bfloat16, device="cuda")
    g_ring = torch.zeros((1, 4, 128), dtype=torch.bfloat16, device="cuda")
    g_raw = bf16_dev(raw)
    p = 0
    while p < L:
        n = int(min(L - p, rng.integers(1, 10)))
        qsa.append_keys(g_raw[p:p + n], to_dev(np.array([0, n], np.int32)), to_dev(np.array([p], np.int32)),
                        g_ring, g_pool, to_dev(pt), P)
        p += n
    direct = torch.zeros_like(g_pool)
    nb = L // 4
    qsa.compress_keys(g_raw[:4 * nb], to_dev(np.arange(nb, dtype=np.int32)), direct,
                      block_req=to_dev(np.zeros(nb, np.int32)), page_table=to_dev(pt), page_size=P)
    assert torch.equal(g_pool, direct)
    assert torch.equal(g_ring[0, (L - 1) % 4], g_raw[L - 1])


# ----------------------------------------------------------------- decode step
@pytest.mark.parametrize("case", ["verify_6rows", "batched_one_row", "multi_request_small_pages"])
def test_decode_step_equals_append_then_indexer(qsa, case):
    """qsa_decode_step (key path, then the fused indexer, the scorer CTAs
    that read no new block not waiting for the key path) gives the same pool,
    ring and slots as the two calls made one after the other."""
    import torch
    if case == "verify_6rows":
        rows, P = [[20_000 - 5 + i for i in range(6)]], 64
    elif case == "batched_one_row":
        rows, P = [[5003], [12_000], [777], [30_001]], 64
    else:
        rows, P = [[4099, 4100, 4101], [9], [2051, 2052]], 16
    rng = np.random.default_rng(81)
    w = decode_workload(82, rows, page_size=P, k_blk=512)
    n_req = w.n_req
    firsts = np.array([min(r) - 1 for r in rows], np.int32)          # each row's own token is appended
    counts = np.array([len(r) for r in rows], np.int32)
    ctx = [int(f + c) for f, c in zip(firsts, counts)]
    raw = [normal_bf16(rng, (L, 128)) for L in ctx]
    # state before the step: blocks completed before first, ring with the rest
    ring0 = np.zeros((n_req, 4, 128), np.uint16)
    blocks_before, reqs_before, raws_before = [], [], []
    for r in range(n_req):
        nb0 = int(firsts[r]) // 4
        blocks_before.append(np.arange(nb0, dtype=np.int32))
        reqs_before.append(np.full(nb0, r, np.int32))
        raws_before.append(raw[r][:4 * nb0])
        for p in range(4 * nb0, int(firsts[r])):
            ring0[r, p % 4] = raw[r][p]
    pool0 = torch.zeros((w.pool_rows, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(bf16_dev(np.concatenate(raws_before)), to_dev(np.concatenate(blocks_before)), pool0,
                      block_req=to_dev(np.concatenate(reqs_before)), page_table=to_dev(w.page_table), page_size=P)
    new = np.concatenate([raw[r][firsts[r]:] for r in range(n_req)])
    rts = to_dev(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32))
    fp, pt = to_dev(firsts), to_dev(w.page_table)
    q, rrs, rl = bf16_dev(w.q), to_dev(w.req_row_start), to_dev(w.row_len)
    # the two calls
    ring_a, pool_a = bf16_dev(ring0), pool0.clone()
    qsa.append_keys(bf16_dev(new), rts, fp, ring_a, pool_a, pt, P)
    out_a = qsa.indexer_select(q, pool_a, rrs, rl, pt, P, w.max_len, w.max_rows_per_req, k_blk=512,
                               want_blocks=True, want_pos=True)
    # one call
    ring_b, pool_b = bf16_dev(ring0), pool0.clone()
    out_b = qsa.decode_step(bf16_dev(new), rts, fp, ring_b, q, pool_b, rrs, rl, pt, P, w.max_len,
                            w.max_rows_per_req, k_blk=512, want_blocks=True, want_pos=True)
    assert torch.equal(ring_a, ring_b) and torch.equal(pool_a, pool_b)
    for key in ("slots", "blocks", "pos"):
        assert torch.equal(out_a[key], out_b[key]), key
    # and the step's selection is the oracle's on the GPU scores of the updated pool
    pool_h = bf16_host(pool_b)
    ld = (w.max_len // 4 + 3) // 4 * 4
    scores = torch.full((w.n_rows, ld), float("nan"), device="cuda")
    qsa.indexer_select(q, pool_b, rrs, rl, pt, P, w.max_len, w.max_rows_per_req, k_blk=512, scores_out=scores)
    sel_ref, _ = oracle.topk(scores.cpu().numpy(), 512, n_valid=w.row_len // 4)
    assert np.array_equal(out_b["blocks"].cpu().numpy(), sel_ref)
    assert pool_h.shape[0] == w.pool_rows
