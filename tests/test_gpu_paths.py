"""GPU parity on launch shapes that reach the less common kernels, and the
headline decode step checked against the oracle end to end.

- Many long rows: more than SMs/2 rows longer than 32,768 entries go to the
  one-CTA streaming selection (select_kernel), in token mode (DSA top-2048
  with slots) and in QSA mode (contexts past 131K tokens).
- Ties at the boundary of the register-resident selection (k <= 1024): the
  k-th key shared by many entries, so only the first `need` of them (lowest
  indices) are taken.
- The 6-row verify step at L = 80,000 as one qsa_decode_step call: the rows'
  own keys (positions 79,994..79,999) complete blocks 19,998 and 19,999
  through the 4-slot ring; the new pool rows against the oracle's key path,
  the scores against the oracle on the same keys, the selection, positions
  and slots bit-exact; also with max_len past the rows.
- One request with max_len far past its rows: the one-request scorer's
  tiles reach page-table entries past the rows (unmapped, past the pool,
  other data's pages) without a fault or a stray score.
- Mixed row lengths in one call (the device row plan), also recorded in a
  CUDA graph (the short rows run on a side stream forked and joined inside
  the call).
- More than two rows per SM with k <= 512 (small CTAs, four per SM): hard
  rows, rows whose evenly spaced 16-byte groups hold the largest values,
  special values, ragged lengths, token and QSA modes.
"""
import numpy as np
import pytest

import oracle
from gpu_util import bf16_dev, bf16_host, key_tolerance, score_tolerance, to_dev
from workloads import c2_verify, decode_workload, topk_workload, TOPK_DISTS

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


# ----------------------------------------------------------------- many long rows
@pytest.mark.parametrize("dist", TOPK_DISTS)
def test_topk_many_long_rows_streaming_selection(qsa, dist):
    """128 DSA rows of 80,000 scores, k = 2048, slots through per-row page
    tables: 128 rows x 2 CTAs exceed the SMs, so every row takes one
    streaming CTA (select_kernel)."""
    w = topk_workload(61, 128, 80_000, k=2048, dist=dist)
    idx, slots = qsa.topk_select(to_dev(w.scores), 2048, n_valid=to_dev(w.n_valid), n_max=80_000,
                                 page_table=to_dev(w.page_table), page_size=w.page_size)
    ref_idx, ref_slots = oracle.topk(w.scores, 2048, n_valid=w.n_valid, page_table=w.page_table,
                                     page_size=w.page_size)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)


def test_select_blocks_many_long_qsa_rows(qsa):
    """96 QSA rows of contexts between 131,073 and 200,000 tokens (more than
    32,768 blocks each) through qsa_select_blocks: the streaming CTA in QSA
    mode (top-512 blocks, expansion with 0-3 pending tokens, slots)."""
    rng = np.random.default_rng(62)
    lens = [int(x) for x in rng.integers(131_073, 200_001, size=96)]
    w = decode_workload(63, [[L] for L in lens], page_size=64, k_blk=512, with_keys=False)
    ld = (w.max_len // 4 + 3) // 4 * 4
    s = rng.standard_normal((w.n_rows, ld)).astype(np.float32)
    out = qsa.select_blocks(to_dev(s), to_dev(w.req_row_start), to_dev(w.row_len), to_dev(w.page_table),
                            w.page_size, w.max_len, k_blk=512, want_blocks=True, want_pos=True)
    sel_ref, _ = oracle.topk(s, 512, n_valid=w.row_len // 4)
    pos_ref, slots_ref = oracle.expand(sel_ref, w.req_row_start, w.row_len, w.page_table, w.page_size)
    assert np.array_equal(out["blocks"].cpu().numpy(), sel_ref)
    assert np.array_equal(out["pos"].cpu().numpy(), pos_ref)
    assert np.array_equal(out["slots"].cpu().numpy(), slots_ref)


# ----------------------------------------------------------------- boundary ties
@pytest.mark.parametrize("n", [3000, 20_000, 32_768])
@pytest.mark.parametrize("k", [512, 1000])
def test_topk_boundary_ties_take_lowest_indices(qsa, n, k):
    """Rows whose k-th largest value is shared by many entries on both sides
    of the cut (some taken, some not): the taken ones are the lowest indices.
    Row 0: k - 40 distinct large values, then 300 copies of one value spread
    over the row.  Row 1: the same with the copies at the front.  Row 2: a
    row of 5 distinct values (massive ties everywhere)."""
    rng = np.random.default_rng(n + k)
    s = (rng.standard_normal((3, n)) * 0.1).astype(np.float32)
    big = rng.permutation(n)[: k - 40]
    s[0, big] = 10.0 + rng.standard_normal(k - 40).astype(np.float32)
    rest = np.setdiff1d(np.arange(n), big)
    s[0, rng.choice(rest, 300, replace=False)] = 5.0
    s[1] = s[0]
    s[1, np.flatnonzero(s[0] == 5.0)] = 0.0
    s[1, rest[:300]] = 5.0
    s[2] = rng.integers(0, 5, n).astype(np.float32)
    nv = np.full(3, n, np.int32)
    idx, _ = qsa.topk_select(to_dev(s), k, n_valid=to_dev(nv), n_max=n)
    ref, _ = oracle.topk(s, k, n_valid=nv)
    assert np.array_equal(idx.cpu().numpy(), ref)


# ----------------------------------------------------------------- the headline step
@pytest.mark.parametrize("max_len", [None, 131_072])
def test_decode_step_c2_verify_against_the_oracle(qsa, max_len):
    """The 6-row verify step at L = 80,000 (rows at positions
    79,994..79,999), as one qsa_decode_step call on a pool holding blocks
    0..19,997 and a ring holding tokens 79,992..79,993.  Also with max_len
    past the rows (a capacity bound, as a captured graph would pass) and the
    table's pages past the rows unmapped: the one-request scorer then builds
    tiles past the rows, which must not fault."""
    import torch
    w = c2_verify(0)
    page_table = w.page_table
    if max_len is None:
        max_len = w.max_len
    else:  # the table covers max_len (the call's contract); pages past the rows unmapped
        page_table = np.full((1, (max_len + w.page_size - 1) // w.page_size), -1, np.int32)
        page_table[0, :w.page_table.shape[1]] = w.page_table[0]
    assert w.n_req == 1 and list(w.row_len) == [79_995 + i for i in range(6)]
    first, count = 79_994, 6
    nb0 = first // 4  # 19,998 blocks complete before the step
    ids = w.block_id
    order = np.argsort(ids)
    raw_tok = w.raw_keys.reshape(-1, 4, 128)[order].reshape(-1, 128)  # token order 0..79,999
    # the state before the step: blocks 0..19,997 compressed (oracle), ring slots 0, 1
    pool0 = np.zeros((w.pool_rows, 128), np.uint16)
    oracle.compress(raw_tok[: 4 * nb0], np.zeros(nb0, np.int32), np.arange(nb0, dtype=np.int32), w.page_table,
                    w.page_size, w.rope_base, pool0)
    ring0 = np.zeros((1, 4, 128), np.uint16)
    for p in range(4 * nb0, first):
        ring0[0, p % 4] = raw_tok[p]
    new = np.ascontiguousarray(raw_tok[first:first + count])
    rts = np.array([0, count], np.int32)
    fp = np.array([first], np.int32)
    # oracle key path
    ring_o, pool_o = oracle.append_keys(new, rts, fp, ring0.copy(), w.page_table, w.page_size, w.rope_base,
                                        pool0.copy())
    # one GPU call
    g_pool, g_ring = bf16_dev(pool0), bf16_dev(ring0)
    ld = (max_len // 4 + 3) // 4 * 4
    scores = torch.full((w.n_rows, ld), float("nan"), device="cuda")
    out = qsa.decode_step(bf16_dev(new), to_dev(rts), to_dev(fp), g_ring, bf16_dev(w.q), g_pool,
                          to_dev(w.req_row_start), to_dev(w.row_len), to_dev(page_table), w.page_size,
                          max_len, w.max_rows_per_req, k_blk=512, rope_base=w.rope_base, want_blocks=True,
                          want_pos=True, scores_out=scores)
    pool_g, ring_g = bf16_host(g_pool), bf16_host(g_ring)
    # ring: the last 4 appended tokens (bit copies)
    assert np.array_equal(ring_g, ring_o)
    # pool: blocks 19,998 and 19,999 written within the key bound, nothing else touched
    new_rows = [oracle.pool_row(w.page_table[0], b, w.page_size) for b in (nb0, nb0 + 1)]
    a_, b_ = oracle.bf16_to_float(pool_g[new_rows]), oracle.bf16_to_float(pool_o[new_rows])
    assert (np.abs(a_ - b_) <= key_tolerance(a_, b_)).all()
    others = np.setdiff1d(np.arange(w.pool_rows), new_rows)
    assert np.array_equal(pool_g[others], pool0[others])
    # scores against the oracle on the GPU's keys (the rule: fed identically)
    s = scores.cpu().numpy()
    want = oracle.index_scores(w.q, pool_g, w.req_row_start, w.row_len, w.page_table, w.page_size, ld)
    tol = score_tolerance(w.q, pool_g, w.req_row_start, w.row_len, w.page_table, w.page_size, ld)
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        err = np.abs(s[t, :nb].astype(np.float64) - want[t, :nb])
        assert (err <= tol[t, :nb]).all(), (t, float(err.max()))
    # selection, positions and slots bit-exact on the GPU's scores
    sel_ref, _ = oracle.topk(s, 512, n_valid=w.row_len // 4)
    pos_ref, slots_ref = oracle.expand(sel_ref, w.req_row_start, w.row_len, w.page_table, w.page_size)
    assert np.array_equal(out["blocks"].cpu().numpy(), sel_ref)
    assert np.array_equal(out["pos"].cpu().numpy(), pos_ref)
    assert np.array_equal(out["slots"].cpu().numpy(), slots_ref)


@pytest.mark.parametrize("rows,table", [([5003, 4099, 5000], "unmapped"), ([5003, 4099, 5000], "past_pool"),
                                        ([5003, 4099, 5000], "other_pages"), ([8190], "unmapped")])
def test_one_request_with_max_len_past_its_rows(qsa, rows, table):
    """One request scored and selected with max_len = 131,072, far past its
    rows (a capacity bound): the one-request scorer's tile list reaches the
    table's entries past the rows -- unmapped (-1), past the pool, or pages
    of other data.  No fault may fire, and scores, selection, positions and
    slots match the oracle."""
    import torch
    max_len = 131_072
    w = decode_workload(71 + len(rows), [rows], page_size=64, k_blk=512, pad_pages=40)
    pool_h = np.zeros((w.pool_rows, 128), np.uint16)
    oracle.compress(w.raw_keys, w.block_req, w.block_id, w.page_table, w.page_size, w.rope_base, pool_h)
    used = (max(rows) + w.page_size - 1) // w.page_size
    pt = np.full((1, max_len // w.page_size), -1, np.int32)
    pt[0, :used] = w.page_table[0, :used]
    if table == "past_pool":
        pt[0, used:] = 1 << 30
    elif table == "other_pages":
        pt[0, used:] = np.random.default_rng(5).integers(0, w.pool_rows * 4 // w.page_size, size=pt.shape[1] - used)
    ld = (max_len // 4 + 3) // 4 * 4
    scores = torch.full((w.n_rows, ld), float("nan"), device="cuda")
    out = qsa.indexer_select(bf16_dev(w.q), bf16_dev(pool_h), to_dev(w.req_row_start), to_dev(w.row_len),
                             to_dev(pt), w.page_size, max_len, w.max_rows_per_req, k_blk=512,
                             want_blocks=True, want_pos=True, scores_out=scores)
    s = scores.cpu().numpy()
    want = oracle.index_scores(w.q, pool_h, w.req_row_start, w.row_len, pt, w.page_size, ld)
    tol = score_tolerance(w.q, pool_h, w.req_row_start, w.row_len, pt, w.page_size, ld)
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        err = np.abs(s[t, :nb].astype(np.float64) - want[t, :nb])
        assert (err <= tol[t, :nb]).all(), (t, float(err.max()))
    sel_ref, _ = oracle.topk(s, 512, n_valid=w.row_len // 4)
    pos_ref, slots_ref = oracle.expand(sel_ref, w.req_row_start, w.row_len, pt, w.page_size)
    assert np.array_equal(out["blocks"].cpu().numpy(), sel_ref)
    assert np.array_equal(out["pos"].cpu().numpy(), pos_ref)
    assert np.array_equal(out["slots"].cpu().numpy(), slots_ref)


# ----------------------------------------------------------------- per-row plan
def _mixed_rows(rng, n_short, lengths_long, short_lo=3000, short_hi=30_000):
    lens = np.concatenate([lengths_long, rng.integers(short_lo, short_hi, size=n_short)]).astype(np.int32)
    return rng.permutation(lens).astype(np.int32)


@pytest.mark.parametrize("k,with_slots", [(2048, True), (512, False)])
def test_topk_mixed_lengths_take_the_row_plan(qsa, k, with_slots):
    """One call with a 1M-entry row, four 80,000-entry rows and 100 short
    rows (3,000-30,000), in random order: the device plan sends the five long
    rows to clusters sized from their count and the short ones to one CTA
    each.  Bit-exact against the oracle, slots included."""
    rng = np.random.default_rng(k)
    nv = _mixed_rows(rng, 100, [1_000_000, 80_000, 80_000, 80_000, 80_000])
    ld = int(nv.max())
    s = rng.standard_normal((nv.size, ld), dtype=np.float32)
    P = 64
    pt = np.stack([rng.permutation((ld + P - 1) // P) for _ in range(nv.size)]).astype(np.int32)
    idx, slots = qsa.topk_select(to_dev(s), k, n_valid=to_dev(nv), n_max=ld,
                                 page_table=to_dev(pt) if with_slots else None, page_size=P)
    ref_idx, ref_slots = oracle.topk(s, k, n_valid=nv, page_table=pt if with_slots else None, page_size=P)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    if with_slots:
        assert np.array_equal(slots.cpu().numpy(), ref_slots)


def test_indexer_mixed_contexts_take_the_row_plan(qsa):
    """The fused indexer on 80 one-row requests, two of them with contexts
    past 131K tokens (more than 32,768 blocks) among short ones, with a
    workspace (so the device plan runs): the selection, positions and slots
    bit-exact against the oracle on the GPU's scores."""
    import torch
    rng = np.random.default_rng(71)
    lens = _mixed_rows(rng, 78, [150_001, 199_998], 4096, 40_000)
    w = decode_workload(72, [[int(L)] for L in lens], page_size=64, k_blk=512, with_keys=False)
    pool = torch.randn((w.pool_rows, 128), device="cuda").to(torch.bfloat16)
    ld = (w.max_len // 4 + 3) // 4 * 4
    scores = torch.full((w.n_rows, ld), float("nan"), device="cuda")
    ws = torch.empty(qsa.indexer_select_workspace_size(w.n_rows, w.max_len, 512), dtype=torch.uint8,
                     device="cuda")
    out = qsa.indexer_select(bf16_dev(w.q), pool, to_dev(w.req_row_start), to_dev(w.row_len),
                             to_dev(w.page_table), w.page_size, w.max_len, w.max_rows_per_req, k_blk=512,
                             want_blocks=True, want_pos=True, scores_out=scores, workspace=ws)
    s = scores.cpu().numpy()
    sel_ref, _ = oracle.topk(s, 512, n_valid=w.row_len // 4)
    pos_ref, slots_ref = oracle.expand(sel_ref, w.req_row_start, w.row_len, w.page_table, w.page_size)
    assert np.array_equal(out["blocks"].cpu().numpy(), sel_ref)
    assert np.array_equal(out["pos"].cpu().numpy(), pos_ref)
    assert np.array_equal(out["slots"].cpu().numpy(), slots_ref)


# ----------------------------------------------------------------- many rows, k <= 512
def _group_sample_positions(n):
    """256 evenly spaced groups of 4 entries: groups floor(j * (n // 4) / 256)
    (a sampled bound read there would sit far above the k-th entry)."""
    g = (np.arange(256, dtype=np.int64) * (n // 4)) // 256
    return (4 * g[:, None] + np.arange(4)).ravel()


@pytest.mark.parametrize("n", [1000, 1537, 3001, 20_000, 32_768])
def test_topk_many_rows_k_up_to_512(qsa, n):
    """More than two rows per SM with k <= 512 (small CTAs).  Ordinary rows,
    rows of one value, three values, one top-bits bin, rows whose evenly
    spaced groups hold the largest values, rows with NaN, +-inf and -0,
    ragged lengths (n not a multiple of 4, fewer entries than k); token mode
    with slots."""
    rng = np.random.default_rng(n + 11)
    rows = []
    for r in range(336):
        kind = r % 6
        if kind == 0:
            x = np.full(n, 1.5, np.float32)
        elif kind == 1:
            x = rng.integers(0, 3, size=n).astype(np.float32)
        elif kind == 2:
            x = (rng.integers(0, 64, size=n) / 64.0 + 1.0).astype(np.float32)
        elif kind == 3:
            x = (rng.standard_normal(n) * 0.01).astype(np.float32)
            x[_group_sample_positions(n)] = 100.0 + rng.standard_normal(1024).astype(np.float32)
        elif kind == 4:
            x = rng.standard_normal(n).astype(np.float32)
            x[rng.choice(n, 40, replace=False)] = np.nan
            x[rng.choice(n, 3, replace=False)] = np.inf
            x[rng.choice(n, 3, replace=False)] = -np.inf
            x[rng.choice(n, 50, replace=False)] = -0.0
            x[rng.choice(n, 50, replace=False)] = 0.0
        else:
            x = rng.standard_normal(n).astype(np.float32)
        rows.append(x)
    s = np.stack(rows)
    nv = np.full(s.shape[0], n, np.int32)
    nv[5] = 100                # fewer entries than k
    nv[11] = n - 3             # ragged tail
    nv[17] = n - 1
    nv[23] = 0
    P = 64
    pt = np.stack([rng.permutation((n + P - 1) // P) for _ in range(s.shape[0])]).astype(np.int32)
    for k in [1, 100, 512]:
        idx, slots = qsa.topk_select(to_dev(s), k, n_valid=to_dev(nv), n_max=n, page_table=to_dev(pt),
                                     page_size=P)
        ref, ref_slots = oracle.topk(s, k, n_valid=nv, page_table=pt, page_size=P)
        assert np.array_equal(idx.cpu().numpy(), ref), k
        assert np.array_equal(slots.cpu().numpy(), ref_slots), k


def test_select_blocks_many_qsa_rows(qsa):
    """400 one-row requests, contexts 1..131,072 tokens (every pending count,
    rows with fewer blocks than k), top-512 blocks expanded to positions and
    slots through the requests' page tables: bit-exact."""
    rng = np.random.default_rng(91)
    lens = rng.integers(1, 131_073, size=400)
    lens[:8] = [1, 3, 4, 2047, 2048, 2051, 6147, 131_072]
    w = decode_workload(92, [[int(L)] for L in lens], page_size=64, k_blk=512, with_keys=False)
    ld = (w.max_len // 4 + 3) // 4 * 4
    s = rng.standard_normal((w.n_rows, ld)).astype(np.float32)
    out = qsa.select_blocks(to_dev(s), to_dev(w.req_row_start), to_dev(w.row_len), to_dev(w.page_table),
                            w.page_size, w.max_len, k_blk=512, want_blocks=True, want_pos=True)
    sel_ref, _ = oracle.topk(s, 512, n_valid=w.row_len // 4)
    pos_ref, slots_ref = oracle.expand(sel_ref, w.req_row_start, w.row_len, w.page_table, w.page_size)
    assert np.array_equal(out["blocks"].cpu().numpy(), sel_ref)
    assert np.array_equal(out["pos"].cpu().numpy(), pos_ref)
    assert np.array_equal(out["slots"].cpu().numpy(), slots_ref)


def test_planned_selection_in_a_cuda_graph(qsa):
    """The planned selection forks its short rows onto a side stream and
    joins them back: recorded in a CUDA graph (after one eager call) and
    replayed on new scores, it matches the oracle every time."""
    import torch
    rng = np.random.default_rng(95)
    nv = _mixed_rows(rng, 80, [100_000, 40_000, 40_000, 40_000], 3000, 8000)
    ld = int(nv.max())
    P = 64
    pt = np.stack([rng.permutation((ld + P - 1) // P) for _ in range(nv.size)]).astype(np.int32)
    k = 2048
    s_dev = torch.empty((nv.size, ld), dtype=torch.float32, device="cuda")
    nv_dev, pt_dev = to_dev(nv), to_dev(pt)
    ws = torch.empty(qsa.lib().topk_select_workspace_size(nv.size, ld, k), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    idx = torch.empty((nv.size, k), dtype=torch.int32, device="cuda")
    slots = torch.empty((nv.size, k), dtype=torch.int32, device="cuda")

    def call():
        qsa.topk_select(s_dev, k, n_valid=nv_dev, n_max=ld, page_table=pt_dev, page_size=P, out_idx=idx,
                        out_slots=slots, workspace=ws)

    s_dev.copy_(torch.from_numpy(rng.standard_normal((nv.size, ld), dtype=np.float32)))
    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    torch.cuda.synchronize()
    for rep in range(2):
        s = rng.standard_normal((nv.size, ld), dtype=np.float32)
        s_dev.copy_(torch.from_numpy(s))
        graph.replay()
        torch.cuda.synchronize()
        ref_idx, ref_slots = oracle.topk(s, k, n_valid=nv, page_table=pt, page_size=P)
        assert np.array_equal(idx.cpu().numpy(), ref_idx), rep
        assert np.array_equal(slots.cpu().numpy(), ref_slots), rep
