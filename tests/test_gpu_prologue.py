"""GPU parity of the prologue tails against the oracle (SGLang GLM-5.2 blog,
"Indexer Prologue Fusion"): the index-query RoPE, the FP8 key quantiser,
the FP8-key scorer and the fused selection on FP8 keys, and the head-gated
score on every scorer.

- RoPE: within one BF16 ulp plus the FP32 rotation's absolute term
  2^-22 (|u| + |v|) per pair (both sides round once to BF16; the GPU's sine
  and cosine and its products are FP32); in place equals out of place to the
  bit; a negative position latches the grouping fault and leaves the row.
- Quantiser: codes and scales bit-exact (both take the same FP32 divisions
  and one round-to-nearest-even to e4m3).
- Scores: within 2e-5 * (1/sqrt(128)) * sum |f16(q) * code * scale| + 1e-6
  of the oracle's FP64 score on the same codes (the GPU multiplies exact
  FP16 x e4m3 products and accumulates in FP32).
- Selection, positions and slots: bit-exact against the oracle on the GPU's
  scores, at small ragged shapes and at the full 32-request batch
  (contexts 4,096..131,072).
"""
import numpy as np
import pytest

import oracle
from gpu_util import SCALE, bf16_dev, bf16_host, key_tolerance, pool_rows_of, to_dev
from workloads import c3_batched, decode_workload, normal_bf16

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


def _deq(codes, scales):
    table = np.array([oracle.e4m3_to_float(c) for c in range(256)])
    return table[codes] * scales[:, None].astype(np.float64)


def fp8_score_tolerance(q_bits, codes, scales, req_row_start, row_len, page_table, page_size, ld):
    qa = np.abs(oracle.bf16_to_float(q_bits)).astype(np.float64).sum(axis=1)  # [n_rows][128]
    tol = np.full((row_len.size, ld), np.inf)
    for r in range(req_row_start.size - 1):
        rows = np.arange(req_row_start[r], req_row_start[r + 1])
        if rows.size == 0:
            continue
        nb = int(row_len[rows].max()) // 4
        prow = pool_rows_of(page_table[r], nb, page_size)
        ka = np.abs(_deq(codes[prow], scales[prow]))
        tol[rows, :nb] = 2e-5 * SCALE * (qa[rows] @ ka.T) + 1e-6
    return tol


# ----------------------------------------------------------------- query RoPE
def test_rope_queries_parity(qsa):
    """37 rows (148 (row, head) units: 5 CTAs, the last ragged) at positions
    from 0 to 2^20, against the oracle's FP64 rotation."""
    rng = np.random.default_rng(81)
    n = 37
    q = normal_bf16(rng, (n, 4, 128))
    q[3] *= 0  # a zero row stays zero
    pos = rng.integers(0, 1 << 20, size=n).astype(np.int32)
    pos[:5] = [0, 1, 79_999, 131_071, (1 << 20) - 1]
    got = bf16_host(qsa.rope_queries(bf16_dev(q), to_dev(pos)))
    want = oracle.rope_queries(q, pos)
    a, b = oracle.bf16_to_float(got).astype(np.float64), oracle.bf16_to_float(want).astype(np.float64)
    u = np.abs(oracle.bf16_to_float(q)).astype(np.float64)
    pair = u[..., :64] + u[..., 64:]
    tol = key_tolerance(a, b) - 2.0 ** -22 + 2.0 ** -22 * np.concatenate([pair, pair], axis=-1)
    assert (np.abs(a - b) <= tol).all(), float(np.abs(a - b).max())
    assert np.array_equal(got[0], q[0])          # position 0: identity, to the bit
    assert (a[3] == 0).all()                     # (either sign of zero)


def test_rope_queries_in_place_and_negative_position(qsa):
    import torch
    rng = np.random.default_rng(82)
    q = normal_bf16(rng, (9, 4, 128))
    pos = rng.integers(0, 200_000, size=9).astype(np.int32)
    ref = bf16_host(qsa.rope_queries(bf16_dev(q), to_dev(pos)))
    g = bf16_dev(q)
    qsa.rope_queries(g, to_dev(pos), out=g)
    assert np.array_equal(bf16_host(g), ref)
    # a negative position: the fault bit, that row untouched, the others rotated
    pos_bad = pos.copy()
    pos_bad[4] = -1
    out = torch.zeros((9, 4, 128), dtype=torch.bfloat16, device="cuda")
    qsa.rope_queries(bf16_dev(q), to_dev(pos_bad), out=out)
    assert qsa.device_status(clear=True) != 0
    got = bf16_host(out)
    assert (got[4] == 0).all()
    keep = np.arange(9) != 4
    assert np.array_equal(got[keep], ref[keep])


# ----------------------------------------------------------------- quantiser
@pytest.mark.parametrize("n", [1, 31, 1003])
def test_quantize_keys_fp8_bit_exact(qsa, n):
    rng = np.random.default_rng(83 + n)
    keys = normal_bf16(rng, (n, 128))
    if n > 8:
        keys[1] = 0                                                    # zero key: scale 0
        keys[2] = oracle.bf16_round_array(rng.standard_normal(128) * 1e-38)  # subnormal scale
        keys[3] = oracle.bf16_round_array(rng.standard_normal(128) * 1e30)
        keys[4] = oracle.bf16_round_array(np.full(128, -0.5))             # every element at the max
    codes, scales = qsa.quantize_keys_fp8(bf16_dev(keys))
    ref_c, ref_s = oracle.quantize_keys_fp8(keys)
    assert np.array_equal(codes.cpu().numpy(), ref_c)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


# ----------------------------------------------------------------- scores
def _fp8_case(qsa, seed, rows_per_req, page_size):
    w = decode_workload(seed, rows_per_req, page_size=page_size, with_keys=False)
    rng = np.random.default_rng(seed + 1)
    pool = normal_bf16(rng, (w.pool_rows, 128))
    codes, scales = qsa.quantize_keys_fp8(bf16_dev(pool))
    return w, codes, scales


@pytest.mark.parametrize("layout", ["mixed_rows", "one_row"])
@pytest.mark.parametrize("page_size", [32, 64])
def test_index_scores_fp8_parity(qsa, page_size, layout):
    """Requests of 1..8 rows (16-key tiles), or of one row each (32-key
    tiles: two or four pages per tile), contexts with ragged tails (several
    tiles plus a partial one, contexts shorter than one tile), n_fill past
    the longest row."""
    import torch
    if layout == "mixed_rows":
        rows = [[1000], [37, 40, 41], [4096 + 4 * i for i in range(8)], [9001, 9002], [12], [2051] * 5]
    else:
        rows = [[L] for L in [12, 37, 128, 129, 1000, 2051, 4096, 4100, 9001, 40_003]]
    w, codes, scales = _fp8_case(qsa, 84, rows, page_size)
    ld = (w.max_len // 4 + 3) // 4 * 4 + 8
    s = qsa.index_scores_fp8(bf16_dev(w.q), codes, scales, to_dev(w.req_row_start), to_dev(w.row_len),
                             to_dev(w.page_table), page_size, w.max_len, w.max_rows_per_req,
                             scores=torch.full((w.n_rows, ld), float("nan"), device="cuda"),
                             n_fill=ld - 3).cpu().numpy()
    c, sc = codes.cpu().numpy(), scales.cpu().numpy()
    want = oracle.index_scores_fp8(w.q, c, sc, w.req_row_start, w.row_len, w.page_table, page_size, ld)
    tol = fp8_score_tolerance(w.q, c, sc, w.req_row_start, w.row_len, w.page_table, page_size, ld)
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        err = np.abs(s[t, :nb].astype(np.float64) - want[t, :nb])
        assert (err <= tol[t, :nb]).all(), (t, float(err.max()))
        assert (s[t, nb:ld - 3] == -np.inf).all()
        assert np.isnan(s[t, ld - 3:]).all()


def test_index_scores_fp8_rejects_unsupported_shapes(qsa):
    w, codes, scales = _fp8_case(qsa, 85, [[256]], 64)
    args = (bf16_dev(w.q), codes, scales, to_dev(w.req_row_start), to_dev(w.row_len), to_dev(w.page_table))
    with pytest.raises(qsa.QSAError):
        qsa.index_scores_fp8(*args, 16, w.max_len)            # 4 keys per page
    w9, c9, s9 = _fp8_case(qsa, 86, [[256] * 9], 64)
    with pytest.raises(qsa.QSAError):                          # 9 rows in one request
        qsa.index_scores_fp8(bf16_dev(w9.q), c9, s9, to_dev(w9.req_row_start), to_dev(w9.row_len),
                             to_dev(w9.page_table), 64, w9.max_len)


# ----------------------------------------------------------------- fused selection
def _check_selection(out, s, w, k_blk):
    sel_ref, _ = oracle.topk(s, k_blk, n_valid=w.row_len // 4)
    pos_ref, slots_ref = oracle.expand(sel_ref, w.req_row_start, w.row_len, w.page_table, w.page_size)
    assert np.array_equal(out["blocks"].cpu().numpy(), sel_ref)
    assert np.array_equal(out["pos"].cpu().numpy(), pos_ref)
    assert np.array_equal(out["slots"].cpu().numpy(), slots_ref)


def test_indexer_select_fp8_small(qsa):
    import torch
    rows = [[3000 + i for i in range(6)], [513], [2047, 2048, 2049], [40_003]]
    w, codes, scales = _fp8_case(qsa, 87, rows, 64)
    ld = (w.max_len // 4 + 3) // 4 * 4
    scores = torch.full((w.n_rows, ld), float("nan"), device="cuda")
    out = qsa.indexer_select_fp8(bf16_dev(w.q), codes, scales, to_dev(w.req_row_start), to_dev(w.row_len),
                                 to_dev(w.page_table), w.page_size, w.max_len, w.max_rows_per_req, k_blk=512,
                                 want_blocks=True, want_pos=True, scores_out=scores)
    s = scores.cpu().numpy()
    c, sc = codes.cpu().numpy(), scales.cpu().numpy()
    want = oracle.index_scores_fp8(w.q, c, sc, w.req_row_start, w.row_len, w.page_table, w.page_size, ld)
    tol = fp8_score_tolerance(w.q, c, sc, w.req_row_start, w.row_len, w.page_table, w.page_size, ld)
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        assert (np.abs(s[t, :nb].astype(np.float64) - want[t, :nb]) <= tol[t, :nb]).all(), t
    _check_selection(out, s, w, 512)
    # without scores_out (the workspace holds them): the same selection
    out2 = qsa.indexer_select_fp8(bf16_dev(w.q), codes, scales, to_dev(w.req_row_start), to_dev(w.row_len),
                                  to_dev(w.page_table), w.page_size, w.max_len, w.max_rows_per_req, k_blk=512,
                                  want_blocks=True, want_pos=True)
    assert np.array_equal(out2["slots"].cpu().numpy(), out["slots"].cpu().numpy())


def test_indexer_select_fp8_full_batch(qsa):
    """The 32-request batch (one row each, contexts 4,096..131,072 tokens):
    scores against the oracle on the GPU's codes, selection bit-exact."""
    import torch
    w = c3_batched(0, with_keys=False)
    rng = np.random.default_rng(88)
    pool = normal_bf16(rng, (w.pool_rows, 128))
    codes, scales = qsa.quantize_keys_fp8(bf16_dev(pool))
    ld = (w.max_len // 4 + 3) // 4 * 4
    scores = torch.full((w.n_rows, ld), float("nan"), device="cuda")
    out = qsa.indexer_select_fp8(bf16_dev(w.q), codes, scales, to_dev(w.req_row_start), to_dev(w.row_len),
                                 to_dev(w.page_table), w.page_size, w.max_len, 1, k_blk=512,
                                 want_blocks=True, want_pos=True, scores_out=scores)
    s = scores.cpu().numpy()
    c, sc = codes.cpu().numpy(), scales.cpu().numpy()
    ref_c, ref_s = oracle.quantize_keys_fp8(pool)
    assert np.array_equal(c, ref_c) and np.array_equal(sc.view(np.uint32), ref_s.view(np.uint32))
    want = oracle.index_scores_fp8(w.q, c, sc, w.req_row_start, w.row_len, w.page_table, w.page_size, ld)
    tol = fp8_score_tolerance(w.q, c, sc, w.req_row_start, w.row_len, w.page_table, w.page_size, ld)
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        assert (np.abs(s[t, :nb].astype(np.float64) - want[t, :nb]) <= tol[t, :nb]).all(), t
    _check_selection(out, s, w, 512)


# ----------------------------------------------------------------- head gates
def gated_score_tolerance(q_bits, gates, pool_bits, req_row_start, row_len, page_table, page_size, ld):
    """2e-5 * (1/sqrt(128)) * sum_{h,d} |g_h q_hd kbar_d| + 1e-6: the score
    bound with each head's terms weighted by |gate|."""
    qa = np.abs(oracle.bf16_to_float(q_bits)).astype(np.float64)  # [rows][4][128]
    qa = (qa * np.abs(gates)[:, :, None]).sum(axis=1)             # [rows][128]
    tol = np.full((row_len.size, ld), np.inf)
    for r in range(req_row_start.size - 1):
        rows = np.arange(req_row_start[r], req_row_start[r + 1])
        if rows.size == 0:
            continue
        nb = int(row_len[rows].max()) // 4
        prow = pool_rows_of(page_table[r], nb, page_size)
        ka = np.abs(oracle.bf16_to_float(pool_bits[prow])).astype(np.float64)
        tol[rows, :nb] = 2e-5 * SCALE * (qa[rows] @ ka.T) + 1e-6
    return tol


@pytest.mark.parametrize("layout,page_size", [("decode_rows", 64), ("prefill_rows", 64), ("one_row_small_pages", 16)])
def test_gated_scores_and_selection(qsa, layout, page_size):
    """Gated scores on each scorer (requests of up to 8 rows: the mma.sync
    decode scorer; a request of 100 rows: the tcgen05 scorer; one-row
    requests on 16-token pages: the CUDA-core scorer) against the oracle,
    gates drawn in [-1, 2] (some negative); the fused gated call's selection
    bit-exact on its own scores; unit gates give the ungated scores to the
    bit."""
    import torch
    if layout == "decode_rows":
        rows = [[3001 + i for i in range(6)], [513], [2047, 2048, 2049], [20_003]]
    elif layout == "prefill_rows":
        rows = [[5000 + i for i in range(100)]]
    else:
        rows = [[L] for L in [37, 1000, 4099, 12_001]]
    w = decode_workload(96, rows, page_size=page_size, with_keys=False)
    rng = np.random.default_rng(97)
    pool_h = normal_bf16(rng, (w.pool_rows, 128))
    gates = rng.uniform(-1, 2, (w.n_rows, 4)).astype(np.float32)
    pool = bf16_dev(pool_h)
    args = (to_dev(w.req_row_start), to_dev(w.row_len), to_dev(w.page_table), w.page_size, w.max_len,
            w.max_rows_per_req)
    ld = (w.max_len // 4 + 3) // 4 * 4
    s = qsa.index_scores_gated(bf16_dev(w.q), to_dev(gates), pool, *args,
                               scores=torch.full((w.n_rows, ld), float("nan"), device="cuda")).cpu().numpy()
    want = oracle.index_scores_gated(w.q, gates, pool_h, w.req_row_start, w.row_len, w.page_table, w.page_size, ld)
    tol = gated_score_tolerance(w.q, gates, pool_h, w.req_row_start, w.row_len, w.page_table, w.page_size, ld)
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        err = np.abs(s[t, :nb].astype(np.float64) - want[t, :nb])
        assert (err <= tol[t, :nb]).all(), (t, float(err.max()))
    # fused call: selection bit-exact on its scores
    scores = torch.full((w.n_rows, ld), float("nan"), device="cuda")
    out = qsa.indexer_select_gated(bf16_dev(w.q), to_dev(gates), pool, *args, k_blk=512, want_blocks=True,
                                   want_pos=True, scores_out=scores)
    sg = scores.cpu().numpy()
    sel_ref, _ = oracle.topk(sg, 512, n_valid=w.row_len // 4)
    pos_ref, slots_ref = oracle.expand(sel_ref, w.req_row_start, w.row_len, w.page_table, w.page_size)
    assert np.array_equal(out["blocks"].cpu().numpy(), sel_ref)
    assert np.array_equal(out["pos"].cpu().numpy(), pos_ref)
    assert np.array_equal(out["slots"].cpu().numpy(), slots_ref)
    # unit gates: the ungated scores, to the bit
    s1 = qsa.index_scores_gated(bf16_dev(w.q), torch.ones((w.n_rows, 4), device="cuda"), pool, *args,
                                scores=torch.full((w.n_rows, ld), float("nan"), device="cuda")).cpu().numpy()
    s0 = qsa.index_scores(bf16_dev(w.q), pool, *args,
                          scores=torch.full((w.n_rows, ld), float("nan"), device="cuda")).cpu().numpy()
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        assert np.array_equal(s1[t, :nb].view(np.uint32), s0[t, :nb].view(np.uint32)), t


def test_gated_decode_step_equals_append_then_gated_indexer(qsa):
    """qsa_decode_step_gated (key path, then the gated fused indexer) gives
    the same pool, ring, scores and slots as qsa_append_keys followed by
    qsa_indexer_select_gated."""
    import torch
    rows, P = [[20_000 - 5 + i for i in range(6)], [5003], [777]], 64
    rng = np.random.default_rng(98)
    w = decode_workload(99, rows, page_size=P, k_blk=512)
    n_req = w.n_req
    firsts = np.array([min(r) - 1 for r in rows], np.int32)
    counts = np.array([len(r) for r in rows], np.int32)
    raw = [normal_bf16(rng, (int(f + c), 128)) for f, c in zip(firsts, counts)]
    ring0 = np.zeros((n_req, 4, 128), np.uint16)
    blocks, reqs, raws = [], [], []
    for r in range(n_req):
        nb0 = int(firsts[r]) // 4
        blocks.append(np.arange(nb0, dtype=np.int32))
        reqs.append(np.full(nb0, r, np.int32))
        raws.append(raw[r][:4 * nb0])
        for p in range(4 * nb0, int(firsts[r])):
            ring0[r, p % 4] = raw[r][p]
    pool0 = torch.zeros((w.pool_rows, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(bf16_dev(np.concatenate(raws)), to_dev(np.concatenate(blocks)), pool0,
                      block_req=to_dev(np.concatenate(reqs)), page_table=to_dev(w.page_table), page_size=P)
    new = np.concatenate([raw[r][firsts[r]:] for r in range(n_req)])
    rts = to_dev(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32))
    fp, pt = to_dev(firsts), to_dev(w.page_table)
    q, rrs, rl = bf16_dev(w.q), to_dev(w.req_row_start), to_dev(w.row_len)
    gates = to_dev(rng.uniform(-1, 2, (w.n_rows, 4)).astype(np.float32))
    ld = (w.max_len // 4 + 3) // 4 * 4
    ring_a, pool_a = bf16_dev(ring0), pool0.clone()
    sa = torch.full((w.n_rows, ld), float("nan"), device="cuda")
    qsa.append_keys(bf16_dev(new), rts, fp, ring_a, pool_a, pt, P)
    out_a = qsa.indexer_select_gated(q, gates, pool_a, rrs, rl, pt, P, w.max_len, w.max_rows_per_req, k_blk=512,
                                     want_blocks=True, want_pos=True, scores_out=sa)
    ring_b, pool_b = bf16_dev(ring0), pool0.clone()
    sb = torch.full((w.n_rows, ld), float("nan"), device="cuda")
    out_b = qsa.decode_step(bf16_dev(new), rts, fp, ring_b, q, pool_b, rrs, rl, pt, P, w.max_len,
                            w.max_rows_per_req, k_blk=512, want_blocks=True, want_pos=True, scores_out=sb,
                            head_gates=gates)
    assert torch.equal(ring_a, ring_b) and torch.equal(pool_a, pool_b)
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        assert torch.equal(sa[t, :nb].view(torch.int32), sb[t, :nb].view(torch.int32)), t
    for key in ("slots", "blocks", "pos"):
        assert torch.equal(out_a[key], out_b[key]), key
    sel_ref, _ = oracle.topk(sb.cpu().numpy(), 512, n_valid=w.row_len // 4)
    assert np.array_equal(out_b["blocks"].cpu().numpy(), sel_ref)
