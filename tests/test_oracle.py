"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- the hand-worked example, closed forms, textbook identities,
a library routine in a special case, brute force on tiny inputs, or
invariants -- chosen so that a dropped term, a wrong sign or index, or a
transposed operand fails at least one of them.

Passages: Qwen3.8-Flash-Next day-0 write-up (theainews.cc), section "Qwen
sparse attention (QSA)" (compressed key, score equation, 512-block budget,
pending tokens, full_slot/4); SGLang GLM-5.2 blog, section "TopK-V2",
Figures 2-4 (exact top-k, page-table transform); vllm-sparse-mla-blackwell,
"Design notes worth knowing" (index >= 0 mask, -1 sentinel).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from workloads import bf16_bits, decode_workload, normal_bf16, topk_workload, TOPK_DISTS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D = 128


def f2b(x):
    """float -> BF16 bits via the generator's FP32 rounding (input prep only)."""
    return bf16_bits(np.asarray(x, np.float32))


def bf16_ulp(x):
    x = abs(float(x))
    if x == 0.0:
        return 2.0 ** -133
    e = math.frexp(x)[1]
    return 2.0 ** max(e - 8, -133)


# ----------------------------------------------------------------- BF16 rounding
def test_bf16_round_matches_torch_on_fp32_values():
    """Special case reducing to a library routine: for values that are exact in
    FP32, one-step FP64->BF16 rounding equals torch's FP32->BF16 RNE."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    # exact halfway cases: BF16 value plus half an ulp, both parities
    base = bf16_bits(rng.standard_normal(2000).astype(np.float32)).astype(np.uint32) << 16
    halfway = (base | 0x8000).view(np.float32)
    tiny = (rng.standard_normal(500) * 1e-39).astype(np.float32)  # FP32 subnormals
    allx = np.concatenate([x, halfway, tiny, np.array([0.0, -0.0, 1.0, -2.5], np.float32)])
    want = torch.from_numpy(allx).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round_array(allx.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_round_double_rounding_case():
    """One-step rounding from FP64: a value just above a BF16 halfway point
    must round up even though FP32 rounding would land exactly on the tie."""
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40   # tie in FP32 (rounds to even = 1.0 via FP32), above tie in FP64
    assert oracle.bf16_round(x) == 0x3F81
    assert oracle.bf16_round(1.0 + 2.0 ** -8) == 0x3F80  # exact tie -> even


# ----------------------------------------------------------------- hand example
def _golden_raw(g):
    raw = np.zeros((3 * 4, D), np.float32)
    for b, dims in g["raw_keys"].items():
        for d, vals in dims.items():
            raw[int(b) * 4: int(b) * 4 + 4, int(d)] = vals
    return f2b(raw)


def _golden_q(g):
    q = np.zeros((1, 4, D), np.float32)
    for h, e in enumerate(g["q_heads_unit_dims"]):
        if e is not None:
            q[0, h, e[0]] = e[1]
    return f2b(q)


def test_hand_example_keys_and_pool_rows():
    g = json.load(open(os.path.join(GOLDEN, "qsa_3block.json")))
    pt = np.array([g["page_table"]], np.int32)
    P = g["page_size"]
    pool = np.zeros((pt.size * P // 4, D), np.uint16)
    oracle.compress(_golden_raw(g), np.zeros(3, np.int32), np.arange(3, dtype=np.int32), pt, P,
                    g["rope_base"], pool)
    for b, (c, s) in enumerate(g["keys_dim0_dim64"]):
        row = g["pool_rows"][b]
        assert oracle.pool_row(pt[0], b, P) == row
        key = oracle.bf16_to_float(pool[row])
        expect = np.zeros(D)
        expect[0], expect[64] = c, s
        assert np.array_equal(key, expect), (b, key[[0, 1, 64]])
    # the pool row not owned by any block stays untouched
    assert not pool[1].any()


def test_hand_example_scores_selection_slots():
    g = json.load(open(os.path.join(GOLDEN, "qsa_3block.json")))
    pt = np.array([g["page_table"]], np.int32)
    P = g["page_size"]
    pool = np.zeros((pt.size * P // 4, D), np.uint16)
    oracle.compress(_golden_raw(g), np.zeros(3, np.int32), np.arange(3, dtype=np.int32), pt, P,
                    g["rope_base"], pool)
    q = _golden_q(g)
    rrs = np.array([0, 1], np.int32)
    rl = np.array([g["row_len"]], np.int32)
    out = oracle.indexer_select(q, pool, rrs, rl, pt, P, k_blk=g["k_blk"])
    want = np.array([eval(e, {"sqrt": math.sqrt}) for e in g["scores_expr"]], np.float32)
    assert np.array_equal(out["scores"][0, :3], want)
    assert out["blocks"][0].tolist() == g["selected_blocks"]
    assert out["pos"][0].tolist() == g["positions"]
    assert out["slots"][0].tolist() == g["slots"]


# ----------------------------------------------------------------- compression
def _theta(p, i, base=10000.0):
    return p * base ** (-2.0 * i / 128.0)


@pytest.mark.parametrize("p", [0, 1, 4, 100, 8188, 79996, 131068])
@pytest.mark.parametrize("j", [0, 1, 5, 31, 63, 64, 65, 100, 127])
def test_rope_closed_form_on_basis_vectors(p, j):
    """All four raw keys = e_j: the normalised mean is e_j and RoPE rotates it
    in the (i, i+64) plane by p * 10000^(-2i/128), i = j mod 64."""
    raw = np.zeros((4, D), np.float32)
    raw[:, j] = 1.0
    key = oracle.bf16_to_float(oracle.compress_block(f2b(raw), p))
    i = j % 64
    c, s = math.cos(_theta(p, i)), math.sin(_theta(p, i))
    expect = np.zeros(D)
    if j < 64:
        expect[i], expect[i + 64] = c, s
    else:
        expect[i], expect[i + 64] = -s, c
    for d in range(D):
        assert abs(key[d] - expect[d]) <= 0.5 * bf16_ulp(expect[d]) + 1e-300, (d, key[d], expect[d])


def test_compress_position_zero_is_normalised_mean():
    """p = 0: RoPE is the identity; each key is m/||m|| rounded once to BF16.
    Raw keys are chosen so that the FP32 block sum is exact."""
    rng = np.random.default_rng(1)
    for _ in range(50):
        raw = (rng.integers(-64, 65, size=(4, D)) / 16.0).astype(np.float32)
        m = raw.astype(np.float64).sum(0) / 4
        u = m / np.linalg.norm(m)
        got = oracle.bf16_to_float(oracle.compress_block(f2b(raw), 0))
        want = oracle.bf16_to_float(oracle.bf16_round_array(u))
        assert np.array_equal(got, want)


def test_compress_invariants():
    """Symmetric in the four raw keys, invariant to a common power-of-two
    scale, unit norm, and a rotation: two keys compressed at the same
    position keep the inner product of their normalised means."""
    rng = np.random.default_rng(2)
    for trial in range(40):
        raw = normal_bf16(rng, (4, D))
        p = int(rng.integers(0, 131072))
        k0 = oracle.compress_block(raw, p)
        assert np.array_equal(oracle.compress_block(raw[[2, 0, 3, 1]], p), k0)
        scaled = f2b(oracle.bf16_to_float(raw) * 4.0)
        assert np.array_equal(oracle.compress_block(scaled, p), k0)
        kf = oracle.bf16_to_float(k0)
        assert abs(np.linalg.norm(kf) - 1.0) < 4e-3
        raw2 = normal_bf16(rng, (4, D))
        k1 = oracle.bf16_to_float(oracle.compress_block(raw2, p))
        m0 = oracle.bf16_to_float(raw).sum(0)
        m1 = oracle.bf16_to_float(raw2).sum(0)
        ip = float(m0 @ m1) / (np.linalg.norm(m0) * np.linalg.norm(m1))
        assert abs(float(kf @ k1) - ip) < 1e-2


def test_compress_relative_position_property():
    """<RoPE_p(u), RoPE_p'(v)> depends only on p - p': shifting both blocks by
    the same multiple of 4 leaves the inner product of the keys unchanged
    (up to BF16 rounding)."""
    rng = np.random.default_rng(3)
    a = normal_bf16(rng, (4, D))
    b = normal_bf16(rng, (4, D))
    base = []
    for shift in [0, 4, 400, 40000]:
        ka = oracle.bf16_to_float(oracle.compress_block(a, 100 + shift))
        kb = oracle.bf16_to_float(oracle.compress_block(b, 36 + shift))
        base.append(float(ka @ kb))
    assert np.ptp(base) < 2e-2
    # while a different offset changes it
    ka = oracle.bf16_to_float(oracle.compress_block(a, 100))
    kb = oracle.bf16_to_float(oracle.compress_block(b, 40))
    assert abs(float(ka @ kb) - base[0]) > 1e-3


def test_compress_zero_block_stays_zero():
    raw = np.zeros((4, D), np.uint16)
    assert (oracle.bf16_to_float(oracle.compress_block(raw, 12)) == 0.0).all()


# ----------------------------------------------------------------- scores
def test_score_closed_form_on_basis_keys():
    """key = e_d: s = sum_h ReLU(q_h[d]) / sqrt(128)."""
    rng = np.random.default_rng(4)
    for d in [0, 7, 64, 127]:
        key = np.zeros(D, np.float32)
        key[d] = 1.0
        for _ in range(20):
            q = normal_bf16(rng, (4, D))
            qd = oracle.bf16_to_float(q)[:, d]
            want = np.float32(np.maximum(qd, 0).sum() / math.sqrt(128))
            assert oracle.score_one(q, f2b(key)) == want


def test_score_identities():
    """ReLU(x) - ReLU(-x) = x gives s(q) - s(-q) = sum_h <q_h, k> / sqrt(128);
    s is positively homogeneous (s(2q) = 2 s(q)) and symmetric in the heads;
    s >= 0."""
    rng = np.random.default_rng(5)
    for _ in range(200):
        q = normal_bf16(rng, (4, D))
        k = normal_bf16(rng, (D,))
        qf, kf = oracle.bf16_to_float(q), oracle.bf16_to_float(k)
        s = oracle.score_one(q, k)
        s_neg = oracle.score_one(q ^ np.uint16(0x8000), k)
        lin = float((qf @ kf).sum()) / math.sqrt(128)
        scale = float(np.abs(qf * kf).sum()) / math.sqrt(128)
        assert abs((s - s_neg) - lin) <= 1e-6 * scale + 1e-7
        assert s >= 0 and s_neg >= 0
        assert oracle.score_one(f2b(qf * 2.0), k) == np.float32(2.0 * s)
        assert oracle.score_one(q[[3, 1, 0, 2]], k) == s
    # all heads anti-aligned with the key -> exactly zero
    k = normal_bf16(rng, (D,))
    q = np.stack([k ^ np.uint16(0x8000)] * 4)
    assert oracle.score_one(q, k) == 0.0


def test_index_scores_visibility_and_paging():
    """Row t scores blocks b < L_t/4 only, reading block b from pool row
    full_slot(4b)/4; compare with scoring each block's key directly."""
    w = decode_workload(7, [[37, 40, 41], [9], [130, 131, 132, 133]], page_size=8, k_blk=4)
    pool = np.zeros((w.pool_rows, D), np.uint16)
    oracle.compress(w.raw_keys, w.block_req, w.block_id, w.page_table, w.page_size, w.rope_base, pool)
    # unpaged copy: block i at row i
    flat = np.zeros((w.n_blocks, D), np.uint16)
    oracle.compress(w.raw_keys, w.block_req, w.block_id, None, 0, w.rope_base, flat)
    s = oracle.index_scores(w.q, pool, w.req_row_start, w.row_len, w.page_table, w.page_size)
    first = {}
    for i, (r, b) in enumerate(zip(w.block_req, w.block_id)):
        first[(int(r), int(b))] = i
    rr = w.row_req()
    for t in range(w.n_rows):
        nb = w.row_len[t] // 4
        for b in range(s.shape[1]):
            if b < nb:
                assert s[t, b] == oracle.score_one(w.q[t], flat[first[(int(rr[t]), b)]])
            else:
                assert np.isnan(s[t, b])


# ----------------------------------------------------------------- top-k
def _brute_topk(row, k):
    """Full sort by (NaN last, value desc, index asc), first k, ascending."""
    keyed = sorted(range(len(row)), key=lambda i: (math.isnan(row[i]),
                                                    -row[i] if not math.isnan(row[i]) else 0.0, i))
    chosen = sorted(keyed[:k])
    return chosen + [-1] * (k - len(chosen))


def test_topk_bruteforce_exhaustive_small():
    vals = [0.0, 1.0, -1.0, 2.0, -2.0]
    for n in range(0, 6):
        for row in itertools.product(vals, repeat=n):
            r = np.array(row, np.float32)
            for k in range(1, n + 2):
                assert oracle.topk_row(r, k).tolist() == _brute_topk(list(row), k), (row, k)


def test_topk_bruteforce_random_up_to_12():
    rng = np.random.default_rng(6)
    vals = np.array([0.0, -0.0, 1.0, -1.0, 2.0, -2.0, np.inf, -np.inf, np.nan], np.float32)
    for _ in range(4000):
        n = int(rng.integers(0, 13))
        r = vals[rng.integers(0, vals.size, size=n)]
        k = int(rng.integers(1, 14))
        got = oracle.topk_row(r, k).tolist()
        want = _brute_topk([float(x) if not (x == 0) else 0.0 for x in r], k)
        assert got == want, (r, k)


def _check_invariants(row, n, k, idx):
    m = min(n, k)
    sel = idx[:m]
    assert (idx[m:] == -1).all()
    assert (sel >= 0).all() and (sel < n).all()
    assert (np.diff(sel) > 0).all()
    if m == n:
        return
    mask = np.zeros(n, bool)
    mask[sel] = True
    v = row[:n].astype(np.float64)
    lo = v[mask].min()
    hi = v[~mask].max()
    assert lo >= hi
    if lo == hi:  # boundary ties: selected ones have the smallest indices
        tie_sel = np.flatnonzero(mask & (v == lo))
        tie_un = np.flatnonzero(~mask & (v == lo))
        assert tie_sel.max() < tie_un.min()


@pytest.mark.parametrize("dist", TOPK_DISTS)
def test_topk_invariants(dist):
    w = topk_workload(8, 6, 6000, k=2048, dist=dist, ragged=True)
    idx, slots = oracle.topk(w.scores, w.k, n_valid=w.n_valid, page_table=w.page_table,
                             page_size=w.page_size)
    for t in range(6):
        _check_invariants(w.scores[t], int(w.n_valid[t]), w.k, idx[t])
        # slot translation inverts through the page table
        inv = {int(p): j for j, p in enumerate(w.page_table[t])}
        good = idx[t] >= 0
        assert (slots[t][~good] == -1).all()
        pages = np.array([inv[int(p)] for p in slots[t][good] // w.page_size], np.int64)
        pos = pages * w.page_size + slots[t][good] % w.page_size
        assert np.array_equal(pos, idx[t][good])


def test_topk_special_cases():
    k = 16
    assert oracle.topk_row(np.full(100, 0.25, np.float32), k).tolist() == list(range(k))
    assert oracle.topk_row(np.arange(5, dtype=np.float32), k).tolist() == list(range(5)) + [-1] * 11
    assert oracle.topk_row(np.zeros(0, np.float32), 4).tolist() == [-1] * 4
    r = np.array([0.0, -0.0, 0.0, -0.0], np.float32)
    assert oracle.topk_row(r, 2).tolist() == [0, 1]
    r = np.array([np.nan, -np.inf, 1.0, np.nan], np.float32)
    assert oracle.topk_row(r, 3).tolist() == [0, 1, 2]
    assert oracle.topk_row(r, 2).tolist() == [1, 2]


# ----------------------------------------------------------------- expansion
@pytest.mark.parametrize("L", [0, 1, 3, 4, 5, 6, 7, 8, 63, 64, 65, 66, 67, 2047, 2048, 2049, 2051])
def test_expand_counts_and_order(L):
    k_blk = 512
    P = 64
    pt = np.random.default_rng(L).permutation(64).astype(np.int32)
    nb = L // 4
    sel = np.full(k_blk, -1, np.int32)
    chosen = np.sort(np.random.default_rng(L + 1).permutation(nb)[:k_blk]).astype(np.int32)
    sel[:chosen.size] = chosen
    pos, slots = oracle.expand_row(sel, L, pt, P)
    assert pos.size == 4 * k_blk + 3
    n_sel = min(nb, k_blk)
    n_out = 4 * n_sel + L % 4
    assert (pos[n_out:] == -1).all() and (pos[:n_out] >= 0).all()
    assert (np.diff(pos[:n_out]) > 0).all()
    assert set(pos[4 * n_sel:n_out].tolist()) == set(range(4 * nb, L))
    for j, b in enumerate(chosen):
        assert pos[4 * j: 4 * j + 4].tolist() == [4 * b, 4 * b + 1, 4 * b + 2, 4 * b + 3]
    inv = np.argsort(pt)
    good = pos >= 0
    assert np.array_equal(inv[slots[good] // P] * P + slots[good] % P, pos[good])
    assert (slots[~good] == -1).all()


def test_indexer_select_composition_and_padding():
    """Whole path on a small paged workload: selection equals top-k of the
    scores; rows with fewer than k visible blocks are padded only at the tail."""
    w = decode_workload(9, [[2048 * 4 + 3, 2000, 17], [1, 4, 5]], page_size=16, k_blk=512)
    pool = np.zeros((w.pool_rows, D), np.uint16)
    oracle.compress(w.raw_keys, w.block_req, w.block_id, w.page_table, w.page_size, w.rope_base, pool)
    out = oracle.indexer_select(w.q, pool, w.req_row_start, w.row_len, w.page_table, w.page_size,
                                k_blk=512)
    for t in range(w.n_rows):
        nb = int(w.row_len[t]) // 4
        want = oracle.topk_row(out["scores"][t, :nb], 512)
        assert np.array_equal(out["blocks"][t], want)
        _check_invariants(out["scores"][t], nb, 512, out["blocks"][t])
        assert ((out["blocks"][t] == -1).sum() > 0) == (nb < 512)


# ------------------------------------------------------------ IndexShare reuse
# Qwen3.8-Flash-Next day-0 write-up, section "IndexShare MTP: reusing the QSA
# selection across draft steps": draft rows read the draft-extend row's
# selection plus the positions drafted since, without a scorer or top-k.
def test_indexshare_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "indexshare_3block.json")))
    pt = np.array(g["page_table"], np.int32)
    for row in g["rows"]:
        pos, slots, flags = oracle.indexshare_row(g["cap_blocks"], g["cap_len"], g["n_extra"], row["L"], pt,
                                                  g["page_size"])
        assert pos.tolist() == row["positions"], row["L"]
        assert slots.tolist() == row["slots"], row["L"]
        assert flags == row["flags"], row["L"]


def _captured(seed, k_blk, cap_len):
    """A captured selection as the selection step makes it: top-k of random
    scores over the capture's complete blocks."""
    nb0 = cap_len // 4
    s = np.random.default_rng(seed).standard_normal(max(nb0, 1)).astype(np.float32)
    return oracle.topk_row(s[:nb0], k_blk)


@pytest.mark.parametrize("cap_len", [0, 3, 4, 13, 14, 15, 16, 2047, 2048, 2051, 5000])
def test_indexshare_without_new_blocks_is_the_plain_expansion(cap_len):
    """While no block completes after the capture, the reused row is exactly
    the expansion of the captured blocks at the row's own length."""
    k_blk, P = 512, 16
    pt = np.random.default_rng(cap_len).permutation(cap_len // P + 4).astype(np.int32)
    sel = _captured(cap_len, k_blk, cap_len)
    for L in range(cap_len, 4 * (cap_len // 4) + 4):
        pos, slots, flags = oracle.indexshare_row(sel, cap_len, 0, L, pt, P)
        epos, eslots = oracle.expand_row(sel, L, pt, P)
        assert flags == 0
        assert np.array_equal(pos, epos) and np.array_equal(slots, eslots)


@pytest.mark.parametrize("cap_len,n_extra", [(14, 3), (16, 1), (2049, 6), (8000, 4), (8003, 9)])
def test_indexshare_equals_expansion_with_every_new_block_kept(cap_len, n_extra):
    """Blocks completed after the capture are visible in full: the reused
    list equals the plain expansion at the row's length of the captured
    blocks plus every block completed since (a wider selection)."""
    k_blk, P = 512, 64
    L_max = cap_len + n_extra
    pt = np.random.default_rng(cap_len + 7).permutation(L_max // P + 2).astype(np.int32)
    sel = _captured(cap_len + 1, k_blk, cap_len)
    nb0 = cap_len // 4
    for L in range(cap_len, L_max + 1):
        pos, slots, flags = oracle.indexshare_row(sel, cap_len, n_extra, L, pt, P)
        assert flags == 0 and pos.size == 4 * k_blk + 3 + n_extra
        new = np.arange(nb0, L // 4, dtype=np.int32)
        wide = np.concatenate([sel[sel >= 0], new]).astype(np.int32)
        epos, eslots = oracle.expand_row(wide, L, pt, P)
        n = int((pos >= 0).sum())
        assert n == int((epos >= 0).sum())
        assert np.array_equal(pos[:n], epos[:n]) and np.array_equal(slots[:n], eslots[:n])
        assert (pos[n:] == -1).all() and (slots[n:] == -1).all()


def test_indexshare_row_before_capture_sees_only_its_past():
    """A row earlier than the capture keeps only the captured positions
    below its own length (ascending, -1 at the tail)."""
    k_blk, P, cap_len = 64, 16, 1000
    pt = np.arange(cap_len // P + 2, dtype=np.int32)[::-1].copy()
    sel = _captured(3, k_blk, cap_len)
    full, _ = oracle.expand_row(sel, cap_len, pt, P)
    for L in [0, 1, 5, 100, 401, 997, 999]:
        pos, slots, flags = oracle.indexshare_row(sel, cap_len, 2, L, pt, P)
        want = [int(p) for p in full if 0 <= p < L]
        n = len(want)
        assert flags == 0 and pos[:n].tolist() == want and (pos[n:] == -1).all()


def test_indexshare_flags_and_request_mapping():
    P = 4
    pt = np.array([[2, 0, 3, 1, 5, 6], [1, 2, 3, 4, 5, 0]], np.int32)
    # a captured block that was not complete at the capture is skipped
    pos, _, flags = oracle.indexshare_row([0, 3], 14, 3, 16, pt[0], P)
    assert flags == 2 and pos.tolist()[:8] == [0, 1, 2, 3, 12, 13, 14, 15]
    # request -> captured row, rows of a request share it; a bad cap_row gives -1
    cap = np.array([[0, 2], [1, -1]], np.int32)
    cap_len = np.array([14, 9], np.int32)
    rrs = np.array([0, 2, 3], np.int32)
    row_len = np.array([15, 17, 11], np.int32)
    pos, slots, flags = oracle.indexshare(cap, cap_len, [0, 1], 3, rrs, row_len, pt, P)
    assert flags == 0
    assert pos[0].tolist() == [0, 1, 2, 3, 8, 9, 10, 11, 12, 13, 14, -1, -1, -1]
    assert pos[2].tolist() == [4, 5, 6, 7, 8, 9, 10] + [-1] * 7
    assert slots[2].tolist() == [8, 9, 10, 11, 12, 13, 14] + [-1] * 7
    pos, slots, flags = oracle.indexshare(cap, cap_len, [0, 2], 3, rrs, row_len, pt, P)
    assert flags == 4 and (pos[2] == -1).all() and (slots[2] == -1).all()


# ------------------------------------------------------------ sparse attention
# Qwen3.8-Flash-Next write-up, "Qwen sparse attention (QSA)": softmax and
# value aggregation over the original K/V at the selected positions;
# vllm-sparse-mla-blackwell, "Design notes worth knowing": the only mask is
# index >= 0, and a fully masked token must not give NaN.
def _attn_case(n_slots=12, h_q=8, h_kv=2, d=128, seed=0):
    rng = np.random.default_rng(seed)
    q = normal_bf16(rng, (1, h_q, d))
    k = normal_bf16(rng, (n_slots, h_kv, d))
    v = normal_bf16(rng, (n_slots, h_kv, d))
    return q, k, v


def _b2f(x):
    return oracle.bf16_to_float(x)


def test_attn_single_slot_returns_its_value_row_per_kv_head():
    q, k, v = _attn_case(h_q=8, h_kv=2)
    out, lse, f = oracle.sparse_attn(q, k, v, np.array([[-1, 5, -1]], np.int32), 0.3)
    assert f == 0
    for h in range(8):  # query heads 0-3 read KV head 0, 4-7 KV head 1
        assert np.array_equal(out[0, h], _b2f(v[5, h // 4]).astype(np.float32))


def test_attn_identical_keys_average_the_values():
    q, k, v = _attn_case(h_q=4, h_kv=1)
    k[:] = k[0]
    slots = np.array([[0, 3, 7, -1, 9]], np.int32)
    out, lse, _ = oracle.sparse_attn(q, k, v, slots, 0.125)
    mean = _b2f(v[[0, 3, 7, 9], 0]).mean(axis=0)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], mean, rtol=1e-6, atol=1e-7)
        dot = float(_b2f(q[0, h]) @ _b2f(k[0, 0]))
        assert abs(lse[0, h] - (0.125 * dot + math.log(4))) < 1e-5 * (1 + abs(dot))


def test_attn_two_slots_closed_form_and_large_logits():
    """q = a e0, k1 = e0, k2 = e0 * (a - 1) / a: logits differ by scale, so
    the weights are sigmoid(scale) and 1 - sigmoid(scale) -- also with logits
    near 1600, far past FP64 exp overflow without the max subtraction."""
    d = 128
    for a, scale in [(2.0, 0.5), (40.0, 1.0)]:
        q = np.zeros((1, 1, d), np.uint16)
        k = np.zeros((2, 1, d), np.uint16)
        q[0, 0, 0] = oracle.bf16_round(a)
        k[0, 0, 0] = oracle.bf16_round(a)
        k[1, 0, 0] = oracle.bf16_round(a - 1.0)
        rng = np.random.default_rng(3)
        v = normal_bf16(rng, (2, 1, d))
        out, lse, _ = oracle.sparse_attn(q, k, v, np.array([[0, 1]], np.int32), scale)
        w1 = 1.0 / (1.0 + math.exp(-scale * a))  # logit gap = scale * a * (a - (a - 1))
        want = w1 * _b2f(v[0, 0]) + (1 - w1) * _b2f(v[1, 0])
        np.testing.assert_allclose(out[0, 0], want, rtol=1e-6, atol=1e-7)
        top = scale * a * a
        assert abs(lse[0, 0] - (top + math.log(1 + math.exp(-scale * a)))) < 1e-6 * max(1.0, top)


def test_attn_zero_query_and_fully_masked_row():
    q, k, v = _attn_case(h_q=2, h_kv=1)
    q[:] = 0
    slots = np.array([[2, 4, 6], [-1, -1, -1]], np.int32)
    out, lse, _ = oracle.sparse_attn(np.concatenate([q, q]), k, v, slots, 1.0)
    np.testing.assert_allclose(out[0, 0], _b2f(v[[2, 4, 6], 0]).mean(axis=0), rtol=1e-6, atol=1e-7)
    assert (out[1] == 0).all() and np.isneginf(lse[1]).all()
    assert not np.isnan(out).any()


def test_attn_permutation_and_duplicates():
    q, k, v = _attn_case(h_q=8, h_kv=2, seed=4)
    a = np.array([[1, -1, 3, 8, -1, 10]], np.int32)
    b = np.array([[10, 8, -1, -1, 1, 3]], np.int32)
    oa, la, _ = oracle.sparse_attn(q, k, v, a, 0.1)
    ob, lb, _ = oracle.sparse_attn(q, k, v, b, 0.1)
    np.testing.assert_allclose(oa, ob, rtol=1e-6, atol=1e-7)
    # the same slot twice is the same softmax average as once
    o1, _, _ = oracle.sparse_attn(q, k, v, np.array([[7]], np.int32), 0.1)
    o2, l2, _ = oracle.sparse_attn(q, k, v, np.array([[7, 7]], np.int32), 0.1)
    np.testing.assert_allclose(o1, o2, rtol=1e-6, atol=1e-7)


def test_attn_slot_past_the_cache_is_flagged_and_skipped():
    q, k, v = _attn_case(n_slots=4, h_q=2, h_kv=1)
    out, lse, f = oracle.sparse_attn(q, k, v, np.array([[4, 1]], np.int32), 0.2)
    o1, _, _ = oracle.sparse_attn(q, k, v, np.array([[1]], np.int32), 0.2)
    assert f == 1 and np.array_equal(out, o1)


# ------------------------------------------------------------ key path (ring)
# Qwen3.8-Flash-Next write-up, "Qwen sparse attention (QSA)": the raw index
# keys of a request's incomplete block wait in a 4-slot ring; a completed
# block is compressed into the pool at full_slot/4.
def _append_in_chunks(raw, chunks, P, pt, n_rows_pool, firsts=None):
    """One request; raw [L][128] u16 appended chunk by chunk."""
    ring = np.zeros((1, 4, D), np.uint16)
    pool = np.zeros((n_rows_pool, D), np.uint16)
    p = 0
    for n in chunks:
        oracle.append_keys(raw[p:p + n], np.array([0, n], np.int32), np.array([p], np.int32), ring, pt[None],
                           P, 10000.0, pool)
        p += n
    return ring, pool


@pytest.mark.parametrize("chunks", [[1] * 23, [6, 6, 6, 5], [3, 9, 4, 1, 2, 4], [23], [2, 2, 11, 8]])
def test_append_keys_equals_direct_compression(chunks):
    """Appending the tokens of a request in any chunking leaves in the pool
    exactly the direct compression of its complete blocks, and in the ring
    the keys of the last positions at slot p mod 4."""
    L, P = sum(chunks), 8
    rng = np.random.default_rng(len(chunks))
    raw = normal_bf16(rng, (L, D))
    pt = rng.permutation(8).astype(np.int32)
    n_rows_pool = 8 * P // 4
    ring, pool = _append_in_chunks(raw, chunks, P, pt, n_rows_pool)
    nb = L // 4
    want = np.zeros_like(pool)
    oracle.compress(raw[:4 * nb], np.zeros(nb, np.int32), np.arange(nb, dtype=np.int32), pt[None], P, 10000.0,
                    want)
    assert np.array_equal(pool, want)
    for p in range(max(0, L - 4), L):
        assert np.array_equal(ring[0, p % 4], raw[p])


def test_append_keys_several_requests_in_one_call():
    """Requests with different first positions and token counts in one call
    (a request completing two blocks, one completing none, one with no
    tokens) match appending each request alone."""
    P = 4
    rng = np.random.default_rng(9)
    firsts = np.array([5, 0, 7, 2], np.int32)
    counts = np.array([7, 2, 0, 3], np.int32)
    rts = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    raw_ctx = [normal_bf16(rng, (int(f + c), D)) for f, c in zip(firsts, counts)]
    pt = rng.permutation(4 * 8).astype(np.int32).reshape(4, 8)
    pool_rows = 32 * P // 4
    ring = np.zeros((4, 4, D), np.uint16)
    pool = np.zeros((pool_rows, D), np.uint16)
    # the tokens before this call, one at a time
    for r in range(4):
        for p in range(int(firsts[r])):
            oracle.append_keys(raw_ctx[r][p:p + 1], np.array([0] * r + [0, 1] + [1] * (3 - r), np.int32),
                               np.where(np.arange(4) == r, p, 0).astype(np.int32), ring, pt, P, 10000.0, pool)
    ring_a, pool_a = ring.copy(), pool.copy()
    new = np.concatenate([raw_ctx[r][firsts[r]:] for r in range(4)])
    oracle.append_keys(new, rts, firsts, ring_a, pt, P, 10000.0, pool_a)
    for r in range(4):  # each request alone
        rs = np.zeros(5, np.int32)
        rs[r + 1:] = counts[r]
        oracle.append_keys(raw_ctx[r][firsts[r]:], rs, firsts, ring, pt, P, 10000.0, pool)
    assert np.array_equal(ring, ring_a) and np.array_equal(pool, pool_a)
    # request 0 completed blocks 1 and 2 (positions 7 and 11)
    for b in (1, 2):
        want = oracle.compress_block(raw_ctx[0][4 * b:4 * b + 4], 4 * b)
        assert np.array_equal(pool_a[oracle.pool_row(pt[0], b, P)], want)


def test_openmp_build_computes_the_same_path():
    """The OpenMP build of the oracle (used only to time the CPU baseline on
    every host core) gives the single-threaded build's scores, selection,
    positions and slots to the bit, on several requests of ragged rows."""
    import subprocess
    from workloads import decode_workload
    w = decode_workload(91, [[4099, 4100, 4101], [1030], [9000, 9002]], page_size=64, k_blk=512)
    pool = np.zeros((w.pool_rows, 128), np.uint16)
    oracle.compress(w.raw_keys, w.block_req, w.block_id, w.page_table, w.page_size, w.rope_base, pool)
    args = (w.q, pool, w.req_row_start, w.row_len, w.page_table, w.page_size)
    one = oracle.indexer_select(*args, k_blk=w.k_blk)
    try:
        many = oracle.indexer_select_threads(*args, k_blk=w.k_blk, threads=4)
    except (OSError, subprocess.CalledProcessError):
        pytest.skip("no OpenMP toolchain")
    for key in ("blocks", "pos", "slots"):
        assert np.array_equal(one[key], many[key]), key
    assert np.array_equal(one["scores"].view(np.uint32), many["scores"].view(np.uint32))
