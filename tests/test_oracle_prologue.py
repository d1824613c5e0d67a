"""Pins of the oracle's prologue-tail functions (CPU only): the query RoPE,
the e4m3 and binary16 encoders, the FP8 key quantiser and the FP8 score.

The encoders are checked against independent implementations of the same
formats (torch's float8_e4m3fn, numpy's float16) and closed forms; the
quantiser against the format's invariants; the FP8 score against closed
forms and against the BF16 score on keys and queries that both formats
represent exactly (then the two must agree to the bit); the query rotation
against closed forms on basis vectors and against the key path's rotation.
"""
import math

import numpy as np
import pytest

import oracle
from workloads import bf16_bits, normal_bf16

SCALE = 1.0 / math.sqrt(128.0)


# ----------------------------------------------------------------- e4m3
def test_e4m3_decodes_like_torch_float8_e4m3fn():
    torch = pytest.importorskip("torch")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([oracle.e4m3_to_float(c) for c in range(256)], np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan].astype(np.float64))


def test_e4m3_rounds_like_torch_within_range():
    """Nearest, ties to even, for |x| <= 448: every code value, every
    midpoint between neighbours (the ties), points just off them, and random
    values over the whole range (torch's cast is the reference there)."""
    torch = pytest.importorskip("torch")
    vals = np.array([oracle.e4m3_to_float(c) for c in range(256)])
    fin = np.sort(np.unique(vals[np.isfinite(vals)]))
    mids = (fin[1:] + fin[:-1]) / 2
    rng = np.random.default_rng(3)
    x = np.concatenate([fin, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                        rng.uniform(-448, 448, 4000), rng.standard_normal(2000) * 0.01]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_round(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, ref), x[got != ref][:5]


def test_e4m3_closed_forms_and_saturation():
    assert oracle.e4m3_round(1.0) == 0x38
    assert oracle.e4m3_round(448.0) == 0x7E
    assert oracle.e4m3_round(500.0) == 0x7E and oracle.e4m3_round(-1e6) == 0xFE  # saturating
    assert oracle.e4m3_round(2.0 ** -9) == 0x01                  # smallest subnormal
    assert oracle.e4m3_round(2.0 ** -10) == 0x00                 # half of it: ties to even (zero)
    assert oracle.e4m3_round(3 * 2.0 ** -10) == 0x02             # 1.5 quanta: to the even 2
    assert oracle.e4m3_round(1.0625) == 0x38                     # between 1 and 1.125: to 1
    assert oracle.e4m3_round(1.1875) == 0x3A                     # between 1.125 and 1.25: to 1.25
    assert oracle.e4m3_round(float("nan")) == 0x7F


# ----------------------------------------------------------------- binary16
def test_f16_rounds_like_numpy_float16():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(3000), rng.standard_normal(1000) * 1e-5,
                        rng.uniform(-65000, 65000, 1000), [2.0 ** -25, 3 * 2.0 ** -25, 65504.0, 65519.0]])
    got = np.array([oracle.f16_round(float(v)) for v in x])
    ref = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(got, ref)
    assert math.isinf(oracle.f16_round(65520.0))  # beyond the largest finite value


# ----------------------------------------------------------------- quantiser
def test_fp8_quantiser_invariants():
    rng = np.random.default_rng(5)
    keys = normal_bf16(rng, (64, 128))
    keys[3] = 0                                       # a zero key
    codes, scales = oracle.quantize_keys_fp8(keys)
    k = oracle.bf16_to_float(keys).astype(np.float64)
    deq = np.vectorize(oracle.e4m3_to_float)(codes) * scales[:, None].astype(np.float64)
    assert scales[3] == 0 and (codes[3] == 0).all()
    for r in range(64):
        if r == 3:
            continue
        mx = np.abs(k[r]).max()
        assert scales[r] == np.float32(np.float32(mx) / np.float32(448.0))
        # the largest element maps to the largest code
        assert np.isin(codes[r][np.abs(k[r]) == mx], [0x7E, 0xFE]).all()
        # nearest value: half an e4m3 step (2^-4 relative in the normal range,
        # 2^-10 * scale absolute among the subnormals)
        q = k[r] / scales[r]
        step = np.where(np.abs(q) >= 2.0 ** -6, np.abs(q) * 2.0 ** -3, 2.0 ** -9)
        assert (np.abs(deq[r] - k[r]) <= 0.5 * step * scales[r] * (1 + 1e-6) + 1e-30).all()
    # scale invariance: doubling the keys doubles the scales, not the codes
    keys2 = bf16_bits(2.0 * k.astype(np.float32))
    codes2, scales2 = oracle.quantize_keys_fp8(keys2)
    assert np.array_equal(codes2, codes) and np.array_equal(scales2, 2 * scales)


# ----------------------------------------------------------------- FP8 score
def test_fp8_score_closed_form():
    """One FP8 key with code 448 on dim 0 and scale 2^-8 (value 1.75): the
    score is 1.75 * sum_h ReLU(q_h0) / sqrt(128)."""
    q = np.zeros((4, 128), np.float32)
    q[:, 0] = [0.5, -2.0, 3.0, 0.25]
    qb = bf16_bits(q)
    codes = np.zeros(128, np.uint8)
    codes[0] = 0x7E
    got = oracle.score_one_fp8(qb, codes, 2.0 ** -8)
    assert got == np.float32(1.75 * (0.5 + 3.0 + 0.25) * SCALE)


def test_fp8_score_equals_the_bf16_score_when_both_formats_are_exact():
    """Keys whose values are e4m3 codes times a power of two and queries
    exact in binary16: FP8 and BF16 scores must agree to the bit."""
    rng = np.random.default_rng(6)
    fin = np.array([oracle.e4m3_to_float(c) for c in range(0x7F)])   # 0 .. 448
    for _ in range(20):
        mag = rng.choice(fin, 128)
        sign = rng.choice([-1.0, 1.0], 128)
        kv = (sign * mag * 2.0 ** -9).astype(np.float32)                # exact in BF16 (4 significant bits)
        kv[rng.integers(0, 128)] = 448 * 2.0 ** -9                      # the maximum is a code value
        key = bf16_bits(kv)
        codes, scales = oracle.quantize_keys_fp8(key[None])
        assert scales[0] == np.float32(2.0 ** -9)
        q = bf16_bits(rng.standard_normal((4, 128)).astype(np.float32))  # 8 bits: exact in binary16
        assert oracle.score_one_fp8(q, codes[0], scales[0]) == oracle.score_one(q, key)


def test_fp8_score_holds_the_query_in_binary16():
    """A query element beyond binary16's range becomes infinity (the FP8
    scorer's query is FP16), and one below its subnormal quantum rounds."""
    q = np.zeros((4, 128), np.float32)
    q[0, 0] = 70000.0
    codes = np.zeros(128, np.uint8)
    codes[0] = 0x38                                  # 1.0
    assert math.isinf(oracle.score_one_fp8(bf16_bits(q), codes, 1.0))
    q[0, 0] = 2.0 ** -20 * (1 + 2.0 ** -7)           # binary16 keeps 2^-20 only
    got = oracle.score_one_fp8(bf16_bits(q), codes, 1.0)
    assert got == np.float32(2.0 ** -20 * SCALE)


# ----------------------------------------------------------------- query RoPE
def test_rope_queries_closed_forms_on_basis_vectors():
    base = 10000.0
    for p in [0, 1, 7, 4095, 79_999, 131_071]:
        for i in [0, 1, 17, 63]:
            q = np.zeros((1, 4, 128), np.float32)
            q[0, 2, i] = 1.0
            out = oracle.bf16_to_float(oracle.rope_queries(bf16_bits(q), np.array([p], np.int32), base))
            th = p * base ** (-2.0 * i / 128)
            assert out[0, 2, i] == oracle.bf16_to_float(np.array([oracle.bf16_round(math.cos(th))]))[0]
            assert out[0, 2, i + 64] == oracle.bf16_to_float(np.array([oracle.bf16_round(math.sin(th))]))[0]
            rest = np.delete(out[0, 2], [i, i + 64])
            assert (rest == 0).all() and (out[0, [0, 1, 3]] == 0).all()


def test_rope_queries_position_zero_is_identity_and_matches_the_key_rotation():
    rng = np.random.default_rng(8)
    q = normal_bf16(rng, (5, 4, 128))
    assert np.array_equal(oracle.rope_queries(q, np.zeros(5, np.int32)), q)
    # a block of four equal unit keys compresses to the rotation of that key
    # at the block's first position: the query rotation must agree
    for p in [4, 8000, 131_068]:
        u = np.zeros(128, np.float32)
        u[rng.integers(0, 128)] = 1.0
        raw = np.tile(bf16_bits(u), (4, 1))
        key = oracle.compress_block(raw, p, 10000.0)
        qq = np.zeros((1, 4, 128), np.uint16)
        qq[0, 1] = bf16_bits(u)
        assert np.array_equal(oracle.rope_queries(qq, np.array([p], np.int32))[0, 1], key)


# ----------------------------------------------------------------- head gate
def test_gated_score_with_unit_gates_is_the_plain_score():
    rng = np.random.default_rng(9)
    ones = np.ones(4, np.float32)
    for _ in range(30):
        q = normal_bf16(rng, (4, 128))
        key = normal_bf16(rng, (128,))
        assert oracle.score_one_gated(q, ones, key) == oracle.score_one(q, key)


def test_gated_score_closed_form_one_head_at_a_time():
    """A basis key e_d and a gate on head h alone: the score is
    g * ReLU(q[h][d]) / sqrt(128)."""
    q = np.zeros((4, 128), np.float32)
    q[:, 5] = [1.5, -2.0, 0.75, 3.0]
    qb = bf16_bits(q)
    key = np.zeros(128, np.float32)
    key[5] = 1.0
    kb = bf16_bits(key)
    for h in range(4):
        g = np.zeros(4, np.float32)
        g[h] = 0.5
        want = np.float32(0.5 * max(float(q[h, 5]), 0.0) * SCALE)
        assert oracle.score_one_gated(qb, g, kb) == want, h


def test_gated_score_odd_in_the_gates_and_scales_with_them():
    """The gate multiplies the rectified dot product: negating every gate
    negates the score and doubling them doubles it, to the bit (a gate
    applied before the ReLU breaks both)."""
    rng = np.random.default_rng(10)
    for _ in range(30):
        q = normal_bf16(rng, (4, 128))
        key = normal_bf16(rng, (128,))
        g = rng.uniform(-2, 2, 4).astype(np.float32)
        s = oracle.score_one_gated(q, g, key)
        assert oracle.score_one_gated(q, -g, key) == -s
        assert oracle.score_one_gated(q, 2 * g, key) == np.float32(2 * s)


def test_gated_block_scores_follow_the_rows_gates():
    """index_scores_gated on a paged pool equals score_one_gated of each
    row's own gates against each visible block's key."""
    rng = np.random.default_rng(11)
    P = 16
    row_len = np.array([13, 40, 9], np.int32)
    rrs = np.array([0, 2, 3], np.int32)
    pt = np.array([[3, 0, 2], [1, 4, 5]], np.int32)
    pool = normal_bf16(rng, (6 * P // 4, 128))
    q = normal_bf16(rng, (3, 4, 128))
    gates = rng.uniform(-1, 2, (3, 4)).astype(np.float32)
    s = oracle.index_scores_gated(q, gates, pool, rrs, row_len, pt, P, ld_scores=12)
    for t, r in [(0, 0), (1, 0), (2, 1)]:
        for b in range(row_len[t] // 4):
            key = pool[oracle.pool_row(pt[r], b, P)]
            assert s[t, b] == np.float32(oracle.score_one_gated(q[t], gates[t], key))
        assert np.isnan(s[t, row_len[t] // 4:]).all()
