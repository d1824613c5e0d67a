"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import math

import numpy as np

import oracle

SCALE = 1.0 / math.sqrt(128.0)


def to_dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.view(dtype) if dtype is not None else t


def bf16_dev(a):
    import torch
    return to_dev(np.ascontiguousarray(a, np.uint16).view(np.int16), torch.bfloat16)


def bf16_host(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# Absolute term of the compressed-key bound.  The GPU rotates the normalised
# mean in FP32: r = u c - v s with |u|, |v|, |c|, |s| <= 1 and u^2 + v^2 <= 1.
# Errors proportional to |r| (the normalisation's scale, the subtraction's
# rounding) are far below an ulp of r.  What is not proportional to |r| is
# bounded by half an FP32 ulp for each of u and v, one for each product and
# about one for sincospif on each of c and s: at most about 3 * 2^-24 in all,
# so 2^-22.  It matters only where u c - v s nearly cancels and an ulp of the
# BF16 result falls below it.
KEY_ABS_TERM = 2.0 ** -22


def key_tolerance(a, b):
    """Compressed-key bound: one BF16 ulp of the larger magnitude (each side
    rounds to BF16 once) plus KEY_ABS_TERM for the FP32 rotation."""
    m = np.maximum(np.maximum(np.abs(a), np.abs(b)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(m)) - 7) + KEY_ABS_TERM


def score_tolerance(q_bits, pool_bits, req_row_start, row_len, page_table, page_size, ld):
    """Per-element bound of the score comparison:
    2e-5 * (1/sqrt(128)) * sum_{h,d} |q[t,h,d] * kbar[b,d]| + 1e-6
    (FP32 accumulation of exact BF16 products against an FP64 reference)."""
    qa = np.abs(oracle.bf16_to_float(q_bits)).sum(axis=1)  # [n_rows][128]: sum over heads
    tol = np.full((row_len.size, ld), np.inf)
    for r in range(req_row_start.size - 1):
        rows = np.arange(req_row_start[r], req_row_start[r + 1])
        if rows.size == 0:
            continue
        nb = int(row_len[rows].max()) // 4
        prow = np.array([oracle.pool_row(page_table[r], b, page_size) for b in range(nb)], np.int64)
        ka = np.abs(oracle.bf16_to_float(pool_bits[prow]))  # [nb][128]
        tol[rows, :nb] = 2e-5 * SCALE * (qa[rows] @ ka.T) + 1e-6
    return tol


def pool_rows_of(page_table_row, nb, page_size):
    return np.array([oracle.pool_row(page_table_row, b, page_size) for b in range(nb)], np.int64)


def attn_tolerance(q_bits, k_bits, v_bits, slots, scale, chunk=256):
    """Per-element bound of the sparse-attention comparison [rows][h_q][d].
    A logit is a tensor-core FP32 accumulation of exact BF16 products:
    d/16 steps, each adding 16 products to the running sum; allowing each
    step 2^-22 of sum|q k| (twice a rounding, for an adder that may
    truncate), plus one step for the scale, its error is at most
    (d/16 + 1) 2^-22 scale sum|q k|; the weights carry twice that relative
    error plus 2^-22 for exp; a warp adds at most chunk/4 weighted rows in
    order.  Bound on |out - out_ref|: that relative error times max_j |v_j|
    (over the valid entries), plus 1e-6."""
    q = oracle.bf16_to_float(q_bits)   # [rows][h_q][d]
    k = oracle.bf16_to_float(k_bits)   # [n_slots][h_kv][d]
    v = oracle.bf16_to_float(v_bits)
    rows, h_q, d = q.shape
    h_kv = k.shape[1]
    g = h_q // h_kv
    tol = np.zeros(q.shape)
    gam = (d / 16 + 1) * 2.0 ** -22
    for t in range(rows):
        sl = slots[t]
        sl = sl[(sl >= 0) & (sl < k.shape[0])]
        if sl.size == 0:
            tol[t] = 1e-6
            continue
        for h in range(h_q):
            kk = k[sl, h // g]                       # [n][d]
            L = abs(scale) * (np.abs(kk) @ np.abs(q[t, h])).max()
            vmax = np.abs(v[sl, h // g]).max(axis=0)  # [d]
            rel = 2 * gam * L + 2.0 ** -22 + (chunk / 4) * 2.0 ** -24 + 4e-6
            tol[t, h] = rel * vmax + 1e-6
    return tol
