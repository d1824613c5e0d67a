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
