"""Capacity of the selection kernels' candidate lists, checked on the CPU.

Three kernels list the entries at or above a lower bound in fixed per-warp
regions of shared memory; a warp whose region would overflow sends its row
(select_fast_kernel, select_rows_kernel) or its CTA's slice
(select_long_kernel) to a slower whole-row path, which is still exact.  These checks replay each kernel's
bound, in the kernel's own layout of entries over warps, on seeded rows of
the benchmark's score distributions, and assert that the per-warp capacity
read from the kernel sources covers the largest count seen with margin.

- select_long_kernel, DSA top-2048 over rows of 80,000 on clusters of 2 CTAs
  (the 64-row C4 launch): the bound is the edge of the top-12-bit bin of the
  r-th largest of 2048 samples (16 runs of 128 spread over the row),
  r = 2 ceil(2048 k / n) + 8; each CTA owns a slice of the row and each of
  its 16 warps a segment of the slice.
- select_fast_kernel, top-512 over QSA block rows of 2,048-32,768 entries:
  the bound is the smallest, over full warps, of the ceil(k/F)-th largest of
  the warp's 32 lane maxima, each lane holding entries 4 (t + 1024 j) + c.
- select_rows_kernel, top-512 over the prefill chunk's rows of up to 32,768
  entries: the bound is the edge of the top-12-bit bin of the r-th largest
  of 1024 samples (32 runs of 32), r = ceil(mu + 3.5 sqrt(mu) + 2) with
  mu = 1024 k / n; each of the 8 warps owns a contiguous segment of the row.
"""
import math
import os
import re

import numpy as np

from workloads.synth import topk_scores

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sparse_attention_indexer_index_gb300", "csrc")


def _const(fname, name):
    src = open(os.path.join(CSRC, fname)).read()
    return int(re.search(rf"constexpr int {name} = (\d+);", src).group(1))


def _keys(x):
    """Order-preserving u32 images of FP32 scores (finite rows here)."""
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    return np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)


def _long_warp_counts(row, k, clusters):
    """Per-warp candidate counts of select_long_kernel on one row."""
    n = row.size
    warps = _const("select_long.cuh", "kSlThreads") // 32
    samples = _const("select_long.cuh", "kSlSamples")
    keys = _keys(row)
    # sampled bound: 16 runs of 128 (one 16-byte group per lane)
    idx = np.concatenate([(((run * n) // warps) & ~3) + np.arange(128) for run in range(warps)])
    r = 2 * ((samples * k + n - 1) // n) + 8
    hist = np.bincount((keys[idx] >> 20).astype(np.int64), minlength=4096)
    above = np.cumsum(hist[::-1])
    bin_ = 4095 - int(np.searchsorted(above, r))
    cand = keys >= (np.uint64(bin_) << 20)
    # slices of the cluster's CTAs, segments of the warps (multiples of 128)
    S = (((n + clusters - 1) // clusters) + 3) & ~3
    counts = []
    for c in range(clusters):
        s0 = min(n, c * S)
        s1 = min(n, s0 + S)
        seg = ((((s1 - s0) + warps - 1) // warps) + 127) & ~127
        for w in range(warps):
            w0 = min(s1, s0 + w * seg)
            w1 = min(s1, w0 + seg)
            counts.append(int(cand[w0:w1].sum()))
    return counts


def _fast_warp_counts(row, k):
    """Per-warp candidate counts of select_fast_kernel on one row."""
    n = row.size
    threads = _const("select_fast.cuh", "kSfThreads")
    runs = _const("select_fast.cuh", "kSfRuns")
    keys = _keys(row).astype(np.int64) + 1
    t = np.arange(threads)
    if n <= 4 * threads:  # short rows: entry t + 1024 c
        idx = np.stack([t + threads * c for c in range(4)], 1)
        has = t < n
    else:
        idx = np.stack([4 * (t + threads * j) + c for j in range(runs) for c in range(4)], 1)
        has = 4 * t < n
    valid = idx < n
    vals = np.where(valid, keys[np.minimum(idx, n - 1)], 0)
    lane_max = np.where(has, vals.max(1), 0)
    full = min(threads, n if n <= 4 * threads else (n + 3) // 4) // 32
    kw = (k + full - 1) // full
    assert kw <= 32
    per_warp = np.sort(lane_max.reshape(threads // 32, 32), axis=1)
    v = max(int(per_warp[:full, 32 - kw].min()), 1)
    cand = (vals >= v) & valid
    return cand.reshape(threads // 32, -1).sum(1)


def _rows_warp_counts(row, k):
    """Per-warp candidate counts of select_rows_kernel on one row."""
    n = row.size
    warps = _const("select_rows.cuh", "kSrThreads") // 32
    keys = _keys(row)
    mu = np.float32(1024.0) * np.float32(k) / np.float32(n)
    r = int(math.ceil(float(mu + np.float32(3.5) * np.sqrt(mu) + np.float32(2.0))))
    cand = np.ones(n, bool)
    if r < 1024:
        idx = np.concatenate([(((run * n) // 32) & ~3) + np.arange(32) for run in range(32)])
        idx = idx[idx < n]
        hist = np.bincount((keys[idx] >> 20).astype(np.int64), minlength=4096)
        above = np.cumsum(hist[::-1])
        bin_ = 4095 - int(np.searchsorted(above, r))
        cand = keys >= (np.uint64(bin_) << 20)
    seg = (((n + warps - 1) // warps) + 127) & ~127
    return [int(cand[min(n, w * seg):min(n, w * seg + seg)].sum()) for w in range(warps)]


def test_small_cta_lists_cover_the_prefill_rows():
    cap = _const("select_rows.cuh", "kSrCandCap") // (_const("select_rows.cuh", "kSrThreads") // 32)
    for dist in ("normal", "relu4"):
        for n in (8000, 20_000, 32_768):
            s, _ = topk_scores(np.random.default_rng(n + 1), 60, n, dist)
            m = max(max(_rows_warp_counts(row, 512)) for row in s)
            assert m <= 0.8 * cap, (dist, n, m, cap)


def test_long_row_lists_cover_the_dsa_rows():
    cap = _const("select_long.cuh", "kSlCandCap") // (_const("select_long.cuh", "kSlThreads") // 32)
    worst = {}
    for dist in ("normal", "relu4", "fp16dup"):
        m = 0
        for seed in (100, 101):
            s, _ = topk_scores(np.random.default_rng(seed), 64, 80_000, dist)
            for row in s:
                m = max(m, max(_long_warp_counts(row, 2048, 2)))
        worst[dist] = m
        assert m <= 0.85 * cap, (dist, m, cap)
    # the ReLU-sum rows are the widest: past the 256 per warp of the
    # capacity before (then one row in ~50 walked its whole slice)
    assert worst["relu4"] > 256, worst


def test_register_resident_lists_cover_qsa_rows():
    cap = _const("select_fast.cuh", "kSfWarpCap")
    for dist in ("normal", "relu4"):
        for n in (2048, 8000, 20_000, 32_768):
            s, _ = topk_scores(np.random.default_rng(n), 40, n, dist)
            m = max(int(_fast_warp_counts(row, 512).max()) for row in s)
            assert m <= 0.75 * cap, (dist, n, m, cap)


def test_bound_replays_hold_at_least_k_candidates():
    """The replayed bounds are lower bounds: at least k entries pass them
    (else the kernels would take the whole-row retry, not the lists)."""
    s, _ = topk_scores(np.random.default_rng(7), 4, 80_000, "relu4")
    for row in s:
        assert sum(_long_warp_counts(row, 2048, 2)) >= 2048
    s, _ = topk_scores(np.random.default_rng(8), 4, 20_000, "normal")
    for row in s:
        assert int(_fast_warp_counts(row, 512).sum()) >= 512
    assert math.isfinite(float(s.sum()))
