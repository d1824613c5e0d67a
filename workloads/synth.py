"""Seeded synthetic workloads for the QSA indexer and the token-level top-k.

Everything is drawn with ``numpy.random.default_rng(seed)`` on the host, so
the oracle and the GPU see the same bytes.  BF16 tensors are produced by
drawing FP32 N(0,1) and rounding to BF16 (nearest, ties to even) and are
returned as ``uint16`` bit patterns.

Shapes follow the indexer's statement of the problem: 4 index query heads of
128 dims, one shared 128-dim index key per token, compression ratio 4,
paged KV with a seeded random page permutation.  Nothing here computes a
compressed key, a score, a selection or a slot.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

D, H, C = 128, 4, 4
__all__ = [
    "D", "H", "C", "bf16_bits", "normal_bf16", "DecodeWorkload", "decode_workload",
    "TopkWorkload", "topk_workload", "c1_decode", "c2_verify", "c2_batched", "c3_batched",
    "c4_dsa_topk", "c5_prefill", "indexshare_mtp", "TOPK_DISTS",
]


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP32 array -> BF16 bit patterns, round to nearest even (finite input)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


@dataclass
class DecodeWorkload:
    """Query rows grouped by request, plus the raw index keys of every
    complete block of every request and a paged KV layout.

    row_len[t] is the number of tokens row t sees (its position + 1); rows of
    request r are req_row_start[r] .. req_row_start[r+1]-1.  Block i of the
    raw-key array is block ``block_id[i]`` of request ``block_req[i]``.
    """
    name: str
    seed: int
    page_size: int
    rope_base: float
    k_blk: int
    row_len: np.ndarray        # int32 [n_rows]
    req_row_start: np.ndarray  # int32 [n_req+1]
    page_table: np.ndarray     # int32 [n_req][ld_pt]
    q: np.ndarray              # uint16 [n_rows][4][128]
    raw_keys: np.ndarray       # uint16 [n_blocks*4][128]
    block_req: np.ndarray      # int32 [n_blocks]
    block_id: np.ndarray       # int32 [n_blocks]
    n_pages: int               # physical pages in the KV pool
    meta: dict = field(default_factory=dict)

    @property
    def n_rows(self) -> int:
        return int(self.row_len.size)

    @property
    def n_req(self) -> int:
        return int(self.req_row_start.size - 1)

    @property
    def n_blocks(self) -> int:
        return int(self.block_id.size)

    @property
    def pool_rows(self) -> int:
        """Rows of the compressed-key pool: one per 4 KV slots."""
        return self.n_pages * self.page_size // C

    @property
    def max_len(self) -> int:
        return int(self.row_len.max()) if self.n_rows else 0

    @property
    def max_rows_per_req(self) -> int:
        return int(np.diff(self.req_row_start).max()) if self.n_req else 0

    def row_req(self) -> np.ndarray:
        return np.repeat(np.arange(self.n_req, dtype=np.int32), np.diff(self.req_row_start))


def decode_workload(seed: int, rows_per_req: list[list[int]], page_size: int = 64,
                    k_blk: int = 512, rope_base: float = 10000.0, name: str = "",
                    pad_pages: int = 0, with_keys: bool = True) -> DecodeWorkload:
    """rows_per_req[r] lists the row lengths (visible tokens) of request r's
    query rows.  A request's context is its longest row; its page table covers
    that context (plus ``pad_pages`` spare pages), drawn as a seeded random
    permutation of the whole pool.  with_keys=False leaves out the raw keys
    (for selection-only cases whose scores are drawn directly)."""
    rng = np.random.default_rng(seed)
    row_len = np.array([L for rows in rows_per_req for L in rows], np.int32)
    counts = np.array([len(rows) for rows in rows_per_req], np.int32)
    req_row_start = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ctx = np.array([max(rows) if rows else 0 for rows in rows_per_req], np.int64)
    pages = (ctx + page_size - 1) // page_size + pad_pages
    n_pages = int(pages.sum())
    ld_pt = max(1, int(pages.max()) if pages.size else 1)
    perm = rng.permutation(n_pages).astype(np.int32)
    page_table = np.zeros((len(rows_per_req), ld_pt), np.int32)
    off = 0
    for r, n in enumerate(pages):
        page_table[r, :n] = perm[off:off + n]
        off += n
    q = normal_bf16(rng, (row_len.size, H, D))
    nb = ctx // C if with_keys else np.zeros_like(ctx)
    block_req = np.repeat(np.arange(len(rows_per_req), dtype=np.int32), nb)
    block_id = np.concatenate([np.arange(n, dtype=np.int32) for n in nb]) if nb.size else \
        np.zeros(0, np.int32)
    raw_keys = normal_bf16(rng, (int(nb.sum()) * C, D))
    return DecodeWorkload(name=name, seed=seed, page_size=page_size, rope_base=rope_base,
                          k_blk=k_blk, row_len=row_len, req_row_start=req_row_start,
                          page_table=page_table, q=q, raw_keys=raw_keys, block_req=block_req,
                          block_id=block_id, n_pages=n_pages)


# --------------------------------------------------------------------------
# The five workloads of the statement of the problem (and one batched
# variant of the verify step).
# --------------------------------------------------------------------------
def c1_decode(seed: int = 0) -> DecodeWorkload:
    """Single request, one decode row at L = 8192 (2048 blocks, no pending)."""
    return decode_workload(seed, [[8192]], name="decode_L8192_1row")


def c2_verify(seed: int = 0, L: int = 80_000, n_rows: int = 6) -> DecodeWorkload:
    """Verify step, batch 1: 1 accepted + 5 draft rows at positions L-6..L-1."""
    rows = [L - n_rows + 1 + i for i in range(n_rows)]
    return decode_workload(seed, [rows], name=f"verify_L{L}_{n_rows}rows")


def c2_batched(seed: int = 0, n_req: int = 32, L: int = 80_000, n_rows: int = 6) -> DecodeWorkload:
    """n_req independent verify steps of the same shape in one call."""
    rows = [L - n_rows + 1 + i for i in range(n_rows)]
    return decode_workload(seed, [list(rows) for _ in range(n_req)],
                           name=f"verify_L{L}_{n_rows}rows_x{n_req}")


def c3_batched(seed: int = 0, n_req: int = 32, lo: int = 4096, hi: int = 131_072,
               with_keys: bool = True) -> DecodeWorkload:
    """Batched decode: n_req requests, one row each, L uniform in [lo, hi]."""
    rng = np.random.default_rng(seed + 1_000_003)
    lens = rng.integers(lo, hi, size=n_req, endpoint=True)
    return decode_workload(seed, [[int(L)] for L in lens], name=f"decode_batched_{n_req}req",
                           with_keys=with_keys)


def indexshare_mtp(seed: int = 0, n_req: int = 32, lo: int = 4096, hi: int = 131_072, n_draft: int = 3,
                   page_size: int = 64) -> DecodeWorkload:
    """One MTP iteration per request: the draft-extend row at L0 (the last
    token the target accepted; L0 uniform in [lo, hi]) followed by the
    n_draft draft rows L0+1 .. L0+n_draft.  Rows of request r: its draft-extend
    row first.  The page table covers the drafted positions."""
    rng = np.random.default_rng(seed + 9000)
    L0 = rng.integers(lo, hi + 1, size=n_req)
    return decode_workload(seed, [[int(l) + j for j in range(n_draft + 1)] for l in L0],
                           page_size=page_size, name=f"indexshare_{n_req}req_{n_draft}draft")


def c5_prefill(seed: int = 0, L: int = 131_072, n_rows: int = 4096) -> DecodeWorkload:
    """Prefill chunk: n_rows consecutive query rows ending at position L-1."""
    rows = [L - n_rows + 1 + i for i in range(n_rows)]
    return decode_workload(seed, [rows], name=f"prefill_L{L}_{n_rows}rows")


TOPK_DISTS = ("normal", "relu4", "fp16dup")


@dataclass
class TopkWorkload:
    name: str
    seed: int
    dist: str
    k: int
    page_size: int
    scores: np.ndarray       # float32 [n_rows][n]
    n_valid: np.ndarray      # int32 [n_rows]
    page_table: np.ndarray   # int32 [n_rows][ld_pt]  (row t uses page-table row t)
    dup_fraction: float = 0.0


def topk_scores(rng: np.random.Generator, n_rows: int, n: int, dist: str):
    """Value distributions for token-level top-k rows.

    normal:  N(0,1) FP32.
    relu4:   sum of 4 ReLU(N(0,1)) / sqrt(128) (about 6% exact zeros).
    fp16dup: N(0,1) rounded to FP16, then 30% of positions overwritten by a
             copy of another seeded-random position (heavy exact ties).
    Returns (scores, measured fraction of entries equal to another entry)."""
    if dist == "normal":
        s = rng.standard_normal(size=(n_rows, n), dtype=np.float32)
    elif dist == "relu4":
        g = rng.standard_normal(size=(n_rows, n, 4), dtype=np.float32)
        s = (np.maximum(g, 0).sum(-1) / np.float32(np.sqrt(128.0))).astype(np.float32)
    elif dist == "fp16dup":
        s = rng.standard_normal(size=(n_rows, n), dtype=np.float32).astype(np.float16).astype(np.float32)
        m = rng.random(size=(n_rows, n)) < 0.30
        src = rng.integers(0, n, size=(n_rows, n))
        rows = np.arange(n_rows)[:, None].repeat(n, 1)
        s = np.where(m, s[rows, src], s).astype(np.float32)
    else:
        raise ValueError(dist)
    dup = 0.0
    if n > 1:
        fr = []
        for row in s[: min(n_rows, 4)]:
            _, inv, cnt = np.unique(row, return_inverse=True, return_counts=True)
            fr.append(float((cnt[inv] > 1).mean()))
        dup = float(np.mean(fr))
    return np.ascontiguousarray(s), dup


def topk_workload(seed: int, n_rows: int, n: int, k: int = 2048, dist: str = "normal",
                  page_size: int = 64, ragged: bool = False, name: str = "") -> TopkWorkload:
    rng = np.random.default_rng(seed)
    scores, dup = topk_scores(rng, n_rows, n, dist)
    if ragged:
        n_valid = rng.integers(0, n, size=n_rows, endpoint=True).astype(np.int32)
    else:
        n_valid = np.full(n_rows, n, np.int32)
    pages = (n + page_size - 1) // page_size
    perm = rng.permutation(n_rows * pages).astype(np.int32)
    page_table = perm.reshape(n_rows, pages)
    return TopkWorkload(name=name or f"topk_{dist}_{n_rows}x{n}_k{k}", seed=seed, dist=dist, k=k,
                        page_size=page_size, scores=scores, n_valid=n_valid,
                        page_table=np.ascontiguousarray(page_table), dup_fraction=dup)


def c4_dsa_topk(seed: int = 0, dist: str = "normal", n_rows: int = 64, n: int = 80_000,
                k: int = 2048) -> TopkWorkload:
    """Token-level top-2048 over 64 FP32 rows of 80,000 scores."""
    return topk_workload(seed, n_rows, n, k, dist, name=f"dsa_topk_{dist}_{n_rows}x{n}")
