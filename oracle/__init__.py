"""CPU oracle for the QSA indexer and its top-k selection.

TEST INFRASTRUCTURE ONLY.  This package is imported by the tests, by the
smoke check and by the benchmark's CPU-baseline leg, and by nothing else.  It
shares no code with the CUDA library: the arithmetic lives in
``qsa_oracle.c`` (plain C, FP64), and this module only compiles it with gcc
and marshals numpy arrays into it.

BF16 values travel as ``uint16`` bit patterns.  All arrays are C-contiguous
host arrays.  Every function cites, in ``qsa_oracle.c``, the passage it
follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libqsa_oracle.so")
_OMP_PATH = os.path.join(_HERE, "libqsa_oracle_omp.so")
_lock = threading.Lock()
_lib = None

# Plain build: no fast-math and no contraction of a*b+c into FMA, so that x86
# and Arm hosts round every step the same way.
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile ``qsa_oracle.c`` into ``libqsa_oracle.so`` next to it."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_omp(force: bool = False) -> str:
    """The same source built with OpenMP: rows and blocks of the whole-path
    call split over the host cores.  Used only to time the oracle on all
    cores (the tests use the plain build)."""
    if force or not os.path.exists(_OMP_PATH) or os.path.getmtime(_OMP_PATH) < os.path.getmtime(_SRC):
        tmp = _OMP_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *_CFLAGS, "-fopenmp", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _OMP_PATH)
    return _OMP_PATH


_omp_lib = None


def indexer_select_threads(q, pool, req_row_start, row_len, page_table, page_size, k_blk=512, threads=1):
    """indexer_select on `threads` host cores (the OpenMP build); returns
    the same dict.  For timing only."""
    global _omp_lib
    with _lock:
        if _omp_lib is None:
            L = ctypes.CDLL(build_omp())
            p, i64 = ctypes.c_void_p, ctypes.c_int64
            L.oracle_indexer_select.restype = None
            L.oracle_indexer_select.argtypes = [p, p, i64, p, p, p, i64, i64, i64, p, i64, p, p, p]
            L.oracle_set_threads.restype = ctypes.c_int
            L.oracle_set_threads.argtypes = [ctypes.c_int]
            _omp_lib = L
    _omp_lib.oracle_set_threads(int(threads))
    return _indexer_select_with(_omp_lib, q, pool, req_row_start, row_len, page_table, page_size, k_blk)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # A test may point the oracle at a deliberately broken copy of the
            # C source (mutation test of the pins); otherwise build our own.
            path = os.environ.get("QSA_ORACLE_LIB")
            if not path:
                path = build()
            L = ctypes.CDLL(path)
            p, i64, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
            sig = {
                "oracle_bf16_round": (ctypes.c_uint16, [d]),
                "oracle_bf16_round_array": (None, [p, i64, p]),
                "oracle_bf16_to_double": (d, [ctypes.c_uint16]),
                "oracle_slot_of": (i64, [p, i64, i64]),
                "oracle_pool_row": (i64, [p, i64, i64]),
                "oracle_compress_block": (None, [p, i64, d, p]),
                "oracle_compress": (None, [p, i64, p, p, p, i64, i64, d, p]),
                "oracle_score_one": (ctypes.c_float, [p, p]),
                "oracle_index_scores": (None, [p, p, i64, p, p, p, i64, i64, p, i64]),
                "oracle_topk_row": (i64, [p, i64, i64, p]),
                "oracle_topk": (None, [p, i64, p, i64, i64, p, i64, p, i64, p, p]),
                "oracle_expand_row": (None, [p, i64, i64, p, i64, p, p]),
                "oracle_expand": (None, [p, i64, i64, p, p, p, i64, i64, p, p]),
                "oracle_indexer_select": (None, [p, p, i64, p, p, p, i64, i64, i64, p, i64, p, p, p]),
                "oracle_indexshare_row": (ctypes.c_int, [p, i64, i64, i64, i64, p, i64, p, p]),
                "oracle_indexshare": (ctypes.c_int, [p, p, i64, p, i64, i64, i64, p, p, p, i64, i64, p, p]),
                "oracle_append_keys": (None, [p, p, p, i64, p, p, i64, i64, d, p]),
                "oracle_sparse_attn_row": (ctypes.c_int, [p, p, p, i64, i64, i64, i64, p, i64, d, p, p]),
                "oracle_sparse_attn": (ctypes.c_int, [p, p, p, i64, i64, i64, i64, i64, p, i64, i64, d, p, p]),
                "oracle_rope_queries": (None, [p, p, i64, d, p]),
                "oracle_e4m3_to_double": (d, [ctypes.c_uint8]),
                "oracle_e4m3_round": (ctypes.c_uint8, [ctypes.c_float]),
                "oracle_quantize_keys_fp8": (None, [p, i64, p, p]),
                "oracle_f16_round": (d, [d]),
                "oracle_score_one_fp8": (ctypes.c_float, [p, p, ctypes.c_float]),
                "oracle_index_scores_fp8": (None, [p, p, p, i64, p, p, p, i64, i64, p, i64]),
                "oracle_score_one_gated": (ctypes.c_float, [p, p, p]),
                "oracle_index_scores_gated": (None, [p, p, p, i64, p, p, p, i64, i64, p, i64]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


D, H, C = 128, 4, 4  # head dim, index query heads, compression ratio


def out_width(k_blk: int) -> int:
    """Entries per expanded row: 4 positions per selected block plus up to 3
    pending tokens."""
    return C * k_blk + (C - 1)


# ---------------------------------------------------------------- scalars
def bf16_round(x: float) -> int:
    return int(_load().oracle_bf16_round(float(x)))


def bf16_round_array(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_bf16_round_array(_ptr(x), x.size, _ptr(out))
    return out


def bf16_to_float(bits) -> np.ndarray:
    """BF16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def slot_of(pt_row, pos: int, page_size: int) -> int:
    pt_row = _c(pt_row, np.int32)
    return int(_load().oracle_slot_of(_ptr(pt_row), int(pos), int(page_size)))


def pool_row(pt_row, b: int, page_size: int) -> int:
    pt_row = _c(pt_row, np.int32)
    return int(_load().oracle_pool_row(_ptr(pt_row), int(b), int(page_size)))


# ---------------------------------------------------------------- compress
def compress_block(raw4, first_pos: int, rope_base: float = 10000.0) -> np.ndarray:
    raw4 = _c(raw4, np.uint16).reshape(C, D)
    out = np.empty(D, np.uint16)
    _load().oracle_compress_block(_ptr(raw4), int(first_pos), float(rope_base), _ptr(out))
    return out


def compress(raw, block_req, block_id, page_table, page_size, rope_base, pool):
    """raw: [n_blocks*4][128] u16.  Writes into ``pool`` ([rows][128] u16) in
    place and returns it.  page_table None -> block i goes to pool row i."""
    raw = _c(raw, np.uint16)
    n_blocks = raw.size // (C * D)
    block_req = _c(block_req, np.int32)
    block_id = _c(block_id, np.int32)
    pt = _c(page_table, np.int32)
    ld_pt = 0 if pt is None else pt.shape[-1]
    assert pool.dtype == np.uint16 and pool.flags.c_contiguous
    _load().oracle_compress(_ptr(raw), n_blocks, _ptr(block_req), _ptr(block_id), _ptr(pt), ld_pt,
                            int(page_size), float(rope_base), _ptr(pool))
    return pool


# ---------------------------------------------------------------- scores
def score_one(q_row, key) -> float:
    q_row = _c(q_row, np.uint16).reshape(H, D)
    key = _c(key, np.uint16).reshape(D)
    return float(_load().oracle_score_one(_ptr(q_row), _ptr(key)))


def index_scores(q, pool, req_row_start, row_len, page_table, page_size, ld_scores=None,
                 fill=np.nan):
    """q: [n_rows][4][128] u16.  Returns scores [n_rows][ld] float32; entries
    b >= row_len/4 hold ``fill``."""
    q = _c(q, np.uint16)
    rrs = _c(req_row_start, np.int32)
    rl = _c(row_len, np.int32)
    pt = _c(page_table, np.int32)
    n_rows = rl.size
    if ld_scores is None:
        ld_scores = max(1, int(rl.max()) // C) if n_rows else 1
    out = np.full((n_rows, ld_scores), fill, np.float32)
    _load().oracle_index_scores(_ptr(q), _ptr(pool), rrs.size - 1, _ptr(rrs), _ptr(rl), _ptr(pt),
                                pt.shape[-1], int(page_size), _ptr(out), ld_scores)
    return out


# ---------------------------------------------------------------- top-k
def topk_row(s, k: int) -> np.ndarray:
    s = _c(s, np.float32)
    out = np.empty(k, np.int32)
    _load().oracle_topk_row(_ptr(s), s.size, int(k), _ptr(out))
    return out


def topk(scores, k, n_valid=None, page_table=None, row_req=None, page_size=0):
    """scores: [n_rows][ld] float32.  Returns (idx [n_rows][k], slots or None)."""
    s = _c(scores, np.float32)
    n_rows, ld = s.shape
    nv = _c(n_valid, np.int32)
    pt = _c(page_table, np.int32)
    rr = _c(row_req, np.int32)
    idx = np.empty((n_rows, k), np.int32)
    slots = np.empty((n_rows, k), np.int32) if pt is not None else None
    _load().oracle_topk(_ptr(s), ld, _ptr(nv), n_rows, int(k), _ptr(pt),
                        0 if pt is None else pt.shape[-1], _ptr(rr), int(page_size), _ptr(idx),
                        _ptr(slots))
    return idx, slots


# ---------------------------------------------------------------- expand
def expand_row(sel, L, pt_row, page_size):
    sel = _c(sel, np.int32)
    pt_row = _c(pt_row, np.int32)
    w = out_width(sel.size)
    pos = np.empty(w, np.int32)
    slots = np.empty(w, np.int32)
    _load().oracle_expand_row(_ptr(sel), sel.size, int(L), _ptr(pt_row), int(page_size),
                              _ptr(pos), _ptr(slots))
    return pos, slots


def expand(sel, req_row_start, row_len, page_table, page_size):
    sel = _c(sel, np.int32)
    n_rows, k_blk = sel.shape
    rrs = _c(req_row_start, np.int32)
    rl = _c(row_len, np.int32)
    pt = _c(page_table, np.int32)
    w = out_width(k_blk)
    pos = np.empty((n_rows, w), np.int32)
    slots = np.empty((n_rows, w), np.int32)
    _load().oracle_expand(_ptr(sel), k_blk, rrs.size - 1, _ptr(rrs), _ptr(rl), _ptr(pt),
                          pt.shape[-1], int(page_size), _ptr(pos), _ptr(slots))
    return pos, slots


# ---------------------------------------------------------------- whole path
def indexer_select(q, pool, req_row_start, row_len, page_table, page_size, k_blk=512):
    """Returns dict(scores, blocks, pos, slots)."""
    return _indexer_select_with(_load(), q, pool, req_row_start, row_len, page_table, page_size, k_blk)


def _indexer_select_with(L, q, pool, req_row_start, row_len, page_table, page_size, k_blk):
    q = _c(q, np.uint16)
    rrs = _c(req_row_start, np.int32)
    rl = _c(row_len, np.int32)
    pt = _c(page_table, np.int32)
    n_rows = rl.size
    ld = max(1, int(rl.max()) // C) if n_rows else 1
    scores = np.full((n_rows, ld), np.nan, np.float32)
    blocks = np.empty((n_rows, k_blk), np.int32)
    w = out_width(k_blk)
    pos = np.empty((n_rows, w), np.int32)
    slots = np.empty((n_rows, w), np.int32)
    L.oracle_indexer_select(_ptr(q), _ptr(pool), rrs.size - 1, _ptr(rrs), _ptr(rl),
                            _ptr(pt), pt.shape[-1], int(page_size), int(k_blk),
                            _ptr(scores), ld, _ptr(blocks), _ptr(pos), _ptr(slots))
    return {"scores": scores, "blocks": blocks, "pos": pos, "slots": slots}


# ---------------------------------------------------------------- IndexShare
def indexshare_width(k_blk: int, n_extra: int) -> int:
    """Entries per reused row: the expanded width plus the drafted columns."""
    return out_width(k_blk) + n_extra


def indexshare_row(cap_sel, cap_len, n_extra, L, pt_row, page_size):
    """Returns (pos, slots, flags) of one draft row reading a captured row."""
    cap_sel = _c(cap_sel, np.int32)
    pt_row = _c(pt_row, np.int32)
    w = indexshare_width(cap_sel.size, n_extra)
    pos = np.empty(w, np.int32)
    slots = np.empty(w, np.int32)
    f = _load().oracle_indexshare_row(_ptr(cap_sel), cap_sel.size, int(cap_len), int(n_extra), int(L),
                                      _ptr(pt_row), int(page_size), _ptr(pos), _ptr(slots))
    return pos, slots, int(f)


def indexshare(cap_sel, cap_len, cap_row, n_extra, req_row_start, row_len, page_table, page_size):
    """cap_sel [n_cap][k_blk], cap_len [n_cap], cap_row [n_req].  Returns
    (pos, slots, flags) for every row."""
    cap_sel = _c(cap_sel, np.int32)
    n_cap, k_blk = cap_sel.shape
    cl = _c(cap_len, np.int32)
    cr = _c(cap_row, np.int32)
    rrs = _c(req_row_start, np.int32)
    rl = _c(row_len, np.int32)
    pt = _c(page_table, np.int32)
    w = indexshare_width(k_blk, n_extra)
    pos = np.empty((rl.size, w), np.int32)
    slots = np.empty((rl.size, w), np.int32)
    f = _load().oracle_indexshare(_ptr(cap_sel), _ptr(cl), n_cap, _ptr(cr), k_blk, int(n_extra),
                                  rrs.size - 1, _ptr(rrs), _ptr(rl), _ptr(pt), pt.shape[-1],
                                  int(page_size), _ptr(pos), _ptr(slots))
    return pos, slots, int(f)


# ---------------------------------------------------------------- sparse attention
def sparse_attn(q, k, v, slots, scale):
    """q [n_rows][H_q][d] u16, k/v [n_slots][H_kv][d] u16, slots [n_rows][n_idx]
    int32 (-1 masked).  Returns (out [n_rows][H_q][d] f32, lse [n_rows][H_q]
    f32, flags)."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sl = _c(slots, np.int32)
    n_rows, h_q, d = q.shape
    n_slots, h_kv, _ = k.shape
    n_idx = sl.shape[1]
    out = np.empty((n_rows, h_q, d), np.float32)
    lse = np.empty((n_rows, h_q), np.float32)
    f = _load().oracle_sparse_attn(_ptr(q), _ptr(k), _ptr(v), n_slots, n_rows, h_q, h_kv, d, _ptr(sl),
                                   n_idx, n_idx, float(scale), _ptr(out), _ptr(lse))
    return out, lse, int(f)


# ---------------------------------------------------------------- key path
def append_keys(new_keys, req_tok_start, req_first_pos, ring, page_table, page_size, rope_base, pool):
    """Appends raw keys per request (ring [n_req][4][128] u16 and pool
    updated in place); returns (ring, pool)."""
    nk = _c(new_keys, np.uint16)
    rts = _c(req_tok_start, np.int32)
    rfp = _c(req_first_pos, np.int32)
    pt = _c(page_table, np.int32)
    assert ring.dtype == np.uint16 and ring.flags.c_contiguous
    assert pool.dtype == np.uint16 and pool.flags.c_contiguous
    _load().oracle_append_keys(_ptr(nk), _ptr(rts), _ptr(rfp), rts.size - 1, _ptr(ring), _ptr(pt),
                               pt.shape[-1], int(page_size), float(rope_base), _ptr(pool))
    return ring, pool


# ---------------------------------------------------------------- prologue tails
def rope_queries(q, pos, rope_base=10000.0):
    """q [n_rows][4][128] u16 (BF16 bits), pos [n_rows] -> the rotated query."""
    q = _c(q, np.uint16)
    pos = _c(pos, np.int32)
    out = np.empty_like(q)
    _load().oracle_rope_queries(_ptr(q), _ptr(pos), pos.size, float(rope_base), _ptr(out))
    return out


def e4m3_to_float(code: int) -> float:
    return float(_load().oracle_e4m3_to_double(int(code)))


def e4m3_round(x: float) -> int:
    return int(_load().oracle_e4m3_round(float(x)))


def f16_round(x: float) -> float:
    return float(_load().oracle_f16_round(float(x)))


def quantize_keys_fp8(keys):
    """keys [n][128] u16 (BF16 bits) -> (codes [n][128] u8, scales [n] f32)."""
    keys = _c(keys, np.uint16)
    n = keys.shape[0]
    codes = np.empty((n, 128), np.uint8)
    scales = np.empty(n, np.float32)
    _load().oracle_quantize_keys_fp8(_ptr(keys), n, _ptr(codes), _ptr(scales))
    return codes, scales


def score_one_fp8(q_row, codes, scale) -> float:
    q_row = _c(q_row, np.uint16)
    codes = _c(codes, np.uint8)
    return float(_load().oracle_score_one_fp8(_ptr(q_row), _ptr(codes), float(scale)))


def index_scores_fp8(q, codes, scales, req_row_start, row_len, page_table, page_size, ld_scores=None):
    """index_scores with FP8 keys (codes [pool_rows][128] u8, scales [pool_rows]);
    entries b >= row_len/4 are NaN."""
    q = _c(q, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    rrs = _c(req_row_start, np.int32)
    rl = _c(row_len, np.int32)
    pt = _c(page_table, np.int32)
    n_rows = rl.size
    if ld_scores is None:
        ld_scores = max(1, int(rl.max()) // C) if n_rows else 1
    out = np.full((n_rows, ld_scores), np.nan, np.float32)
    _load().oracle_index_scores_fp8(_ptr(q), _ptr(codes), _ptr(scales), rrs.size - 1, _ptr(rrs), _ptr(rl),
                                    _ptr(pt), pt.shape[-1], int(page_size), _ptr(out), ld_scores)
    return out


def score_one_gated(q_row, gates, key) -> float:
    """(1/sqrt(128)) sum_h gates[h] ReLU(<q_h, key>): q_row [4][128] and key
    [128] u16 (BF16 bits), gates [4] float32."""
    q_row = _c(q_row, np.uint16)
    gates = _c(gates, np.float32)
    key = _c(key, np.uint16)
    return float(_load().oracle_score_one_gated(_ptr(q_row), _ptr(gates), _ptr(key)))


def index_scores_gated(q, gates, pool, req_row_start, row_len, page_table, page_size, ld_scores=None):
    """index_scores with a gate per row and head (gates [n_rows][4] float32);
    entries b >= row_len/4 are NaN."""
    q = _c(q, np.uint16)
    gates = _c(gates, np.float32)
    pool = _c(pool, np.uint16)
    rrs = _c(req_row_start, np.int32)
    rl = _c(row_len, np.int32)
    pt = _c(page_table, np.int32)
    n_rows = rl.size
    if ld_scores is None:
        ld_scores = max(1, int(rl.max()) // C) if n_rows else 1
    out = np.full((n_rows, ld_scores), np.nan, np.float32)
    _load().oracle_index_scores_gated(_ptr(q), _ptr(gates), _ptr(pool), rrs.size - 1, _ptr(rrs), _ptr(rl),
                                      _ptr(pt), pt.shape[-1], int(page_size), _ptr(out), ld_scores)
    return out
