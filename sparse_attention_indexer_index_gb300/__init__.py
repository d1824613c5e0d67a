"""GB300-native QSA sparse-attention indexer and top-k selection.

A thin Python binding over the C ABI of ``libqsa.so`` (declared in
``include/qsa.h``).  Every step of the path runs in the library's CUDA
kernels; this module only checks tensor placement and dtypes, passes raw
device pointers and the current CUDA stream, and turns a non-zero status into
an exception.  PyTorch provides device memory and streams.

There is no CPU fallback: if the library is missing the import of the
functions below fails loudly.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB_PATH, build  # noqa: F401

__all__ = [
    "build", "lib", "QSAError", "compress_keys", "index_scores", "topk_select", "expand_slots",
    "indexer_select", "indexer_select_workspace_size", "device_status", "out_width",
    "select_blocks", "indexshare_slots", "indexshare_width", "sparse_attn", "append_keys", "decode_step",
    "rope_queries", "quantize_keys_fp8", "index_scores_fp8", "indexer_select_fp8", "index_scores_gated",
    "indexer_select_gated",
    "HEAD_DIM", "HEADS", "BLOCK", "MAX_K",
]

HEAD_DIM, HEADS, BLOCK, MAX_K = 128, 4, 4, 2048
_lib = None


class QSAError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} failed: {lib().qsa_status_string(status).decode()} (status {status})")
        self.status = status


def lib():
    """The loaded ``libqsa.so`` (ctypes), with argument types declared."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libqsa.so not built at {LIB_PATH}: run build() first "
                              "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        p, i32, i64, sz, d = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t,
                              ctypes.c_double)
        sig = {
            "qsa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "qsa_version": (ctypes.c_int, []),
            "qsa_device_status": (ctypes.c_int, [p, ctypes.c_int, p]),
            "qsa_compress_keys": (ctypes.c_int, [p, p, p, i64, i32, p, i64, i32, d, p, i64, p]),
            "qsa_append_keys": (ctypes.c_int, [p, p, p, i32, p, p, i64, i32, d, p, i64, p]),
            "qsa_decode_step": (ctypes.c_int, [p, p, p, p, d, p, p, i64, i32, p, i32, p, i32, i32, p, i64, i32,
                                               i32, p, p, p, p, i64, p, sz, p]),
            "qsa_index_scores": (ctypes.c_int, [p, p, i64, i32, p, i32, p, i32, i32, p, i64, i32, p,
                                                i64, i64, p]),
            "topk_select_workspace_size": (sz, [i32, i32, i32]),
            "topk_select": (ctypes.c_int, [p, i64, p, i32, i32, i32, p, i64, p, i32, p, p, p, sz, p]),
            "qsa_expand_slots": (ctypes.c_int, [p, i32, i32, p, i32, p, p, i64, i32, p, p, p]),
            "qsa_select_blocks": (ctypes.c_int, [p, i64, i32, p, i32, p, i32, p, i64, i32, i32, p, p, p,
                                                 p]),
            "qsa_indexshare_slots": (ctypes.c_int, [p, p, i32, p, i32, i32, i32, p, i32, p, p, i64, i32,
                                                    p, p, p]),
            "qsa_sparse_attn_workspace_size": (sz, [i32, i32, i32, i32]),
            "qsa_sparse_attn": (ctypes.c_int, [p, p, p, i64, i32, i32, i32, i32, p, i64, i32,
                                               ctypes.c_float, p, p, p, sz, p]),
            "qsa_indexer_select_workspace_size": (sz, [i32, i32, i32]),
            "qsa_indexer_select": (ctypes.c_int, [p, p, i64, i32, p, i32, p, i32, i32, p, i64, i32,
                                                  i32, p, p, p, p, i64, p, sz, p]),
            "qsa_rope_queries": (ctypes.c_int, [p, p, i32, d, p, p]),
            "qsa_quantize_keys_fp8": (ctypes.c_int, [p, i64, p, p, p]),
            "qsa_index_scores_fp8": (ctypes.c_int, [p, p, p, i64, i32, p, i32, p, i32, i32, p, i64, i32, p,
                                                    i64, i64, p]),
            "qsa_indexer_select_fp8": (ctypes.c_int, [p, p, p, i64, i32, p, i32, p, i32, i32, p, i64, i32,
                                                      i32, p, p, p, p, i64, p, sz, p]),
            "qsa_index_scores_gated": (ctypes.c_int, [p, p, p, i64, i32, p, i32, p, i32, i32, p, i64, i32, p,
                                                      i64, i64, p]),
            "qsa_decode_step_gated": (ctypes.c_int, [p, p, p, p, d, p, p, p, i64, i32, p, i32, p, i32, i32, p,
                                                     i64, i32, i32, p, p, p, p, i64, p, sz, p]),
            "qsa_indexer_select_gated": (ctypes.c_int, [p, p, p, i64, i32, p, i32, p, i32, i32, p, i64, i32,
                                                        i32, p, p, p, p, i64, p, sz, p]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ----------------------------------------------------------------- helpers
def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else t.data_ptr()


_raw_stream = None


def _stream(stream=None, device=None):
    """The CUDA stream handle: `stream`'s, else the current stream of
    `device` (a tensor's device; the current device if None)."""
    global _raw_stream
    torch = _torch()
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is None:  # the raw query avoids building a Stream object per call
        _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", False)
    if _raw_stream:
        idx = device.index if device is not None and device.index is not None else torch.cuda.current_device()
        return _raw_stream(idx)
    return torch.cuda.current_stream(device).cuda_stream


def _dev(t, dtype, name, ndim=None):
    # one pass of cheap attribute checks; the precise message only on failure
    try:
        ok = t.is_cuda and t.dtype is dtype and t.is_contiguous() and (ndim is None or t.dim() == ndim)
    except AttributeError:
        ok = False
    if not ok:
        _dev_error(t, dtype, name, ndim)
    return t


def _dev_error(t, dtype, name, ndim):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    raise ValueError(f"{name} must have {ndim} dims")


_fast = None


def _call(fn, *args):
    """Call the C entry point `fn`: through the CPython entry points of
    _fastcall.c when they were built (the per-step calls), else ctypes."""
    global _fast
    if _fast is None:
        lib()
        try:
            from . import _fastcall as m
        except ImportError:
            m = False
        _fast = m
    f = getattr(_fast, fn, None) if _fast else None
    return (f or getattr(lib(), fn))(*args)


def _check(fn, status):
    if status != 0:
        raise QSAError(fn, status)


def out_width(k_blk: int) -> int:
    """Entries per expanded row: 4 positions per block plus 3 pending slots."""
    return BLOCK * k_blk + (BLOCK - 1)


# ----------------------------------------------------------------- entry points
def device_status(clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return the device fault bits (0 = none)."""
    bits = ctypes.c_uint32(0)
    lib().qsa_device_status(_stream(stream), int(clear), ctypes.byref(bits))
    return int(bits.value)


def compress_keys(raw, block_id, pool, block_req=None, page_table=None, page_size=0,
                  rope_base=10000.0, stream=None):
    """raw [n_blocks*4][128] bf16 -> pool rows (in place).  With a page table,
    block i of request block_req[i] goes to pool row slot(4*block_id[i])/4."""
    torch = _torch()
    _dev(raw, torch.bfloat16, "raw", 2)
    _dev(block_id, torch.int32, "block_id", 1)
    _dev(pool, torch.bfloat16, "pool", 2)
    n_blocks = block_id.numel()
    if raw.shape[0] != 4 * n_blocks or raw.shape[1] != HEAD_DIM:
        raise ValueError("raw must be [4*n_blocks][128]")
    n_req, ld_pt = 0, 0
    if page_table is not None:
        _dev(page_table, torch.int32, "page_table", 2)
        _dev(block_req, torch.int32, "block_req", 1)
        n_req, ld_pt = page_table.shape
    _check("qsa_compress_keys", lib().qsa_compress_keys(
        _ptr(raw), _ptr(block_req), _ptr(block_id), n_blocks, n_req, _ptr(page_table), ld_pt,
        int(page_size), float(rope_base), _ptr(pool), pool.shape[0], _stream(stream)))
    return pool


def append_keys(new_keys, req_tok_start, req_first_pos, ring, pool, page_table, page_size, rope_base=10000.0,
                stream=None):
    """Decode key path: appends raw keys [n_tok][128] bf16 per request into
    the 4-slot ring [n_req][4][128] and compresses the completed blocks into
    the pool (both updated in place)."""
    torch = _torch()
    _dev(new_keys, torch.bfloat16, "new_keys", 2)
    _dev(req_tok_start, torch.int32, "req_tok_start", 1)
    _dev(req_first_pos, torch.int32, "req_first_pos", 1)
    _dev(ring, torch.bfloat16, "ring", 3)
    _dev(pool, torch.bfloat16, "pool", 2)
    _dev(page_table, torch.int32, "page_table", 2)
    n_req = req_first_pos.numel()
    if req_tok_start.numel() != n_req + 1 or tuple(ring.shape) != (n_req, BLOCK, HEAD_DIM):
        raise ValueError("req_tok_start must have n_req+1 entries and ring be [n_req][4][128]")
    _check("qsa_append_keys", lib().qsa_append_keys(
        _ptr(new_keys), _ptr(req_tok_start), _ptr(req_first_pos), n_req, _ptr(ring), _ptr(page_table),
        page_table.shape[1], int(page_size), float(rope_base), _ptr(pool), pool.shape[0], _stream(stream)))
    return ring, pool


def decode_step(new_keys, req_tok_start, req_first_pos, ring, q, pool, req_row_start, row_len, page_table,
                page_size, max_len, max_rows_per_req=None, k_blk=512, rope_base=10000.0, want_blocks=False,
                want_pos=False, out_slots=None, scores_out=None, workspace=None, stream=None, head_gates=None):
    """Key path (append_keys) then the fused indexer (indexer_select) in one
    call; returns dict(slots, blocks?, pos?) like indexer_select.  head_gates
    [n_rows][4] float32: gated scores (qsa_decode_step_gated)."""
    torch = _torch()
    if head_gates is not None:
        _gates(head_gates, row_len)
    for t, nm in [(new_keys, "new_keys"), (q, "q"), (pool, "pool"), (ring, "ring")]:
        _dev(t, torch.bfloat16, nm)
    for t, nm in [(req_tok_start, "req_tok_start"), (req_first_pos, "req_first_pos"),
                  (req_row_start, "req_row_start"), (row_len, "row_len"), (page_table, "page_table")]:
        _dev(t, torch.int32, nm)
    n_req = req_row_start.numel() - 1
    if req_first_pos.numel() != n_req or req_tok_start.numel() != n_req + 1:
        raise ValueError("req_first_pos / req_tok_start must describe the same requests as req_row_start")
    n_rows = row_len.numel()
    if max_rows_per_req is None:
        max_rows_per_req = n_rows
    dev = q.device
    w = out_width(k_blk)
    if out_slots is None:
        out_slots = torch.empty((n_rows, w), dtype=torch.int32, device=dev)
    blocks = torch.empty((n_rows, k_blk), dtype=torch.int32, device=dev) if want_blocks else None
    pos = torch.empty((n_rows, w), dtype=torch.int32, device=dev) if want_pos else None
    ld = 0
    if scores_out is not None:
        _dev(scores_out, torch.float32, "scores_out", 2)
        ld = scores_out.shape[1]
    elif workspace is None:
        nbytes = indexer_select_workspace_size(n_rows, max_len, k_blk)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    fn = "qsa_decode_step" if head_gates is None else "qsa_decode_step_gated"
    gate_args = () if head_gates is None else (_ptr(head_gates),)
    _check(fn, _call(
        fn, _ptr(new_keys), _ptr(req_tok_start), _ptr(req_first_pos), _ptr(ring), float(rope_base), _ptr(q),
        *gate_args, _ptr(pool), pool.shape[0], n_req, _ptr(req_row_start), n_rows, _ptr(row_len), int(max_len),
        int(max_rows_per_req), _ptr(page_table), page_table.shape[1], int(page_size), int(k_blk), _ptr(blocks),
        _ptr(pos), _ptr(out_slots), _ptr(scores_out), ld, _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream, q.device)))
    out = {"slots": out_slots}
    if blocks is not None:
        out["blocks"] = blocks
    if pos is not None:
        out["pos"] = pos
    return out


def index_scores(q, pool, req_row_start, row_len, page_table, page_size, max_len,
                 max_rows_per_req=None, scores=None, n_fill=0, stream=None):
    """Block scores [n_rows][ld] float32 (entries b < row_len/4 written,
    [row_len/4, n_fill) set to -inf)."""
    torch = _torch()
    _dev(pool, torch.bfloat16, "pool", 2)
    return _index_scores_call("qsa_index_scores", (_ptr(pool),), pool.shape[0], q, req_row_start, row_len,
                              page_table, page_size, max_len, max_rows_per_req, scores, n_fill, stream)


def index_scores_fp8(q, codes, scales, req_row_start, row_len, page_table, page_size, max_len,
                     max_rows_per_req=None, scores=None, n_fill=0, stream=None):
    """index_scores on FP8 keys: codes [pool_rows][128] uint8 (e4m3) and
    scales [pool_rows] float32 from quantize_keys_fp8."""
    torch = _torch()
    _dev(codes, torch.uint8, "codes", 2)
    _dev(scales, torch.float32, "scales", 1)
    if scales.numel() != codes.shape[0]:
        raise ValueError("scales must have one entry per key")
    return _index_scores_call("qsa_index_scores_fp8", (_ptr(codes), _ptr(scales)), codes.shape[0], q,
                              req_row_start, row_len, page_table, page_size, max_len, max_rows_per_req,
                              scores, n_fill, stream)


def index_scores_gated(q, head_gates, pool, req_row_start, row_len, page_table, page_size, max_len,
                       max_rows_per_req=None, scores=None, n_fill=0, stream=None):
    """index_scores with a gate per row and head: head_gates [n_rows][4]
    float32 multiplies each head's rectified dot product before the sum."""
    torch = _torch()
    _dev(pool, torch.bfloat16, "pool", 2)
    _gates(head_gates, row_len)
    return _index_scores_call("qsa_index_scores_gated", (_ptr(head_gates), _ptr(pool)), pool.shape[0], q,
                              req_row_start, row_len, page_table, page_size, max_len, max_rows_per_req, scores,
                              n_fill, stream)


def _gates(head_gates, row_len):
    torch = _torch()
    _dev(head_gates, torch.float32, "head_gates", 2)
    if head_gates.shape[1] != HEADS or head_gates.shape[0] != row_len.numel():
        raise ValueError("head_gates must be [n_rows][4]")


def _index_scores_call(fn, key_ptrs, pool_rows, q, req_row_start, row_len, page_table, page_size, max_len,
                       max_rows_per_req, scores, n_fill, stream):
    torch = _torch()
    _dev(q, torch.bfloat16, "q", 3)
    _dev(req_row_start, torch.int32, "req_row_start", 1)
    _dev(row_len, torch.int32, "row_len", 1)
    _dev(page_table, torch.int32, "page_table", 2)
    n_rows = row_len.numel()
    if max_rows_per_req is None:
        max_rows_per_req = n_rows
    if scores is None:
        ld = max(1, (max(int(max_len) // BLOCK, int(n_fill)) + 3) // 4 * 4)
        scores = torch.empty((n_rows, ld), dtype=torch.float32, device=q.device)
    _dev(scores, torch.float32, "scores", 2)
    _check(fn, _call(
        fn, _ptr(q), *key_ptrs, pool_rows, req_row_start.numel() - 1, _ptr(req_row_start), n_rows,
        _ptr(row_len), int(max_len), int(max_rows_per_req), _ptr(page_table), page_table.shape[1],
        int(page_size), _ptr(scores), scores.shape[1], int(n_fill), _stream(stream)))
    return scores


def rope_queries(q, pos, out=None, rope_base=10000.0, stream=None):
    """Index-query RoPE: q [n_rows][4][128] bf16 rotated (rotate-half) at
    pos [n_rows] int32; out may be q itself.  Returns out."""
    torch = _torch()
    _dev(q, torch.bfloat16, "q", 3)
    _dev(pos, torch.int32, "pos", 1)
    if pos.numel() != q.shape[0]:
        raise ValueError("pos must have one entry per row")
    if out is None:
        out = torch.empty_like(q)
    _dev(out, torch.bfloat16, "out", 3)
    _check("qsa_rope_queries", lib().qsa_rope_queries(
        _ptr(q), _ptr(pos), q.shape[0], float(rope_base), _ptr(out), _stream(stream)))
    return out


def quantize_keys_fp8(keys, codes=None, scales=None, stream=None):
    """Compressed keys [n][128] bf16 -> (codes [n][128] uint8 e4m3,
    scales [n] float32), scale = max|k| / 448 per key."""
    torch = _torch()
    _dev(keys, torch.bfloat16, "keys", 2)
    n = keys.shape[0]
    if codes is None:
        codes = torch.empty((n, keys.shape[1]), dtype=torch.uint8, device=keys.device)
    if scales is None:
        scales = torch.empty(n, dtype=torch.float32, device=keys.device)
    _dev(codes, torch.uint8, "codes", 2)
    _dev(scales, torch.float32, "scales", 1)
    _check("qsa_quantize_keys_fp8", lib().qsa_quantize_keys_fp8(
        _ptr(keys), n, _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


def topk_select(scores, k, n_valid=None, n_max=None, page_table=None, row_req=None, page_size=0,
                out_idx=None, out_slots=None, want_slots=None, workspace=None, stream=None):
    """Exact top-k per row, ascending indices, -1 padded; optionally slots.
    workspace: None (allocated from the size query: room for the device row
    plan), or a uint8 tensor (an empty one: no plan).  Returns (idx, slots or
    None)."""
    torch = _torch()
    _dev(scores, torch.float32, "scores", 2)
    n_rows, ld = scores.shape
    if n_valid is not None:
        _dev(n_valid, torch.int32, "n_valid", 1)
    if n_max is None:
        n_max = ld
    if page_table is not None:
        _dev(page_table, torch.int32, "page_table", 2)
    if row_req is not None:
        _dev(row_req, torch.int32, "row_req", 1)
    if want_slots is None:
        want_slots = page_table is not None
    if out_idx is None:
        out_idx = torch.empty((n_rows, k), dtype=torch.int32, device=scores.device)
    if want_slots and out_slots is None:
        out_slots = torch.empty((n_rows, k), dtype=torch.int32, device=scores.device)
    if workspace is None:
        ws_bytes = lib().topk_select_workspace_size(n_rows, int(n_max), int(k))
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=scores.device) if ws_bytes else None
    else:
        ws_bytes = workspace.numel() * workspace.element_size()
        ws = workspace if ws_bytes else None
    _check("topk_select", lib().topk_select(
        _ptr(scores), ld, _ptr(n_valid), n_rows, int(n_max), int(k), _ptr(page_table),
        0 if page_table is None else page_table.shape[1], _ptr(row_req), int(page_size),
        _ptr(out_idx), _ptr(out_slots), _ptr(ws), ws_bytes, _stream(stream)))
    return out_idx, out_slots


def expand_slots(sel_blocks, req_row_start, row_len, page_table, page_size, want_pos=True,
                 stream=None):
    """Selected blocks [n_rows][k] -> (positions or None, slots) [n_rows][4k+3]."""
    torch = _torch()
    _dev(sel_blocks, torch.int32, "sel_blocks", 2)
    _dev(req_row_start, torch.int32, "req_row_start", 1)
    _dev(row_len, torch.int32, "row_len", 1)
    _dev(page_table, torch.int32, "page_table", 2)
    n_rows, k = sel_blocks.shape
    w = out_width(k)
    slots = torch.empty((n_rows, w), dtype=torch.int32, device=sel_blocks.device)
    pos = torch.empty((n_rows, w), dtype=torch.int32, device=sel_blocks.device) if want_pos else None
    _check("qsa_expand_slots", lib().qsa_expand_slots(
        _ptr(sel_blocks), k, req_row_start.numel() - 1, _ptr(req_row_start), n_rows, _ptr(row_len),
        _ptr(page_table), page_table.shape[1], int(page_size), _ptr(pos), _ptr(slots),
        _stream(stream)))
    return pos, slots


def indexshare_width(k_blk: int, n_extra: int) -> int:
    """Entries per reused row: the expanded width plus the drafted columns."""
    return out_width(k_blk) + int(n_extra)


def indexshare_slots(cap_blocks, cap_len, cap_row, n_extra, req_row_start, row_len, page_table,
                     page_size, want_pos=True, out_slots=None, stream=None):
    """Draft rows read a kept selection (IndexShare): cap_blocks [n_cap][k]
    with cap_len [n_cap]; request r reads kept row cap_row[r].
    Returns (positions or None, slots) [n_rows][4k+3+n_extra]."""
    torch = _torch()
    _dev(cap_blocks, torch.int32, "cap_blocks", 2)
    _dev(cap_len, torch.int32, "cap_len", 1)
    _dev(cap_row, torch.int32, "cap_row", 1)
    _dev(req_row_start, torch.int32, "req_row_start", 1)
    _dev(row_len, torch.int32, "row_len", 1)
    _dev(page_table, torch.int32, "page_table", 2)
    n_cap, k = cap_blocks.shape
    if cap_len.numel() != n_cap or cap_row.numel() != req_row_start.numel() - 1:
        raise ValueError("cap_len must have n_cap entries and cap_row one per request")
    n_rows = row_len.numel()
    w = indexshare_width(k, n_extra)
    dev = cap_blocks.device
    if out_slots is None:
        out_slots = torch.empty((n_rows, w), dtype=torch.int32, device=dev)
    _dev(out_slots, torch.int32, "out_slots", 2)
    pos = torch.empty((n_rows, w), dtype=torch.int32, device=dev) if want_pos else None
    _check("qsa_indexshare_slots", lib().qsa_indexshare_slots(
        _ptr(cap_blocks), _ptr(cap_len), n_cap, _ptr(cap_row), k, int(n_extra),
        req_row_start.numel() - 1, _ptr(req_row_start), n_rows, _ptr(row_len), _ptr(page_table),
        page_table.shape[1], int(page_size), _ptr(pos), _ptr(out_slots), _stream(stream)))
    return pos, out_slots


def sparse_attn(q, k_cache, v_cache, slots, scale=None, n_idx=None, out=None, lse=None, want_lse=True,
                workspace=None, stream=None):
    """Softmax attention of q [n_rows][h_q][d] over the K/V rows
    [n_slots][h_kv][d] (bf16) at slots [n_rows][w] (int32, -1 skipped).
    Returns (out [n_rows][h_q][d] float32, lse [n_rows][h_q] or None)."""
    torch = _torch()
    _dev(q, torch.bfloat16, "q", 3)
    _dev(k_cache, torch.bfloat16, "k_cache", 3)
    _dev(v_cache, torch.bfloat16, "v_cache", 3)
    _dev(slots, torch.int32, "slots", 2)
    n_rows, h_q, d = q.shape
    n_slots, h_kv, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape) or slots.shape[0] != n_rows:
        raise ValueError("q, k_cache, v_cache and slots shapes disagree")
    if n_idx is None:
        n_idx = slots.shape[1]
    if scale is None:
        scale = d ** -0.5
    dev = q.device
    if out is None:
        out = torch.empty((n_rows, h_q, d), dtype=torch.float32, device=dev)
    if want_lse and lse is None:
        lse = torch.empty((n_rows, h_q), dtype=torch.float32, device=dev)
    ws_bytes = lib().qsa_sparse_attn_workspace_size(n_rows, h_q, d, int(n_idx))
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _check("qsa_sparse_attn", lib().qsa_sparse_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), n_slots, n_rows, h_q, h_kv, d, _ptr(slots), slots.shape[1],
        int(n_idx), float(scale), _ptr(out), _ptr(lse if want_lse else None), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream)))
    return out, (lse if want_lse else None)


def select_blocks(scores, req_row_start, row_len, page_table, page_size, max_len, k_blk=512,
                  want_blocks=False, want_pos=False, out_slots=None, stream=None):
    """Top-k_blk blocks of given scores -> expand -> slots.
    Returns dict(slots, blocks?, pos?)."""
    torch = _torch()
    _dev(scores, torch.float32, "scores", 2)
    _dev(req_row_start, torch.int32, "req_row_start", 1)
    _dev(row_len, torch.int32, "row_len", 1)
    _dev(page_table, torch.int32, "page_table", 2)
    n_rows = row_len.numel()
    dev = scores.device
    w = out_width(k_blk)
    if out_slots is None:
        out_slots = torch.empty((n_rows, w), dtype=torch.int32, device=dev)
    blocks = torch.empty((n_rows, k_blk), dtype=torch.int32, device=dev) if want_blocks else None
    pos = torch.empty((n_rows, w), dtype=torch.int32, device=dev) if want_pos else None
    _check("qsa_select_blocks", lib().qsa_select_blocks(
        _ptr(scores), scores.shape[1], req_row_start.numel() - 1, _ptr(req_row_start), n_rows,
        _ptr(row_len), int(max_len), _ptr(page_table), page_table.shape[1], int(page_size), int(k_blk),
        _ptr(blocks), _ptr(pos), _ptr(out_slots), _stream(stream)))
    out = {"slots": out_slots}
    if blocks is not None:
        out["blocks"] = blocks
    if pos is not None:
        out["pos"] = pos
    return out


def indexer_select_workspace_size(n_rows, max_len, k_blk=512) -> int:
    return int(lib().qsa_indexer_select_workspace_size(int(n_rows), int(max_len), int(k_blk)))


def indexer_select(q, pool, req_row_start, row_len, page_table, page_size, max_len,
                   max_rows_per_req=None, k_blk=512, want_blocks=False, want_pos=False,
                   scores_out=None, workspace=None, out_slots=None, stream=None):
    """Fused decode path: score -> top-k_blk blocks -> expand -> slots.
    Returns dict(slots, blocks?, pos?, scores?)."""
    torch = _torch()
    _dev(pool, torch.bfloat16, "pool", 2)
    return _indexer_select_call("qsa_indexer_select", (_ptr(pool),), pool.shape[0], q, req_row_start,
                                row_len, page_table, page_size, max_len, max_rows_per_req, k_blk,
                                want_blocks, want_pos, scores_out, workspace, out_slots, stream)


def indexer_select_fp8(q, codes, scales, req_row_start, row_len, page_table, page_size, max_len,
                       max_rows_per_req=None, k_blk=512, want_blocks=False, want_pos=False,
                       scores_out=None, workspace=None, out_slots=None, stream=None):
    """indexer_select on FP8 keys (codes, scales from quantize_keys_fp8)."""
    torch = _torch()
    _dev(codes, torch.uint8, "codes", 2)
    _dev(scales, torch.float32, "scales", 1)
    if scales.numel() != codes.shape[0]:
        raise ValueError("scales must have one entry per key")
    return _indexer_select_call("qsa_indexer_select_fp8", (_ptr(codes), _ptr(scales)), codes.shape[0], q,
                                req_row_start, row_len, page_table, page_size, max_len, max_rows_per_req,
                                k_blk, want_blocks, want_pos, scores_out, workspace, out_slots, stream)


def indexer_select_gated(q, head_gates, pool, req_row_start, row_len, page_table, page_size, max_len,
                         max_rows_per_req=None, k_blk=512, want_blocks=False, want_pos=False,
                         scores_out=None, workspace=None, out_slots=None, stream=None):
    """indexer_select with a gate per row and head (head_gates [n_rows][4]
    float32)."""
    torch = _torch()
    _dev(pool, torch.bfloat16, "pool", 2)
    _gates(head_gates, row_len)
    return _indexer_select_call("qsa_indexer_select_gated", (_ptr(head_gates), _ptr(pool)), pool.shape[0], q,
                                req_row_start, row_len, page_table, page_size, max_len, max_rows_per_req, k_blk,
                                want_blocks, want_pos, scores_out, workspace, out_slots, stream)


def _indexer_select_call(fn, key_ptrs, pool_rows, q, req_row_start, row_len, page_table, page_size,
                         max_len, max_rows_per_req, k_blk, want_blocks, want_pos, scores_out, workspace,
                         out_slots, stream):
    torch = _torch()
    _dev(q, torch.bfloat16, "q", 3)
    _dev(req_row_start, torch.int32, "req_row_start", 1)
    _dev(row_len, torch.int32, "row_len", 1)
    _dev(page_table, torch.int32, "page_table", 2)
    n_rows = row_len.numel()
    dev = q.device
    if max_rows_per_req is None:
        max_rows_per_req = n_rows
    w = out_width(k_blk)
    if out_slots is None:
        out_slots = torch.empty((n_rows, w), dtype=torch.int32, device=dev)
    blocks = torch.empty((n_rows, k_blk), dtype=torch.int32, device=dev) if want_blocks else None
    pos = torch.empty((n_rows, w), dtype=torch.int32, device=dev) if want_pos else None
    ld = 0
    ws_bytes = 0
    if scores_out is not None:
        _dev(scores_out, torch.float32, "scores_out", 2)
        ld = scores_out.shape[1]
        if workspace is not None:  # may still hold the device row plan
            ws_bytes = workspace.numel() * workspace.element_size()
    else:
        ws_bytes = indexer_select_workspace_size(n_rows, max_len, k_blk)
        if workspace is None and ws_bytes:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        elif workspace is not None:
            ws_bytes = workspace.numel() * workspace.element_size()
    _check(fn, _call(
        fn, _ptr(q), *key_ptrs, pool_rows, req_row_start.numel() - 1, _ptr(req_row_start), n_rows,
        _ptr(row_len), int(max_len), int(max_rows_per_req), _ptr(page_table), page_table.shape[1],
        int(page_size), int(k_blk), _ptr(blocks), _ptr(pos), _ptr(out_slots), _ptr(scores_out), ld,
        _ptr(workspace), ws_bytes, _stream(stream, q.device)))
    out = {"slots": out_slots}
    if blocks is not None:
        out["blocks"] = blocks
    if pos is not None:
        out["pos"] = pos
    if scores_out is not None:
        out["scores"] = scores_out
    return out
