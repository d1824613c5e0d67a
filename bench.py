"""Benchmark of the QSA indexer hot path on GB300.

One step = one decode verify step of the indexer at L = 80,000: compress the
blocks that the step's tokens completed, then the fused indexer call (score
all visible compressed blocks for the 6 query rows, keep the best 512 per
row, expand to token positions plus pending tokens, translate to physical KV
slots).  The reported value is query rows per second.

Timing: the L2 cache (129 MB) is flushed before every timed step, outside the
timed region: a 256 MB buffer is written, then another 256 MB buffer is read,
so the step starts with none of its data in L2 and with no dirty lines of the
flush left for the step to write back; each step is bracketed by CUDA
events on the launching stream.  W untimed warm-up steps come first.  Under
torchrun every rank runs an independent replica (the path shards by request
with no exchange), and the time is the maximum over ranks.

--workload picks another decode workload for the primary line (profiling
runs use it); the default is the 6-row verify step above.

--impl reference times the CPU oracle (plain C, FP64) on the host cores, on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import (c1_decode, c2_batched, c2_verify, c3_batched, c4_dsa_topk, indexshare_mtp,  # noqa: E402
                       c5_prefill)

METRIC = "indexer+top-k query rows/sec at L=80k decode; achieved HBM GB/s vs roofline"
NOMINAL_HBM_GBS = 7900.0  # the GB300's nominal HBM3e bandwidth (context; the measured copy peak is the denominator)


def add_nominal_fractions(out):
    """Beside every fraction of the measured HBM peak, the same bytes as a
    fraction of the nominal bandwidth: the step's and each variant's."""
    if "step_alg_GBps" in out:
        out["step_frac_hbm_nominal"] = out["step_alg_GBps"] / NOMINAL_HBM_GBS
    for v in out.get("variants", {}).values():
        if isinstance(v, dict) and "alg_GBps" in v and "frac_hbm" in v:
            v["frac_hbm_nominal"] = v["alg_GBps"] / NOMINAL_HBM_GBS
    return out
L2_FLUSH_BYTES = 256 << 20


def captured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    capture (profiles/traffic.json), or None once the kernel's source no
    longer matches the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec or workload not in rec:
        return None
    m = hashlib.sha256()
    for f in rec["sources"]:
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None
        m.update(open(fp, "rb").read())
    if m.hexdigest() != rec["csrc_sha256"]:
        return None
    w = rec[workload]
    return int(w["dram_read_bytes"]) + int(w["dram_write_bytes"])


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 6:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for name, v in zip(names, f[2:6]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_time(local_ms: float, world_size: int, backend_device=None) -> float:
    """Max over ranks of a per-rank time (a timing collective only)."""
    if world_size <= 1:
        return local_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_ms], dtype=torch.float64,
                     device=backend_device if backend_device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world_size):
    if world_size > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- GPU arm
class Gpu:
    def __init__(self, device):
        import torch
        import sparse_attention_indexer_index_gb300 as qsa
        self.torch, self.qsa, self.dev = torch, qsa, device
        self.flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.flush_sum = torch.empty((), dtype=torch.float32, device=device)
        self.stream = torch.cuda.current_stream(device)

    def flush(self):
        """Evict the step's data from L2: write 256 MB, then read 256 MB of
        another buffer (the written lines are cleaned here, not in the step)."""
        self.flush_buf.fill_(1.0)
        self.torch.sum(self.flush_read, 0, out=self.flush_sum)

    def h2d(self, a, dtype=None):
        t = self.torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)
        return t.view(dtype) if dtype is not None else t

    def bf16(self, a):
        return self.h2d(np.ascontiguousarray(a, np.uint16).view(np.int16), self.torch.bfloat16)

    def capture(self, fn):
        """Record fn's launches into a CUDA graph (after fn has run eagerly, so
        every one-time set-up is done outside the capture)."""
        torch = self.torch
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        torch.cuda.synchronize()
        return graph.replay

    def timed(self, fn, iters, warmup, flush=True, graph=True, pre=None):
        """Per-iteration CUDA-event times (ms) with an L2 flush before each.
        With graph=True the step is replayed from a CUDA graph, so the events
        see device time rather than Python launch overhead.  pre(), if given,
        runs before every iteration outside the timed region (state resets)."""
        torch = self.torch
        for _ in range(warmup):
            if pre is not None:
                pre()
            if flush:
                self.flush()
            fn()
        torch.cuda.synchronize()
        run = self.capture(fn) if graph else fn
        for _ in range(2):
            if pre is not None:
                pre()
            run()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(iters)]
        for s, e in ev:
            if pre is not None:
                pre()
            if flush:
                self.flush()
            s.record(self.stream)
            run()
            e.record(self.stream)
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in ev]


def setup_decode(g: Gpu, w, new_blocks: int):
    """Device-resident state of a decode workload: the compressed-key pool
    (built by the library's own compress kernel), metadata, and the raw keys
    of the blocks completed by this step."""
    torch, qsa = g.torch, g.qsa
    st = {"w": w}
    st["pool"] = torch.zeros((w.pool_rows, 128), dtype=torch.bfloat16, device=g.dev)
    st["rrs"] = g.h2d(w.req_row_start)
    st["row_len"] = g.h2d(w.row_len)
    st["pt"] = g.h2d(w.page_table)
    st["q"] = g.bf16(w.q)
    # compress every complete block once (setup)
    qsa.compress_keys(g.bf16(w.raw_keys), g.h2d(w.block_id), st["pool"], block_req=g.h2d(w.block_req),
                      page_table=st["pt"], page_size=w.page_size, rope_base=w.rope_base)
    # the step's own compress work: the last `new_blocks` blocks of each request
    sel = []
    for r in range(w.n_req):
        idx = np.flatnonzero(w.block_req == r)
        sel.extend(idx[-new_blocks:].tolist())
    sel = np.array(sel, np.int64)
    st["new_raw_h"] = np.ascontiguousarray(w.raw_keys.reshape(-1, 4, 128)[sel].reshape(-1, 128))
    st["new_id_h"] = w.block_id[sel].copy()
    st["new_req_h"] = w.block_req[sel].copy()
    st["new_raw"] = g.bf16(st["new_raw_h"])
    st["new_id"] = g.h2d(st["new_id_h"])
    st["new_req"] = g.h2d(st["new_req_h"])
    ld = (w.max_len // 4 + 3) // 4 * 4
    st["ws"] = torch.empty(qsa.indexer_select_workspace_size(w.n_rows, w.max_len, w.k_blk),
                           dtype=torch.uint8, device=g.dev)
    st["slots"] = torch.empty((w.n_rows, 4 * w.k_blk + 3), dtype=torch.int32, device=g.dev)
    st["scores"] = torch.empty((w.n_rows, ld), dtype=torch.float32, device=g.dev)
    torch.cuda.synchronize()
    return st


def decode_step(g: Gpu, st):
    w = st["w"]
    g.qsa.compress_keys(st["new_raw"], st["new_id"], st["pool"], block_req=st["new_req"],
                        page_table=st["pt"], page_size=w.page_size, rope_base=w.rope_base)
    g.qsa.indexer_select(st["q"], st["pool"], st["rrs"], st["row_len"], st["pt"], w.page_size,
                         w.max_len, w.max_rows_per_req, k_blk=w.k_blk, workspace=st["ws"],
                         out_slots=st["slots"])


def scores_only(g: Gpu, st):
    w = st["w"]
    g.qsa.index_scores(st["q"], st["pool"], st["rrs"], st["row_len"], st["pt"], w.page_size,
                       w.max_len, w.max_rows_per_req, scores=st["scores"])


def compress_only(g: Gpu, st):
    w = st["w"]
    g.qsa.compress_keys(st["new_raw"], st["new_id"], st["pool"], block_req=st["new_req"],
                        page_table=st["pt"], page_size=w.page_size, rope_base=w.rope_base)


def select_only(g: Gpu, st):
    """The selection half of the fused call on the scores left in st["scores"]
    by scores_only (the kernel the fused call runs after the scorer)."""
    w = st["w"]
    g.qsa.select_blocks(st["scores"], st["rrs"], st["row_len"], st["pt"], w.page_size, w.max_len,
                        k_blk=w.k_blk, out_slots=st["slots"])


def kernel_names(w, sm_count=152):
    """Kernels the library dispatches to for this workload (the launch rules
    of qsa_api.cu: requests of up to 8 rows on pages holding a multiple of 8
    compressed keys use the mma.sync decode scorer, requests with more rows
    the tensor-core tile scorer (fed by TMA on such pages, by cp.async on
    smaller ones), one-row requests on small pages the CUDA-core scorer; rows
    of more than 32768 blocks take a cluster of 2-16 CTAs per row when
    rows * 2 <= SMs (one streaming CTA per row otherwise), more than two rows
    per SM take small CTAs (four per SM), other rows (k <= 1024) one
    register-resident CTA per row)."""
    kpp = w.page_size // 4
    if kpp % 8 == 0 and w.max_rows_per_req <= 8:
        score = "score_mma_kernel"
    elif w.max_rows_per_req >= 2:
        score = "score_tc_kernel" if kpp % 8 == 0 and w.pool_rows % 8 == 0 else "score_tc_cpasync_kernel"
    else:
        score = "score_decode_kernel"
    return {"compress": "compress_keys_kernel", "append": "append_keys_kernel", "score": score,
            "select": topk_kernel_name(w.n_rows, w.max_len // 4, sm_count, w.k_blk)}


def kernel_bytes(w, new_blocks):
    """Algorithmic HBM bytes per launch of each kernel of the step.
    compress: per new block 4 raw keys read (1 KB), one key written (256 B),
      its id, request and page-table entry (12 B);
    score: decode_bytes' keys + q + page table + the FP32 scores written;
    select: the FP32 scores read, the page-table entries of the context, the
      slot rows written."""
    by = decode_bytes(w)
    n_new = new_blocks * w.n_req
    return {"compress": n_new * (4 * 256 + 256 + 12),
            "score": by["keys"] + by["q"] + by["page_table"] + by["scores_fp32"],
            "select": by["scores_fp32"] + by["page_table"] + by["slots"]}


def append_bytes(st):
    """Algorithmic HBM bytes of one key-path launch (qsa_append_keys) as set
    up by setup_key_path: per request, the appended raw keys read (256 B
    each); per block they complete, its keys from earlier calls read from
    the ring, the compressed key written (256 B) and its page-table entry
    (4 B); the last 4 appended keys written to the ring; the request's
    metadata (12 B)."""
    total = 0
    rts, first = st["kp_rts_h"], st["kp_first_h"]
    for r in range(len(first)):
        n, p0 = int(rts[r + 1] - rts[r]), int(first[r])
        done = [p // 4 for p in range(p0, p0 + n) if p % 4 == 3]
        from_ring = sum(max(0, p0 - 4 * b) for b in done)
        total += 256 * n + 256 * from_ring + (256 + 4) * len(done) + 256 * min(n, 4) + 12
    return total


def decode_bytes(w):
    """Algorithmic HBM bytes of one fused indexer call: every visible
    compressed key of a request read once (256 B), the query rows (1 KB
    each), the page-table entries covering the context, and the slot rows
    written (4 B x (4k+3))."""
    nb_req = [int(w.row_len[w.req_row_start[r]:w.req_row_start[r + 1]].max()) // 4
              for r in range(w.n_req)]
    keys = 256 * sum(nb_req)
    pt = 4 * sum((int(w.row_len[w.req_row_start[r]:w.req_row_start[r + 1]].max()) + w.page_size - 1)
                 // w.page_size for r in range(w.n_req))
    return {"keys": keys, "q": 1024 * w.n_rows, "page_table": pt,
            "slots": 4 * (4 * w.k_blk + 3) * w.n_rows,
            "scores_fp32": 4 * sum(int(L) // 4 for L in w.row_len)}


def e2e_decode(g: Gpu, st, iters, warmup):
    """The same step through the public API with HOST buffers: the step's
    inputs (q, the appended raw keys, their positions and the row metadata)
    packed in one pinned host buffer and copied in with one transfer, one
    decode_step call on views of the device copy, the slots copied back,
    all inside the timed region (the ring is put back before each step,
    outside it)."""
    torch = g.torch
    w = st["w"]
    parts = {
        "q": np.ascontiguousarray(w.q).view(np.uint8).reshape(-1),
        "keys": np.ascontiguousarray(st["kp_keys_h"]).view(np.uint8).reshape(-1),
        "rts": st["kp_rts_h"].view(np.uint8),
        "first": st["kp_first_h"].view(np.uint8),
        "rrs": np.ascontiguousarray(w.req_row_start).view(np.uint8),
        "rl": np.ascontiguousarray(w.row_len).view(np.uint8),
    }
    off, pos = {}, 0
    for k, v in parts.items():  # 16-byte aligned pieces
        off[k] = pos
        pos += (v.size + 15) // 16 * 16
    packed = np.zeros(pos, np.uint8)
    for k, v in parts.items():
        packed[off[k]:off[k] + v.size] = v
    host = torch.from_numpy(packed).pin_memory()
    dev = torch.empty_like(host, device=g.dev)

    def view(k, dtype):
        return dev[off[k]:off[k] + parts[k].size].view(dtype)

    q_d, keys_d = view("q", torch.bfloat16).view(-1, 4, 128), view("keys", torch.bfloat16).view(-1, 128)
    rts_d, first_d = view("rts", torch.int32), view("first", torch.int32)
    rrs_d, rl_d = view("rrs", torch.int32), view("rl", torch.int32)
    out_h = torch.empty(st["slots"].shape, dtype=torch.int32).pin_memory()
    h2d = int(host.numel())
    d2h = out_h.numel() * 4

    def step():
        dev.copy_(host, non_blocking=True)
        g.qsa.decode_step(keys_d, rts_d, first_d, st["kp_ring"], q_d, st["pool"], rrs_d, rl_d, st["pt"],
                          w.page_size, w.max_len, w.max_rows_per_req, k_blk=w.k_blk, rope_base=w.rope_base,
                          workspace=st["ws"], out_slots=st["slots"])
        out_h.copy_(st["slots"], non_blocking=True)

    times = g.timed(step, iters, warmup, graph=False, pre=lambda: restore_ring(st))
    return times, h2d, d2h


def setup_key_path(g, st):
    """The decode key path of the step: every query row's own token is
    appended (request r: positions row_len - 1 of its rows, consecutive)
    through the 4-slot ring, which holds the earlier positions of the
    block.  Raw keys come from the workload where it has them (complete
    blocks), seeded N(0,1) BF16 otherwise."""
    w = st["w"]
    rng = np.random.default_rng(777)
    raw_of = {}
    for i in range(w.n_blocks):
        raw_of[(int(w.block_req[i]), int(w.block_id[i]))] = i

    def raw_key(r, p):
        i = raw_of.get((r, p // 4))
        if i is None:
            return bf16_bits_of(rng.standard_normal(128).astype(np.float32))
        return w.raw_keys[4 * i + p % 4]

    keys, first, counts = [], [], []
    ring = np.zeros((w.n_req, 4, 128), np.uint16)
    for r in range(w.n_req):
        pos = sorted(int(L) - 1 for L in w.row_len[w.req_row_start[r]:w.req_row_start[r + 1]])
        p0 = pos[0]
        first.append(p0)
        counts.append(len(pos))
        keys.extend(raw_key(r, p) for p in range(p0, p0 + len(pos)))
        for p in range(4 * (p0 // 4), p0):
            ring[r, p % 4] = raw_key(r, p)
    st["kp_keys_h"] = np.stack(keys)
    st["kp_rts_h"] = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    st["kp_first_h"] = np.array(first, np.int32)
    st["kp_keys"] = g.bf16(st["kp_keys_h"])
    st["kp_rts"] = g.h2d(st["kp_rts_h"])
    st["kp_first"] = g.h2d(st["kp_first_h"])
    st["kp_ring"] = g.bf16(ring)
    st["kp_ring0"] = st["kp_ring"].clone()  # the ring before the step (restored between replays)


def bf16_bits_of(x):
    from workloads import bf16_bits
    return bf16_bits(np.asarray(x, np.float32))


def append_only(g, st):
    """The key path alone (ring append + compression of the completed
    blocks); restore_ring() puts the ring back between replays."""
    w = st["w"]
    g.qsa.append_keys(st["kp_keys"], st["kp_rts"], st["kp_first"], st["kp_ring"], st["pool"], st["pt"],
                      w.page_size, w.rope_base)


def restore_ring(st):
    st["kp_ring"].copy_(st["kp_ring0"])


def decode_step_ring(g, st):
    """One decode step in one call (qsa_decode_step): the rows' own tokens
    appended through the ring (completing their blocks), then the fused
    indexer; scorer CTAs that read no new block do not wait for the key
    path."""
    w = st["w"]
    g.qsa.decode_step(st["kp_keys"], st["kp_rts"], st["kp_first"], st["kp_ring"], st["q"], st["pool"], st["rrs"],
                      st["row_len"], st["pt"], w.page_size, w.max_len, w.max_rows_per_req, k_blk=w.k_blk,
                      rope_base=w.rope_base, workspace=st["ws"], out_slots=st["slots"])


def bench_variant_decode(g, w, new_blocks, iters, warmup, peaks):
    """One decode step of workload w as the library's one-call decode step
    (qsa_decode_step: the rows' own index keys through the 4-slot ring, the
    blocks they complete compressed, then the fused indexer), L2 flushed
    before every step; beside it the same work as two calls (compress the
    step's new blocks, then qsa_indexer_select) and each kernel alone."""
    st = setup_decode(g, w, new_blocks)
    t_two = g.timed(lambda: decode_step(g, st), iters, warmup)
    t_score = g.timed(lambda: scores_only(g, st), iters, warmup)
    t_select = g.timed(lambda: select_only(g, st), iters, warmup)
    setup_key_path(g, st)
    t_append = g.timed(lambda: append_only(g, st), iters, warmup, pre=lambda: restore_ring(st))
    t_step = g.timed(lambda: decode_step_ring(g, st), iters, warmup, pre=lambda: restore_ring(st))
    t_compress = g.timed(lambda: compress_only(g, st), iters, warmup) if new_blocks > 0 else None
    by = decode_bytes(w)
    alg = by["keys"] + by["q"] + by["page_table"] + by["slots"]
    ms = statistics.mean(t_step)
    ms_sc = statistics.mean(t_score)
    res = {"workload": w.name, "rows": w.n_rows, "us_per_call": 1e3 * ms,
           "step": "one qsa_decode_step call (ring append + compression of completed blocks + fused indexer)",
           "rows_per_s": w.n_rows / (ms * 1e-3), "alg_bytes": alg,
           "alg_GBps": alg / (ms * 1e-3) / 1e9, "frac_hbm": alg / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
           "score_kernel_us": 1e3 * ms_sc, "select_kernel_us": 1e3 * statistics.mean(t_select),
           "key_path_append_us": 1e3 * statistics.mean(t_append),
           "two_calls_us": 1e3 * statistics.mean(t_two),
           "compress_kernel_us": 1e3 * statistics.mean(t_compress) if t_compress else None,
           "kernels": kernel_names(w),
           "score_alg_GBps": (by["keys"] + by["q"] + by["page_table"] + by["scores_fp32"]) /
                             (ms_sc * 1e-3) / 1e9}
    del st
    return res


def bench_variant_decode_fp8(g, w, iters, warmup, peaks):
    """The fused indexer call on FP8 index keys (e4m3 codes + one FP32 scale
    per compressed key: 132 B a key instead of 256 B) beside the same call
    on BF16 keys, L2 flushed before every call; plus the scorer alone on
    each, and how many of the BF16 call's selected blocks the FP8 call also
    selects (the quality cost of the smaller keys)."""
    torch, qsa = g.torch, g.qsa
    st = setup_decode(g, w, 0)
    codes, scales = qsa.quantize_keys_fp8(st["pool"])
    args = (st["rrs"], st["row_len"], st["pt"], w.page_size, w.max_len, w.max_rows_per_req)

    def bf16_call():
        qsa.indexer_select(st["q"], st["pool"], *args, k_blk=w.k_blk, workspace=st["ws"], out_slots=st["slots"])

    def fp8_call():
        qsa.indexer_select_fp8(st["q"], codes, scales, *args, k_blk=w.k_blk, workspace=st["ws"],
                               out_slots=st["slots"])

    t_bf16 = g.timed(bf16_call, iters, warmup)
    t_fp8 = g.timed(fp8_call, iters, warmup)
    t_sc_bf16 = g.timed(lambda: qsa.index_scores(st["q"], st["pool"], *args, scores=st["scores"]), iters, warmup)
    t_sc_fp8 = g.timed(lambda: qsa.index_scores_fp8(st["q"], codes, scales, *args, scores=st["scores"]),
                       iters, warmup)
    sel = {}
    for name, fn in (("bf16", qsa.indexer_select), ("fp8", qsa.indexer_select_fp8)):
        keys = (st["pool"],) if name == "bf16" else (codes, scales)
        sel[name] = fn(st["q"], *keys, *args, k_blk=w.k_blk, want_blocks=True)["blocks"].cpu().numpy()
    overlap = [len(np.intersect1d(a[a >= 0], b[b >= 0])) / max(1, int((a >= 0).sum()))
               for a, b in zip(sel["bf16"], sel["fp8"])]
    by = decode_bytes(w)
    keys8 = by["keys"] // 256 * (128 + 4)
    alg = keys8 + by["q"] + by["page_table"] + by["slots"]
    ms, ms16 = statistics.mean(t_fp8), statistics.mean(t_bf16)
    res = {"workload": w.name + "_fp8_keys", "rows": w.n_rows, "us_per_call": 1e3 * ms,
           "bf16_keys_us_per_call": 1e3 * ms16, "speedup_vs_bf16_keys": ms16 / ms,
           "alg_bytes": alg, "alg_GBps": alg / (ms * 1e-3) / 1e9,
           "frac_hbm": alg / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
           "score_kernel_us": 1e3 * statistics.mean(t_sc_fp8),
           "score_kernel_bf16_keys_us": 1e3 * statistics.mean(t_sc_bf16),
           "selection_overlap_with_bf16_keys": float(np.mean(overlap))}
    del st
    torch.cuda.synchronize()
    return res


def topk_kernel_name(n_rows, n, sm_count=152, k=2048):
    """The selection kernel for n_rows rows of n scores and k winners."""
    if n > 32768:
        return "select_long_kernel" if n_rows * 2 <= sm_count else "select_kernel"
    if n_rows > 2 * sm_count:
        return "select_rows_kernel"
    if k <= 1024:
        return "select_fast_kernel"
    if n_rows * 8 <= sm_count:
        return "select_cluster_kernel"
    return "select_resident_kernel"


def bench_variant_topk(g, w, iters, warmup, peaks):
    torch, qsa = g.torch, g.qsa
    s = g.h2d(w.scores)
    nv = g.h2d(w.n_valid)
    pt = g.h2d(w.page_table)
    out_i = torch.empty((s.shape[0], w.k), dtype=torch.int32, device=g.dev)
    out_s = torch.empty_like(out_i)
    fn = lambda: qsa.topk_select(s, w.k, n_valid=nv, n_max=int(w.n_valid.max()), page_table=pt,
                                 page_size=w.page_size, out_idx=out_i, out_slots=out_s)
    t = g.timed(fn, iters, warmup)
    ms = statistics.mean(t)
    alg = w.scores.nbytes + 2 * out_i.numel() * 4 + w.page_table.nbytes
    return {"workload": w.name, "rows": int(s.shape[0]), "us_per_call": 1e3 * ms,
            "rows_per_s": s.shape[0] / (ms * 1e-3), "alg_bytes": alg,
            "alg_GBps": alg / (ms * 1e-3) / 1e9, "frac_hbm": alg / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "dup_fraction": w.dup_fraction,
            "kernel": topk_kernel_name(int(s.shape[0]), int(w.n_valid.max()), k=w.k)}


def bench_variant_topk_mixed(g, iters, warmup, peaks, seed=0, k=2048, page_size=64):
    """DSA top-2048 with slots on a mixed batch in one call: one row of
    1,000,000 scores, four of 80,000 and 100 of 3,000-30,000 (seeded, in
    shuffled order; N(0,1) scores drawn on the device).  The library plans the
    rows on the device (long rows on clusters, short ones one CTA each);
    beside it the same rows as two calls, the long ones and the short ones."""
    torch, qsa = g.torch, g.qsa
    rng = np.random.default_rng(seed + 77)
    lens = np.array([1_000_000] + [80_000] * 4 + list(rng.integers(3000, 30_000, size=100)), np.int32)
    nv_h = rng.permutation(lens).astype(np.int32)
    ld = int(nv_h.max())
    gen = torch.Generator(device=g.dev)
    gen.manual_seed(seed + 78)
    s = torch.randn((nv_h.size, ld), generator=gen, device=g.dev)
    pt_h = np.stack([rng.permutation((ld + page_size - 1) // page_size) for _ in range(nv_h.size)]).astype(np.int32)
    nv, pt = g.h2d(nv_h), g.h2d(pt_h)
    long_i = np.flatnonzero(nv_h > 32768)
    short_i = np.flatnonzero(nv_h <= 32768)
    s_long, s_short = s[g.h2d(long_i)].contiguous(), s[g.h2d(short_i)][:, :32768].contiguous()
    nv_long, nv_short = g.h2d(nv_h[long_i]), g.h2d(nv_h[short_i])
    pt_long, pt_short = g.h2d(pt_h[long_i]), g.h2d(pt_h[short_i])
    n_short_max = int(nv_h[short_i].max())
    outs = {}
    for name, rows in (("mixed", nv_h.size), ("long", long_i.size), ("short", short_i.size)):
        outs[name] = (torch.empty((rows, k), dtype=torch.int32, device=g.dev),
                      torch.empty((rows, k), dtype=torch.int32, device=g.dev))
    fn_mixed = lambda: qsa.topk_select(s, k, n_valid=nv, n_max=ld, page_table=pt, page_size=page_size,
                                       out_idx=outs["mixed"][0], out_slots=outs["mixed"][1])
    fn_long = lambda: qsa.topk_select(s_long, k, n_valid=nv_long, n_max=ld, page_table=pt_long,
                                      page_size=page_size, out_idx=outs["long"][0], out_slots=outs["long"][1])
    fn_short = lambda: qsa.topk_select(s_short, k, n_valid=nv_short, n_max=n_short_max, page_table=pt_short,
                                       page_size=page_size, out_idx=outs["short"][0], out_slots=outs["short"][1])
    no_ws = torch.empty(0, dtype=torch.uint8, device=g.dev)
    fn_noplan = lambda: qsa.topk_select(s, k, n_valid=nv, n_max=ld, page_table=pt, page_size=page_size,
                                        out_idx=outs["mixed"][0], out_slots=outs["mixed"][1], workspace=no_ws)
    t_noplan = 1e3 * statistics.mean(g.timed(fn_noplan, iters, warmup))
    t_mixed = 1e3 * statistics.mean(g.timed(fn_mixed, iters, warmup))
    t_long = 1e3 * statistics.mean(g.timed(fn_long, iters, warmup))
    t_short = 1e3 * statistics.mean(g.timed(fn_short, iters, warmup))
    alg = int(nv_h.sum()) * 4 + 2 * nv_h.size * k * 4 + int(sum((n + page_size - 1) // page_size for n in nv_h)) * 4
    ms = t_mixed * 1e-3
    return {"workload": "dsa_topk_mixed_1x1M_4x80K_100short", "rows": int(nv_h.size), "us_per_call": t_mixed,
            "rows_per_s": nv_h.size / (ms * 1e-3), "alg_bytes": alg, "alg_GBps": alg / (ms * 1e-3) / 1e9,
            "frac_hbm": alg / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "classes_apart_us": {"long_5_rows": t_long, "short_100_rows": t_short, "sum": t_long + t_short},
            "without_plan_us": t_noplan,
            "without_plan": "no workspace for the plan: the host rule from the longest row and the row count "
                            "(every row on one streaming CTA)"}


def bench_variant_indexshare(g, w, iters, warmup, peaks):
    """One draft step of an MTP iteration with IndexShare: each request's
    draft row reads the selection kept at its draft-extend row
    (qsa_indexshare_slots) instead of running the indexer.  The indexer call
    the same draft rows would otherwise make is timed beside it."""
    torch, qsa = g.torch, g.qsa
    ext_rows = w.req_row_start[:-1]
    ext_len = np.ascontiguousarray(w.row_len[ext_rows])
    d_rows = ext_rows + 1  # the first draft step: position L0 + 1
    d_len = np.ascontiguousarray(w.row_len[d_rows])
    n_req = w.n_req
    st = setup_decode(g, w, 0)
    rrs1 = g.h2d(np.arange(n_req + 1, dtype=np.int32))
    pt = st["pt"]
    ext = qsa.indexer_select(g.bf16(w.q[ext_rows]), st["pool"], rrs1, g.h2d(ext_len), pt, w.page_size,
                             int(ext_len.max()), 1, k_blk=w.k_blk, want_blocks=True)
    kept, kept_len = ext["blocks"], g.h2d(ext_len)
    cap_row = g.h2d(np.arange(n_req, dtype=np.int32))
    n_extra = int(w.max_rows_per_req)  # the draft depth + 1
    d_len_t = g.h2d(d_len)
    out = torch.empty((n_req, qsa.indexshare_width(w.k_blk, n_extra)), dtype=torch.int32, device=g.dev)
    t_share = g.timed(lambda: qsa.indexshare_slots(kept, kept_len, cap_row, n_extra, rrs1, d_len_t, pt,
                                                   w.page_size, want_pos=False, out_slots=out),
                      iters, warmup)
    q_d = g.bf16(w.q[d_rows])
    ws = torch.empty(qsa.indexer_select_workspace_size(n_req, int(d_len.max()), w.k_blk), dtype=torch.uint8,
                     device=g.dev)
    slots = torch.empty((n_req, 4 * w.k_blk + 3), dtype=torch.int32, device=g.dev)
    t_full = g.timed(lambda: qsa.indexer_select(q_d, st["pool"], rrs1, d_len_t, pt, w.page_size,
                                                int(d_len.max()), 1, k_blk=w.k_blk, workspace=ws,
                                                out_slots=slots), iters, warmup)
    ms, ms_full = statistics.mean(t_share), statistics.mean(t_full)
    width = 4 * w.k_blk + 3 + n_extra
    # kept blocks and row lengths read, one page-table entry per kept block
    # and per tail page, the slot rows written
    alg = n_req * (4 * w.k_blk + 8 + 4 * w.k_blk + 4 * width)
    del st
    return {"workload": w.name + "_draft_step", "rows": n_req, "us_per_call": 1e3 * ms,
            "rows_per_s": n_req / (ms * 1e-3), "alg_bytes": alg, "alg_GBps": alg / (ms * 1e-3) / 1e9,
            "indexer_us_same_rows": 1e3 * ms_full, "indexer_over_indexshare": ms_full / ms,
            "kernel": "indexshare_kernel"}


def bench_variant_prefill(g, w, iters, warmup, peaks):
    st = setup_decode(g, w, 0)
    t = g.timed(lambda: g.qsa.indexer_select(st["q"], st["pool"], st["rrs"], st["row_len"], st["pt"],
                                             w.page_size, w.max_len, w.max_rows_per_req, k_blk=w.k_blk,
                                             workspace=st["ws"], out_slots=st["slots"]),
                iters, warmup)
    t_score = g.timed(lambda: scores_only(g, st), max(2, iters), warmup)
    t_select = g.timed(lambda: select_only(g, st), max(2, iters), warmup)
    ms = statistics.mean(t)
    pairs = int(sum(int(L) // 4 for L in w.row_len))
    flop = 2 * 4 * 128 * pairs
    return {"workload": w.name, "rows": w.n_rows, "us_per_call": 1e3 * ms,
            "rows_per_s": w.n_rows / (ms * 1e-3), "flop": flop,
            "TFLOPs": flop / (ms * 1e-3) / 1e12,
            "frac_tensor": flop / (ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
            "score_kernel_us": 1e3 * statistics.mean(t_score), "select_kernel_us": 1e3 * statistics.mean(t_select),
            "score_TFLOPs": flop / (statistics.mean(t_score) * 1e-3) / 1e12,
            "path": "tensor-core scorer (tcgen05 MMA, TMA-fed key tiles) + small-CTA row selection"}


def cpu_oracle_rate(w, budget_s=10.0):
    """Oracle rows/s on a bounded sample: whole steps of the workload (all its
    rows) repeated until half the budget is used, first on one host core (the
    plain build), then on every core of this process's affinity mask (the
    same source built with OpenMP: blocks of a row and rows split over the
    cores).  The all-core rate is the line's value."""
    import oracle
    oracle.build()
    pool = np.zeros((w.pool_rows, 128), np.uint16)
    oracle.compress(w.raw_keys, w.block_req, w.block_id, w.page_table, w.page_size, w.rope_base, pool)
    cores = len(os.sched_getaffinity(0))

    def rate(fn, budget):
        fn()  # first call: loads and warms the library
        rows, n, t0 = 0, 0, time.perf_counter()
        while True:
            fn()
            rows += w.n_rows
            n += 1
            el = time.perf_counter() - t0
            if el >= budget:
                return rows / el, n, el

    args = (w.q, pool, w.req_row_start, w.row_len, w.page_table, w.page_size)
    v1, n1, e1 = rate(lambda: oracle.indexer_select(*args, k_blk=w.k_blk), budget_s / 2)
    try:
        vn, nn, en = rate(lambda: oracle.indexer_select_threads(*args, k_blk=w.k_blk, threads=cores), budget_s / 2)
    except (OSError, subprocess.CalledProcessError):  # no OpenMP toolchain: single core only
        vn, nn, en, cores = v1, n1, e1, 1
    return {"value": vn, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{nn} full steps of {w.name} ({w.n_rows} rows each) in {en:.1f} s on {cores} host "
                      f"cores (OpenMP over blocks and rows); key compression excluded",
            "single_core": {"value": v1, "unit": "rows/s", "cores": 1,
                            "sample": f"{n1} full steps in {e1:.1f} s on one core"}}


def run_reference(args):
    """The reference arm: the CPU oracle (plain C, FP64) on this process's
    host cores (OpenMP build), on the primary workload's verify steps."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = c2_verify(0)
    import oracle
    oracle.build()
    pool = np.zeros((w.pool_rows, 128), np.uint16)
    oracle.compress(w.raw_keys, w.block_req, w.block_id, w.page_table, w.page_size, w.rope_base, pool)
    cores = len(os.sched_getaffinity(0))
    args_ = (w.q, pool, w.req_row_start, w.row_len, w.page_table, w.page_size)
    try:
        step = lambda: oracle.indexer_select_threads(*args_, k_blk=w.k_blk, threads=cores)
        step()
    except (OSError, subprocess.CalledProcessError):  # no OpenMP toolchain: single core
        cores = 1
        step = lambda: oracle.indexer_select(*args_, k_blk=w.k_blk)
    for _ in range(args.warmup):
        step()
    t = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        t.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(t)
    v = w.n_rows / (ms * 1e-3)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "rows": w.n_rows, "L": 80000, "k_blk": 512, "page_size": 64,
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": v, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} verify steps of {w.n_rows} rows on {cores} host cores, "
                                   "key compression excluded"},
        "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


WORKLOADS = {
    "c2": lambda seed: (c2_verify(seed), 2),
    "c1": lambda seed: (c1_decode(seed), 1),
    "c2x32": lambda seed: (c2_batched(seed), 2),
    "c3": lambda seed: (c3_batched(seed), 1),
}


def bench_variant_attn(g, w, iters, warmup, peaks, h_q=16, h_kv=2, d=256):
    """Sparse attention over the slots the fused indexer selects for w's
    rows (synthetic BF16 K/V cache covering every slot of the page pool,
    drawn on the device from a seeded generator): the consumer of the
    selection.  Timed alone; the indexer + attention pair timed too."""
    torch, qsa = g.torch, g.qsa
    st = setup_decode(g, w, 0)
    qsa.indexer_select(st["q"], st["pool"], st["rrs"], st["row_len"], st["pt"], w.page_size, w.max_len,
                       w.max_rows_per_req, k_blk=w.k_blk, workspace=st["ws"], out_slots=st["slots"])
    n_slots = w.n_pages * w.page_size
    gen = torch.Generator(device=g.dev)
    gen.manual_seed(1234)
    k = torch.randn((n_slots, h_kv, d), generator=gen, device=g.dev).to(torch.bfloat16)
    v = torch.randn((n_slots, h_kv, d), generator=gen, device=g.dev).to(torch.bfloat16)
    qa = torch.randn((w.n_rows, h_q, d), generator=gen, device=g.dev).to(torch.bfloat16)
    slots = st["slots"]
    out = torch.empty((w.n_rows, h_q, d), dtype=torch.float32, device=g.dev)
    lse = torch.empty((w.n_rows, h_q), dtype=torch.float32, device=g.dev)
    n_idx = slots.shape[1]
    ws = torch.empty(max(1, qsa.lib().qsa_sparse_attn_workspace_size(w.n_rows, h_q, d, n_idx)),
                     dtype=torch.uint8, device=g.dev)
    fn = lambda: qsa.sparse_attn(qa, k, v, slots, d ** -0.5, out=out, lse=lse, workspace=ws)
    t_attn = g.timed(fn, iters, warmup)
    both = lambda: (qsa.indexer_select(st["q"], st["pool"], st["rrs"], st["row_len"], st["pt"], w.page_size,
                                       w.max_len, w.max_rows_per_req, k_blk=w.k_blk, workspace=st["ws"],
                                       out_slots=slots), fn())
    t_both = g.timed(both, iters, warmup)
    valid = int((slots >= 0).sum().item())
    # K and V rows of every valid entry, the queries, the slot rows, the outputs
    alg = valid * h_kv * d * 2 * 2 + w.n_rows * h_q * d * 2 + slots.numel() * 4 + w.n_rows * h_q * (d + 1) * 4
    ms, ms_both = statistics.mean(t_attn), statistics.mean(t_both)
    del st
    return {"workload": w.name + f"_attn_h{h_q}kv{h_kv}d{d}", "rows": w.n_rows, "us_per_call": 1e3 * ms,
            "rows_per_s": w.n_rows / (ms * 1e-3), "alg_bytes": alg, "alg_GBps": alg / (ms * 1e-3) / 1e9,
            "frac_hbm": alg / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], "indexer_plus_attn_us": 1e3 * ms_both,
            "kernel": "sparse_attn_kernel<8, 256> + sparse_attn_merge_kernel<256>",
            "kv": "synthetic BF16 N(0,1), 16 query / 2 KV heads, head dim 256 (the pages give no shape)"}


def variant_table(g, it, warmup, peaks):
    """The secondary workloads of the JSON line: name -> a call measuring it."""
    return {
        "c1_decode_L8192": lambda: bench_variant_decode(g, c1_decode(0), 1, it, warmup, peaks),
        "c2_b32_verify_x32": lambda: bench_variant_decode(g, c2_batched(0), 2, it, warmup, peaks),
        "c3_batched_32req": lambda: bench_variant_decode(g, c3_batched(0), 1, it, warmup, peaks),
        "c3_batched_32req_fp8_keys": lambda: bench_variant_decode_fp8(g, c3_batched(0), it, warmup, peaks),
        "c4_dsa_topk_normal": lambda: bench_variant_topk(g, c4_dsa_topk(0, "normal"), it, warmup, peaks),
        "c4_dsa_topk_relu4": lambda: bench_variant_topk(g, c4_dsa_topk(0, "relu4"), it, warmup, peaks),
        "c4_dsa_topk_fp16dup": lambda: bench_variant_topk(g, c4_dsa_topk(0, "fp16dup"), it, warmup, peaks),
        # the verify shape of the TopK-V2 latency figure (6 rows) at 80K and 1M tokens
        "dsa_topk_verify_6x80000": lambda: bench_variant_topk(g, c4_dsa_topk(0, "normal", n_rows=6), it, warmup,
                                                              peaks),
        "dsa_topk_verify_6x1M": lambda: bench_variant_topk(g, c4_dsa_topk(0, "normal", n_rows=6, n=1_000_000), it,
                                                           warmup, peaks),
        "dsa_topk_mixed_1M_4x80K_100short": lambda: bench_variant_topk_mixed(g, it, warmup, peaks),
        "c5_prefill_4096rows": lambda: bench_variant_prefill(g, c5_prefill(0), 3, 3, peaks),
        "indexshare_32req_draft": lambda: bench_variant_indexshare(g, indexshare_mtp(0), it, warmup, peaks),
        "sparse_attn_32req": lambda: bench_variant_attn(g, c3_batched(0), it, warmup, peaks),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c2", choices=sorted(WORKLOADS),
                    help="decode workload of the primary line (default: the 6-row verify step)")
    ap.add_argument("--no-variants", action="store_true", help="primary workload only")
    ap.add_argument("--variant", default=None,
                    help="measure this one secondary workload only and print its line")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time (0: skip)")
    ap.add_argument("--clock-window", type=float, default=1.5,
                    help="seconds of untimed steps run under the clock sampler before timing")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    if args.variant is not None:
        g = Gpu(torch.device("cuda", 0))
        fns = variant_table(g, max(10, min(args.steps, 30)), args.warmup, load_peaks())
        if args.variant not in fns:
            raise SystemExit(f"unknown variant {args.variant}; one of {sorted(fns)}")
        print(json.dumps({"variant": args.variant, **fns[args.variant]()}))
        return 0
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import sparse_attention_indexer_index_gb300 as qsa
    qsa.build()
    peaks = load_peaks()
    g = Gpu(device)

    # ---- primary: one decode step of the chosen workload ------------------
    # (qsa_decode_step: the rows' own index keys appended through the ring,
    # the blocks they complete compressed, then the fused indexer; the ring
    # is put back before every step, outside the timed region)
    w, new_blocks = WORKLOADS[args.workload](rank)
    st = setup_decode(g, w, new_blocks=new_blocks)
    setup_key_path(g, st)
    for _ in range(args.warmup):
        restore_ring(st)
        g.flush()
        decode_step_ring(g, st)
    torch.cuda.synchronize()
    replay = g.capture(lambda: decode_step_ring(g, st))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        t_end = time.perf_counter() + args.clock_window
        while time.perf_counter() < t_end:  # untimed: clocks settle, sampler starts
            for _ in range(20):
                restore_ring(st)
                g.flush()
                replay()
            torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for s, e in ev:
            restore_ring(st)
            g.flush()
            s.record(g.stream)
            replay()
            e.record(g.stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        barrier(ws)
    step_ms = [s.elapsed_time(e) for s, e in ev]
    local_ms = statistics.mean(step_ms)
    ms = aggregate_time(local_ms, ws, device)
    value = ws * w.n_rows / (ms * 1e-3)

    # ---- each kernel of the step alone, timed the same way; the roofline
    # object describes the one that takes longest -------------------------
    names = kernel_names(w, torch.cuda.get_device_properties(device).multi_processor_count)
    kbytes = kernel_bytes(w, new_blocks)
    kbytes["append"] = append_bytes(st)
    del kbytes["compress"]
    scores_only(g, st)  # the selection below reads these scores
    kms = {
        "append": statistics.mean(g.timed(lambda: append_only(g, st), args.steps, args.warmup,
                                          pre=lambda: restore_ring(st))),
        "score": statistics.mean(g.timed(lambda: scores_only(g, st), args.steps, args.warmup)),
        "select": statistics.mean(g.timed(lambda: select_only(g, st), args.steps, args.warmup)),
    }
    kernels = {names[k]: {"us_per_launch": 1e3 * v, "alg_bytes_per_launch": kbytes[k],
                          "achieved_GBps": kbytes[k] / (v * 1e-3) / 1e9,
                          "frac": kbytes[k] / (v * 1e-3) / 1e9 / peaks["hbm_gbs"]}
               for k, v in kms.items()}
    dom = max(kms, key=kms.get)
    achieved = kbytes[dom] / (kms[dom] * 1e-3) / 1e9
    by = decode_bytes(w)
    step_bytes = by["keys"] + by["q"] + by["page_table"] + by["slots"]

    # ---- end to end through the API with host buffers ---------------------
    t_e2e, h2d, d2h = e2e_decode(g, st, min(args.steps, 100), args.warmup)
    e2e_ms = aggregate_time(statistics.mean(t_e2e), ws, device)

    # ---- the timing method's own floor: a graph of one trivial kernel (a
    # one-element add), timed like the step (L2 flushed, events around it)
    tiny = torch.zeros(1, device=device)
    floor_ms = statistics.mean(g.timed(lambda: tiny.add_(1.0), min(args.steps, 50), args.warmup))

    out = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "rows": w.n_rows, "requests": w.n_req,
                   "L": int(w.max_len), "k_blk": w.k_blk, "page_size": w.page_size,
                   "step": f"one qsa_decode_step call: the rows' {int(st['kp_rts_h'][-1])} own index "
                           "key(s) appended through the 4-slot ring (the blocks they complete "
                           "compressed) + fused score/top-512/expand/slots, replayed from a CUDA graph",
                   "l2": "flushed before every timed step (256 MB written, then 256 MB of another buffer read)",
                   "parallelism": f"replicas x{ws}"},
        "us_per_step": 1e3 * ms,
        "us_per_step_median": 1e3 * statistics.median(step_ms),
        "step_alg_bytes": step_bytes,
        "step_alg_GBps": step_bytes / (ms * 1e-3) / 1e9,
        "step_frac_hbm": step_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "roofline": {"bound": "hbm", "kernel": names[dom], "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": captured_traffic(names[dom], w.name),
                     "alg_bytes_per_launch": kbytes[dom],
                     "us_per_launch": 1e3 * kms[dom],
                     "timing": "CUDA events around the kernel's own API call replayed from a CUDA "
                               "graph, L2 flushed before each launch, mean over the timed launches",
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, burst)"},
        "kernels": kernels,
        "e2e": {"value": ws * w.n_rows / (e2e_ms * 1e-3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "how": "one pinned host buffer of the step's inputs copied in, one eager decode_step "
                       "call, slots copied back; no graph"},
        "gpu_launches": 3 * args.steps,
        "timing_floor_us": {"value": 1e3 * floor_ms,
                            "how": "a CUDA graph of one trivial kernel (a one-element add) timed like the "
                                   "step: L2 flushed before it, CUDA events around the replay"},
        "clocks": clocks.summary(),
        "wall_s_timed_region": wall,
    }
    del st
    if rank == 0 and not args.no_variants:
        it = max(10, min(args.steps, 30))
        out["variants"] = {name: fn() for name, fn in variant_table(g, it, args.warmup, peaks).items()}
    if rank == 0:
        if args.cpu_budget > 0:
            out["cpu_baseline"] = cpu_oracle_rate(w, args.cpu_budget)
        print(json.dumps(add_nominal_fractions(out)))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
