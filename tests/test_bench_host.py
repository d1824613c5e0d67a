"""Host-side logic of the benchmark without a GPU: the max-over-ranks timing
used when every rank runs an independent replica (world size 2, gloo), the
algorithmic byte counts, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.aggregate_time(1.0 + rank, world)  # rank 1 is the slow one
    bench.barrier(world)
    q.put((rank, t))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 2000)
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 2.0, 1: 2.0}
    assert all(p.exitcode == 0 for p in ps)


def test_decode_bytes_c2():
    import bench
    from workloads import c2_verify
    w = c2_verify(0)
    by = bench.decode_bytes(w)
    assert by["keys"] == 20000 * 256          # keys read once for all 6 rows
    assert by["q"] == 6 * 1024
    assert by["slots"] == 6 * 2051 * 4
    assert by["page_table"] == 1250 * 4


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "rows/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_kernel_names_follow_the_dispatch_rules():
    import bench
    from workloads import c2_verify, c3_batched
    n2 = bench.kernel_names(c2_verify(0))  # 6 rows per request, 64-token pages
    assert n2 == {"compress": "compress_keys_kernel", "append": "append_keys_kernel",
                  "score": "score_mma_kernel", "select": "select_fast_kernel"}
    n3 = bench.kernel_names(c3_batched(0))  # one row per request, 32 rows
    assert n3["score"] == "score_mma_kernel" and n3["select"] == "select_fast_kernel"
    from workloads import c5_prefill
    n5 = bench.kernel_names(c5_prefill(0))  # 4096 rows of one request
    assert n5["score"] == "score_tc_kernel" and n5["select"] == "select_rows_kernel"


def test_kernel_bytes_c2():
    import bench
    from workloads import c2_verify
    w = c2_verify(0)
    kb = bench.kernel_bytes(w, 2)
    nb = [int(L) // 4 for L in w.row_len]
    assert kb["compress"] == 2 * (4 * 256 + 256 + 12)
    assert kb["select"] == 4 * sum(nb) + 4 * (80000 // 64) + 6 * 4 * (4 * 512 + 3)
    assert kb["score"] == 256 * max(nb) + 1024 * 6 + 4 * (80000 // 64) + 4 * sum(nb)


def test_append_bytes_verify_step():
    import bench
    import numpy as np
    # 6 tokens at 79994..79999: blocks 19998 (2 keys from the ring) and 19999 complete
    st = {"kp_rts_h": np.array([0, 6], np.int32), "kp_first_h": np.array([79994], np.int32)}
    assert bench.append_bytes(st) == 256 * 6 + 256 * 2 + 260 * 2 + 256 * 4 + 12
    # one token that completes nothing: its key read, the ring written
    st = {"kp_rts_h": np.array([0, 1], np.int32), "kp_first_h": np.array([8], np.int32)}
    assert bench.append_bytes(st) == 256 + 256 + 12


def test_long_rows_take_the_cluster_selection():
    import bench
    assert bench.topk_kernel_name(6, 80_000) == "select_long_kernel"
    assert bench.topk_kernel_name(64, 80_000) == "select_long_kernel"
    assert bench.topk_kernel_name(100, 80_000) == "select_kernel"
    assert bench.topk_kernel_name(6, 20_000) == "select_cluster_kernel"
    assert bench.topk_kernel_name(64, 20_000) == "select_resident_kernel"
    assert bench.topk_kernel_name(200, 20_000) == "select_resident_kernel"
    assert bench.topk_kernel_name(400, 20_000) == "select_rows_kernel"
    # k <= 1024: one register-resident CTA per row
    assert bench.topk_kernel_name(6, 20_000, k=512) == "select_fast_kernel"
    assert bench.topk_kernel_name(200, 32_768, k=1024) == "select_fast_kernel"
    assert bench.topk_kernel_name(400, 20_000, k=512) == "select_rows_kernel"


def test_nominal_fractions_beside_the_measured_ones():
    """Every fraction of the measured HBM peak in the line gets its
    companion against the nominal bandwidth (the same bytes, the same time)."""
    import bench
    out = {"step_alg_GBps": 790.0, "step_frac_hbm": 790.0 / 6683.8,
           "variants": {"a": {"alg_GBps": 3950.0, "frac_hbm": 3950.0 / 6683.8}, "b": {"us_per_call": 1.0},
                        "c": {"alg_GBps": 10.0}}}
    bench.add_nominal_fractions(out)
    assert abs(out["step_frac_hbm_nominal"] - 0.1) < 1e-12
    assert abs(out["variants"]["a"]["frac_hbm_nominal"] - 0.5) < 1e-12
    assert "frac_hbm_nominal" not in out["variants"]["b"]
    assert "frac_hbm_nominal" not in out["variants"]["c"]
