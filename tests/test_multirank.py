"""The N > 1 host logic of bench.py on CPU: two gloo ranks over 127.0.0.1.

The decode path shards by batch with no exchange (replicas), so the only
cross-rank steps are the barrier, the max of the timed regions and the sum of
the bytes; rank 0 alone prints, and the reference arm does its work on rank 0
only while the other ranks exit cleanly.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist

    import bench
    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    mx = bench.max_over_ranks(float(rank + 1) * 1.5, w)
    sm = bench.sum_over_ranks(float(10 * (rank + 1)), w)

    class A:  # reference-arm arguments: rank != 0 must return without work
        steps, warmup, workload, cpu_budget = 1, 0, "llama32_1b_tiny", 0.1
    ref = bench.run_reference(A, w, r) if r != 0 else "skipped"
    q.put((rank, mx, sm, ref))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_only_rank0_works():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got[0][1] == pytest.approx(3.0) and got[1][1] == pytest.approx(3.0)   # max over ranks
    assert got[0][2] == pytest.approx(30.0) and got[1][2] == pytest.approx(30.0)  # sum over ranks
    assert got[1][3] is None                                                     # rank 1 did no work


def test_byte_accounting_counts_visible_keys_once_per_kv_head():
    import bench
    cfg = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=64, kv_dtype="bf16", io_dtype="bf16",
               out_dtype="f32", window=0)
    assert bench.partial_bytes(cfg, [10, 20]) == (10 + 20) * 2 * (128 + 128)
    cfg_w = dict(cfg, window=15)
    assert bench.partial_bytes(cfg_w, [10, 20]) == (10 + 15) * 2 * 256
    cfg_q = dict(cfg, kv_dtype="vq8")
    assert bench.partial_bytes(cfg_q, [5]) == 5 * 2 * (128 + 64 + 4)
    small = 2 * (8 + 4) * 64 * 2 + 2 * 2 * 256 + 2 * 8 * 64 * 4
    assert bench.decode_step_bytes(cfg, [9, 19]) == bench.partial_bytes(cfg, [10, 20]) + small


def test_byte_accounting_for_q8_and_chunks():
    """q8 rows are D codes plus a 4-byte scale for keys and values alike; a step of
    T tokens reads each visible key once (lengths grow by T) and moves T times
    the small rows (q, k, v in; appended rows; outputs)."""
    import bench
    cfg = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, kv_dtype="q8", io_dtype="bf16",
               out_dtype="f32", window=0)
    assert bench.partial_bytes(cfg, [10, 20]) == (10 + 20) * 2 * (2 * (128 + 4))
    chunk = dict(cfg, kv_dtype="bf16", q_len=4)
    small = 4 * (2 * (8 + 4) * 128 * 2 + 2 * 2 * (256 + 256) + 2 * 8 * 128 * 4)
    assert bench.decode_step_bytes(chunk, [9, 19]) == bench.partial_bytes(chunk, [13, 23]) + small
    # with a window each token sees its own last W keys: the step reads the union of
    # the rows' windows, W + T - 1 keys, once
    win = dict(chunk, window=5)
    assert bench.partial_bytes(win, [13, 23]) == (8 + 8) * 2 * 512


def test_clock_summary_uses_samples_inside_the_timed_region():
    """The reported SM clock and throttle reasons come from the nvidia-smi
    samples taken between mark_start and mark_end; without such a sample (a
    region shorter than the sampling period) all samples count, and the line
    says so with under_load = 0."""
    import datetime

    import bench
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    base = datetime.datetime(2026, 1, 2, 3, 4, 5)
    c.lines = []
    for i in range(12):
        t = base + datetime.timedelta(milliseconds=20 * i)
        sm = 1980 if 3 <= i <= 8 else 2070                      # the loaded samples run slower
        cap = "Active" if i == 5 else "Not Active"
        c.lines.append(f"{t:%Y/%m/%d %H:%M:%S}.{t.microsecond // 1000:03d}, {sm}, 2070, 900.0, 0x4, "
                       f"Not Active, Not Active, Not Active, {cap}")
    c.lines.append("garbage line")
    c.t0 = base + datetime.timedelta(milliseconds=55)
    c.t1 = base + datetime.timedelta(milliseconds=170)
    s = c.summary()
    assert s == {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 12,
                 "under_load": 6}
    c.t0 = c.t1 = None
    s = c.summary()
    assert s["under_load"] == 0 and s["samples"] == 12 and s["sm_mhz"] == 2025.0
