"""Host-side logic of bench.py on CPU: FLOP/byte accounting, the reduction
over ranks (gloo, two processes), and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

import bench
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("nq,nk,causal", [(7, 7, True), (5, 2, True), (2, 5, True), (9, 4, False),
                                          (1, 700, True), (517, 200, True), (300, 300, True)])
def test_attended_pairs_brute_force(nq, nk, causal):
    p = workloads.make_prefill(1, 3, 1, nq, nk, 8, causal=causal, seed=1)
    brute = 3 * sum(1 for i in range(nq) for j in range(nk) if (not causal or j <= i + nk - nq))
    assert bench.attended_pairs(p) == brute


@pytest.mark.parametrize("nq,nk,causal,window", [(7, 7, True, (2, -1)), (5, 9, False, (1, 2)),
                                                 (9, 5, False, (0, 0)), (300, 700, True, (128, 5)),
                                                 (40, 40, False, (-1, 3)), (3, 50, False, (60, 60))])
def test_attended_pairs_window_brute_force(nq, nk, causal, window):
    p = workloads.make_prefill(1, 2, 1, nq, nk, 8, causal=causal, seed=1, window=window)
    left, right = window
    def keep(i, j):
        c = i + nk - nq
        return ((not causal or j <= c) and (left < 0 or j >= c - left) and (right < 0 or j <= c + right))
    brute = 2 * sum(1 for i in range(nq) for j in range(nk) if keep(i, j))
    assert bench.attended_pairs(p) == brute


def test_mha_causal_flops():
    p = workloads.make_prefill(4, 16, 16, 4096, 4096, 128, causal=True, seed=1)
    assert bench.prefill_flops(p) == 4 * 128 * 64 * 4096 * 4097 // 2
    assert bench.prefill_flops_literal(p) == 4 * 4096 * 4096 * 128 * 64 / 2


def test_decode_bytes():
    d = workloads.make_decode([17, 32], 8, 2, 128, num_pages=8, seed=1)
    kv = (17 + 32) * 2 * 128 * 2 * 2
    assert bench.decode_bytes(d) == kv + 2 * 2 * 8 * 128 * 2 + 4 * 2 * 8 + 4 * (2 + 2) + 4 * 2


def test_backward_flops():
    p = workloads.make_prefill(4, 16, 16, 4096, 4096, 128, causal=True, seed=1)
    assert bench.backward_flops(p) == 2.5 * bench.prefill_flops(p)


def test_kvcache_bytes():
    p = workloads.make_kvcache_decode([17, 32], 3, 8, 2, 128, num_pages=8, seed=1, append=True)
    kv = (17 + 32) * 2 * 128 * 2 * 2
    new = 2 * (2 * 2 * 3 * 2 * 128 * 2)
    assert bench.kvcache_bytes(p) == kv + new + 2 * 2 * 3 * 8 * 128 * 2 + 4 * 2 * 8 * 3 + 4 * (2 + 2) + 4 * 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t, u = bench.reduce_max_sum(world, 10.0 + rank, 100.0 * (rank + 1))
    bench.barrier(world)
    q.put((rank, t, u))
    dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, u in got:
        assert t == 11.0 and u == 300.0


def test_reference_arm_json_line():
    env = dict(os.environ, ATTN_REFERENCE_STEP_SECONDS="0.3")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny", "--steps", "2", "--warmup", "1"], capture_output=True, text=True, env=env,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the arm's own step time (each step is one bounded sample of ~0.3 s) and the
    # whole workload's time at the measured rate
    assert 0.1e3 < line["ms_per_step"] < 60e3
    assert line["ms_per_full_step_extrapolated"] > 0


def test_clock_summary_windows_and_reasons():
    """The clock record keeps only the samples of the timed window, reports
    their median and the union of the clock-event reasons, and the whole run
    beside it."""
    c = bench.ClockSampler(0)
    c.source = "test"
    c.samples = [(0.0, 1000.0, 2070.0, set()), (1.0, 2070.0, 2070.0, set()), (2.0, 2055.0, 2070.0, {"sw_power_cap"}),
                 (3.0, 2070.0, 2070.0, set()), (9.0, 800.0, 2070.0, {"hw_slowdown"})]
    rec = c.record(1.0, 3.0)
    assert rec["samples"] == 3 and rec["sm_mhz"] == 2070.0 and rec["sm_min_mhz"] == 2055.0
    assert rec["reasons"] == ["sw_power_cap"] and rec["source"] == "test"
    assert rec["whole_run"]["samples"] == 5 and rec["whole_run"]["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_sampler_without_a_gpu_records_nothing():
    with bench.ClockSampler(0) as c:
        pass
    rec = c.record(0.0, 1e18)
    assert rec["samples"] == rec["whole_run"]["samples"] == len(c.samples)
