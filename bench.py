"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * attn_fwd on the MHA causal prefill workload (B=4, Hq=Hkv=16, N=4096,
    d=128, bottom-right causal), and
  * attn_decode_paged on the paged split-KV decode workload (B=64, Hq=32,
    Hkv=8, d=128, lengths U[4096, 32768], 16-token pages, 200k-page pool).
`value` is the prefill throughput in TFLOP/s (exact attended query-key pairs
x 4 x d, i.e. causal-adjusted); the decode bandwidth in GB/s (algorithmic
bytes: every K/V row the sequences own, read once, plus q, out, lse and the
block-table rows) is reported beside it.  Both are timed per call with CUDA
events on the launching stream; L2 is flushed (a 256 MB write) between steps,
outside the timed calls.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl libattn|reference]
                  [--workload hot_path|mha_causal|gqa_causal|varlen_chunked|swa_causal|tiny|
                              paged_decode|paged_decode_small|spec_decode|mha_causal_bwd|gqa_causal_bwd]

--impl reference times the fp64 CPU oracle on the host cores (bounded row
samples of the same workload, same metric and unit).  Under torchrun each rank
runs an independent replica on its own GPU (the path needs no exchange);
rank 0 prints one JSON line with the max time over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

PREFILL_WORKLOADS = ("mha_causal", "gqa_causal", "varlen_chunked", "swa_causal", "tiny")
BWD_WORKLOADS = {"mha_causal_bwd": "mha_causal", "gqa_causal_bwd": "gqa_causal"}  # backward of a prefill workload
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0}
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------- accounting
def attended_pairs(p) -> int:
    """Exact number of (query, key) pairs the mask allows, over all heads:
    row i of a sequence keeps keys [c - left, c + right] inside [0, nk) with
    c = i + nk - nq (a side < 0 unbounded; causal caps right at 0)."""
    left, right = (int(x) for x in getattr(p, "window", (-1, -1)))
    if p.causal:
        right = 0
    total = 0
    for nq, nk in p.seq_lens():
        if nq <= 0 or nk <= 0:
            continue
        c = np.arange(nq, dtype=np.int64) + (nk - nq)
        lo = np.maximum(c - left, 0) if left >= 0 else np.zeros_like(c)
        hi = np.minimum(c + right, nk - 1) if right >= 0 else np.full_like(c, nk - 1)
        total += int(np.maximum(hi - lo + 1, 0).sum())
    return total * p.Hq


def prefill_flops(p) -> float:
    return 4.0 * p.d * attended_pairs(p)


def prefill_flops_literal(p) -> float:
    """4*Nq*Nk*d*H*B, halved for causal (the coarse textbook count)."""
    tot = sum(4.0 * nq * nk * p.d for nq, nk in p.seq_lens()) * p.Hq
    return tot / 2 if p.causal else tot


def prefill_bytes(p) -> float:
    tq = sum(nq for nq, _ in p.seq_lens())
    tk = sum(nk for _, nk in p.seq_lens())
    return 2.0 * p.d * (2 * tq * p.Hq + 2 * tk * p.Hkv) + 4.0 * tq * p.Hq


def decode_bytes(d) -> float:
    """Algorithmic bytes of one decode call: each sequence's K and V rows once,
    q and out, lse, and the block-table entries the sequences use."""
    lens = d.seq_lens.cpu().tolist()
    kv = sum(lens) * d.Hkv * d.d * 2 * 2
    pages = sum(-(-L // d.page_size) for L in lens)
    return float(kv + 2 * d.B * d.Hq * d.d * 2 + 4 * d.B * d.Hq + 4 * pages + 4 * d.B)


def kvcache_bytes(p) -> float:
    """Algorithmic bytes of one multi-query decode call with append: every
    key and value row of each sequence once (the appended rows included),
    the new K/V rows read and written once, q and out, lse, and the
    block-table entries the sequences use."""
    lens = p.seq_lens.cpu().tolist()
    kv = sum(lens) * p.Hkv * p.d * 2 * 2
    new = 0 if p.k_new is None else 2 * (2 * p.B * p.Nq * p.Hkv * p.d * 2)
    pages = sum(-(-L // p.page_size) for L in lens)
    return float(kv + new + 2 * p.B * p.Nq * p.Hq * p.d * 2 + 4 * p.B * p.Hq * p.Nq + 4 * pages + 4 * p.B)


def is_kvcache(d) -> bool:
    return isinstance(d, workloads.KVCacheDecode)


def backward_flops(p) -> float:
    """Algorithmic FLOPs of one backward call: the five products of the
    recomputation (S, dP, dV, dS^T Q, dS K), 2 * d per attended pair each."""
    return 10.0 * p.d * attended_pairs(p)


KERNEL_SOURCES = {
    "attn_fwd": ["exact_io_aware_04_gb300/csrc/fwd.cu", "exact_io_aware_04_gb300/csrc/ptx.cuh"],
    "attn_bwd": ["exact_io_aware_04_gb300/csrc/bwd.cu", "exact_io_aware_04_gb300/csrc/ptx.cuh"],
    "attn_decode_paged": ["exact_io_aware_04_gb300/csrc/decode.cu", "exact_io_aware_04_gb300/csrc/ptx.cuh"],
    "attn_decode_kvcache": ["exact_io_aware_04_gb300/csrc/decode.cu", "exact_io_aware_04_gb300/csrc/ptx.cuh"],
}


def source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from profiles/traffic.json (an ncu capture), or
    None when no capture exists for this workload or the kernel source has
    changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(kernel, {}).get(workload)
    except Exception:
        return None
    if not rec or rec.get("source_sha256") != source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return {k: float(j[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
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
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max_sum(world, t_max: float, units: float, device=None):
    """(max over ranks of t_max, sum over ranks of units)."""
    if world <= 1:
        return t_max, units
    import torch.distributed as dist
    dev = device if device is not None else torch.device("cpu")
    a = torch.tensor([t_max], dtype=torch.float64, device=dev)
    b = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(a, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(a.item()), float(b.item())


# ---------------------------------------------------------------- oracle timing (CPU)
def oracle_sample_rate(p, target_s: float, seed: int, max_rows: int = 1 << 20):
    """Times the oracle on seeded rows of prefill problem p; grows the sample
    until it takes about target_s.  Returns (flops/s, rows, seconds, threads)."""
    import numpy as np
    import oracle
    threads = oracle.num_threads()
    lens = [nq for nq, _ in p.seq_lens()]
    g = torch.Generator().manual_seed(seed)
    n = 64
    while True:
        b = torch.randint(0, p.B, (n,), generator=g)
        h = torch.randint(0, p.Hq, (n,), generator=g)
        i = (torch.rand(n, generator=g) * torch.tensor([lens[x] for x in b.tolist()], dtype=torch.float32)).long()
        rows = torch.stack([b, h, i], 1).numpy().astype(np.int32)
        t0 = time.perf_counter()
        oracle.prefill(p, rows, threads=threads)
        dt = time.perf_counter() - t0
        fl = 4.0 * p.d * sum(row_keys(p, int(r[0]), int(r[2])) for r in rows)
        if dt >= target_s * 0.5 or n >= max_rows:
            return fl / dt, n, dt, threads, fl
        n = min(max_rows, int(n * max(2.0, target_s / max(dt, 1e-3))))


def row_keys(p, b, i):
    """Keys row i of sequence b keeps (the attended_pairs rule for one row)."""
    nq, nk = p.seq_lens()[b]
    left, right = (int(x) for x in getattr(p, "window", (-1, -1)))
    if p.causal:
        right = 0
    c = i + nk - nq
    lo = max(c - left, 0) if left >= 0 else 0
    hi = min(c + right, nk - 1) if right >= 0 else nk - 1
    return max(0, hi - lo + 1)


def oracle_kvcache_rate(p, target_s: float, seed: int):
    """Times the oracle on seeded (b, h, i) rows of a multi-query decode
    problem (cache already appended); bytes = the K/V rows each row reads."""
    import oracle
    threads = oracle.num_threads()
    g = torch.Generator().manual_seed(seed)
    n = 32
    lens = p.seq_lens.cpu().tolist()
    while True:
        b = torch.randint(0, p.B, (n,), generator=g)
        h = torch.randint(0, p.Hq, (n,), generator=g)
        i = torch.randint(0, p.Nq, (n,), generator=g)
        rows = torch.stack([b, h, i], 1).numpy().astype(np.int32)
        t0 = time.perf_counter()
        oracle.decode_multi_rows(p.q, p.k_cache, p.v_cache, p.block_table, p.seq_lens, scale=p.scale,
                                 causal=p.causal, rows=rows, threads=threads)
        dt = time.perf_counter() - t0
        keys = [lens[int(r[0])] - (p.Nq - 1 - int(r[2]) if p.causal else 0) for r in rows]
        byts = sum(max(0, k) * p.d * 2 * 2 for k in keys)
        if dt >= target_s * 0.5 or n >= p.B * p.Hq * p.Nq * 8:
            return byts / dt, n, dt, threads
        n = int(n * max(2.0, target_s / max(dt, 1e-3)))


def appended_host_copy(p):
    """Host copy of a multi-query decode problem with its append applied."""
    import oracle
    host = p.to("cpu")
    if host.k_new is not None:
        oracle.append_kv(host.k_cache, host.v_cache, host.block_table, host.seq_lens, host.k_new, host.v_new,
                         inplace=True)
    return host


def oracle_bwd_rate(p, g, target_s: float, seed: int):
    """Times the oracle backward on seeded (sequence, K/V head) pairs, one per
    host thread, over every row_stride-th query row; halves row_stride until
    the sample takes about target_s.  Returns (flops/s, sample text, seconds,
    threads); flops = 10 d x the keys of the rows processed."""
    import oracle
    threads = oracle.num_threads()
    gen = torch.Generator().manual_seed(seed)
    all_pairs = [(b, h) for b in range(p.B) for h in range(p.Hkv)]
    n = min(len(all_pairs), max(1, threads))
    idx = torch.randperm(len(all_pairs), generator=gen)[:n].tolist()
    pairs = [all_pairs[i] for i in idx]
    group = p.Hq // p.Hkv
    stride = max(1, p.Nq // 8)
    while True:
        t0 = time.perf_counter()
        oracle.backward(p, g, pairs=pairs, threads=threads, row_stride=stride)
        dt = time.perf_counter() - t0
        keys = sum(row_keys(p, b, i) for b, _ in pairs for i in range(0, p.seq_lens()[b][0], stride))
        flops = 10.0 * p.d * keys * group
        if dt >= target_s * 0.5 or stride == 1:
            return flops / dt, f"{n} pairs, every {stride}-th row", dt, min(threads, n)
        stride = max(1, int(stride / max(2.0, target_s / max(dt, 1e-3))))


def oracle_decode_rate(d, target_s: float, seed: int):
    import numpy as np
    import oracle
    threads = oracle.num_threads()
    g = torch.Generator().manual_seed(seed)
    n = 32
    lens = d.seq_lens.cpu().tolist()
    while True:
        b = torch.randint(0, d.B, (n,), generator=g)
        h = torch.randint(0, d.Hq, (n,), generator=g)
        rows = torch.stack([b, h], 1).numpy().astype(np.int32)
        t0 = time.perf_counter()
        oracle.decode(d, rows, threads=threads)
        dt = time.perf_counter() - t0
        byts = sum(lens[int(r[0])] * d.d * 2 * 2 for r in rows)
        if dt >= target_s * 0.5 or n >= d.B * d.Hq * 8:
            return byts / dt, n, dt, threads
        n = int(n * max(2.0, target_s / max(dt, 1e-3)))


# ---------------------------------------------------------------- main
def make_workloads(name, device):
    prefill = decode = None
    if name in ("hot_path",) + PREFILL_WORKLOADS:
        pname = "mha_causal" if name == "hot_path" else name
        prefill = getattr(workloads, pname)() if pname != "tiny" else workloads.tiny(True)
    if name in ("hot_path", "paged_decode"):
        decode = workloads.paged_decode(device=device)
    if name == "paged_decode_small":
        decode = workloads.paged_decode_small(device=device)
    if name == "spec_decode":
        decode = workloads.spec_decode(device=device)
    return prefill, decode


def run_reference(args, world, rank):
    """fp64 CPU oracle on bounded samples of the same workload."""
    if rank != 0:
        return 0
    # the headline of the hot-path step is the prefill metric; the CPU arm
    # times that part (the decode pool would not fit a bounded CPU sample)
    name = "mha_causal" if args.workload == "hot_path" else args.workload
    # each step is a bounded sample: about 4 s, but the whole --steps/--warmup run stays near
    # 150 s of oracle work however many steps are asked for
    per_step = float(os.environ.get("ATTN_REFERENCE_STEP_SECONDS", "4.0"))
    per_step = max(0.02, min(per_step, 150.0 / max(1, args.steps + args.warmup)))
    if name in BWD_WORKLOADS:
        prefill = getattr(workloads, BWD_WORKLOADS[name])()
        decode = None
        grad = workloads.randn_bf16(tuple(prefill.q.shape), seed=prefill.seed + 900)
    else:
        prefill, decode = make_workloads(name, "cpu")
    if name in BWD_WORKLOADS:
        rate_fn = lambda s: oracle_bwd_rate(prefill, grad, per_step, seed=s)[0]
        unit, metric_scale = "TFLOP/s", 1e-12
    elif prefill is not None:
        rate_fn = lambda s: oracle_sample_rate(prefill, per_step, seed=s)[0]
        unit, metric_scale = "TFLOP/s", 1e-12
    elif is_kvcache(decode):
        decode = appended_host_copy(decode)
        rate_fn = lambda s: oracle_kvcache_rate(decode, per_step, seed=s)[0]
        unit, metric_scale = "GB/s", 1e-9
    else:
        rate_fn = lambda s: oracle_decode_rate(decode, per_step, seed=s)[0]
        unit, metric_scale = "GB/s", 1e-9
    for w in range(args.warmup):
        rate_fn(10_000 + w)
    rates = [rate_fn(20_000 + s) for s in range(args.steps)]
    value = statistics.median(rates) * metric_scale
    import oracle
    cores = oracle.num_threads()
    wname = prefill.name if prefill else decode.name
    metric = METRIC
    if name in BWD_WORKLOADS:
        wname += "_backward"
        metric = BWD_METRIC
    sample = (f"each step: seeded rows of the {wname} workload, "
              f"about {per_step:.2f} s of fp64 oracle work, rate = work/seconds")
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wname},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


METRIC = "fwd TFLOP/s & % bf16 tensor peak; split-KV decode GB/s & % HBM peak"
BWD_METRIC = "bwd TFLOP/s (5 recomputation products per attended pair) & % bf16 tensor peak"


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["libattn", "reference"], default="libattn")
    ap.add_argument("--workload", default="hot_path",
                    choices=["hot_path", "paged_decode", "paged_decode_small", "spec_decode"]
                    + list(PREFILL_WORKLOADS) + list(BWD_WORKLOADS))
    ap.add_argument("--cpu-baseline-seconds", type=float, default=15.0)
    args = ap.parse_args(argv)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import exact_io_aware_04_gb300 as la
    la.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks, peaks_kind = load_peaks()
    if args.workload in BWD_WORKLOADS:
        return run_backward(args, la, dev, stream, world, rank, local, peaks, peaks_kind)

    prefill, decode = make_workloads(args.workload, dev)
    # ---- device-resident inputs
    if prefill is not None:
        pg = prefill.to(dev)
        if prefill.varlen:
            fargs = (pg.q, pg.k, pg.v)
            fkw = dict(causal=pg.causal, scale=pg.scale, cu_seqlens_q=pg.cu_q, cu_seqlens_k=pg.cu_k)
        else:
            fargs = (pg.q.view(pg.B, pg.Nq, pg.Hq, pg.d), pg.k.view(pg.B, pg.Nk, pg.Hkv, pg.d),
                     pg.v.view(pg.B, pg.Nk, pg.Hkv, pg.d))
            fkw = dict(causal=pg.causal, scale=pg.scale)
        if tuple(prefill.window) != (-1, -1):
            fkw["window"] = tuple(prefill.window)
        f_out = torch.empty_like(fargs[0])
        f_lse = torch.empty((pg.Hq, pg.q.shape[0]) if prefill.varlen else (pg.B, pg.Hq, pg.Nq),
                            dtype=torch.float32, device=dev)
        fkw.update(out=f_out, lse=f_lse)
        p_flops = prefill_flops(prefill)
    d_kernel, d_fn, d_launches = None, None, 0
    if decode is not None and is_kvcache(decode):
        ws = torch.empty(la.attn_decode_kvcache_workspace_size(decode.B, decode.Nq, decode.Hq, decode.Hkv,
                                                               decode.d, decode.page_size, decode.max_pages, 0),
                         dtype=torch.uint8, device=dev)
        d_out = torch.empty_like(decode.q)
        d_lse = torch.empty((decode.B, decode.Hq, decode.Nq), dtype=torch.float32, device=dev)
        dargs = (decode.q, decode.k_cache, decode.v_cache, decode.block_table, decode.seq_lens)
        dkw = dict(k_new=decode.k_new, v_new=decode.v_new, causal=decode.causal, scale=decode.scale, out=d_out,
                   lse=d_lse, workspace=ws)
        d_bytes = kvcache_bytes(decode)
        d_kernel, d_fn, d_launches = "attn_decode_kvcache", la.attn_decode_kvcache, 2 + (decode.k_new is not None)
    elif decode is not None:
        ws = torch.empty(la.attn_decode_workspace_size(decode.B, decode.Hq, decode.Hkv, decode.d,
                                                       decode.page_size, decode.max_pages, 0),
                         dtype=torch.uint8, device=dev)
        d_out = torch.empty_like(decode.q)
        d_lse = torch.empty((decode.B, decode.Hq), dtype=torch.float32, device=dev)
        dargs = (decode.q, decode.k_cache, decode.v_cache, decode.block_table, decode.seq_lens)
        dkw = dict(scale=decode.scale, out=d_out, lse=d_lse, workspace=ws)
        d_bytes = decode_bytes(decode)
        d_kernel, d_fn, d_launches = "attn_decode_paged", la.attn_decode_paged, 2
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(ev=None):
        flush.fill_(1)
        if ev is not None:
            ev[0].record(stream)
        if prefill is not None:
            la.attn_fwd(*fargs, **fkw)
        if ev is not None:
            ev[1].record(stream)
        if decode is not None:
            d_fn(*dargs, **dkw)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if la.attn_get_device_status() != 0:
        raise RuntimeError("device error during warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            step(events[i])
        torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier(world)
    st = la.attn_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {la.attn_status_string(st)} after the timed region")
    f_ms = [e[0].elapsed_time(e[1]) for e in events]
    d_ms = [e[1].elapsed_time(e[2]) for e in events]
    f_tot, d_tot = sum(f_ms), sum(d_ms)
    step_ms = (f_tot + d_tot) / args.steps

    # whole-job figures (max time over ranks, units summed over ranks)
    rooflines = {}
    line = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) rounded to bf16)"}
    if prefill is not None:
        f_max, f_units = reduce_max_sum(world, f_tot, p_flops * args.steps, dev)
        value = f_units / (f_max * 1e-3) / 1e12
        ach = p_flops / (f_tot / args.steps * 1e-3) / 1e12
        rooflines["attn_fwd"] = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                                 "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
                                 "frac_nominal": ach / NOMINAL["bf16_tflops"],
                                 "traffic": measured_traffic("attn_fwd", prefill.name),
                                 "compulsory_bytes": prefill_bytes(prefill),
                                 "peak_source": f"{peaks_kind} bf16 burst",
                                 "ms_per_launch_median": statistics.median(f_ms),
                                 "ms_per_launch_p95": sorted(f_ms)[int(0.95 * (len(f_ms) - 1))],
                                 "flops_per_launch": p_flops,
                                 "flops_per_launch_literal_formula": prefill_flops_literal(prefill)}
        line.update(value=value, unit="TFLOP/s")
    if decode is not None:
        d_max, d_units = reduce_max_sum(world, d_tot, d_bytes * args.steps, dev)
        dval = d_units / (d_max * 1e-3) / 1e9
        ach = d_bytes / (d_tot / args.steps * 1e-3) / 1e9
        rooflines[d_kernel] = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": ach / peaks["hbm_gbs"], "frac_nominal": ach / NOMINAL["hbm_gbs"],
                               "traffic": measured_traffic(d_kernel, decode.name),
                               "peak_source": f"{peaks_kind} copy bandwidth",
                               "ms_per_call_median": statistics.median(d_ms),
                               "ms_per_call_p95": sorted(d_ms)[int(0.95 * (len(d_ms) - 1))],
                               "bytes_per_call": d_bytes, "launches_per_call": d_launches}
        line["decode"] = {"value": dval, "unit": "GB/s", "frac_of_measured_hbm": dval / world / peaks["hbm_gbs"],
                          "frac_of_8TBs": dval / world / NOMINAL["hbm_gbs"]}
        if prefill is None:
            line.update(value=dval, unit="GB/s")
    dominant = max(rooflines, key=lambda k: (f_tot if k == "attn_fwd" else d_tot))
    line["roofline"] = dict(rooflines[dominant], kernel=dominant)
    line["rooflines"] = rooflines
    line["ms_per_step"] = step_ms
    line["gpu_launches"] = args.steps * ((1 if prefill is not None else 0) + d_launches)
    cfg = {"workload": ("mha_causal_b4_h16_n4096_d128 + paged_decode_b64_hq32_hkv8_d128"
                        if args.workload == "hot_path" else (prefill or decode).name),
           "l2": "flushed between steps (256 MB write, outside the timed calls)",
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    if prefill is not None:
        cfg.update(prefill={"B": prefill.B, "Hq": prefill.Hq, "Hkv": prefill.Hkv, "Nq": prefill.Nq,
                            "Nk": prefill.Nk, "d": prefill.d, "causal": prefill.causal,
                            "varlen": prefill.varlen})
    if decode is not None:
        cfg.update(decode={"B": decode.B, "Hq": decode.Hq, "Hkv": decode.Hkv, "d": decode.d,
                           "page_size": decode.page_size, "num_pages": decode.num_pages,
                           "tokens": int(decode.seq_lens.sum())})
        if is_kvcache(decode):
            cfg["decode"].update(Nq=decode.Nq, causal=decode.causal, append=decode.k_new is not None)
    line["config"] = cfg
    line["clocks"] = clocks.summary()
    line["wall_s_timed_region"] = t_wall

    # ---- end to end through the public API with pinned host buffers
    line["e2e"] = measure_e2e(la, prefill, decode, fargs if prefill is not None else None,
                              fkw if prefill is not None else None, dargs if decode is not None else None,
                              dkw if decode is not None else None, stream, world, dev,
                              steps=min(args.steps, 20), d_fn=d_fn)

    if rank == 0 and world == 1 and args.cpu_baseline_seconds > 0:
        line["cpu_baseline"] = cpu_baseline(prefill, decode, args.cpu_baseline_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_backward(args, la, dev, stream, world, rank, local, peaks, peaks_kind):
    """The backward of a prefill workload: attn_bwd (D, dK/dV, dQ kernels)
    with q, k, v, the forward's out and lse and a seeded dO resident."""
    p = getattr(workloads, BWD_WORKLOADS[args.workload])()
    g_host = workloads.randn_bf16(tuple(p.q.shape), seed=p.seed + 900)
    pg = p.to(dev)
    shape_q = (p.B, p.Nq, p.Hq, p.d)
    shape_k = (p.B, p.Nk, p.Hkv, p.d)
    q, k, v = pg.q.view(shape_q), pg.k.view(shape_k), pg.v.view(shape_k)
    out, lse = la.attn_fwd(q, k, v, causal=p.causal, scale=p.scale)
    g = g_host.to(dev).view(shape_q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(la.lib().attn_bwd_workspace_size(p.B, p.Hq, p.Nq, 0), dtype=torch.uint8, device=dev)
    kw = dict(causal=p.causal, scale=p.scale, dq=dq, dk=dk, dv=dv, workspace=ws)
    flops = backward_flops(p)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(ev=None):
        flush.fill_(1)
        if ev is not None:
            ev[0].record(stream)
        la.attn_bwd(q, k, v, out, lse, g, **kw)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if la.attn_get_device_status() != 0:
        raise RuntimeError("device error during warm-up")
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            step(events[i])
        torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier(world)
    st = la.attn_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {la.attn_status_string(st)} after the timed region")
    ms = [e[0].elapsed_time(e[1]) for e in events]
    tot = sum(ms)
    t_max, units = reduce_max_sum(world, tot, flops * args.steps, dev)
    value = units / (t_max * 1e-3) / 1e12
    ach = flops / (tot / args.steps * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": ach / peaks["bf16_tflops"], "frac_nominal": ach / NOMINAL["bf16_tflops"],
            "traffic": measured_traffic("attn_bwd", p.name), "peak_source": f"{peaks_kind} bf16 burst",
            "ms_per_call_median": statistics.median(ms), "ms_per_call_p95": sorted(ms)[int(0.95 * (len(ms) - 1))],
            "flops_per_call": flops, "flops_executed_per_call": 14.0 * p.d * attended_pairs(p),
            "launches_per_call": 3, "kernel": "attn_bwd"}
    line = {"metric": BWD_METRIC,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) rounded to bf16)",
            "value": value, "unit": "TFLOP/s", "roofline": roof, "ms_per_step": tot / args.steps,
            "gpu_launches": 3 * args.steps,
            "config": {"workload": p.name + "_backward", "l2": "flushed between steps (256 MB write, outside the timed calls)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "prefill": {"B": p.B, "Hq": p.Hq, "Hkv": p.Hkv, "Nq": p.Nq, "Nk": p.Nk, "d": p.d,
                                   "causal": p.causal}},
            "clocks": clocks.summary(), "wall_s_timed_region": t_wall}
    # end to end: q, k, v, out, lse, dO from pinned host memory, dq/dk/dv back
    src = [q, k, v, out, lse, g]
    host_in = [t.cpu().pin_memory() for t in src]
    bkw = {x: y for x, y in kw.items() if x not in ("dq", "dk", "dv")}
    out_shapes = [(tuple(t.shape), t.dtype) for t in (dq, dk, dv)]

    def compute(b, dev_in, dev_out):
        la.attn_bwd(*dev_in[:5], dev_in[5], dq=dev_out[0], dk=dev_out[1], dv=dev_out[2], **bkw)
    n_e2e = min(args.steps, 20)
    barrier(world)
    ms_e2e, host_out = run_streamed(host_in, compute, out_shapes, n_e2e, stream, dev)
    e_max, e_units = reduce_max_sum(world, ms_e2e, flops * n_e2e, dev)
    line["e2e"] = {"value": e_units / (e_max * 1e-3) / 1e12, "unit": "TFLOP/s",
                   "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host_in),
                   "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_out), "steps": n_e2e,
                   "note": "q, k, v, out, lse and dO copied from pinned host memory and dq, dk, dv copied back "
                           "every step (transfers overlap neighbouring steps)"}
    if rank == 0 and world == 1 and args.cpu_baseline_seconds > 0:
        try:
            rate, what, dt, threads = oracle_bwd_rate(p, g_host, args.cpu_baseline_seconds, seed=4242)
            line["cpu_baseline"] = {"value": rate * 1e-12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                    "sample": f"seeded (sequence, K/V head) pairs of {p.name}: {what}, "
                                              f"in {dt:.1f} s"}
        except Exception as e:
            line["cpu_baseline"] = {"value": None, "unit": None, "cores": None, "kind": "oracle",
                                    "sample": f"failed: {e}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_streamed(host_in, compute, out_shapes, steps, stream, dev, depth=2):
    """End-to-end steps with the transfers of neighbouring steps overlapped,
    as a streaming caller would run them: step i+1's inputs upload on one
    copy stream while step i computes on `stream` and step i-1's results
    download on another.  Every step still moves all of its inputs host ->
    device and all of its results device -> host inside the timed region.
    Device buffers are `depth`-deep; `compute(b, dev_in, dev_out)` runs step
    buffer b.  Returns the elapsed ms between an event on `stream` before the
    first upload and one after the last download (after 3 untimed steps)."""
    dev_in = [[torch.empty(h.shape, dtype=h.dtype, device=dev) for h in host_in] for _ in range(depth)]
    dev_out = [[torch.empty(sh, dtype=dt, device=dev) for sh, dt in out_shapes] for _ in range(depth)]
    host_out = [torch.empty(sh, dtype=dt).pin_memory() for sh, dt in out_shapes]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    in_ready = [ev() for _ in range(depth)]
    comp_done = [ev() for _ in range(depth)]
    out_done = [ev() for _ in range(depth)]

    def run(n):
        start = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        up.wait_event(start)
        down.wait_event(start)
        for i in range(n):
            b = i % depth
            with torch.cuda.stream(up):
                if i >= depth:
                    up.wait_event(comp_done[b])   # step i-depth has read these inputs
                for h, d in zip(host_in, dev_in[b]):
                    d.copy_(h, non_blocking=True)
                in_ready[b].record(up)
            stream.wait_event(in_ready[b])
            if i >= depth:
                stream.wait_event(out_done[b])    # step i-depth's results have left
            compute(b, dev_in[b], dev_out[b])
            comp_done[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(comp_done[b])
                for h, d in zip(host_out, dev_out[b]):
                    h.copy_(d, non_blocking=True)
                out_done[b].record(down)
        stream.wait_event(out_done[(n - 1) % depth])
        end = torch.cuda.Event(enable_timing=True)
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    run(3)
    return run(steps), host_out


def measure_e2e(la, prefill, decode, fargs, fkw, dargs, dkw, stream, world, dev, steps, d_fn=None):
    """The headline metric through the public API with the step's inputs in
    pinned host memory: H2D copies, the call, and a D2H read of the result,
    all inside the timed region (transfers of neighbouring steps overlap,
    see run_streamed)."""
    if prefill is not None:
        host_in = [t.cpu().pin_memory() for t in fargs]
        kw = {k: v for k, v in fkw.items() if k not in ("out", "lse")}
        out_shapes = [(tuple(fkw["out"].shape), fkw["out"].dtype), (tuple(fkw["lse"].shape), fkw["lse"].dtype)]

        def compute(b, dev_in, dev_out):
            la.attn_fwd(*dev_in, out=dev_out[0], lse=dev_out[1], **kw)
        units, unit, scale = prefill_flops(prefill), "TFLOP/s", 1e-12
        note = "prefill q, k, v copied from pinned host memory and out, lse copied back every step"
    else:
        # the step's inputs: the queries (and the new tokens' K/V when appending)
        names = ["q"] + [k for k in ("k_new", "v_new") if dkw.get(k) is not None]
        src = {"q": dargs[0], **{k: dkw[k] for k in names[1:]}}
        host_in = [src[k].cpu().pin_memory() for k in names]
        kw = {k: v for k, v in dkw.items() if k not in ("out", "lse", "k_new", "v_new")}
        out_shapes = [(tuple(dkw["out"].shape), dkw["out"].dtype), (tuple(dkw["lse"].shape), dkw["lse"].dtype)]

        def compute(b, dev_in, dev_out):
            extra = dict(zip(names[1:], dev_in[1:]))
            d_fn(dev_in[0], *dargs[1:], out=dev_out[0], lse=dev_out[1], **extra, **kw)
        units = kvcache_bytes(decode) if is_kvcache(decode) else decode_bytes(decode)
        unit, scale = "GB/s", 1e-9
        note = "decode queries (and new K/V rows) copied each step; the paged cache stays resident"
    barrier(world)
    ms, host_out = run_streamed(host_in, compute, out_shapes, steps, stream, dev)
    t_max, tot_units = reduce_max_sum(world, ms, units * steps, dev)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    return {"value": tot_units / (t_max * 1e-3) * scale, "unit": unit, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "note": note + " (transfers overlap neighbouring steps)"}


def cpu_baseline(prefill, decode, seconds):
    try:
        if prefill is not None:
            host = prefill.to("cpu")
            rate, n, dt, threads, fl = oracle_sample_rate(host, seconds, seed=4242)
            return {"value": rate * 1e-12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                    "sample": f"{n} seeded query rows of {prefill.name} ({fl / 1e9:.1f} GFLOP fp64) in {dt:.1f} s"}
        if is_kvcache(decode):
            host = appended_host_copy(decode)
            rate, n, dt, threads = oracle_kvcache_rate(host, seconds, seed=4242)
            return {"value": rate * 1e-9, "unit": "GB/s", "cores": threads, "kind": "oracle",
                    "sample": f"{n} seeded (sequence, head, query) rows of {decode.name} in {dt:.1f} s"}
        host = decode.to("cpu")
        rate, n, dt, threads = oracle_decode_rate(host, seconds, seed=4242)
        return {"value": rate * 1e-9, "unit": "GB/s", "cores": threads, "kind": "oracle",
                "sample": f"{n} seeded (sequence, head) rows of {decode.name} in {dt:.1f} s"}
    except Exception as e:  # the baseline never blocks the GPU line
        return {"value": None, "unit": None, "cores": None, "kind": "oracle", "sample": f"failed: {e}"}


if __name__ == "__main__":
    sys.exit(main())
