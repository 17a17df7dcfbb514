"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
attn_fwd on each single-GPU prefill configuration and attn_decode_paged on the
paged decode configuration, all inputs resident in HBM:
  * GQA causal prefill  B=2, Hq=32, Hkv=8, N=8192, d=128, one K channel x3
    (the largest configuration: it carries the headline `value`),
  * MHA causal prefill  B=4, Hq=Hkv=16, N=4096, d=128,
  * varlen chunked prefill  16 sequences, Nk ~ U[1024, 16384], Nq = min(512, Nk),
    Hq=32, Hkv=8, d=128, packed with cu_seqlens,
  * paged split-KV decode  B=64, Hq=32, Hkv=8, d=128, lengths U[4096, 32768],
    16-token pages in a 200k-page pool.
Prefill throughput is TFLOP/s of exact attended query-key pairs x 4 x d
(causal-adjusted); decode bandwidth is GB/s of algorithmic bytes (every K/V
row the sequences own, read once, plus q, out, lse and the block-table rows).
Every call is timed with CUDA events on the launching stream; L2 is flushed
at the start of each step, outside the timed calls: a 256 MB write, then a
256 MB read that writes the flush's dirty lines back before the call starts.  Each
configuration gets its own roofline record and, on rank 0 with one GPU, an
accuracy record against the fp64 oracle on a seeded row sample (the CPU
baseline leg).  After the step, the next rows (backward, local window,
several queries with the in-place append) are timed on their own.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl libattn|reference]
                  [--workload hot_path|mha_causal|gqa_causal|varlen_chunked|swa_causal|tiny|
                              paged_decode|paged_decode_small|spec_decode|spec_decode_small|
                              mha_causal_bwd|gqa_causal_bwd|
                              gqa_causal_fp8|mha_causal_fp8|varlen_chunked_fp8]
                  [--no-next]

--impl reference times the fp64 CPU oracle on the host cores (bounded row
samples of the headline workload, same metric and unit).  Under torchrun each
rank runs an independent replica on its own GPU (the path needs no exchange);
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
    "attn_fwd_fp8": ["exact_io_aware_04_gb300/csrc/fwd.cu", "exact_io_aware_04_gb300/csrc/ptx.cuh"],
    "attn_quantize_fp8": ["exact_io_aware_04_gb300/csrc/quant.cu", "exact_io_aware_04_gb300/csrc/ptx.cuh"],
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
    """SM clock, its maximum and the clock-event (throttle) reasons, sampled
    about every `period_ms` while the region runs, each sample stamped with
    the host clock so that the samples of a window (the timed region) can be
    summarised on their own.  Reads NVML directly (the driver's
    libnvidia-ml, through ctypes: a query takes microseconds, so even a
    50 ms timed region gets dozens of samples); where NVML cannot be loaded it
    falls back to `nvidia-smi -lms`.  Reading only: no setting is changed."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits (nvmlClocksEventReason*), the ones reported
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, gpu_index: int, period_ms: float = 1.0):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.nvml = None
        self.stop = threading.Event()
        self.thread = None
        self.samples = []   # (host time, sm MHz, max sm MHz, set of reasons)
        self.source = None
        self.pci = None

    def _open_nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        handle = ctypes.c_void_p()
        # the CUDA device's PCI address picks the NVML device (NVML may order
        # the GPUs differently); its index is the fallback
        found = False
        try:
            pr = torch.cuda.get_device_properties(self.gpu)
            self.pci = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
            found = lib.nvmlDeviceGetHandleByPciBusId_v2(self.pci.encode(), ctypes.byref(handle)) == 0
        except Exception:
            self.pci = None
        if not found and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(handle)) != 0:
            lib.nvmlShutdown()
            raise RuntimeError("no NVML handle")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mhz, mx, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        SM = ctypes.c_int(1)   # NVML_CLOCK_SM

        def query():
            if lib.nvmlDeviceGetClockInfo(handle, SM, ctypes.byref(mhz)) != 0:
                return None
            if lib.nvmlDeviceGetMaxClockInfo(handle, SM, ctypes.byref(mx)) != 0:
                return None
            if reasons_fn(handle, ctypes.byref(bits)) != 0:
                return None
            return float(mhz.value), float(mx.value), {n for n, b in self.REASON_BITS.items() if bits.value & b}
        if query() is None:
            lib.nvmlShutdown()
            raise RuntimeError("NVML queries failed")
        self.nvml = (lib, query)

    def _poll_nvml(self):
        query = self.nvml[1]
        while not self.stop.is_set():
            r = query()
            if r is not None:
                self.samples.append((time.perf_counter(),) + r)
            time.sleep(self.period_ms * 1e-3)

    def __enter__(self):
        try:
            self._open_nvml()
            self.source = "nvml"
            self.thread = threading.Thread(target=self._poll_nvml, daemon=True)
            self.thread.start()
            return self
        except Exception:
            self.nvml = None
        try:
            self.period_ms = 20
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            f = [x.strip() for x in line.strip().split(",")]
            if len(f) < 9:
                continue
            try:
                sm, mx = float(f[1]), float(f[2])
            except ValueError:
                continue
            reasons = {n for n, v in zip(names, f[5:9]) if v.lower().startswith("active")}
            self.samples.append((time.perf_counter(), sm, mx, reasons))

    def __exit__(self, *exc):
        self.stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        if self.nvml is not None:
            self.nvml[0].nvmlShutdown()

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock and throttle reasons of the samples taken
        in [t0, t1] (all samples when no window is given)."""
        sm, mx, reasons = [], [], set()
        for t, s, m, r in list(self.samples):
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            sm.append(s)
            mx.append(m)
            reasons |= r
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "sm_min_mhz": min(sm),
                "reasons": sorted(reasons), "samples": len(sm)}

    def record(self, t0, t1):
        """The timed window's summary, with the whole run (warm-up included,
        sampler started before it) beside it."""
        rec = self.summary(t0, t1)
        rec["period_ms"] = self.period_ms
        rec["source"] = self.source
        if self.pci:
            rec["gpu_pci"] = self.pci
        rec["whole_run"] = self.summary()
        return rec


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
# The default step: the three single-GPU prefill configurations (the largest,
# GQA causal N8192, first: it carries the headline value) and the paged decode.
HOT_PREFILL = ("gqa_causal", "mha_causal", "varlen_chunked")
DECODE_WORKLOADS = ("paged_decode", "paged_decode_small", "spec_decode", "spec_decode_small")
# Measured after the step on their own (backward, window, several queries with append).
NEXT_ROWS = ("mha_causal_bwd", "gqa_causal_bwd", "swa_causal", "spec_decode", "gqa_causal_fp8", "mha_causal_fp8",
             "gqa_causal_quantize_fp8")
FP8_WORKLOADS = {"gqa_causal_fp8": "gqa_causal", "mha_causal_fp8": "mha_causal", "varlen_chunked_fp8": "varlen_chunked"}


def make_workloads(name, device):
    """(prefill problems on the host, decode problem on `device` or None)."""
    if name == "hot_path":
        return [getattr(workloads, n)() for n in HOT_PREFILL], workloads.paged_decode(device=device)
    if name == "tiny":
        return [workloads.tiny(True)], None
    if name in PREFILL_WORKLOADS:
        return [getattr(workloads, name)()], None
    return [], getattr(workloads, name)(device=device)


class PrefillCall:
    """attn_fwd on one prefill problem with device-resident inputs and outputs."""
    kind, kernel, unit, unit_scale, launches, bound = "prefill", "attn_fwd", "TFLOP/s", 1e-12, 1, "tensor"

    def __init__(self, la, p, dev):
        self.la, self.p, self.name = la, p, p.name
        g = p.to(dev)
        if p.varlen:
            self.args = (g.q, g.k, g.v)
            self.kw = dict(causal=p.causal, scale=p.scale, cu_seqlens_q=g.cu_q, cu_seqlens_k=g.cu_k)
        else:
            self.args = (g.q.view(p.B, p.Nq, p.Hq, p.d), g.k.view(p.B, p.Nk, p.Hkv, p.d),
                         g.v.view(p.B, p.Nk, p.Hkv, p.d))
            self.kw = dict(causal=p.causal, scale=p.scale)
        if tuple(p.window) != (-1, -1):
            self.kw["window"] = tuple(p.window)
        self.out = torch.empty_like(self.args[0])
        self.lse = torch.empty((p.Hq, g.q.shape[0]) if p.varlen else (p.B, p.Hq, p.Nq), dtype=torch.float32,
                               device=dev)
        self.units = prefill_flops(p)

    def __call__(self):
        self.la.attn_fwd(*self.args, out=self.out, lse=self.lse, **self.kw)

    def describe(self):
        p = self.p
        return {"B": p.B, "Hq": p.Hq, "Hkv": p.Hkv, "Nq": p.Nq, "Nk": p.Nk, "d": p.d, "causal": p.causal,
                "varlen": p.varlen, "window": list(p.window)}

    def roofline_extra(self):
        return {"flops_per_launch": self.units, "flops_per_launch_literal_formula": prefill_flops_literal(self.p),
                "compulsory_bytes": prefill_bytes(self.p)}

    def e2e_parts(self):
        """(host inputs, compute(dev_in, dev_out), output shapes, note)."""
        host_in = [t.cpu().pin_memory() for t in self.args]
        kw = dict(self.kw)

        def compute(dev_in, dev_out):
            self.la.attn_fwd(*dev_in, out=dev_out[0], lse=dev_out[1], **kw)
        shapes = [(tuple(self.out.shape), self.out.dtype), (tuple(self.lse.shape), self.lse.dtype)]
        return host_in, compute, shapes, "prefill q, k, v copied from pinned host memory and out, lse copied back every step"


class DecodeCall:
    """attn_decode_paged (one query) or attn_decode_kvcache (several, with the
    append) on a decode problem whose paged cache stays resident."""
    kind, unit, unit_scale, bound = "decode", "GB/s", 1e-9, "hbm"

    def __init__(self, la, d, dev):
        self.la, self.d, self.name = la, d, d.name
        self.dargs = (d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens)
        self.out = torch.empty_like(d.q)
        if is_kvcache(d):
            ws = la.attn_decode_kvcache_workspace_size(d.B, d.Nq, d.Hq, d.Hkv, d.d, d.page_size, d.max_pages, 0)
            self.lse = torch.empty((d.B, d.Hq, d.Nq), dtype=torch.float32, device=dev)
            self.dkw = dict(k_new=d.k_new, v_new=d.v_new, causal=d.causal, scale=d.scale)
            self.fn, self.kernel = la.attn_decode_kvcache, "attn_decode_kvcache"
            self.units, self.launches = kvcache_bytes(d), 2 + (d.k_new is not None)
        else:
            ws = la.attn_decode_workspace_size(d.B, d.Hq, d.Hkv, d.d, d.page_size, d.max_pages, 0)
            self.lse = torch.empty((d.B, d.Hq), dtype=torch.float32, device=dev)
            self.dkw = dict(scale=d.scale)
            self.fn, self.kernel = la.attn_decode_paged, "attn_decode_paged"
            self.units, self.launches = decode_bytes(d), 2
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.fn(*self.dargs, out=self.out, lse=self.lse, workspace=self.ws, **self.dkw)

    def describe(self):
        d = self.d
        r = {"B": d.B, "Hq": d.Hq, "Hkv": d.Hkv, "d": d.d, "page_size": d.page_size, "num_pages": d.num_pages,
             "tokens": int(d.seq_lens.sum())}
        if is_kvcache(d):
            r.update(Nq=d.Nq, causal=d.causal, append=d.k_new is not None)
        return r

    def roofline_extra(self):
        return {"bytes_per_call": self.units, "launches_per_call": self.launches}

    def e2e_parts(self):
        names = ["q"] + [k for k in ("k_new", "v_new") if self.dkw.get(k) is not None]
        src = {"q": self.dargs[0], **{k: self.dkw[k] for k in names[1:]}}
        host_in = [src[k].cpu().pin_memory() for k in names]
        kw = {k: v for k, v in self.dkw.items() if k not in ("k_new", "v_new")}

        def compute(dev_in, dev_out):
            extra = dict(zip(names[1:], dev_in[1:]))
            self.fn(dev_in[0], *self.dargs[1:], out=dev_out[0], lse=dev_out[1], workspace=self.ws, **extra, **kw)
        shapes = [(tuple(self.out.shape), self.out.dtype), (tuple(self.lse.shape), self.lse.dtype)]
        return host_in, compute, shapes, "decode queries (and new K/V rows) copied each step; the paged cache stays resident"


class L2Flush:
    """Run between steps, outside the timed calls.  A 256 MB write evicts
    every input from the 126 MB L2; a 256 MB read of a second buffer then
    evicts the write's dirty lines, so their write-back happens here and not
    inside the next timed call (a short HBM-bound call, such as the 300 MB
    quantization, would otherwise pay for up to an L2's worth of it)."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.fill_(1)
        torch.amax(self.r, dim=0, out=self.sink)


L2_NOTE = ("flushed between steps (256 MB write, then a 256 MB read so the write's dirty lines are written back; "
           "outside the timed calls)")


def time_calls(calls, steps, warmup, stream, flush, sampler=None):
    """W untimed steps, then `steps` timed ones.  A step flushes L2
    (L2Flush) and runs every call once; each call is bracketed by CUDA events on
    the launching stream.  Returns (ms per call per step, wall seconds and
    host window of the timed region)."""
    def step(ev=None):
        flush()
        for c, fn in enumerate(calls):
            if ev is not None:
                ev[c][0].record(stream)
            fn()
            if ev is not None:
                ev[c][1].record(stream)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in calls]
              for _ in range(steps)]
    t0 = time.perf_counter()
    for i in range(steps):
        step(events[i])
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    ms = [[events[i][c][0].elapsed_time(events[i][c][1]) for i in range(steps)] for c in range(len(calls))]
    return ms, t1 - t0, (t0, t1)


def call_roofline(call, ms, peaks, peaks_kind):
    """Roofline record of one call from its per-step CUDA-event times."""
    mean = sum(ms) / len(ms)
    ach = call.units / (mean * 1e-3) * call.unit_scale
    peak_scale = getattr(call, "peak_scale", 1.0)
    peak = (peaks["bf16_tflops"] if call.bound == "tensor" else peaks["hbm_gbs"]) * peak_scale
    nominal = (NOMINAL["bf16_tflops"] if call.bound == "tensor" else NOMINAL["hbm_gbs"]) * peak_scale
    rec = {"kernel": call.kernel, "bound": call.bound, "achieved": ach, "peak": peak, "unit": call.unit,
           "frac": ach / peak, "frac_nominal": nominal and ach / nominal,
           "traffic": measured_traffic(call.kernel, call.name),
           "peak_source": getattr(call, "peak_note", None) or
                          (f"{peaks_kind} " + ("bf16 burst" if call.bound == "tensor" else "copy bandwidth")),
           "ms_mean": mean, "ms_median": statistics.median(ms), "ms_p95": sorted(ms)[int(0.95 * (len(ms) - 1))]}
    rec.update(call.roofline_extra())
    return rec


def kernel_roofline(calls, ms, peaks, peaks_kind):
    """The dominant kernel (most device time in the step) over all its
    launches: achieved = algorithmic work per launch / average launch time,
    i.e. the total work of its launches over their total time."""
    by_kernel = {}
    for c, call in enumerate(calls):
        by_kernel.setdefault(call.kernel, []).append(c)
    kern = max(by_kernel, key=lambda k: sum(sum(ms[c]) for c in by_kernel[k]))
    idx = by_kernel[kern]
    first = calls[idx[0]]
    tot_ms = sum(sum(ms[c]) for c in idx)
    steps = len(ms[idx[0]])
    units = sum(calls[c].units for c in idx) * steps
    ach = units / (tot_ms * 1e-3) * first.unit_scale
    peak = (peaks["bf16_tflops"] if first.bound == "tensor" else peaks["hbm_gbs"]) * getattr(first, "peak_scale", 1.0)
    traffic = [measured_traffic(calls[c].kernel, calls[c].name) for c in idx]
    n_launch = sum(calls[c].launches for c in idx)
    return {"kernel": kern, "bound": first.bound, "achieved": ach, "peak": peak, "unit": first.unit,
            "frac": ach / peak, "peak_source": getattr(first, "peak_note", None) or
                                               (f"{peaks_kind} " + ("bf16 burst" if first.bound == "tensor"
                                                                    else "copy bandwidth")),
            "traffic": (sum(traffic) / len(traffic)) if all(t is not None for t in traffic) else None,
            "launches_per_step": n_launch, "configs": [calls[c].name for c in idx],
            "ms_per_launch_mean": tot_ms / (steps * len(idx))}


def run_reference(args, world, rank):
    """fp64 CPU oracle on bounded samples of the same workload."""
    if rank != 0:
        return 0
    # the headline of the default step is the largest prefill configuration;
    # the CPU arm times that part (the decode pool would not fit a bounded CPU sample)
    name = HOT_PREFILL[0] if args.workload == "hot_path" else args.workload
    # each step is a bounded sample: about 4 s, but the whole --steps/--warmup run stays near
    # 150 s of oracle work however many steps are asked for
    per_step = float(os.environ.get("ATTN_REFERENCE_STEP_SECONDS", "4.0"))
    per_step = max(0.02, min(per_step, 150.0 / max(1, args.steps + args.warmup)))
    if name in BWD_WORKLOADS:
        prefill = getattr(workloads, BWD_WORKLOADS[name])()
        decode = None
        grad = workloads.randn_bf16(tuple(prefill.q.shape), seed=prefill.seed + 900)
    else:
        prefills, decode = make_workloads(name, "cpu")
        prefill = prefills[0] if prefills else None
    if name in BWD_WORKLOADS:
        rate_fn = lambda s: oracle_bwd_rate(prefill, grad, per_step, seed=s)[0]
        unit, metric_scale, full_units = "TFLOP/s", 1e-12, backward_flops(prefill)
    elif prefill is not None:
        rate_fn = lambda s: oracle_sample_rate(prefill, per_step, seed=s)[0]
        unit, metric_scale, full_units = "TFLOP/s", 1e-12, prefill_flops(prefill)
    elif is_kvcache(decode):
        decode = appended_host_copy(decode)
        rate_fn = lambda s: oracle_kvcache_rate(decode, per_step, seed=s)[0]
        unit, metric_scale, full_units = "GB/s", 1e-9, kvcache_bytes(decode)
    else:
        rate_fn = lambda s: oracle_decode_rate(decode, per_step, seed=s)[0]
        unit, metric_scale, full_units = "GB/s", 1e-9, decode_bytes(decode)
    for w in range(args.warmup):
        rate_fn(10_000 + w)
    rates, walls = [], []
    for s in range(args.steps):
        t0 = time.perf_counter()
        rates.append(rate_fn(20_000 + s))
        walls.append(time.perf_counter() - t0)
    value = statistics.median(rates) * metric_scale
    import oracle
    cores = oracle.num_threads()
    wname = prefill.name if prefill else decode.name
    metric = METRIC
    if name in BWD_WORKLOADS:
        wname += "_backward"
        metric = BWD_METRIC
    sample = (f"each step: seeded rows of the {wname} workload, "
              f"about {per_step:.2f} s of fp64 oracle work, rate = work/seconds; ms_per_step is the "
              f"sample's wall time, ms_per_full_step_extrapolated the whole workload at that rate")
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(walls),
        "ms_per_full_step_extrapolated": (1e3 * full_units / (value / metric_scale)) if value > 0 else None,
        "higher_is_better": True,
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
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["libattn", "reference"], default="libattn")
    ap.add_argument("--workload", default="hot_path",
                    choices=["hot_path"] + list(DECODE_WORKLOADS) + list(PREFILL_WORKLOADS) + list(BWD_WORKLOADS)
                    + list(FP8_WORKLOADS))
    ap.add_argument("--cpu-baseline-seconds", type=float, default=15.0)
    ap.add_argument("--no-next", action="store_true", help="skip the separately timed next rows")
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

    if args.workload in FP8_WORKLOADS:
        prefills, decode = [getattr(workloads, FP8_WORKLOADS[args.workload])()], None
        calls = [Fp8Call(la, prefills[0], dev, peaks_kind)]
    else:
        prefills, decode = make_workloads(args.workload, dev)
        calls = [PrefillCall(la, p, dev) for p in prefills] + ([DecodeCall(la, decode, dev)] if decode else [])
    head = calls[0]   # the headline: the largest prefill configuration (or the one workload asked for)
    flush = L2Flush(dev)

    barrier(world)
    with ClockSampler(local) as clocks:   # started before the warm-up
        ms, t_wall, window = time_calls(calls, args.steps, args.warmup, stream, flush)
    barrier(world)
    st = la.attn_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {la.attn_status_string(st)} after the timed region")

    # whole-job figures (max time over ranks, units summed over ranks)
    h_max, h_units = reduce_max_sum(world, sum(ms[0]), head.units * args.steps, dev)
    value = h_units / (h_max * 1e-3) * head.unit_scale
    rooflines = {call.name: call_roofline(call, ms[c], peaks, peaks_kind) for c, call in enumerate(calls)}
    line = {"metric": METRIC, "value": value, "unit": head.unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sum(sum(m) for m in ms) / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) rounded to bf16)"}
    line["roofline"] = kernel_roofline(calls, ms, peaks, peaks_kind)
    line["rooflines"] = rooflines
    line["headline"] = {"config": head.name, "kernel": head.kernel, "value": value, "unit": head.unit,
                        "frac_of_measured_peak": rooflines[head.name]["frac"]}
    dcall = None
    if decode is not None and head.kind != "decode":
        dcall = calls[-1]
        d_max, d_units = reduce_max_sum(world, sum(ms[-1]), dcall.units * args.steps, dev)
        dval = d_units / (d_max * 1e-3) * 1e-9
        line["decode"] = {"config": dcall.name, "value": dval, "unit": "GB/s",
                          "frac_of_measured_hbm": dval / world / peaks["hbm_gbs"],
                          "frac_of_8TBs": dval / world / NOMINAL["hbm_gbs"]}
    line["gpu_launches"] = args.steps * sum(c.launches for c in calls)
    line["config"] = {"workload": " + ".join(c.name for c in calls), "headline": head.name,
                      "l2": L2_NOTE + "; every input is also larger than L2",
                      "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                      "calls": {c.name: c.describe() for c in calls}}
    line["clocks"] = clocks.record(*window)
    line["wall_s_timed_region"] = t_wall

    # ---- end to end through the public API with pinned host buffers (the headline call)
    line["e2e"] = measure_e2e(head, stream, world, dev, steps=min(args.steps, 20))

    # ---- the CPU baseline leg (rank 0, one GPU): the oracle timed on the host
    # cores, and each configuration's GPU output checked on a seeded row sample
    if rank == 0 and world == 1 and args.cpu_baseline_seconds > 0:
        line["cpu_baseline"] = cpu_baseline(head, args.cpu_baseline_seconds)
        line["accuracy"] = {c.name: accuracy(c) for c in calls}

    # ---- the next rows, each timed on its own after the step
    if world == 1 and not args.no_next and args.workload == "hot_path":
        calls.clear()   # free the step's device buffers (the 13 GB decode pool among them)
        head = decode = prefills = dcall = None
        torch.cuda.empty_cache()
        line["next_rows"] = measure_next_rows(la, dev, stream, flush, min(args.steps, 20), args.warmup,
                                              peaks, peaks_kind)
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
    flush = L2Flush(dev)

    def step(ev=None):
        flush()
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
            "traffic": measured_traffic("attn_bwd", p.name + "_backward"), "peak_source": f"{peaks_kind} bf16 burst",
            "ms_per_call_median": statistics.median(ms), "ms_per_call_p95": sorted(ms)[int(0.95 * (len(ms) - 1))],
            "flops_per_call": flops, "flops_executed_per_call": 14.0 * p.d * attended_pairs(p),
            "launches_per_call": 3, "kernel": "attn_bwd"}
    line = {"metric": BWD_METRIC,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) rounded to bf16)",
            "value": value, "unit": "TFLOP/s", "roofline": roof, "ms_per_step": tot / args.steps,
            "gpu_launches": 3 * args.steps,
            "config": {"workload": p.name + "_backward", "l2": L2_NOTE,
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


def measure_e2e(call, stream, world, dev, steps):
    """The call's metric through the public API with the step's inputs in
    pinned host memory: H2D copies, the call, and a D2H read of the result,
    all inside the timed region (transfers of neighbouring steps overlap,
    see run_streamed)."""
    host_in, compute, out_shapes, note = call.e2e_parts()
    barrier(world)
    ms, host_out = run_streamed(host_in, lambda b, dev_in, dev_out: compute(dev_in, dev_out), out_shapes, steps,
                                stream, dev)
    t_max, tot_units = reduce_max_sum(world, ms, call.units * steps, dev)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    return {"value": tot_units / (t_max * 1e-3) * call.unit_scale, "unit": call.unit, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "config": call.name,
            "note": note + " (transfers overlap neighbouring steps)"}


class BwdCall:
    """attn_bwd on the backward of a prefill problem: q, k, v, the forward's
    out and lse, and a seeded dO resident on the device."""
    kind, kernel, unit, unit_scale, launches, bound = "backward", "attn_bwd", "TFLOP/s", 1e-12, 3, "tensor"

    def __init__(self, la, p, dev):
        self.la, self.p, self.name = la, p, p.name + "_backward"
        pg = p.to(dev)
        self.q = pg.q.view(p.B, p.Nq, p.Hq, p.d)
        self.k, self.v = pg.k.view(p.B, p.Nk, p.Hkv, p.d), pg.v.view(p.B, p.Nk, p.Hkv, p.d)
        self.out, self.lse = la.attn_fwd(self.q, self.k, self.v, causal=p.causal, scale=p.scale)
        self.g = workloads.randn_bf16(tuple(p.q.shape), seed=p.seed + 900).to(dev).view(self.q.shape)
        ws = torch.empty(la.lib().attn_bwd_workspace_size(p.B, p.Hq, p.Nq, 0), dtype=torch.uint8, device=dev)
        self.kw = dict(causal=p.causal, scale=p.scale, dq=torch.empty_like(self.q), dk=torch.empty_like(self.k),
                       dv=torch.empty_like(self.v), workspace=ws)
        self.units = backward_flops(p)

    def __call__(self):
        self.la.attn_bwd(self.q, self.k, self.v, self.out, self.lse, self.g, **self.kw)

    def describe(self):
        p = self.p
        return {"B": p.B, "Hq": p.Hq, "Hkv": p.Hkv, "Nq": p.Nq, "Nk": p.Nk, "d": p.d, "causal": p.causal}

    def roofline_extra(self):
        return {"flops_per_call": self.units, "flops_executed_per_call": 14.0 * self.p.d * attended_pairs(self.p),
                "launches_per_call": 3}


class Fp8Call(PrefillCall):
    """attn_fwd_fp8 on the per-tile E4M3 quantization of a prefill problem
    (quantized on the device by attn_quantize_fp8_qkv before timing).  Work is
    the same 4 d FLOP per attended pair; the S product runs at the 8-bit rate
    and the PV product at the 16-bit rate, so the peak for this kernel is
    4/3 of the bf16 peak (half the FLOPs at twice the rate)."""
    kernel, peak_scale = "attn_fwd_fp8", 4.0 / 3.0

    def __init__(self, la, p, dev, peaks_kind="measured"):
        super().__init__(la, p, dev)
        self.name = p.name + "_fp8"
        q, k, v = self.args
        kw = dict(cu_seqlens_q=self.kw["cu_seqlens_q"], cu_seqlens_k=self.kw["cu_seqlens_k"]) if p.varlen else {}
        (self.q8, self.qs), (self.k8, self.ks), (self.v8, self.vs) = la.attn_quantize_fp8_qkv(q, k, v, **kw)
        self.fkw = {x: y for x, y in self.kw.items() if x != "window"}
        self.peak_note = (f"{peaks_kind} bf16 burst x 4/3 (S at the 8-bit rate, nominally 2x bf16; "
                          "PV at the 16-bit rate)")

    def __call__(self):
        self.la.attn_fwd_fp8(self.q8, self.k8, self.v8, self.qs, self.ks, self.vs, out=self.out, lse=self.lse,
                             **self.fkw)

    def e2e_parts(self):
        src = [self.q8, self.k8, self.v8, self.qs, self.ks, self.vs]
        host_in = [t.cpu().pin_memory() for t in src]
        kw = dict(self.fkw)

        def compute(dev_in, dev_out):
            self.la.attn_fwd_fp8(*dev_in, out=dev_out[0], lse=dev_out[1], **kw)
        shapes = [(tuple(self.out.shape), self.out.dtype), (tuple(self.lse.shape), self.lse.dtype)]
        return host_in, compute, shapes, ("8-bit q, k, v codes and their scales copied from pinned host memory "
                                          "and out, lse copied back every step")


class QuantizeCall:
    """attn_quantize_fp8_qkv on q, k and v of a prefill problem (one launch):
    every bf16 element read once, every code written once, plus the scales."""
    kind, kernel, unit, unit_scale, launches, bound = "quantize", "attn_quantize_fp8", "GB/s", 1e-9, 1, "hbm"

    def __init__(self, la, p, dev):
        self.la, self.p, self.name = la, p, p.name + "_quantize_fp8"
        g = p.to(dev)
        self.xs = [g.q, g.k, g.v]
        self.cu = [g.cu_q, g.cu_k, g.cu_k]
        self.outs = []
        for x, cu in zip(self.xs, self.cu):
            T, H, d = x.shape
            B = p.B
            self.outs.append((torch.empty_like(x, dtype=torch.uint8),
                              torch.zeros((H, la.attn_fp8_scale_count(B, T)), dtype=torch.float32, device=dev)))
        self.units = float(sum(3 * x.numel() + 4 * o[1].numel() for x, o in zip(self.xs, self.outs)))

    def __call__(self):
        p = self.p
        outs = tuple(o8 for o8, _ in self.outs)
        scales = tuple(osc for _, osc in self.outs)
        if p.varlen:
            self.la.attn_quantize_fp8_qkv(*self.xs, cu_seqlens_q=self.cu[0], cu_seqlens_k=self.cu[1], out=outs,
                                          scales=scales)
        else:
            xs = [x.view(p.B, x.shape[0] // p.B, *x.shape[1:]) for x in self.xs]
            self.la.attn_quantize_fp8_qkv(*xs, out=tuple(o.view(x.shape) for o, x in zip(outs, xs)), scales=scales)

    def describe(self):
        return {"B": self.p.B, "tokens_q": int(self.xs[0].shape[0]), "tokens_k": int(self.xs[1].shape[0]),
                "Hq": self.p.Hq, "Hkv": self.p.Hkv, "d": self.p.d}

    def roofline_extra(self):
        return {"bytes_per_call": self.units, "launches_per_call": 1}


def measure_next_rows(la, dev, stream, flush, steps, warmup, peaks, peaks_kind):
    """Each next row (backward, local window, several queries with the
    append) timed on its own with CUDA events, after the step's buffers are
    freed; a row that fails reports its error instead of a number."""
    rows = {}
    for name in NEXT_ROWS:
        call = None
        try:
            if name in BWD_WORKLOADS:
                call = BwdCall(la, getattr(workloads, BWD_WORKLOADS[name])(), dev)
            elif name in FP8_WORKLOADS:
                call = Fp8Call(la, getattr(workloads, FP8_WORKLOADS[name])(), dev, peaks_kind)
            elif name.endswith("_quantize_fp8"):
                call = QuantizeCall(la, getattr(workloads, name[:-len("_quantize_fp8")])(), dev)
            elif name in PREFILL_WORKLOADS:
                call = PrefillCall(la, getattr(workloads, name)(), dev)
            else:
                call = DecodeCall(la, getattr(workloads, name)(device=dev), dev)
            ms, wall, _ = time_calls([call], steps, warmup, stream, flush)
            st = la.attn_get_device_status()
            if st != 0:
                raise RuntimeError(f"device status {la.attn_status_string(st)}")
            rec = call_roofline(call, ms[0], peaks, peaks_kind)
            rec.update(value=rec["achieved"], steps=steps, gpu_launches=steps * call.launches,
                       config=call.describe())
            rows[call.name] = rec
        except Exception as e:   # a next row never blocks the step's line
            rows[name] = {"error": f"{type(e).__name__}: {e}"}
        finally:
            call = None
            torch.cuda.empty_cache()
    return rows


def _gather_prefill(p, out, lse, rows):
    """GPU results at rows (b, h, i) of a prefill problem (host arrays)."""
    o = out.reshape(-1, p.Hq, p.d)
    if p.varlen:
        tok = p.cu_q.cpu().numpy().astype(np.int64)[rows[:, 0]] + rows[:, 2]
        li = rows[:, 1].astype(np.int64) * o.shape[0] + tok
    else:
        tok = rows[:, 0].astype(np.int64) * p.Nq + rows[:, 2]
        li = (rows[:, 0].astype(np.int64) * p.Hq + rows[:, 1]) * p.Nq + rows[:, 2]
    go = o[torch.as_tensor(tok).to(out.device), torch.as_tensor(rows[:, 1].astype(np.int64)).to(out.device)]
    gl = lse.reshape(-1)[torch.as_tensor(li).to(lse.device)]
    return go.float().cpu().numpy().astype(np.float64), gl.float().cpu().numpy().astype(np.float64)


TOL = {"o_max_abs": 1e-2, "o_rel_rms": 5e-3, "lse_abs": 1e-3}


def _compare(got_o, got_lse, ref_o, ref_lse):
    err = np.abs(got_o - ref_o)
    denom = float(np.sqrt((ref_o ** 2).sum()))
    fin = np.isfinite(ref_lse)
    rec = {"o_max_abs": float(err.max(initial=0.0)),
           "o_rel_rms": float(np.sqrt((err ** 2).sum()) / denom) if denom > 0 else float(np.sqrt((err ** 2).sum())),
           "lse_abs": float(np.abs(got_lse[fin] - ref_lse[fin]).max(initial=0.0)),
           "finite": bool(np.isfinite(got_o).all() and (np.isfinite(got_lse) == fin).all())}
    rec["within_tolerance"] = rec["finite"] and all(rec[k] <= v for k, v in TOL.items())
    rec["tolerance"] = TOL
    return rec


def accuracy(call):
    """The call's GPU output from the timed run against the fp64 oracle:
    prefill on a seeded row sample per (sequence, head) that always holds the
    first, last and tile-boundary rows; decode on every (sequence, head) row."""
    import oracle
    t0 = time.perf_counter()
    try:
        if call.kind == "prefill":
            p = call.p
            per = 16 if p.varlen else 64
            rows = workloads.sample_rows(None, [nq for nq, _ in p.seq_lens()], p.Hq, per,
                                         seed=p.seed + 700).numpy()
            if isinstance(call, Fp8Call):   # against the values the oracle's own 8-bit codes stand for
                ref_o, ref_lse = oracle.prefill_fp8(p, rows)
            else:
                ref_o, ref_lse = oracle.prefill(p, rows)
            got_o, got_lse = _gather_prefill(p, call.out, call.lse, rows)
            what = f"{len(rows)} seeded rows ({per} per sequence and head)"
        elif is_kvcache(call.d):
            host = appended_host_copy(call.d)
            rows = np.asarray([(b, h, i) for b in range(host.B) for h in range(host.Hq) for i in range(host.Nq)],
                              dtype=np.int32)
            ref_o, ref_lse = oracle.decode_multi_rows(host.q, host.k_cache, host.v_cache, host.block_table,
                                                      host.seq_lens, scale=host.scale, causal=host.causal, rows=rows)
            got_o = call.out.float().cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]].astype(np.float64)
            got_lse = call.lse.cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
            what = f"all {len(rows)} (sequence, head, query) rows"
        else:
            host = call.d.to("cpu")
            ref_o, ref_lse = oracle.decode(host)
            got_o = call.out.float().cpu().numpy().reshape(-1, host.d).astype(np.float64)
            got_lse = call.lse.cpu().numpy().reshape(-1).astype(np.float64)
            what = f"all {len(ref_lse)} (sequence, head) rows"
        rec = _compare(got_o, got_lse, ref_o, ref_lse)
        rec["sample"] = what
        rec["seconds"] = time.perf_counter() - t0
        return rec
    except Exception as e:   # the accuracy record never blocks the GPU line
        return {"error": f"{type(e).__name__}: {e}"}


def cpu_baseline(call, seconds):
    """The oracle as it stands, timed on the host cores on a bounded sample of
    the headline configuration."""
    try:
        if call.kind == "prefill":
            rate, n, dt, threads, fl = oracle_sample_rate(call.p, seconds, seed=4242)
            return {"value": rate * 1e-12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                    "sample": f"{n} seeded query rows of {call.name} ({fl / 1e9:.1f} GFLOP fp64) in {dt:.1f} s"}
        if is_kvcache(call.d):
            host = appended_host_copy(call.d)
            rate, n, dt, threads = oracle_kvcache_rate(host, seconds, seed=4242)
            return {"value": rate * 1e-9, "unit": "GB/s", "cores": threads, "kind": "oracle",
                    "sample": f"{n} seeded (sequence, head, query) rows of {call.name} in {dt:.1f} s"}
        host = call.d.to("cpu")
        rate, n, dt, threads = oracle_decode_rate(host, seconds, seed=4242)
        return {"value": rate * 1e-9, "unit": "GB/s", "cores": threads, "kind": "oracle",
                "sample": f"{n} seeded (sequence, head) rows of {call.name} in {dt:.1f} s"}
    except Exception as e:  # the baseline never blocks the GPU line
        return {"value": None, "unit": None, "cores": None, "kind": "oracle", "sample": f"failed: {e}"}


if __name__ == "__main__":
    sys.exit(main())
