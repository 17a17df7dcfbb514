"""CPU fp64 oracle for exact scaled dot-product attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path (the CUDA
library in ``exact_io_aware_04_gb300``) never imports this package, and this
package imports nothing from it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, one row at a time, the
definition written out); this module only compiles it and marshals arrays.

Parity status of each function (what pins it, see ``tests/test_oracle.py``):
  prefill_rows -- pinned: the two-tile worked example and the normaliser
                  example (printed values), keep matrices for both causal
                  corners, the GQA head map, torch SDPA fp64 MATH backend with
                  an explicit bottom-right keep mask, shift invariance, the
                  log-sum-exp merge identity, rows summing to one; the local
                  window through its special cases (unbounded = full, right 0
                  = causal corner, (0, 0) = the single diagonal key, a window
                  covering every key = full, left-only window with causal =
                  causal minus the far keys).
  decode_rows  -- pinned: equals prefill_rows on the keys gathered through the
                  block table as the paged-gather example describes, and the
                  example's gathered shape.
  decode_multi_rows -- pinned: Nq = 1 equals decode_rows; the printed
                  bottom-right keep matrices read through a paged cache; equals
                  prefill_rows (bottom-right causal, Nq queries) on the
                  gathered keys.
  append_kv    -- pinned: brute-force gather of the written positions through
                  the block table; untouched slots keep their bytes.
  e4m3_value, e4m3_from_float -- pinned: torch's float8_e4m3fn casts (a
                  library routine) on every code and on every finite bf16
                  value below the saturation point; saturation at 448.
  quantize_fp8 -- pinned: every tile's largest magnitude lands on the code
                  448; the round trip is within half a step of the E4M3 grid
                  at each value's own scale; tiles start at sequence starts
                  and at multiples of 128 tokens inside a sequence (an
                  outlier moves the codes of its own tile only); all-zero
                  tiles give zero codes.
  prefill_rows_f64 -- pinned: bit-identical to prefill_rows on inputs
                  that bf16 holds exactly (the same code path).
  backward     -- pinned: torch autograd through SDPA's fp64 MATH backend with
                  an explicit keep mask; central finite differences of
                  <G, O> on inputs whose perturbations are exact in bf16;
                  sum_j dV_j = sum_i G_i over nonempty rows; sum_j dK_j = 0
                  without a mask; empty rows pass no gradient.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_long
            D = ctypes.c_double
            lib.oracle_prefill_rows.argtypes = [P, P, P, I, I, I, I, I, I, D, I, P, P, P, L, P, P, I]
            lib.oracle_prefill_rows.restype = I
            lib.oracle_prefill_rows_window.argtypes = [P, P, P, I, I, I, I, I, I, D, I, I, I, P, P, P, L, P, P, I]
            lib.oracle_prefill_rows_window.restype = I
            lib.oracle_decode_rows.argtypes = [P, P, P, P, I, P, I, I, I, I, I, D, P, L, P, P, I]
            lib.oracle_decode_rows.restype = I
            lib.oracle_decode_multi_rows.argtypes = [P, P, P, P, I, P, I, I, I, I, I, I, D, I, P, L, P, P, I]
            lib.oracle_decode_multi_rows.restype = I
            lib.oracle_backward.argtypes = [P, P, P, P, I, I, I, I, I, I, D, I, I, I, P, P, P, L, L, P, P, P, I]
            lib.oracle_backward.restype = I
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = I
            lib.oracle_prefill_rows_f64.argtypes = [P, P, P, I, I, I, I, I, I, D, I, I, I, P, P, P, L, P, P, I]
            lib.oracle_prefill_rows_f64.restype = I
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = D
            lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
            lib.oracle_quantize_fp8.argtypes = [P, I, I, I, I, P, P, P, L]
            lib.oracle_quantize_fp8.restype = I
            lib.oracle_dequantize_fp8.argtypes = [P, P, L, I, I, I, I, P, P]
            lib.oracle_dequantize_fp8.restype = I
            _lib = lib
    return _lib


def num_threads() -> int:
    """CPUs this process may run on (sched_getaffinity)."""
    return int(_load().oracle_num_threads())


def _bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype != torch.bfloat16:
        raise TypeError("oracle inputs are bf16 tensors")
    return np.ascontiguousarray(t.detach().to("cpu").contiguous().view(torch.int16).numpy())


def _i32(t) -> np.ndarray:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.int32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def prefill_rows(q, k, v, *, B, Hq, Hkv, Nq, Nk, scale, causal, rows,
                 cu_q=None, cu_k=None, window=(-1, -1), threads: int = 0):
    """Rows (b, h, i) of softmax(QK^T*scale + mask) V and their lse, fp64.

    q [T_q, Hq, d], k/v [T_k, Hkv, d] bf16; rows int [n, 3]; window =
    (left, right) local window, -1 = unbounded on that side.
    Returns (out [n, d] float64, lse [n] float64)."""
    d = int(q.shape[-1])
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    r = _i32(rows).reshape(-1, 3)
    n = r.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    cq, ck = _i32(cu_q), _i32(cu_k)
    left, right = (int(x) for x in window)
    rc = _load().oracle_prefill_rows_window(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Nq, Nk, d,
                                            float(scale), int(bool(causal)), left, right, _ptr(cq), _ptr(ck),
                                            _ptr(r), n, _ptr(out), _ptr(lse),
                                            threads if threads > 0 else num_threads())
    if rc != 0:
        raise ValueError(f"oracle_prefill_rows rejected its arguments (status {rc})")
    return out, lse


def decode_rows(q, k_cache, v_cache, block_table, seq_lens, *, scale, rows, threads: int = 0):
    """Rows (b, h) of paged single-query attention, fp64.

    q [B, Hq, d]; caches [num_pages, page, Hkv, d]; block_table int [B, max_pages];
    seq_lens int [B]; rows int [n, 2].  Returns (out [n, d], lse [n])."""
    B, Hq, d = (int(x) for x in q.shape)
    page, Hkv = int(k_cache.shape[1]), int(k_cache.shape[2])
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    r = _i32(rows).reshape(-1, 2)
    n = r.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = _load().oracle_decode_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(bt), int(bt.shape[1]),
                                    _ptr(sl), B, Hq, Hkv, d, page, float(scale), _ptr(r), n,
                                    _ptr(out), _ptr(lse), threads if threads > 0 else num_threads())
    if rc != 0:
        raise ValueError(f"oracle_decode_rows rejected its arguments (status {rc})")
    return out, lse


def all_rows(p) -> np.ndarray:
    """Every (b, h, i) row of a prefill problem (small problems only)."""
    out = []
    for b, (nq, _) in enumerate(p.seq_lens()):
        for h in range(p.Hq):
            for i in range(nq):
                out.append((b, h, i))
    return np.asarray(out, dtype=np.int32).reshape(-1, 3)


def prefill(p, rows=None, threads: int = 0):
    """prefill_rows over a workloads.Prefill problem (all rows by default)."""
    if rows is None:
        rows = all_rows(p)
    return prefill_rows(p.q, p.k, p.v, B=p.B, Hq=p.Hq, Hkv=p.Hkv, Nq=p.Nq, Nk=p.Nk,
                        scale=p.scale, causal=p.causal, rows=rows, cu_q=p.cu_q, cu_k=p.cu_k,
                        window=getattr(p, "window", (-1, -1)), threads=threads)


def decode(p, rows=None, threads: int = 0):
    """decode_rows over a workloads.Decode problem (all (b, h) by default)."""
    if rows is None:
        rows = np.asarray([(b, h) for b in range(p.B) for h in range(p.Hq)], dtype=np.int32)
    return decode_rows(p.q, p.k_cache, p.v_cache, p.block_table, p.seq_lens, scale=p.scale,
                       rows=rows, threads=threads)


def decode_multi_rows(q, k_cache, v_cache, block_table, seq_lens, *, scale, causal, rows, threads: int = 0):
    """Rows (b, h, i) of Nq-query paged attention, fp64.

    q [B, Nq, Hq, d] (query i of sequence b is position seq_lens[b] - Nq + i);
    caches [num_pages, page, Hkv, d]; rows int [n, 3].  Returns (out [n, d], lse [n])."""
    B, Nq, Hq, d = (int(x) for x in q.shape)
    page, Hkv = int(k_cache.shape[1]), int(k_cache.shape[2])
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    r = _i32(rows).reshape(-1, 3)
    n = r.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = _load().oracle_decode_multi_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(bt), int(bt.shape[1]),
                                          _ptr(sl), B, Nq, Hq, Hkv, d, page, float(scale), int(bool(causal)),
                                          _ptr(r), n, _ptr(out), _ptr(lse),
                                          threads if threads > 0 else num_threads())
    if rc != 0:
        raise ValueError(f"oracle_decode_multi_rows rejected its arguments (status {rc})")
    return out, lse


def append_kv(k_cache, v_cache, block_table, seq_lens, k_new, v_new, inplace=False):
    """The in-place cache update (on copies unless inplace): new row i of
    sequence b goes to position seq_lens[b] - Nq + i, i.e. page
    block_table[b][pos // page] at slot pos % page.  Positions below zero, and
    page ids outside the pool, are skipped.  k_new/v_new [B, Nq, Hkv, d].
    Returns (k_cache', v_cache')."""
    kc, vc = (k_cache, v_cache) if inplace else (k_cache.clone(), v_cache.clone())
    B, Nq = int(k_new.shape[0]), int(k_new.shape[1])
    page, pool = int(kc.shape[1]), int(kc.shape[0])
    bt = block_table.cpu()
    lens = [int(x) for x in seq_lens.cpu().tolist()]
    for b in range(B):
        for i in range(Nq):
            pos = lens[b] - Nq + i
            if pos < 0 or pos // page >= bt.shape[1]:
                continue
            pg = int(bt[b, pos // page])
            if 0 <= pg < pool:
                kc[pg, pos % page] = k_new[b, i]
                vc[pg, pos % page] = v_new[b, i]
    return kc, vc


def decode_kvcache(p, rows=None, threads: int = 0):
    """decode_multi_rows over a workloads.KVCacheDecode problem, on the cache
    after its append (all (b, h, i) rows by default)."""
    kc, vc = p.k_cache, p.v_cache
    if p.k_new is not None:
        kc, vc = append_kv(kc, vc, p.block_table, p.seq_lens, p.k_new, p.v_new)
    if rows is None:
        rows = np.asarray([(b, h, i) for b in range(p.B) for h in range(p.Hq) for i in range(p.Nq)],
                          dtype=np.int32)
    return decode_multi_rows(p.q, kc, vc, p.block_table, p.seq_lens, scale=p.scale, causal=p.causal,
                             rows=rows, threads=threads)


def backward(p, g, pairs=None, threads: int = 0, row_stride: int = 1):
    """dQ, dK, dV (fp64 numpy, shaped like q, k, v) of L = <g, O> for a
    workloads.Prefill problem; g is bf16 like q.  pairs: (b, kv head) pairs
    to compute (default: all); rows outside them are zero.  row_stride > 1
    processes every row_stride-th query row only (a timing sample)."""
    qb, kb, vb, gb = _bits(p.q), _bits(p.k), _bits(p.v), _bits(g)
    if pairs is None:
        pairs = [(b, h) for b in range(p.B) for h in range(p.Hkv)]
    pr = _i32(pairs).reshape(-1, 2)
    dq = np.zeros(tuple(p.q.shape), dtype=np.float64)
    dk = np.zeros(tuple(p.k.shape), dtype=np.float64)
    dv = np.zeros(tuple(p.v.shape), dtype=np.float64)
    left, right = (int(x) for x in getattr(p, "window", (-1, -1)))
    rc = _load().oracle_backward(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), p.B, p.Hq, p.Hkv, p.Nq, p.Nk,
                                 int(p.d), float(p.scale), int(bool(p.causal)), left, right,
                                 _ptr(_i32(p.cu_q)), _ptr(_i32(p.cu_k)), _ptr(pr), pr.shape[0], int(row_stride),
                                 _ptr(dq), _ptr(dk), _ptr(dv), threads if threads > 0 else num_threads())
    if rc != 0:
        raise ValueError(f"oracle_backward rejected its arguments (status {rc})")
    return dq, dk, dv



# ---------------------------------------------------------------------------
# 8-bit (E4M3) per-tile quantization and attention on the values it stands for
# ---------------------------------------------------------------------------
def fp8_scale_count(B: int, T: int) -> int:
    """Scale entries per head for T tokens in B sequences (tiles of 128 tokens
    counted from each sequence's first token; tile t of sequence b is entry
    T_b // 128 + b + t, T_b the sequence's first token)."""
    return T // 128 + B


def e4m3_value(code: int) -> float:
    return float(_load().oracle_e4m3_value(int(code)))


def e4m3_from_float(x: float) -> int:
    return int(_load().oracle_e4m3_from_float(float(x)))


def _seq_args(T, B, N, cu):
    if cu is None:
        if N is None or B * N != T:
            raise ValueError("dense layout needs B * N == T")
        return int(N), None
    c = _i32(cu)
    if c.shape[0] != B + 1 or int(c[-1]) != T:
        raise ValueError("cu must have B + 1 entries ending at T")
    return 0, c


def quantize_fp8(x, *, B, N=None, cu=None):
    """Per-tile E4M3 quantization of x [T, H, d] bf16 (see oracle.c).
    Returns (codes uint8 [T, H, d], scales float32 [H, fp8_scale_count(B, T)]);
    scale entries between sequences are 0."""
    T, H, d = (int(v) for v in x.shape)
    n, c = _seq_args(T, B, N, cu)
    xb = _bits(x)
    codes = np.zeros((T, H, d), dtype=np.uint8)
    ns = fp8_scale_count(B, T)
    scales = np.zeros((H, ns), dtype=np.float32)
    rc = _load().oracle_quantize_fp8(_ptr(xb), B, H, n, d, _ptr(c), _ptr(codes), _ptr(scales), ns)
    if rc != 0:
        raise ValueError(f"oracle_quantize_fp8 rejected its arguments (status {rc})")
    return codes, scales


def dequantize_fp8(codes, scales, *, B, N=None, cu=None):
    """The fp64 values E4M3 codes [T, H, d] with their per-tile scales stand for."""
    codes = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    scales = np.ascontiguousarray(np.asarray(scales, dtype=np.float32))
    T, H, d = codes.shape
    n, c = _seq_args(T, B, N, cu)
    out = np.zeros((T, H, d), dtype=np.float64)
    rc = _load().oracle_dequantize_fp8(_ptr(codes), _ptr(scales), int(scales.shape[1]), B, H, n, d, _ptr(c),
                                       _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_dequantize_fp8 rejected its arguments (status {rc})")
    return out


def prefill_rows_f64(q, k, v, *, B, Hq, Hkv, Nq, Nk, scale, causal, rows, cu_q=None, cu_k=None,
                     window=(-1, -1), threads: int = 0):
    """prefill_rows on fp64 inputs q [T_q, Hq, d], k/v [T_k, Hkv, d]."""
    f = lambda a: np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    qd, kd, vd = f(q), f(k), f(v)
    d = int(qd.shape[-1])
    r = _i32(rows).reshape(-1, 3)
    n = r.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    cq, ck = _i32(cu_q), _i32(cu_k)
    left, right = (int(x) for x in window)
    rc = _load().oracle_prefill_rows_f64(_ptr(qd), _ptr(kd), _ptr(vd), B, Hq, Hkv, Nq, Nk, d, float(scale),
                                         int(bool(causal)), left, right, _ptr(cq), _ptr(ck), _ptr(r), n,
                                         _ptr(out), _ptr(lse), threads if threads > 0 else num_threads())
    if rc != 0:
        raise ValueError(f"oracle_prefill_rows_f64 rejected its arguments (status {rc})")
    return out, lse


def quantize_problem_fp8(p):
    """Per-tile E4M3 codes and scales of a workloads.Prefill problem's q, k, v:
    {"q": (codes, scales), "k": ..., "v": ...}."""
    tq = sum(nq for nq, _ in p.seq_lens())
    tk = sum(nk for _, nk in p.seq_lens())
    if p.varlen:
        return {"q": quantize_fp8(p.q, B=p.B, cu=p.cu_q), "k": quantize_fp8(p.k, B=p.B, cu=p.cu_k),
                "v": quantize_fp8(p.v, B=p.B, cu=p.cu_k)}
    return {"q": quantize_fp8(p.q, B=p.B, N=p.Nq), "k": quantize_fp8(p.k, B=p.B, N=p.Nk),
            "v": quantize_fp8(p.v, B=p.B, N=p.Nk)}


def prefill_fp8(p, rows=None, quantized=None, threads: int = 0):
    """Attention of a workloads.Prefill problem on the values its per-tile
    E4M3 quantization stands for: rows (b, h, i) of softmax(QK^T*scale +
    mask) V over the dequantized q, k, v, fp64.  Returns (out, lse)."""
    if quantized is None:
        quantized = quantize_problem_fp8(p)
    if rows is None:
        rows = all_rows(p)
    seq = dict(B=p.B, cu=p.cu_q) if p.varlen else dict(B=p.B, N=p.Nq)
    seqk = dict(B=p.B, cu=p.cu_k) if p.varlen else dict(B=p.B, N=p.Nk)
    q = dequantize_fp8(*quantized["q"], **seq)
    k = dequantize_fp8(*quantized["k"], **seqk)
    v = dequantize_fp8(*quantized["v"], **seqk)
    return prefill_rows_f64(q, k, v, B=p.B, Hq=p.Hq, Hkv=p.Hkv, Nq=p.Nq, Nk=p.Nk, scale=p.scale, causal=p.causal,
                            rows=rows, cu_q=p.cu_q, cu_k=p.cu_k, window=getattr(p, "window", (-1, -1)),
                            threads=threads)
