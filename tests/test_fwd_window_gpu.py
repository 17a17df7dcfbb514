"""GPU parity of the local-window prefill (attn_fwd_window) against the fp64
oracle, through the C ABI.  The band: query row i keeps keys
[i + Nk - Nq - left, i + Nk - Nq + right] inside [0, Nk), a side of -1 being
unbounded, intersected with the causal corner when causal ("Deep Dive -
FlashAttention", section "Causal 2.1 is the decode gotcha", paragraph on local
attention)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_close, gather_prefill, one_hot_check, run_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    import exact_io_aware_04_gb300 as m
    m.build()
    torch.cuda.set_device(0)
    yield m
    assert m.attn_get_device_status() == 0


def check_all_rows(la, p):
    out, lse = run_prefill(la, p)
    torch.cuda.synchronize()
    rows = oracle.all_rows(p)
    ref_o, ref_lse = oracle.prefill(p, rows)
    go, gl = gather_prefill(p, out, lse, rows)
    return assert_close(p.name, go, gl, ref_o, ref_lse)


# (B, Hq, Hkv, Nq, Nk, d, causal, (left, right))
WINDOWS = [
    (2, 4, 2, 700, 700, 128, True, (200, -1)),      # causal sliding window, ragged tail
    (1, 4, 4, 600, 600, 128, False, (100, 100)),    # symmetric band
    (1, 2, 2, 300, 1000, 128, True, (127, 0)),      # Nq < Nk, a window of exactly one tile
    (1, 2, 2, 1000, 300, 64, False, (50, 10)),      # Nq > Nk: leading rows see no key
    (1, 2, 1, 517, 517, 64, True, (0, 0)),          # the diagonal key only
    (2, 8, 2, 384, 900, 128, False, (-1, 64)),      # right side only
    (1, 2, 2, 256, 256, 128, False, (1000, 1000)),  # wider than the keys
    (1, 4, 1, 1024, 1024, 128, True, (128, -1)),    # left = a tile, MQA
    (1, 2, 2, 2000, 2000, 64, True, (257, 0)),
    (1, 2, 2, 129, 4000, 128, False, (0, 3000)),    # band starts at the corner and runs right
]


def _id(c):
    return "B{}_Hq{}_Hkv{}_Nq{}_Nk{}_d{}_{}_w{}_{}".format(*c[:6], "c" if c[6] else "n", *c[7])


@pytest.mark.parametrize("cfg", WINDOWS, ids=_id)
def test_window_small_problems_all_rows(la, cfg):
    B, Hq, Hkv, Nq, Nk, d, causal, window = cfg
    p = workloads.make_prefill(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=hash(cfg) % 10_000, window=window)
    check_all_rows(la, p)


VARLEN = [
    ([5, 300, 0, 129, 1000, 1], [5, 300, 17, 700, 1000, 1], 128, True, (100, -1)),
    ([256, 3, 600], [100, 3, 2000], 128, False, (64, 32)),
    ([77, 512, 512], [1024, 1500, 512], 64, True, (300, 0)),
]


@pytest.mark.parametrize("cfg", VARLEN, ids=lambda c: f"varlen_{len(c[0])}seq_d{c[2]}_w{c[4][0]}_{c[4][1]}")
def test_window_varlen_all_rows(la, cfg):
    ql, kl, d, causal, window = cfg
    p = workloads.make_varlen(ql, kl, 4, 2, d, causal=causal, seed=sum(ql) + 7, window=window)
    check_all_rows(la, p)


def test_window_one_hot_attended_keys(la):
    """Which keys each row attends, bit for bit, with both band edges inside
    tiles and across tile boundaries."""
    p = workloads.make_prefill(1, 4, 2, 300, 600, 64, causal=False, seed=41, window=(70, 45))
    one_hot_check(la, p, [0, 64, 128, 200, 300, 400, 536])
    p = workloads.make_varlen([300, 129], [500, 129], 4, 2, 64, causal=True, seed=42, window=(150, -1))
    one_hot_check(la, p, [0, 64, 128, 190, 256, 380, 436])


def _bits(la, p):
    out, lse = run_prefill(la, p)
    torch.cuda.synchronize()
    return out.clone(), lse.clone()


def test_window_reductions_are_bit_identical(la):
    """Windows that allow the same keys give the same bits: (-1, -1) is
    attn_fwd, a window wider than every sequence is no window, and with causal
    the right side does not matter."""
    for causal in (False, True):
        base = workloads.make_prefill(2, 4, 2, 500, 700, 128, causal=causal, seed=51)
        o0, l0 = _bits(la, base)
        for w in [(-1, -1), (5000, 5000), (700, -1), (-1, 700)]:
            o1, l1 = _bits(la, dataclasses.replace(base, window=w))
            if w == (-1, -1):   # run_prefill takes attn_fwd for it: call the window entry explicitly
                g = base.to("cuda")
                o1, l1 = la.attn_fwd(g.q.view(2, 500, 4, 128), g.k.view(2, 700, 2, 128), g.v.view(2, 700, 2, 128),
                                     causal=causal, scale=base.scale, window=(-1, -1))
                torch.cuda.synchronize()
            assert torch.equal(o0.view(-1), o1.reshape(-1)) and torch.equal(l0, l1), (causal, w)
    c0 = workloads.make_prefill(1, 2, 2, 400, 400, 64, causal=True, seed=52, window=(90, 0))
    o0, l0 = _bits(la, c0)
    o1, l1 = _bits(la, dataclasses.replace(c0, window=(90, 37)))
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_window_empty_rows(la):
    """A band that misses every key of some rows: those rows give O = 0 and
    lse = -inf, the others match the oracle."""
    p = workloads.make_prefill(1, 2, 2, 600, 200, 128, causal=True, seed=53, window=(30, -1))
    stats = check_all_rows(la, p)
    out, lse = run_prefill(la, p)
    torch.cuda.synchronize()
    assert torch.isneginf(lse[0, :, :400]).all()
    assert (out.view(600, 2, 128)[:400] == 0).all()


def test_window_full_size_sampled_rows(la):
    p = workloads.swa_causal()
    out, lse = run_prefill(la, p)
    torch.cuda.synchronize()
    lens = [nq for nq, _ in p.seq_lens()]
    rows = workloads.sample_rows(None, lens, p.Hq, 512, seed=p.seed + 500)
    ref_o, ref_lse = oracle.prefill(p, rows.numpy())
    go, gl = gather_prefill(p, out, lse, rows.numpy())
    stats = assert_close(p.name, go, gl, ref_o, ref_lse)
    print(p.name, stats)


def test_tensors_past_4gib(la):
    """q and out hold 2^31 elements (4 GiB) each, so the last rows sit past
    every 32-bit element and byte offset.  A causal band of 128 keys keeps
    the work small.  The rows checked sit at both ends of the tensors:
    first rows that a wrapped offset would overwrite, and last rows that
    only 64-bit arithmetic reaches."""
    B, Hq, Hkv, N, d = 1, 64, 8, 262144, 128
    p = workloads.make_prefill(B, Hq, Hkv, N, N, d, causal=True, seed=1237, window=(127, 0))
    assert p.q.numel() == 1 << 31
    out, lse = run_prefill(la, p)
    torch.cuda.synchronize()
    toks = [0, 1, 127, 128, 131071, 200003, N - 129, N - 128, N - 2, N - 1]
    rows = np.array([(0, h, t) for h in (0, 37, Hq - 1) for t in toks], dtype=np.int32)
    ref_o, ref_lse = oracle.prefill(p, rows)
    go, gl = gather_prefill(p, out, lse, rows)
    assert_close("past 4 GiB", go, gl, ref_o, ref_lse)
