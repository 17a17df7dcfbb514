"""Comparison helpers for GPU-vs-oracle parity tests.

Tolerances (fixed by the project's accuracy contract, fp64 oracle on the
bf16-rounded inputs):
  O   : max |O - O*| <= 1e-2  and  ||O - O*||_2 / ||O*||_2 <= 5e-3
  lse : |lse - lse*| <= 1e-3   (both -inf on empty rows)
Which keys are attended is checked bit-exactly (one-hot tests).
"""
import numpy as np
import torch

import oracle
import workloads

O_MAX_ABS = 1e-2
O_REL_RMS = 5e-3
LSE_ABS = 1e-3


def assert_close(name, got_o, got_lse, ref_o, ref_lse):
    got_o = np.asarray(got_o, dtype=np.float64)
    got_lse = np.asarray(got_lse, dtype=np.float64)
    assert got_o.shape == ref_o.shape, (got_o.shape, ref_o.shape)
    assert np.isfinite(got_o).all(), f"{name}: non-finite output values"
    err = np.abs(got_o - ref_o)
    max_abs = float(err.max(initial=0.0))
    denom = float(np.sqrt((ref_o ** 2).sum()))
    rel = float(np.sqrt((err ** 2).sum()) / denom) if denom > 0 else float(np.sqrt((err ** 2).sum()))
    fin = np.isfinite(ref_lse)
    assert (np.isfinite(got_lse) == fin).all(), f"{name}: lse finite pattern differs"
    assert (got_lse[~fin] == -np.inf).all(), f"{name}: empty rows must have lse -inf"
    lse_err = float(np.abs(got_lse[fin] - ref_lse[fin]).max(initial=0.0))
    assert max_abs <= O_MAX_ABS, f"{name}: O max abs err {max_abs:.3e}"
    assert rel <= O_REL_RMS, f"{name}: O rel-RMS {rel:.3e}"
    assert lse_err <= LSE_ABS, f"{name}: lse err {lse_err:.3e}"
    return {"max_abs": max_abs, "rel_rms": rel, "lse_abs": lse_err}


def gather_prefill(p, out, lse, rows):
    """GPU results at oracle rows (b, h, i) of a workloads.Prefill problem."""
    rows = np.asarray(rows)
    o = out.reshape(-1, p.Hq, p.d)
    if p.varlen:
        cq = p.cu_q.cpu().numpy().astype(np.int64)
        tok = cq[rows[:, 0]] + rows[:, 2]
        li = torch.as_tensor(rows[:, 1] * o.shape[0] + tok)
        l = lse.reshape(-1)[li.to(lse.device)]
    else:
        tok = rows[:, 0].astype(np.int64) * p.Nq + rows[:, 2]
        li = torch.as_tensor((rows[:, 0].astype(np.int64) * p.Hq + rows[:, 1]) * p.Nq + rows[:, 2])
        l = lse.reshape(-1)[li.to(lse.device)]
    ti = torch.as_tensor(tok).to(out.device)
    hi = torch.as_tensor(rows[:, 1].astype(np.int64)).to(out.device)
    go = o[ti, hi].float().cpu().numpy()
    return go, l.float().cpu().numpy()


def run_prefill(la, p, device="cuda"):
    """attn_fwd on a workloads.Prefill problem; returns (out, lse) on device."""
    g = p.to(device)
    window = None if tuple(p.window) == (-1, -1) else tuple(p.window)
    if p.varlen:
        return la.attn_fwd(g.q, g.k, g.v, causal=p.causal, scale=p.scale, window=window,
                           cu_seqlens_q=g.cu_q, cu_seqlens_k=g.cu_k)
    q = g.q.view(p.B, p.Nq, p.Hq, p.d)
    k = g.k.view(p.B, p.Nk, p.Hkv, p.d)
    v = g.v.view(p.B, p.Nk, p.Hkv, p.d)
    return la.attn_fwd(q, k, v, causal=p.causal, scale=p.scale, window=window)


def run_decode(la, d, device="cuda", num_splits=0):
    g = d.to(device)
    return la.attn_decode_paged(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, scale=d.scale,
                                num_splits=num_splits)


def one_hot_check(la, p, bases):
    """Q = 0 and V one-hot over a window of d keys: the nonzero pattern of O
    must equal the oracle's allowed set exactly, the magnitude must name the
    K/V head, and exp(lse) must be the allowed-key count."""
    for base in bases:
        ph = workloads.one_hot_values(p, base)
        out, lse = run_prefill(la, ph)
        torch.cuda.synchronize()
        rows = oracle.all_rows(ph)
        ref_o, ref_lse = oracle.prefill(ph, rows)
        go, gl = gather_prefill(ph, out, lse, rows)
        assert np.array_equal(go != 0, ref_o != 0), f"base {base}: attended-key pattern differs"
        cnt = np.where(np.isfinite(ref_lse), np.rint(np.exp(ref_lse)), 0)
        g_of_h = (rows[:, 1] // (p.Hq // p.Hkv)) + 1
        nz = go != 0
        assert np.array_equal(np.rint((go * cnt[:, None])[nz]), np.broadcast_to(g_of_h[:, None], go.shape)[nz]), \
            f"base {base}: K/V head map differs"
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(gl), fin)
        assert np.array_equal(np.rint(np.exp(gl[fin])), cnt[fin]), f"base {base}: allowed-key count differs"
