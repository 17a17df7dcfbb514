"""GPU parity of attn_bwd (gradients by recomputation) against the fp64
oracle's gradients of the same bf16 inputs, through the C ABI.  The forward
output and lse come from attn_fwd; dO is seeded.

Tolerance (the accuracy contract states none for gradients): the kernels
round P, dS and the three outputs to bf16 (relative 2^-9 each) and build D
from the bf16 forward output, so every gradient element carries a few bf16
roundings of terms of its own size.  A single bf16 rounding of uniformly
distributed relative position has an RMS of 2^-9/sqrt(3) = 1.1e-3; the
measured relative RMS is 2.2-2.6e-3 on every case (two to three such
roundings), bounded here at 5e-3 per tensor.  max |err| <= 1e-2 * max |ref|
(measured at most 0.52%: a single worst element may sit on several rounding
errors of the same sign), plus an absolute floor of 1e-4 for the
fp32 residue of exact cancellations (a row with a single key has dS = 0 in
exact arithmetic; dP and D = G.O are then two fp32 dot products of d terms
that agree to ~1e-6)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import run_prefill

pytestmark = pytest.mark.gpu

REL_RMS = 5e-3
MAX_REL = 1e-2
ABS_FLOOR = 1e-4


@pytest.fixture(scope="module")
def la():
    import exact_io_aware_04_gb300 as m
    m.build()
    torch.cuda.set_device(0)
    yield m
    assert m.attn_get_device_status() == 0


def run_bwd(la, p, g):
    """attn_fwd then attn_bwd on device copies; returns (dq, dk, dv) as host fp64 arrays shaped like q, k, v."""
    gp = p.to("cuda")
    out, lse = run_prefill(la, p)
    window = None if tuple(p.window) == (-1, -1) else tuple(p.window)
    gd = g.to("cuda")
    if p.varlen:
        dq, dk, dv = la.attn_bwd(gp.q, gp.k, gp.v, out, lse, gd, causal=p.causal, scale=p.scale, window=window,
                                 cu_seqlens_q=gp.cu_q, cu_seqlens_k=gp.cu_k)
    else:
        q4 = gp.q.view(p.B, p.Nq, p.Hq, p.d)
        k4 = gp.k.view(p.B, p.Nk, p.Hkv, p.d)
        v4 = gp.v.view(p.B, p.Nk, p.Hkv, p.d)
        dq, dk, dv = la.attn_bwd(q4, k4, v4, out, lse, gd.view(p.B, p.Nq, p.Hq, p.d), causal=p.causal,
                                 scale=p.scale, window=window)
    torch.cuda.synchronize()
    f = lambda t, like: t.float().cpu().double().numpy().reshape(like.shape)
    return f(dq, p.q), f(dk, p.k), f(dv, p.v)


def grad_stats(name, got, ref, mask=None):
    if mask is not None:
        got, ref = got[mask], ref[mask]
    assert np.isfinite(got).all(), f"{name}: non-finite gradient"
    err = np.abs(got - ref)
    denom = float(np.sqrt((ref ** 2).sum()))
    rel = float(np.sqrt((err ** 2).sum()) / denom) if denom > ABS_FLOOR else 0.0
    mx = float(err.max(initial=0.0))
    scale = float(np.abs(ref).max(initial=0.0))
    return rel, mx, scale


def check(la, p, g=None, pairs=None):
    if g is None:
        g = workloads.randn_bf16(tuple(p.q.shape), seed=p.seed + 900)
    dq, dk, dv = run_bwd(la, p, g)
    rq, rk, rv = oracle.backward(p, g, pairs=pairs)
    out = {}
    masks = (None, None, None)
    if pairs is not None:   # compare only the rows of the computed (b, kv head) pairs
        masks = sampled_masks(p, pairs)
    for name, got, ref, m in (("dq", dq, rq, masks[0]), ("dk", dk, rk, masks[1]), ("dv", dv, rv, masks[2])):
        rel, mx, sc = grad_stats(name, got, ref, m)
        out[name] = (rel, mx, sc)
        assert rel <= REL_RMS, f"{p.name} {name}: relative RMS error {rel:.3e}"
        assert mx <= MAX_REL * sc + ABS_FLOOR, f"{p.name} {name}: max abs error {mx:.3e} (max |ref| {sc:.3e})"
    print(p.name, {k: f"rel {v[0]:.2e} max {v[1]:.2e} / {v[2]:.2e}" for k, v in out.items()})
    return dq, dk, dv


def sampled_masks(p, pairs):
    group = p.Hq // p.Hkv
    mq = np.zeros(tuple(p.q.shape), dtype=bool)
    mk = np.zeros(tuple(p.k.shape), dtype=bool)
    lens = p.seq_lens()
    cq = np.cumsum([0] + [a for a, _ in lens])
    ck = np.cumsum([0] + [b for _, b in lens])
    for b, g in pairs:
        mq[cq[b]:cq[b + 1], g * group:(g + 1) * group] = True
        mk[ck[b]:ck[b + 1], g] = True
    return mq, mk, mk


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_all_rows(la, causal):
    check(la, workloads.tiny(causal))


# (B, Hq, Hkv, Nq, Nk, d, causal)
SMALL = [
    (2, 4, 4, 300, 300, 128, True),
    (2, 4, 4, 300, 300, 128, False),
    (1, 2, 2, 200, 517, 128, True),     # Nq < Nk
    (1, 2, 2, 517, 200, 128, True),     # Nq > Nk: leading rows have no key
    (1, 2, 2, 517, 200, 64, False),
    (2, 8, 2, 384, 384, 64, True),      # GQA 4:1, exact tile multiple
    (1, 6, 1, 129, 1000, 128, True),    # MQA, one row past a tile
    (3, 2, 1, 1, 700, 128, True),       # single query row
    (1, 4, 2, 640, 640, 64, False),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: "B{}_Hq{}_Hkv{}_Nq{}_Nk{}_d{}_{}".format(*c[:6], "c" if c[6] else "n"))
def test_small_problems(la, cfg):
    B, Hq, Hkv, Nq, Nk, d, causal = cfg
    check(la, workloads.make_prefill(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=hash(cfg) % 10_000))


@pytest.mark.parametrize("window,causal", [((100, -1), True), ((40, 25), False), ((0, 0), False)])
def test_window(la, window, causal):
    p = workloads.make_prefill(1, 4, 2, 400, 700, 128, causal=causal, seed=61, window=window)
    dq, dk, dv = check(la, p)
    if window == (100, -1):   # keys no query sees get zero gradients
        unseen = 700 - 400 - 100
        assert (dk[:unseen] == 0).all() and (dv[:unseen] == 0).all()


VARLEN = [
    ([5, 300, 0, 129, 1000, 1], [5, 300, 17, 700, 1000, 1], 128, True),
    ([256, 3, 600], [100, 3, 2000], 128, True),
    ([77, 512, 512], [1024, 1500, 512], 64, True),
    ([77, 400, 33], [300, 400, 1000], 128, False),
]


@pytest.mark.parametrize("cfg", VARLEN, ids=lambda c: f"varlen_{len(c[0])}seq_d{c[2]}_{'c' if c[3] else 'n'}")
def test_varlen(la, cfg):
    ql, kl, d, causal = cfg
    check(la, workloads.make_varlen(ql, kl, 4, 2, d, causal=causal, seed=sum(ql) + 3))


def test_deterministic(la):
    p = workloads.make_prefill(1, 8, 2, 700, 900, 128, causal=True, seed=71)
    g = workloads.randn_bf16(tuple(p.q.shape), seed=72)
    a = run_bwd(la, p, g)
    b = run_bwd(la, p, g)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_full_size_mha_sampled_heads(la):
    p = workloads.mha_causal()
    check(la, p, pairs=[(0, 0), (3, 15), (1, 7)])


def test_full_size_gqa_one_kv_head(la):
    """The full GQA causal workload (B2 Hq32 Hkv8 N8192, hot channel): every
    row of one (sequence, K/V head) pair and its four query heads, so dK and
    dV sum over the whole group."""
    check(la, workloads.gqa_causal(), pairs=[(1, 7)])


def test_varlen_many_sequences(la):
    """The packed-mode tile lookup scans cu_seqlens 32 sequences at a time:
    100 sequences take several rounds."""
    g = torch.Generator().manual_seed(91)
    ql = torch.randint(0, 300, (100,), generator=g).tolist()
    kl = [q + int(x) for q, x in zip(ql, torch.randint(0, 200, (100,), generator=g).tolist())]
    check(la, workloads.make_varlen(ql, kl, 2, 1, 64, causal=True, seed=92))


def test_varlen_window(la):
    check(la, workloads.make_varlen([200, 5, 300], [700, 5, 300], 4, 2, 128, causal=False, seed=93,
                                    window=(90, 40)))


def test_tensors_past_4gib(la):
    """q, dO, out and dQ hold 2^31 elements (4 GiB) each, so the last rows
    sit past every 32-bit element and byte offset.  With a causal band of
    128 keys each gradient depends only on nearby rows and keys, and the
    tiles of the last 1024 tokens line up with those of a run on those
    tokens alone: the big run's tail must equal that run bit for bit (the
    kernels are deterministic), and the small run is checked against the
    oracle.  The big tensors repeat a seeded 2^24-element block, which keeps
    their generation quick."""
    N, Hq, Hkv, d, W, T = 262144, 64, 8, 128, 127, 1024
    scale = 1.0 / np.sqrt(d)
    rep = lambda seed: workloads.randn_bf16((1 << 24,), seed=seed).repeat((N * Hq * d) >> 24)
    q = rep(1301).view(1, N, Hq, d).cuda()
    g = rep(1302).view(1, N, Hq, d).cuda()
    k = workloads.randn_bf16((1, N, Hkv, d), seed=1303).cuda()
    v = workloads.randn_bf16((1, N, Hkv, d), seed=1304).cuda()
    assert q.numel() == 1 << 31
    kw = dict(causal=True, scale=scale, window=(W, 0))
    out, lse = la.attn_fwd(q, k, v, **kw)
    dq, dk, dv = la.attn_bwd(q, k, v, out, lse, g, **kw)
    torch.cuda.synchronize()
    t0 = N - T
    tail = lambda x: x[:, t0:].contiguous()
    qs, ks, vs, gs = tail(q), tail(k), tail(v), tail(g)
    out_s, lse_s = la.attn_fwd(qs, ks, vs, **kw)
    dq_s, dk_s, dv_s = la.attn_bwd(qs, ks, vs, out_s, lse_s, gs, **kw)
    torch.cuda.synchronize()
    # rows from W on see the same keys in both runs; keys W .. T-W-2 are seen
    # by the same rows, all of them from W on
    assert torch.equal(out[:, t0 + W:], out_s[:, W:])
    assert torch.equal(lse[:, :, t0 + W:], lse_s[:, :, W:])
    assert torch.equal(dq[:, t0 + W:], dq_s[:, W:])
    assert torch.equal(dk[:, t0 + W:N - W - 1], dk_s[:, W:T - W - 1])
    assert torch.equal(dv[:, t0 + W:N - W - 1], dv_s[:, W:T - W - 1])
    p = workloads.Prefill("tail_1024", qs.view(T, Hq, d).cpu(), ks.view(T, Hkv, d).cpu(), vs.view(T, Hkv, d).cpu(),
                          1, Hq, Hkv, T, T, d, scale, True, seed=1301, window=(W, 0))
    rq, rk, rv = oracle.backward(p, gs.view(T, Hq, d).cpu())
    f = lambda t, like: t.float().cpu().double().numpy().reshape(like.shape)
    for name, got, ref in (("dq", f(dq_s, rq), rq), ("dk", f(dk_s, rk), rk), ("dv", f(dv_s, rv), rv)):
        rel, mx, sc = grad_stats(name, got, ref)
        assert rel <= REL_RMS, f"tail {name}: relative RMS error {rel:.3e}"
        assert mx <= MAX_REL * sc + ABS_FLOOR, f"tail {name}: max abs error {mx:.3e} (max |ref| {sc:.3e})"
