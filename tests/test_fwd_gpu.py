"""GPU parity of attn_fwd against the fp64 oracle (through the C ABI)."""
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


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_workload_all_rows(la, causal):
    check_all_rows(la, workloads.tiny(causal))


# (B, Hq, Hkv, Nq, Nk, d, causal): several tiles, ragged tails, both corners
SMALL = [
    (2, 4, 4, 300, 300, 128, True),
    (2, 4, 4, 300, 300, 128, False),
    (1, 2, 2, 200, 517, 128, True),     # Nq < Nk: short query block over a long cache
    (1, 2, 2, 517, 200, 128, True),     # Nq > Nk: leading rows have no key
    (1, 2, 2, 517, 200, 64, False),
    (2, 8, 2, 384, 384, 64, True),      # GQA 4:1, exact tile multiple
    (1, 6, 1, 129, 1000, 128, True),    # MQA, one row past a tile
    (3, 2, 1, 1, 700, 128, True),       # single query row (decode-like prefill)
    (1, 2, 2, 1000, 3000, 128, True),
    (1, 4, 2, 640, 640, 64, False),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: "B{}_Hq{}_Hkv{}_Nq{}_Nk{}_d{}_{}".format(*c[:6], "c" if c[6] else "n"))
def test_small_problems_all_rows(la, cfg):
    B, Hq, Hkv, Nq, Nk, d, causal = cfg
    p = workloads.make_prefill(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=hash(cfg) % 10_000)
    check_all_rows(la, p)


# Score ladders: the running max of a row holds, rises by less than the
# rescale threshold over a whole block (row sums of p far above 2^8), jumps
# far above it, and falls, tile after tile (workloads.score_ladder).
LADDER = [
    (1, 4, 2, 300, 1100, 128, False),
    (1, 4, 2, 300, 1100, 128, True),
    (2, 4, 4, 260, 700, 64, False),
]


@pytest.mark.parametrize("cfg", LADDER, ids=lambda c: "B{}_Hq{}_Hkv{}_Nq{}_Nk{}_d{}_{}".format(*c[:6], "c" if c[6] else "n"))
def test_score_ladder_all_rows(la, cfg):
    B, Hq, Hkv, Nq, Nk, d, causal = cfg
    p = workloads.make_prefill(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=31 + Nk + d)
    check_all_rows(la, workloads.score_ladder(p))


# Peaked rows: q and k times 8 (exact in bf16) put the scores' spread near
# +-100 in natural units, so each row's probability mass sits on a few keys and
# the exponentials of most keys underflow to zero; whole tiles contribute
# nothing after the first, and the running max jumps by tens of octaves.  O is
# then a few single V rows rather than an average, so V is scaled by 1/4
# (exact): at |O| >= 2.56 a bf16 output's half step alone exceeds the 1e-2
# absolute bound.
PEAKED = [
    (1, 4, 2, 300, 1100, 128, False),
    (1, 4, 2, 300, 1100, 128, True),
    (2, 4, 1, 260, 700, 64, True),
]


@pytest.mark.parametrize("cfg", PEAKED, ids=lambda c: "B{}_Hq{}_Hkv{}_Nq{}_Nk{}_d{}_{}".format(*c[:6], "c" if c[6] else "n"))
def test_peaked_softmax_all_rows(la, cfg):
    B, Hq, Hkv, Nq, Nk, d, causal = cfg
    p = workloads.make_prefill(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=41 + Nk + d)
    p = dataclasses.replace(p, q=p.q * 8, k=p.k * 8, v=p.v * 0.25)
    check_all_rows(la, p)


VARLEN = [
    ([5, 300, 0, 129, 1000, 1], [5, 300, 17, 700, 1000, 1], 128, True),
    ([256, 3, 600], [100, 3, 2000], 128, True),     # a sequence with Nq > Nk
    ([77, 512, 512], [1024, 1500, 512], 64, True),
    ([77, 400, 33], [300, 400, 1000], 128, False),
]


@pytest.mark.parametrize("cfg", VARLEN, ids=lambda c: f"varlen_{len(c[0])}seq_d{c[2]}_{'c' if c[3] else 'n'}")
def test_varlen_all_rows(la, cfg):
    ql, kl, d, causal = cfg
    p = workloads.make_varlen(ql, kl, 4, 2, d, causal=causal, seed=sum(ql) + sum(kl))
    check_all_rows(la, p)


def test_no_keys_gives_zero_rows(la):
    p = workloads.make_varlen([3, 40], [0, 0], 2, 2, 128, causal=False, seed=3)
    out, lse = run_prefill(la, p)
    torch.cuda.synchronize()
    assert (out == 0).all() and torch.isneginf(lse).all()


# ---------------------------------------------------------------- one-hot: which keys are attended
def test_one_hot_tiny_all_windows(la):
    for causal in (False, True):
        p = workloads.tiny(causal)
        one_hot_check(la, p, range(0, p.Nk, p.d))


def test_one_hot_gqa_unequal_lengths(la):
    p = workloads.make_prefill(2, 8, 2, 200, 517, 128, causal=True, seed=12)
    one_hot_check(la, p, [0, 128, 256, 389, 517 - 128])


def test_one_hot_varlen(la):
    p = workloads.make_varlen([5, 300, 129, 600], [5, 300, 700, 200], 4, 2, 64, causal=True, seed=13)
    one_hot_check(la, p, [0, 64, 128, 192, 300, 450, 636])


# ---------------------------------------------------------------- mixed shapes in one process
def test_shape_order_independence(la):
    """Shape A then B then A again: identical bits for A, both match the
    oracle (a kernel keyed only on the GQA ratio would mix these up)."""
    a = workloads.make_prefill(1, 4, 2, 256, 256, 128, causal=True, seed=21)  # Hq 4, Hkv 2
    b = workloads.make_prefill(1, 2, 1, 256, 256, 128, causal=True, seed=22)  # Hq 2, Hkv 1
    oa1, la1 = run_prefill(la, a)
    ob, lb = run_prefill(la, b)
    oa2, la2 = run_prefill(la, a)
    torch.cuda.synchronize()
    assert torch.equal(oa1, oa2) and torch.equal(la1, la2)
    for p, (o, l) in ((a, (oa1, la1)), (b, (ob, lb))):
        rows = oracle.all_rows(p)
        ref_o, ref_lse = oracle.prefill(p, rows)
        go, gl = gather_prefill(p, o, l, rows)
        assert_close(p.name, go, gl, ref_o, ref_lse)


# ---------------------------------------------------------------- full-size workloads, sampled rows
@pytest.mark.parametrize("name", ["mha_causal", "gqa_causal", "varlen_chunked"])
def test_full_size_sampled_rows(la, name):
    p = getattr(workloads, name)()
    out, lse = run_prefill(la, p)
    torch.cuda.synchronize()
    per = 64 if name == "varlen_chunked" else 512
    lens = [nq for nq, _ in p.seq_lens()]
    rows = workloads.sample_rows(None, lens, p.Hq, per, seed=p.seed + 500)
    ref_o, ref_lse = oracle.prefill(p, rows.numpy())
    go, gl = gather_prefill(p, out, lse, rows.numpy())
    stats = assert_close(p.name, go, gl, ref_o, ref_lse)
    print(p.name, stats)


def test_varlen_many_sequences_natural_order(la):
    """More (sequence, pair) entries than the in-kernel sort takes (1024): the
    items run in their natural order.  1200 sequences of 0..599 rows."""
    g = torch.Generator().manual_seed(81)
    ql = torch.randint(0, 600, (1200,), generator=g).tolist()
    kl = [q + int(x) for q, x in zip(ql, torch.randint(0, 300, (1200,), generator=g).tolist())]
    p = workloads.make_varlen(ql, kl, 2, 1, 64, causal=True, seed=82)
    n_pairs = sum((q + 255) // 256 for q in ql)
    assert n_pairs > 1024
    out, lse = run_prefill(la, p)
    torch.cuda.synchronize()
    rows = workloads.sample_rows(None, ql, p.Hq, 4, seed=83)
    ref_o, ref_lse = oracle.prefill(p, rows.numpy())
    go, gl = gather_prefill(p, out, lse, rows.numpy())
    assert_close(p.name, go, gl, ref_o, ref_lse)


def test_varlen_thousands_of_sequences_every_row_written(la):
    """3000 packed sequences (about 3000 (sequence, pair) entries, natural
    order) -- short prompts, and every 100th a 512-query chunk over a long
    prefix: with out and lse prefilled with NaN, every row is written once the
    call returns (no entry is lost, none runs into another's rows), and
    sampled rows match the oracle."""
    g = torch.Generator().manual_seed(84)
    B = 3000
    ql = torch.randint(1, 300, (B,), generator=g).tolist()
    kl = [q + int(x) for q, x in zip(ql, torch.randint(0, 200, (B,), generator=g).tolist())]
    for b in range(0, B, 100):
        ql[b] = 512
        kl[b] = 512 + int(torch.randint(4000, 20000, (1,), generator=g))
    p = workloads.make_varlen(ql, kl, 2, 1, 64, causal=True, seed=85)
    gp = p.to("cuda")
    out = torch.full_like(gp.q, float("nan"))
    lse = torch.full((p.Hq, gp.q.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
    la.attn_fwd(gp.q, gp.k, gp.v, causal=True, scale=p.scale, cu_seqlens_q=gp.cu_q, cu_seqlens_k=gp.cu_k,
                out=out, lse=lse)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    rows = workloads.sample_rows(None, ql, p.Hq, 2, seed=86)
    ref_o, ref_lse = oracle.prefill(p, rows.numpy())
    go, gl = gather_prefill(p, out, lse, rows.numpy())
    assert_close(p.name, go, gl, ref_o, ref_lse)


def test_long_sequence_65536(la):
    """One causal sequence of 65,536 tokens (GQA 8:2, q doubled for larger
    logits and more rescales): the last rows run the recurrence over all
    512 K/V tiles.  Rows at both ends, around tile boundaries, in the
    middle, and seeded draws, against the oracle."""
    N, Hq, Hkv, d = 65536, 8, 2, 128
    p = workloads.make_prefill(1, Hq, Hkv, N, N, d, causal=True, seed=2100)
    p = dataclasses.replace(p, q=(p.q.float() * 2.0).to(torch.bfloat16))
    out, lse = run_prefill(la, p)
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(2101)
    fixed = [0, 1, 127, 128, 129, N // 2 - 1, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = [(0, h, i) for h in range(Hq) for i in sorted(set(fixed + torch.randint(0, N, (12,), generator=g).tolist()))]
    rows = np.asarray(rows, dtype=np.int32)
    ref_o, ref_lse = oracle.prefill(p, rows)
    go, gl = gather_prefill(p, out, lse, rows)
    print(assert_close("long_65536", go, gl, ref_o, ref_lse))
