"""GPU parity of the 8-bit (E4M3) path through the C ABI.

attn_quantize_fp8 must reproduce the oracle's per-tile quantization bit for
bit (codes and scales).  attn_fwd_fp8 is compared with the fp64 oracle run on
the values the oracle's own codes stand for (E4M3(code) * tile scale), at the
tolerances of every other forward test: the quantization of the inputs is the
caller's choice of representation, not an error of the kernel; what the
kernel adds (fp32 accumulation of the 8-bit products, f16 probabilities,
bf16 output) must stay within max-abs 1e-2, relative RMS 5e-3 and lse 1e-3.
Which keys are attended is checked bit-exactly with one-hot values."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import LSE_ABS, O_REL_RMS, assert_close, gather_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    import exact_io_aware_04_gb300 as m
    m.build()
    torch.cuda.set_device(0)
    yield m
    assert m.attn_get_device_status() == 0


def gpu_quantize(la, x, B, N=None, cu=None):
    """attn_quantize_fp8 on a host bf16 tensor [T, H, d]; returns host numpy (codes, scales)."""
    g = x.to("cuda")
    if cu is None:
        codes, scales = la.attn_quantize_fp8(g.view(B, N, g.shape[1], g.shape[2]))
    else:
        codes, scales = la.attn_quantize_fp8(g, cu_seqlens=cu.to("cuda"))
    torch.cuda.synchronize()
    return codes.cpu().numpy().reshape(x.shape), scales.cpu().numpy()


@pytest.mark.parametrize("d", [64, 128])
def test_quantize_dense_bit_exact(la, d):
    x = workloads.randn_bf16((2 * 300, 3, d), seed=51)
    spread = torch.logspace(-4, 3, x.shape[0])[:, None, None]
    x = (x.float() * spread).to(torch.bfloat16)
    x[128:256, 1] = 0.0                       # an all-zero tile of one head
    x[300 + 5, 2, 7] = -300.0                 # an outlier
    ref_c, ref_s = oracle.quantize_fp8(x, B=2, N=300)
    got_c, got_s = gpu_quantize(la, x, 2, N=300)
    assert np.array_equal(got_c, ref_c)
    assert np.array_equal(got_s.view(np.uint32), ref_s.view(np.uint32))


def test_quantize_packed_bit_exact(la):
    lens = [130, 1, 0, 257, 128, 3000]
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    x = workloads.randn_bf16((int(cu[-1]), 2, 128), seed=52)
    x[140:200, 0] *= 1e-30                    # tiny values: subnormal codes
    ref_c, ref_s = oracle.quantize_fp8(x, B=len(lens), cu=cu)
    got_c, got_s = gpu_quantize(la, x, len(lens), cu=cu)
    assert np.array_equal(got_c, ref_c)
    assert np.array_equal(got_s.view(np.uint32), ref_s.view(np.uint32))


def gpu_quantize_qkv(la, q, k, v, B, Nq=None, Nk=None, cu_q=None, cu_k=None, sentinel=None):
    """attn_quantize_fp8_qkv on host bf16 tensors [T, H, d]; returns host numpy
    ((q codes, q scales), (k ...), (v ...)).  With `sentinel`, the scale arrays
    start filled with it, so entries the call must leave alone can be checked."""
    g = [x.to("cuda") for x in (q, k, v)]
    scales = None
    if sentinel is not None:
        Tq, Tk = q.shape[0], k.shape[0]
        scales = tuple(torch.full((x.shape[1], la.attn_fp8_scale_count(B, T)), sentinel, dtype=torch.float32,
                                  device="cuda") for x, T in ((q, Tq), (k, Tk), (v, Tk)))
    if cu_q is None:
        res = la.attn_quantize_fp8_qkv(g[0].view(B, Nq, *q.shape[1:]), g[1].view(B, Nk, *k.shape[1:]),
                                       g[2].view(B, Nk, *v.shape[1:]), scales=scales)
    else:
        res = la.attn_quantize_fp8_qkv(*g, cu_seqlens_q=cu_q.to("cuda"), cu_seqlens_k=cu_k.to("cuda"), scales=scales)
    torch.cuda.synchronize()
    return [(c.cpu().numpy().reshape(x.shape), sc.cpu().numpy()) for (c, sc), x in zip(res, (q, k, v))]


def assert_quantized_equal(got, ref, what):
    got_c, got_s = got
    ref_c, ref_s = ref
    assert np.array_equal(got_c, np.asarray(ref_c).reshape(got_c.shape)), f"{what}: codes differ"
    assert np.array_equal(got_s.view(np.uint32), np.asarray(ref_s, dtype=np.float32).view(np.uint32)
                          .reshape(got_s.shape)), f"{what}: scales differ"


@pytest.mark.parametrize("d", [64, 128])
def test_quantize_qkv_dense_bit_exact(la, d):
    """One launch over q (Hq heads, Nq tokens) and k, v (Hkv heads, Nk
    tokens) gives the oracle's codes and scales for each of the three."""
    B, Nq, Nk, Hq, Hkv = 3, 300, 517, 6, 2
    q = workloads.randn_bf16((B * Nq, Hq, d), seed=81)
    k = workloads.randn_bf16((B * Nk, Hkv, d), seed=82)
    v = (workloads.randn_bf16((B * Nk, Hkv, d), seed=83).float()
         * torch.logspace(-5, 4, B * Nk)[:, None, None]).to(torch.bfloat16)
    q[128:256, 4] = 0.0                       # an all-zero tile of one head
    k[Nk + 3, 1, 5] = 400.0                   # an outlier
    got = gpu_quantize_qkv(la, q, k, v, B, Nq=Nq, Nk=Nk)
    for name, x, n, g in (("q", q, Nq, got[0]), ("k", k, Nk, got[1]), ("v", v, Nk, got[2])):
        assert_quantized_equal(g, oracle.quantize_fp8(x, B=B, N=n), f"dense d={d} {name}")


def test_quantize_qkv_packed_bit_exact_and_gaps_untouched(la):
    """Packed sequences of unequal q and k lengths (some empty, some a single
    token, some crossing many tiles); the scale entries between sequences keep
    the sentinel."""
    q_lens = [130, 1, 0, 257, 128, 3000, 5]
    k_lens = [900, 64, 7, 0, 129, 3000, 1]
    cq = torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32)
    ck = torch.tensor([0] + list(np.cumsum(k_lens)), dtype=torch.int32)
    q = workloads.randn_bf16((int(cq[-1]), 8, 128), seed=84)
    k = workloads.randn_bf16((int(ck[-1]), 2, 128), seed=85)
    v = workloads.randn_bf16((int(ck[-1]), 2, 128), seed=86)
    v[1000:1100, 0] *= 1e-30                  # tiny values: subnormal codes
    sentinel = -7.0
    got = gpu_quantize_qkv(la, q, k, v, len(q_lens), cu_q=cq, cu_k=ck, sentinel=sentinel)
    for name, x, cu, g in (("q", q, cq, got[0]), ("k", k, ck, got[1]), ("v", v, ck, got[2])):
        ref_c, ref_s = oracle.quantize_fp8(x, B=len(q_lens), cu=cu)
        assert np.array_equal(g[0], np.asarray(ref_c).reshape(g[0].shape)), f"packed {name}: codes differ"
        written = np.zeros(g[1].shape[1], dtype=bool)
        for b in range(len(q_lens)):
            first, last = int(cu[b]), int(cu[b + 1])
            base = first // 128 + b
            written[base:base + (last - first + 127) // 128] = True
        assert np.array_equal(g[1][:, written].view(np.uint32),
                              np.asarray(ref_s, dtype=np.float32)[:, written].view(np.uint32)), \
            f"packed {name}: scales differ"
        assert (g[1][:, ~written] == sentinel).all(), f"packed {name}: an entry between sequences was written"


def test_quantize_qkv_many_short_sequences(la):
    """2,000 packed sequences of 0-300 tokens: many more (entry, head) units
    than CTAs, with gaps between sequences everywhere."""
    gen = torch.Generator().manual_seed(87)
    lens = torch.randint(0, 301, (2000,), generator=gen).tolist()
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    q = workloads.randn_bf16((int(cu[-1]), 4, 64), seed=88)
    k = workloads.randn_bf16((int(cu[-1]), 1, 64), seed=89)
    v = workloads.randn_bf16((int(cu[-1]), 1, 64), seed=90)
    got = gpu_quantize_qkv(la, q, k, v, len(lens), cu_q=cu, cu_k=cu)
    for name, x, g in (("q", q, got[0]), ("k", k, got[1]), ("v", v, got[2])):
        ref_c, ref_s = oracle.quantize_fp8(x, B=len(lens), cu=cu)
        assert np.array_equal(g[0], np.asarray(ref_c).reshape(g[0].shape)), f"{name}: codes differ"
        for b in range(0, len(lens), 97):       # every 97th sequence's entries
            first, last = int(cu[b]), int(cu[b + 1])
            base, n = first // 128 + b, (last - first + 127) // 128
            assert np.array_equal(g[1][:, base:base + n].view(np.uint32),
                                  np.asarray(ref_s, dtype=np.float32)[:, base:base + n].view(np.uint32)), name


def test_quantize_qkv_no_keys(la):
    """Nk == 0 quantizes q alone; k, v and their codes may be empty."""
    q = workloads.randn_bf16((2 * 200, 4, 128), seed=91)
    g = q.to("cuda").view(2, 200, 4, 128)
    e = torch.empty((2, 0, 2, 128), dtype=torch.bfloat16, device="cuda")
    (q8, qs), _, _ = la.attn_quantize_fp8_qkv(g, e, e)
    torch.cuda.synchronize()
    assert_quantized_equal((q8.cpu().numpy().reshape(q.shape), qs.cpu().numpy()),
                           oracle.quantize_fp8(q, B=2, N=200), "q alone")


def fp8_inputs(p, device="cuda"):
    """The oracle's codes and scales of a prefill problem, uploaded, as
    attn_fwd_fp8 arguments; and the quantized dict for the oracle."""
    qz = oracle.quantize_problem_fp8(p)
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    (qc, qs), (kc, ks), (vc, vs) = qz["q"], qz["k"], qz["v"]
    if p.varlen:
        args = (up(qc), up(kc), up(vc), up(qs), up(ks), up(vs))
        kw = dict(cu_seqlens_q=p.cu_q.to(device), cu_seqlens_k=p.cu_k.to(device))
    else:
        args = (up(qc).view(p.B, p.Nq, p.Hq, p.d), up(kc).view(p.B, p.Nk, p.Hkv, p.d),
                up(vc).view(p.B, p.Nk, p.Hkv, p.d), up(qs), up(ks), up(vs))
        kw = {}
    return args, kw, qz


def check_fp8(la, p, rows=None):
    args, kw, qz = fp8_inputs(p)
    if tuple(getattr(p, "window", (-1, -1))) != (-1, -1):
        kw["window"] = tuple(p.window)
    out, lse = la.attn_fwd_fp8(*args, causal=p.causal, scale=p.scale, **kw)
    torch.cuda.synchronize()
    if rows is None:
        rows = oracle.all_rows(p)
    ref_o, ref_lse = oracle.prefill_fp8(p, rows, quantized=qz)
    go, gl = gather_prefill(p, out, lse, rows)
    return assert_close(p.name + " fp8", go, gl, ref_o, ref_lse)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_tiny_all_rows(la, causal, d):
    """The tiny configuration (B1, H2, N256; d = 64 as configured, and d = 128)."""
    p = workloads.make_prefill(1, 2, 2, 256, 256, d, causal=causal, seed=1000, name=f"tiny_d{d}")
    check_fp8(la, p)


@pytest.mark.parametrize("causal", [False, True])
def test_peaked_softmax_all_rows(la, causal):
    """q and k times 8 (the codes are unchanged, the tile scales grow 8x):
    score spreads near +-100, most exponentials underflow and the reference
    max jumps by tens of octaves, with the per-tile score coefficients.  V
    times 1/4 keeps |O| where the 1e-2 absolute bound is above a bf16
    output's rounding (O is a few single V rows here, not an average)."""
    p = workloads.make_prefill(1, 4, 2, 300, 1100, 128, causal=causal, seed=43 + causal)
    check_fp8(la, dataclasses.replace(p, q=p.q * 8, k=p.k * 8, v=p.v * 0.25))


# (B, Hq, Hkv, Nq, Nk, causal)
SMALL = [
    (2, 4, 4, 300, 300, True),
    (2, 4, 4, 300, 300, False),
    (1, 2, 2, 200, 517, True),      # Nq < Nk
    (1, 2, 2, 517, 200, True),      # Nq > Nk: leading rows have no key
    (2, 8, 2, 384, 384, True),      # GQA 4:1, exact tile multiple
    (1, 6, 1, 129, 1000, True),     # MQA, one row past a tile
    (3, 2, 1, 1, 700, True),        # single query row
    (1, 4, 2, 640, 640, False),
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: "B{}_Hq{}_Hkv{}_Nq{}_Nk{}_{}".format(*c[:5], "c" if c[5] else "n"))
def test_small_problems(la, cfg, d):
    B, Hq, Hkv, Nq, Nk, causal = cfg
    check_fp8(la, workloads.make_prefill(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=sum(cfg[:5]) + 7 + d))


@pytest.mark.parametrize("q_lens,k_lens", [
    ([5, 1, 33, 0, 130, 300], [5, 9, 200, 4, 130, 1000]),
    ([512, 512, 100], [1024, 4000, 100]),
    ([7, 0, 300], [3, 0, 2]),                 # Nq > Nk and an empty sequence
])
def test_varlen(la, q_lens, k_lens):
    check_fp8(la, workloads.make_varlen(q_lens, k_lens, 4, 2, 128, causal=True, seed=len(q_lens) + 60))


def test_varlen_d64(la):
    check_fp8(la, workloads.make_varlen([5, 1, 33, 0, 130, 300], [5, 9, 200, 4, 130, 1000], 4, 2, 64, causal=True,
                                        seed=161))


def test_no_keys_gives_zero_rows(la):
    p = workloads.make_varlen([40, 3], [0, 0], 2, 1, 128, causal=True, seed=64)
    check_fp8(la, p)


@pytest.mark.parametrize("causal", [True, False])
def test_score_ladder_all_rows(la, causal):
    """Tile maxima that hold, rise a little, jump and fall, with per-tile
    scales that differ from tile to tile: every branch of the rescale runs
    on its own tile coefficient."""
    p = workloads.score_ladder(workloads.make_prefill(1, 4, 2, 256, 1024, 128, causal=causal, seed=65))
    check_fp8(la, p)


@pytest.mark.parametrize("d", [64, 128])
def test_one_hot_attended_keys(la, d):
    """Q = 0 (every allowed key weighs 1/|A_i|), V one-hot by key index over a
    window of d keys: the nonzero pattern of O is the allowed set exactly,
    its magnitude names the K/V head, and exp(lse) is the allowed count."""
    p = workloads.make_varlen([3, 130, 200], [70, 300, 128], 4, 2, d, causal=True, seed=66)
    for base in (0, 60, 200):
        ph = workloads.one_hot_values(p, base)
        args, kw, qz = fp8_inputs(ph)
        out, lse = la.attn_fwd_fp8(*args, causal=True, scale=ph.scale, **kw)
        torch.cuda.synchronize()
        rows = oracle.all_rows(ph)
        ref_o, ref_lse = oracle.prefill_fp8(ph, rows, quantized=qz)
        go, gl = gather_prefill(ph, out, lse, rows)
        assert np.array_equal(go != 0, ref_o != 0), f"base {base}: attended-key pattern differs"
        cnt = np.where(np.isfinite(ref_lse), np.rint(np.exp(ref_lse)), 0)
        g_of_h = (rows[:, 1] // (p.Hq // p.Hkv)) + 1
        nz = go != 0
        assert np.array_equal(np.rint((go * cnt[:, None])[nz]), np.broadcast_to(g_of_h[:, None], go.shape)[nz])
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.rint(np.exp(gl[fin])), cnt[fin])


@pytest.mark.parametrize("d", [64, 128])
def test_quantize_then_forward_end_to_end(la, d):
    """The GPU's own quantization feeds the GPU forward; the oracle quantizes
    the same bf16 inputs itself."""
    p = workloads.make_varlen([300, 77], [900, 77], 8, 2, d, causal=True, seed=67)
    g = p.to("cuda")
    (q8, qs), (k8, ks), (v8, vs) = la.attn_quantize_fp8_qkv(g.q, g.k, g.v, cu_seqlens_q=g.cu_q, cu_seqlens_k=g.cu_k)
    out, lse = la.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True, scale=p.scale, cu_seqlens_q=g.cu_q,
                               cu_seqlens_k=g.cu_k)
    torch.cuda.synchronize()
    rows = oracle.all_rows(p)
    ref_o, ref_lse = oracle.prefill_fp8(p, rows)
    go, gl = gather_prefill(p, out, lse, rows)
    assert_close(p.name + " fp8 end to end", go, gl, ref_o, ref_lse)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mha_causal", "gqa_causal", "varlen_chunked"])
def test_full_size_sampled_rows(la, name):
    p = getattr(workloads, name)()
    per = 32 if name == "varlen_chunked" else 128
    rows = workloads.sample_rows(None, [nq for nq, _ in p.seq_lens()], p.Hq, per, seed=p.seed + 800).numpy()
    print(name, check_fp8(la, p, rows))


def check_rows_on_own_scale(la, p, row_bound=2e-2):
    """Every row of attn_fwd_fp8 against the oracle, each on its own scale.

    For inputs whose tiles differ by powers of two the outputs span many
    octaves, so the absolute bound of the other tests says nothing; instead
    the relative RMS over all rows, the lse, and each row's error norm over
    its reference norm are bounded.  The per-row bound is 2e-2: a bf16 output
    rounds each element by at most 2^-9 relative (2e-3), the f16 weights by
    2^-12, and the rest leaves room for rows whose values partly cancel.  A
    row whose weight sits on tiles with small V scales has a small output,
    which the global measures cannot see; the per-row one does."""
    args, kw, qz = fp8_inputs(p)
    out, lse = la.attn_fwd_fp8(*args, causal=p.causal, scale=p.scale, **kw)
    torch.cuda.synchronize()
    rows = oracle.all_rows(p)
    ref_o, ref_lse = oracle.prefill_fp8(p, rows, quantized=qz)
    go, gl = gather_prefill(p, out, lse, rows)
    go = np.asarray(go, dtype=np.float64)
    gl = np.asarray(gl, dtype=np.float64)
    assert np.isfinite(go).all(), "non-finite output values"
    fin = np.isfinite(ref_lse)
    assert (np.isfinite(gl) == fin).all() and (gl[~fin] == -np.inf).all()
    lse_err = float(np.abs(gl[fin] - ref_lse[fin]).max(initial=0.0))
    rel = float(np.sqrt(((go - ref_o) ** 2).sum() / (ref_o ** 2).sum()))
    ref_n = np.sqrt((ref_o ** 2).sum(axis=1))
    err_n = np.sqrt(((go - ref_o) ** 2).sum(axis=1))
    nz = ref_n > 0
    assert (err_n[~nz] == 0).all(), "rows whose reference is zero must be zero"
    worst = float((err_n[nz] / ref_n[nz]).max(initial=0.0))
    assert rel <= O_REL_RMS, f"O rel-RMS {rel:.3e}"
    assert lse_err <= LSE_ABS, f"lse err {lse_err:.3e}"
    assert worst <= row_bound, f"worst row relative error {worst:.3e}"
    return {"rel_rms": rel, "lse_abs": lse_err, "worst_row": worst}


@pytest.mark.parametrize("causal", [True, False])
def test_tile_scales_spanning_many_octaves(la, causal):
    """V tiles whose values (hence scales) differ by up to 2^+-20, so that the
    ratio of a tile's scale to the largest reaches 2^-40, far below f16's
    normal range; Q and K tiles differ by up to 2^+-3, so that each K tile's
    score coefficient differs while the logits stay in the range an fp32
    softmax resolves.  Values are multiplied by powers of two, exact in bf16,
    so the inputs stay on the oracle's grid."""
    p = workloads.make_varlen([300, 77], [900, 300], 4, 2, 128, causal=causal, seed=68)
    g = torch.Generator().manual_seed(69)
    for t, lens, span in ((p.q, [300, 77], 3), (p.k, [900, 300], 3), (p.v, [900, 300], 20)):
        start = 0
        for L in lens:
            for r0 in range(0, L, 128):
                e = int(torch.randint(-span, span + 1, (1,), generator=g))
                t[start + r0:start + min(L, r0 + 128)] = (t[start + r0:start + min(L, r0 + 128)].float()
                                                          * 2.0 ** e).to(torch.bfloat16)
            start += L
    check_rows_on_own_scale(la, p)


@pytest.mark.parametrize("causal", [True, False])
def test_outlier_value_tile_with_little_weight(la, causal):
    """The first K/V tile of every sequence holds V values 2^16 times larger
    than the rest but scores about 14 below them (q . k = -160 on channel 0
    at scale 1/sqrt(128)), so its weights are about 2^-20 of the others': the
    rows' outputs come from tiles whose V scales are 2^-16 of the item's
    largest.  Each row must still be right on its own scale."""
    p = workloads.make_varlen([300, 200], [700, 400], 4, 2, 128, causal=causal, seed=70)
    q = p.q.float() * 0.25
    k = p.k.float() * 0.25
    v = p.v.float()
    q[:, :, 0] = 16.0
    cq, ck = p.cu_q.tolist(), p.cu_k.tolist()
    for b in range(p.B):
        k[ck[b]:ck[b + 1], :, 0] = 0.0
        k[ck[b]:ck[b] + 128, :, 0] = -10.0
        v[ck[b]:ck[b] + 128] *= 2.0 ** 16
    p = dataclasses.replace(p, q=q.to(torch.bfloat16), k=k.to(torch.bfloat16), v=v.to(torch.bfloat16))
    check_rows_on_own_scale(la, p)


def test_large_value_tile_unseen_by_early_rows(la):
    """Causal, 128 queries over 300 keys: row i sees keys up to i + 172, so
    rows 0..83 never see the last K/V tile (keys 256..299), whose values are
    2^30 times larger.  The V scale those rows' weights are normalised to
    must come from tiles they see, or their outputs vanish in f16."""
    p = workloads.make_prefill(2, 4, 2, 128, 300, 128, causal=True, seed=71)
    v = p.v.float().reshape(p.B, p.Nk, p.Hkv, p.d)
    v[:, 256:] *= 2.0 ** 30
    p = dataclasses.replace(p, v=v.reshape(-1, p.Hkv, p.d).to(torch.bfloat16))
    check_rows_on_own_scale(la, p)


@pytest.mark.parametrize("name", ["gqa_causal", "varlen_chunked"])
def test_quantize_full_size_bit_exact(la, name):
    """The quantizer on the q, k and v of the full workloads the benchmark
    times (GQA causal with its hot channel; the packed chunked prefill), bit
    for bit against the oracle's codes and scales."""
    p = getattr(workloads, name)()
    qz = oracle.quantize_problem_fp8(p)
    if p.varlen:
        qkv = gpu_quantize_qkv(la, p.q, p.k, p.v, p.B, cu_q=p.cu_q, cu_k=p.cu_k)
    else:
        qkv = gpu_quantize_qkv(la, p.q, p.k, p.v, p.B, Nq=p.Nq, Nk=p.Nk)
    for i, (key, x, n) in enumerate((("q", p.q, p.Nq), ("k", p.k, p.Nk), ("v", p.v, p.Nk))):
        if p.varlen:
            one = gpu_quantize(la, x, p.B, cu=p.cu_q if key == "q" else p.cu_k)
        else:
            one = gpu_quantize(la, x, p.B, N=n)
        assert_quantized_equal(one, qz[key], f"{name} {key}")
        assert_quantized_equal(qkv[i], qz[key], f"{name} {key} (one launch for q, k, v)")


@pytest.mark.parametrize("window,causal", [((100, -1), True), ((40, 25), False), ((0, 0), False), ((300, 300), False)])
def test_window_dense(la, window, causal):
    """attn_fwd_fp8_window on a dense problem: the band of attn_fwd_window
    (Nq < Nk, both edges inside and across tiles), every row."""
    check_fp8(la, workloads.make_prefill(1, 4, 2, 400, 700, 128, causal=causal, seed=1950, window=window))


@pytest.mark.parametrize("d", [64, 128])
def test_window_varlen(la, d):
    check_fp8(la, workloads.make_varlen([200, 5, 300, 0], [700, 5, 300, 9], 4, 2, d, causal=False, seed=1951,
                                        window=(90, 40)))


def test_window_attended_keys_one_hot(la):
    """Which keys each row attends under a two-sided band, bit for bit: Q = 0
    (codes 0, scale 1) and V one-hot by key index (exact in E4M3)."""
    p = workloads.make_prefill(1, 4, 2, 300, 500, 128, causal=False, seed=1952, window=(70, 30))
    for base in (0, 128, 250):
        ph = workloads.one_hot_values(p, base)
        args, kw, qz = fp8_inputs(ph)
        out, lse = la.attn_fwd_fp8(*args, causal=False, scale=ph.scale, window=(70, 30))
        torch.cuda.synchronize()
        rows = oracle.all_rows(ph)
        ref_o, ref_lse = oracle.prefill_fp8(ph, rows, quantized=qz)
        go, gl = gather_prefill(ph, out, lse, rows)
        assert np.array_equal(go != 0, ref_o != 0), f"base {base}: attended-key pattern differs"
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(gl), fin)
