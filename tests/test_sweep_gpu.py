"""Seeded sweeps over random problem shapes, every row against the fp64
oracle, through the C ABI.

The hand-picked cases of the other GPU files cover each edge on purpose;
these draw the combinations nobody picked: head groupings, head dims, ragged
lengths on both sides, causal or not, two-sided windows, packed sequences
with empty ones, decode lengths and split counts, several queries with and
without the append, the backward, and the 8-bit path.  Each configuration is
a fixed function of its index (numpy RandomState), so a failure names a
reproducible case.  Tolerances are the ones every other test uses."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_close, gather_prefill, one_hot_check, run_decode, run_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    import exact_io_aware_04_gb300 as m
    m.build()
    torch.cuda.set_device(0)
    yield m
    assert m.attn_get_device_status() == 0


def heads(r, max_hq=16):
    hkv = int(r.choice([1, 2, 4]))
    group = int(r.choice([g for g in (1, 2, 4, 8) if hkv * g <= max_hq]))
    return hkv * group, hkv


def window(r):
    """None, or (left, right) with each side unbounded (-1) or bounded."""
    if r.rand() < 0.5:
        return None
    left = -1 if r.rand() < 0.3 else int(r.randint(0, 300))
    right = -1 if r.rand() < 0.3 else int(r.randint(0, 120))
    return (left, right)


def prefill_case(i, fp8=False, bwd=False):
    r = np.random.RandomState(7100 + 97 * i + (5000 if fp8 else 0) + (9000 if bwd else 0))
    Hq, Hkv = heads(r, 8 if bwd else 16)
    d = int(r.choice([64, 128]))
    causal = bool(r.rand() < 0.6)
    win = window(r)
    if win is not None and causal:
        win = (win[0], 0)   # causal fixes the right side at 0
    lim_q, lim_k = (300, 400) if bwd else (700, 1500)
    seed = 7300 + i
    if r.rand() < 0.4:   # packed sequences, some empty
        n = int(r.randint(1, 6))
        ql = [int(x) for x in r.randint(0, lim_q // 2, n)]
        kl = [int(x) for x in r.randint(0, lim_k // 2, n)]
        if sum(ql) == 0:
            ql[0] = 1
        p = workloads.make_varlen(ql, kl, Hq, Hkv, d, causal=causal, seed=seed, window=win or (-1, -1))
    else:
        B = int(r.randint(1, 4))
        Nq = int(r.randint(1, lim_q))
        Nk = int(r.randint(1, lim_k))
        p = workloads.make_prefill(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=seed, window=win or (-1, -1))
    return p


@pytest.mark.parametrize("i", range(64))
def test_forward(la, i):
    p = prefill_case(i)
    out, lse = run_prefill(la, p)
    torch.cuda.synchronize()
    rows = oracle.all_rows(p)
    ref_o, ref_lse = oracle.prefill(p, rows)
    go, gl = gather_prefill(p, out, lse, rows)
    assert_close(f"sweep {i}", go, gl, ref_o, ref_lse)


@pytest.mark.parametrize("i", range(12))
def test_forward_attended_keys_one_hot(la, i):
    """Which keys each row attends, bit for bit (Q = 0, V one-hot by key)."""
    one_hot_check(la, prefill_case(100 + i), bases=(0, 100))


def decode_case(i):
    r = np.random.RandomState(8100 + 31 * i)
    Hq, Hkv = heads(r, 64)
    d = int(r.choice([64, 128]))
    B = int(r.randint(1, 12))
    lens = [int(x) for x in r.randint(0, 3000, B)]
    num_pages = sum(-(-L // 16) for L in lens) + int(r.randint(1, 40))
    splits = int(r.choice([0, 0, 1, 2, 5, 13]))
    return workloads.make_decode(lens, Hq, Hkv, d, num_pages=num_pages, seed=8300 + i, nan_fill_unused=True), splits


@pytest.mark.parametrize("i", range(32))
def test_paged_decode(la, i):
    dd, splits = decode_case(i)
    out, lse = run_decode(la, dd, num_splits=splits)
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.decode(dd)
    assert_close(f"decode sweep {i}", out.float().cpu().numpy().reshape(-1, dd.d), lse.cpu().numpy().reshape(-1),
                 ref_o, ref_lse)


@pytest.mark.parametrize("i", range(24))
def test_decode_several_queries(la, i):
    r = np.random.RandomState(8600 + 13 * i)
    Hq, Hkv = heads(r, 32)
    d = int(r.choice([64, 128]))
    Nq = int(r.randint(1, 17))
    append = bool(r.rand() < 0.7)
    causal = bool(r.rand() < 0.7)
    B = int(r.randint(1, 8))
    lens = [int(x) for x in r.randint(Nq, 2500, B)]
    num_pages = sum(-(-L // 16) for L in lens) + int(r.randint(1, 30))
    splits = int(r.choice([0, 0, 1, 3, 9]))
    p = workloads.make_kvcache_decode(lens, Nq, Hq, Hkv, d, num_pages=num_pages, seed=8800 + i, causal=causal,
                                      append=append, nan_fill_unused=True)
    g = p.to("cuda")
    out, lse = la.attn_decode_kvcache(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, k_new=g.k_new,
                                      v_new=g.v_new, causal=p.causal, scale=p.scale, num_splits=splits)
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.decode_kvcache(p)
    if append:
        rk, rv = oracle.append_kv(p.k_cache, p.v_cache, p.block_table, p.seq_lens, p.k_new, p.v_new)
        assert torch.equal(g.k_cache.cpu().view(torch.int16), rk.view(torch.int16))
        assert torch.equal(g.v_cache.cpu().view(torch.int16), rv.view(torch.int16))
    go = out.float().cpu().permute(0, 2, 1, 3).reshape(-1, p.d).numpy()
    assert_close(f"kvcache sweep {i}", go, lse.cpu().reshape(-1).numpy(), ref_o, ref_lse)


@pytest.mark.parametrize("i", range(16))
def test_backward(la, i):
    from test_bwd_gpu import check
    check(la, prefill_case(i, bwd=True))


@pytest.mark.parametrize("i", range(16))
def test_fp8_forward(la, i):
    from test_fp8_gpu import check_fp8
    check_fp8(la, prefill_case(i, fp8=True))


@pytest.mark.parametrize("i", range(24))
def test_quantize_qkv(la, i):
    """The one-launch q, k, v quantizer on the sweep's prefill shapes (d = 64
    or 128, dense or packed with empty sequences), bit for bit against the
    oracle's codes and scales, with a tile of zeros and a spread of
    magnitudes across the tokens drawn in."""
    r = np.random.RandomState(8800 + i)
    p = prefill_case(i + 100)
    tq, tk = p.q.shape[0], p.k.shape[0]
    spread = torch.from_numpy(10.0 ** r.uniform(-6, 4, size=(tq, 1, 1))).float()
    q = (p.q.float() * spread).to(torch.bfloat16)
    v = p.v.clone()
    if tk > 130:
        v[128:256 if tk >= 256 else tk, int(r.randint(0, p.Hkv))] = 0.0
    from test_fp8_gpu import gpu_quantize_qkv, assert_quantized_equal
    if p.varlen:
        got = gpu_quantize_qkv(la, q, p.k, v, p.B, cu_q=p.cu_q, cu_k=p.cu_k)
        seq = [dict(B=p.B, cu=p.cu_q), dict(B=p.B, cu=p.cu_k), dict(B=p.B, cu=p.cu_k)]
    else:
        got = gpu_quantize_qkv(la, q, p.k, v, p.B, Nq=p.Nq, Nk=p.Nk)
        seq = [dict(B=p.B, N=p.Nq), dict(B=p.B, N=p.Nk), dict(B=p.B, N=p.Nk)]
    for name, x, kw, g in zip(("q", "k", "v"), (q, p.k, v), seq, got):
        assert_quantized_equal(g, oracle.quantize_fp8(x, **kw), f"sweep {i} {name}")
