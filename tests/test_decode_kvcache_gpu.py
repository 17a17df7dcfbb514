"""GPU parity of attn_decode_kvcache (several new queries per sequence over
the paged cache, with the in-place append) against the fp64 oracle, through
the C ABI.  Query i of Nq is position seq_lens[b] - Nq + i and, with causal,
sees keys up to that position ("Deep Dive - FlashAttention", sections "Causal
2.1 is the decode gotcha" and "Paged KV is a lookup, not a cache manager")."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    import exact_io_aware_04_gb300 as m
    m.build()
    torch.cuda.set_device(0)
    yield m
    assert m.attn_get_device_status() == 0


def run(la, p, num_splits=0):
    """The call on device copies; returns (out, lse, k_cache, v_cache) on the host."""
    g = p.to("cuda")
    out, lse = la.attn_decode_kvcache(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, k_new=g.k_new,
                                      v_new=g.v_new, causal=p.causal, scale=p.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu(), g.k_cache.cpu(), g.v_cache.cpu()


def gpu_rows(p, out, lse):
    """GPU results in the oracle's (b, h, i) row order."""
    o = out.float().permute(0, 2, 1, 3).reshape(-1, p.d).numpy()   # [B, Nq, Hq, d] -> (b, h, i)
    return o, lse.reshape(-1).numpy()                               # [B, Hq, Nq]


def check(la, p, num_splits=0):
    out, lse, kc, vc = run(la, p, num_splits)
    ref_o, ref_lse = oracle.decode_kvcache(p)
    if p.k_new is not None:   # the cache after the call is the oracle's append, bit for bit
        rk, rv = oracle.append_kv(p.k_cache, p.v_cache, p.block_table, p.seq_lens, p.k_new, p.v_new)
        assert torch.equal(kc.view(torch.int16), rk.view(torch.int16))
        assert torch.equal(vc.view(torch.int16), rv.view(torch.int16))
    go, gl = gpu_rows(p, out, lse)
    return assert_close(p.name, go, gl, ref_o, ref_lse)


LENS = [1, 2, 3, 15, 16, 17, 31, 33, 255, 257, 1000, 4095, 0, 2500]


@pytest.mark.parametrize("nq,hq,hkv,d", [(4, 32, 8, 128), (8, 32, 8, 128), (16, 8, 8, 128), (3, 16, 2, 128),
                                         (16, 64, 8, 64), (2, 8, 2, 64), (1, 32, 8, 128)])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_lengths_with_append(la, nq, hq, hkv, d, causal):
    p = workloads.make_kvcache_decode(LENS, nq, hq, hkv, d, num_pages=900, seed=nq * 100 + hq + d,
                                      causal=causal, append=True, nan_fill_unused=True)
    check(la, p)


@pytest.mark.parametrize("causal", [True, False])
def test_without_append(la, causal):
    p = workloads.make_kvcache_decode(LENS, 5, 32, 8, 128, num_pages=900, seed=77, causal=causal, append=False,
                                      nan_fill_unused=True)
    check(la, p)


@pytest.mark.parametrize("num_splits", [1, 2, 7, 64])
def test_fixed_split_counts(la, num_splits):
    p = workloads.make_kvcache_decode([3000, 17, 800, 4096], 6, 8, 2, 128, num_pages=700, seed=num_splits,
                                      nan_fill_unused=True, max_pages=256)
    check(la, p, num_splits=num_splits)


def test_one_query_no_append_is_attn_decode_paged(la):
    d = workloads.make_decode(LENS, 32, 8, 128, num_pages=900, seed=91, nan_fill_unused=True)
    g = d.to("cuda")
    o1, l1 = la.attn_decode_paged(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, scale=d.scale)
    o2, l2 = la.attn_decode_kvcache(g.q[:, None], g.k_cache, g.v_cache, g.block_table, g.seq_lens,
                                    causal=True, scale=d.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2[:, 0]) and torch.equal(l1, l2[:, :, 0])


def test_one_hot_attended_positions(la):
    """Q = 0 and V one-hot by position: the nonzero pattern of each query's
    output is exactly the set of positions it may see, appended ones included."""
    lens = [40, 128, 300, 7, 3]
    nq = 4
    p = workloads.make_kvcache_decode(lens, nq, 8, 2, 128, num_pages=64, seed=95, append=True, causal=True,
                                      nan_fill_unused=True)
    for base in (0, 100, 172, 250):
        q = torch.zeros_like(p.q)
        v = torch.where(torch.isnan(p.v_cache), p.v_cache, torch.zeros_like(p.v_cache))
        vn = torch.zeros_like(p.v_new)
        for b, L in enumerate(lens):
            for c in range(p.d):
                t = base + c
                if t < L:
                    if t >= L - nq:
                        vn[b, t - (L - nq), :, c] = 1.0
                    else:
                        v[int(p.block_table[b, t // 16]), t % 16, :, c] = 1.0
        ph = dataclasses.replace(p, q=q, v_cache=v, v_new=vn)
        out, lse, _, _ = run(la, ph)
        ref_o, ref_lse = oracle.decode_kvcache(ph)
        go, gl = gpu_rows(ph, out, lse)
        assert np.array_equal(go != 0, ref_o != 0), f"base {base}: attended positions differ"
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(gl), fin)
        assert np.array_equal(np.rint(np.exp(gl[fin])), np.rint(np.exp(ref_lse[fin])))


def test_append_with_bad_pages_writes_nothing_outside(la):
    """New positions whose table entry is outside the pool are skipped (and
    reported with validation on); nothing else in the pool changes."""
    p = workloads.make_kvcache_decode([40, 20, 5], 4, 4, 2, 128, num_pages=16, seed=97, append=True)
    bt = p.block_table.clone()
    bt[0, 2] = 10_000_000     # positions 36..39 of sequence 0
    bt[1, 1] = -3             # positions 16..19 of sequence 1
    bad = dataclasses.replace(p, block_table=bt)
    prev = la.attn_set_validation(True)
    try:
        g = bad.to("cuda")
        la.attn_decode_kvcache(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, k_new=g.k_new,
                               v_new=g.v_new, causal=True, scale=p.scale)
        st = la.attn_get_device_status()
    finally:
        la.attn_set_validation(prev)
    assert st == la.ATTN_ERR_BAD_INDEX
    rk, rv = oracle.append_kv(p.k_cache, p.v_cache, bt, p.seq_lens, p.k_new, p.v_new)
    assert torch.equal(g.k_cache.cpu().view(torch.int16), rk.view(torch.int16))
    assert torch.equal(g.v_cache.cpu().view(torch.int16), rv.view(torch.int16))


def test_full_size_spec_decode(la):
    # NaN in every unused slot, and in the slots the append fills until it writes them
    p = workloads.spec_decode(device="cuda", nan_fill_unused=True)
    host = p.to("cpu")   # the inputs, before the call writes the device cache
    out, lse = la.attn_decode_kvcache(p.q, p.k_cache, p.v_cache, p.block_table, p.seq_lens, k_new=p.k_new,
                                      v_new=p.v_new, causal=True, scale=p.scale)
    torch.cuda.synchronize()
    lens = host.seq_lens.tolist()
    for b in range(p.B):   # the written slots (the pool is 13 GB)
        for i in range(p.Nq):
            pos = lens[b] - p.Nq + i
            pg = int(host.block_table[b, pos // 16])
            assert torch.equal(p.k_cache[pg, pos % 16].cpu(), host.k_new[b, i])
            assert torch.equal(p.v_cache[pg, pos % 16].cpu(), host.v_new[b, i])
    kc, vc = oracle.append_kv(host.k_cache, host.v_cache, host.block_table, host.seq_lens, host.k_new, host.v_new,
                              inplace=True)
    rows = np.asarray([(b, h, i) for b in range(p.B) for h in range(p.Hq) for i in range(p.Nq)], dtype=np.int32)
    ref_o, ref_lse = oracle.decode_multi_rows(host.q, kc, vc, host.block_table, host.seq_lens, scale=p.scale,
                                              causal=True, rows=rows)
    go, gl = gpu_rows(p, out.cpu(), lse.cpu())
    stats = assert_close(p.name, go, gl, ref_o, ref_lse)
    print(p.name, stats)


def test_more_sequences_than_one_grid_dimension(la):
    """70,000 sequences, two new tokens each with the append: the split
    kernel's units run over two grid dimensions; outputs and the cache after
    the append against the oracle."""
    g = torch.Generator().manual_seed(2010)
    lens = torch.randint(2, 41, (70_000,), generator=g).tolist()
    num_pages = sum(-(-L // 16) for L in lens) + 5
    p = workloads.make_kvcache_decode(lens, 2, 4, 1, 64, num_pages=num_pages, seed=2011, causal=True, append=True)
    # V/4 (exact in bf16): rows over a few keys keep |O| below 2, where the
    # 1e-2 bound is larger than a bf16 output's rounding
    p = dataclasses.replace(p, v_cache=p.v_cache * 0.25, v_new=p.v_new * 0.25)
    check(la, p)
