"""CUDA graph capture of the library's calls.

A serving loop captures its step once and replays it with new inputs copied
into the captured buffers.  The calls allocate nothing, never synchronise,
and launch their kernels (programmatic dependent launches included) on the
caller's stream, so they can be captured after one eager call (which sets the
kernels' launch attributes).  Each test checks every replay: against the
oracle, or bit for bit against an eager call of the deterministic kernels."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_close, gather_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    import exact_io_aware_04_gb300 as m
    m.build()
    torch.cuda.set_device(0)
    yield m
    assert m.attn_get_device_status() == 0


def capture(step):
    """One eager call on a side stream, then the capture of a second."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    return g


def test_forward_and_backward_in_one_graph(la):
    B, Hq, Hkv, Nq, Nk, d = 2, 8, 2, 300, 700, 128
    shp_q, shp_k = (B, Nq, Hq, d), (B, Nk, Hkv, d)
    q = torch.empty(shp_q, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(shp_k, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    dout = torch.empty_like(q)
    out, lse = torch.empty_like(q), torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(la.lib().attn_bwd_workspace_size(B, Hq, Nq, 0), dtype=torch.uint8, device="cuda")
    scale = d ** -0.5

    def load(seed):
        p = workloads.make_prefill(B, Hq, Hkv, Nq, Nk, d, causal=True, seed=seed)
        q.copy_(p.q.view(shp_q))
        k.copy_(p.k.view(shp_k))
        v.copy_(p.v.view(shp_k))
        dout.copy_(workloads.randn_bf16(shp_q, seed=seed + 1))
        return p

    def step():
        la.attn_fwd(q, k, v, causal=True, scale=scale, out=out, lse=lse)
        la.attn_bwd(q, k, v, out, lse, dout, causal=True, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    load(1500)
    g = capture(step)
    for rep in range(3):
        p = load(1510 + 10 * rep)
        g.replay()
        torch.cuda.synchronize()
        rows = oracle.all_rows(p)
        ref_o, ref_lse = oracle.prefill(p, rows)
        go, gl = gather_prefill(p, out, lse, rows)
        assert_close(f"graph replay {rep}", go, gl, ref_o, ref_lse)
        got = [t.clone() for t in (out, lse, dq, dk, dv)]
        step()   # eager, the same inputs: the kernels are deterministic
        torch.cuda.synchronize()
        for a, b in zip(got, (out, lse, dq, dk, dv)):
            assert torch.equal(a, b)


def test_decode_steps_with_append_in_a_graph(la):
    """Each replay appends Nq new tokens per sequence and attends over the
    cache: the lengths advance between replays through the captured
    seq_lens buffer.  Every step is checked against the oracle (output, lse
    and the cache after the append, bit for bit)."""
    B, Nq, Hq, Hkv, d, steps = 4, 2, 16, 4, 128, 3
    lens0 = [100, 517, 33, 1000]
    final = [L + steps * Nq for L in lens0]
    num_pages = sum(-(-L // 16) for L in final) + 7
    base = workloads.make_decode(final, Hq, Hkv, d, num_pages=num_pages, seed=1600)
    kc, vc = base.k_cache.cuda(), base.v_cache.cuda()
    table = base.block_table.cuda()
    seq_lens = torch.tensor(lens0, dtype=torch.int32, device="cuda")
    q = torch.empty((B, Nq, Hq, d), dtype=torch.bfloat16, device="cuda")
    kn = torch.empty((B, Nq, Hkv, d), dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    out, lse = torch.empty_like(q), torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    ws = torch.empty(la.attn_decode_kvcache_workspace_size(B, Nq, Hq, Hkv, d, 16, int(table.shape[1]), 0),
                     dtype=torch.uint8, device="cuda")

    def step():
        la.attn_decode_kvcache(q, kc, vc, table, seq_lens, k_new=kn, v_new=vn, causal=True, out=out, lse=lse,
                               workspace=ws)

    # capture on a scratch copy of the cache state (the warm-up call appends)
    seq_lens.copy_(torch.tensor([L + Nq for L in lens0], dtype=torch.int32))
    q.zero_(); kn.zero_(); vn.zero_()
    saved = kc.clone(), vc.clone()
    g = capture(step)
    kc.copy_(saved[0]); vc.copy_(saved[1])
    for s in range(steps):
        lens = [L + (s + 1) * Nq for L in lens0]
        seed = 1610 + 10 * s
        q.copy_(workloads.randn_bf16(tuple(q.shape), seed=seed))
        kn.copy_(workloads.randn_bf16(tuple(kn.shape), seed=seed + 1))
        vn.copy_(workloads.randn_bf16(tuple(vn.shape), seed=seed + 2))
        seq_lens.copy_(torch.tensor(lens, dtype=torch.int32))
        before = kc.cpu(), vc.cpu()
        g.replay()
        torch.cuda.synchronize()
        p = workloads.KVCacheDecode("graph_step", q.cpu(), kn.cpu(), vn.cpu(), before[0], before[1], table.cpu(),
                                    seq_lens.cpu(), B, Nq, Hq, Hkv, d, 16, num_pages, d ** -0.5, True, seed=seed)
        ref_o, ref_lse = oracle.decode_kvcache(p)
        rk, rv = oracle.append_kv(before[0], before[1], p.block_table, p.seq_lens, p.k_new, p.v_new)
        assert torch.equal(kc.cpu().view(torch.int16), rk.view(torch.int16))
        assert torch.equal(vc.cpu().view(torch.int16), rv.view(torch.int16))
        go = out.float().cpu().permute(0, 2, 1, 3).reshape(-1, d).numpy()
        assert_close(f"graph decode step {s}", go, lse.cpu().reshape(-1).numpy(), ref_o, ref_lse)


def test_noalloc_decode_in_a_graph(la):
    """The no-allocation entry point, captured after its first call, replays
    with new queries and equals attn_decode_paged bit for bit."""
    dd = workloads.make_decode([300, 2000, 17, 900, 4096], 32, 8, 128, num_pages=700, seed=1700,
                               nan_fill_unused=True)
    g_ = dd.to("cuda")
    q = g_.q.clone()
    out, lse = torch.empty_like(q), torch.empty((dd.B, dd.Hq), dtype=torch.float32, device="cuda")

    def step():
        la.attn_decode_paged_noalloc(q, g_.k_cache, g_.v_cache, g_.block_table, g_.seq_lens, out=out, lse=lse)

    g = capture(step)
    for rep in range(3):
        q.copy_(workloads.randn_bf16(tuple(q.shape), seed=1710 + rep))
        g.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = la.attn_decode_paged(q, g_.k_cache, g_.v_cache, g_.block_table, g_.seq_lens)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_quantize_and_fp8_forward_in_one_graph(la):
    """The 8-bit path as a serving step: q, k, v quantized in one launch, then
    the 8-bit forward, captured once and replayed on new bf16 inputs.  Each
    replay's codes and scales equal the oracle's bit for bit, and its output
    meets the forward tolerances against the oracle on those codes."""
    B, Hq, Hkv, Nq, Nk, d = 2, 8, 2, 300, 700, 128
    shp_q, shp_k = (B, Nq, Hq, d), (B, Nk, Hkv, d)
    q = torch.empty(shp_q, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(shp_k, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    codes = tuple(torch.empty(x.shape, dtype=torch.uint8, device="cuda") for x in (q, k, v))
    scales = (torch.zeros((Hq, la.attn_fp8_scale_count(B, B * Nq)), dtype=torch.float32, device="cuda"),
              torch.zeros((Hkv, la.attn_fp8_scale_count(B, B * Nk)), dtype=torch.float32, device="cuda"),
              torch.zeros((Hkv, la.attn_fp8_scale_count(B, B * Nk)), dtype=torch.float32, device="cuda"))
    out, lse = torch.empty_like(q), torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    scale = d ** -0.5

    def step():
        la.attn_quantize_fp8_qkv(q, k, v, out=codes, scales=scales)
        la.attn_fwd_fp8(*codes, *scales, causal=True, scale=scale, out=out, lse=lse)

    def load(seed):
        p = workloads.make_prefill(B, Hq, Hkv, Nq, Nk, d, causal=True, seed=seed)
        q.copy_(p.q.view(shp_q))
        k.copy_(p.k.view(shp_k))
        v.copy_(p.v.view(shp_k))
        return p

    load(1800)
    g = capture(step)
    for rep in range(3):
        p = load(1810 + 10 * rep)
        g.replay()
        torch.cuda.synchronize()
        qz = oracle.quantize_problem_fp8(p)
        for name, c, sc in zip(("q", "k", "v"), codes, scales):
            ref_c, ref_s = qz[name]
            assert np.array_equal(c.cpu().numpy().reshape(np.asarray(ref_c).shape), ref_c), f"replay {rep} {name}"
            assert np.array_equal(sc.cpu().numpy().view(np.uint32),
                                  np.asarray(ref_s, dtype=np.float32).view(np.uint32)), f"replay {rep} {name}"
        rows = oracle.all_rows(p)
        ref_o, ref_lse = oracle.prefill_fp8(p, rows, quantized=qz)
        go, gl = gather_prefill(p, out, lse, rows)
        assert_close(f"fp8 graph replay {rep}", go, gl, ref_o, ref_lse)
