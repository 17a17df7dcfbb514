"""Malformed index arrays: never a fault, and reported when validation is on.

Every entry point clamps packed offsets and page indices into the buffers the
ABI describes, so garbage in cu_seqlens, block tables or seq_lens cannot move
an access outside them.  With attn_set_validation(1) the same inputs are
reported as ATTN_ERR_BAD_INDEX through attn_get_device_status; with it off
the call completes with status OK (the results are unspecified).  The
quantizer's outputs sit inside larger buffers whose tails must keep their
sentinel bytes."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

BAD_CU = {
    "decreasing": [0, 300, 100, 500],
    "past_the_end": [0, 200, 900, 500],
    "negative": [0, -50, 300, 500],
    "end_short": [0, 100, 200, 400],
}


@pytest.fixture(scope="module")
def la():
    import exact_io_aware_04_gb300 as m
    m.build()
    torch.cuda.set_device(0)
    yield m
    assert m.attn_get_device_status() == 0


def with_validation(la, on, fn):
    prev = la.attn_set_validation(on)
    try:
        fn()
        return la.attn_get_device_status()
    finally:
        la.attn_set_validation(prev)


@pytest.mark.parametrize("bad", sorted(BAD_CU))
def test_forward_and_backward_packed(la, bad):
    T, Hq, Hkv, d = 500, 4, 2, 128
    q = workloads.randn_bf16((T, Hq, d), seed=1900).cuda()
    k = workloads.randn_bf16((T, Hkv, d), seed=1901).cuda()
    v = workloads.randn_bf16((T, Hkv, d), seed=1902).cuda()
    g = workloads.randn_bf16((T, Hq, d), seed=1903).cuda()
    cu_bad = torch.tensor(BAD_CU[bad], dtype=torch.int32, device="cuda")
    cu_ok = torch.tensor([0, 100, 300, 500], dtype=torch.int32, device="cuda")
    for cq, ck in ((cu_bad, cu_ok), (cu_ok, cu_bad)):
        def fwd():
            return la.attn_fwd(q, k, v, causal=True, cu_seqlens_q=cq, cu_seqlens_k=ck)
        assert with_validation(la, True, fwd) == la.ATTN_ERR_BAD_INDEX
        assert with_validation(la, False, fwd) == la.ATTN_OK
        out, lse = la.attn_fwd(q, k, v, causal=True, cu_seqlens_q=cu_ok, cu_seqlens_k=cu_ok)

        def bwd():
            la.attn_bwd(q, k, v, out, lse, g, causal=True, cu_seqlens_q=cq, cu_seqlens_k=ck)
        assert with_validation(la, True, bwd) == la.ATTN_ERR_BAD_INDEX
        assert with_validation(la, False, bwd) == la.ATTN_OK


@pytest.mark.parametrize("bad", sorted(BAD_CU))
def test_quantizer_packed_stays_inside_its_buffers(la, bad):
    T, H, d = 500, 3, 128
    x = workloads.randn_bf16((T, H, d), seed=1910).cuda()
    cu = torch.tensor(BAD_CU[bad], dtype=torch.int32, device="cuda")
    B = cu.numel() - 1
    n_scale = la.attn_fp8_scale_count(B, T)
    codes = torch.full((T + 256, H, d), 0x5A, dtype=torch.uint8, device="cuda")
    scales = torch.full((H * n_scale + 256,), -7.0, dtype=torch.float32, device="cuda")

    def quant():
        la.attn_quantize_fp8(x, cu_seqlens=cu, out=codes[:T], scale=scales[:H * n_scale].view(H, n_scale))
    for on in (True, False):
        st = with_validation(la, on, quant)
        assert st == (la.ATTN_ERR_BAD_INDEX if on else la.ATTN_OK)
        assert bool((codes[T:] == 0x5A).all()), "a code was written past the tensor"
        assert bool((scales[H * n_scale:] == -7.0).all()), "a scale was written past the array"


@pytest.mark.parametrize("bad", sorted(BAD_CU))
def test_quantizer_qkv_packed_stays_inside_its_buffers(la, bad):
    """The one-launch q, k, v quantizer with malformed offsets for the keys:
    nothing is written past any of the six outputs."""
    T, Hq, Hkv, d = 500, 4, 2, 128
    cu_ok = torch.tensor([0, 100, 300, 500], dtype=torch.int32, device="cuda")
    cu = torch.tensor(BAD_CU[bad], dtype=torch.int32, device="cuda")
    B = cu.numel() - 1
    n_scale = la.attn_fp8_scale_count(B, T)
    xs = [workloads.randn_bf16((T, H, d), seed=1940 + i).cuda() for i, H in enumerate((Hq, Hkv, Hkv))]
    codes = [torch.full((T + 256, H, d), 0x5A, dtype=torch.uint8, device="cuda") for H in (Hq, Hkv, Hkv)]
    scales = [torch.full((H * n_scale + 256,), -7.0, dtype=torch.float32, device="cuda") for H in (Hq, Hkv, Hkv)]

    def quant():
        la.attn_quantize_fp8_qkv(*xs, cu_seqlens_q=cu_ok, cu_seqlens_k=cu, out=tuple(c[:T] for c in codes),
                                 scales=tuple(s[:H * n_scale].view(H, n_scale) for s, H in zip(scales, (Hq, Hkv, Hkv))))
    for on in (True, False):
        st = with_validation(la, on, quant)
        assert st == (la.ATTN_ERR_BAD_INDEX if on else la.ATTN_OK)
        for c, s, H in zip(codes, scales, (Hq, Hkv, Hkv)):
            assert bool((c[T:] == 0x5A).all()), "a code was written past the tensor"
            assert bool((s[H * n_scale:] == -7.0).all()), "a scale was written past the array"


def test_decode_lengths_past_the_table(la):
    dd = workloads.make_decode([100, 300, 50], 8, 2, 128, num_pages=64, seed=1920).to("cuda")
    lens = torch.tensor([100, 300 + 16 * 64, 50], dtype=torch.int32, device="cuda")   # beyond max_pages * 16

    def dec():
        la.attn_decode_paged(dd.q, dd.k_cache, dd.v_cache, dd.block_table, lens)
    assert with_validation(la, True, dec) == la.ATTN_ERR_BAD_INDEX
    assert with_validation(la, False, dec) == la.ATTN_OK


@pytest.mark.parametrize("bad", sorted(BAD_CU))
def test_fp8_forward_packed(la, bad):
    T, Hq, Hkv, d = 500, 4, 2, 128
    cu_ok = torch.tensor([0, 100, 300, 500], dtype=torch.int32, device="cuda")
    cu_bad = torch.tensor(BAD_CU[bad], dtype=torch.int32, device="cuda")
    q8, qs = la.attn_quantize_fp8(workloads.randn_bf16((T, Hq, d), seed=1930).cuda(), cu_seqlens=cu_ok)
    k8, ks = la.attn_quantize_fp8(workloads.randn_bf16((T, Hkv, d), seed=1931).cuda(), cu_seqlens=cu_ok)
    v8, vs = la.attn_quantize_fp8(workloads.randn_bf16((T, Hkv, d), seed=1932).cuda(), cu_seqlens=cu_ok)
    for cq, ck in ((cu_bad, cu_ok), (cu_ok, cu_bad)):
        def fwd():
            la.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True, cu_seqlens_q=cq, cu_seqlens_k=ck)
        assert with_validation(la, True, fwd) == la.ATTN_ERR_BAD_INDEX
        assert with_validation(la, False, fwd) == la.ATTN_OK
