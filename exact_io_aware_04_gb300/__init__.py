"""libattn: exact scaled dot-product attention on one GB300 (sm_103a).

This package is a thin binding over the C ABI declared in include/attn.h: it
marshals torch tensors (device memory, streams) into pointers and sizes and
calls the shared library; every step of the computation runs in the library's
CUDA kernels.  There is no CPU path: without the built library, or without a
CUDA device, the calls raise.

    out, lse = attn_fwd(q, k, v, causal=True)                       # dense THD/BSHD
    out, lse = attn_fwd(q, k, v, causal=True, cu_seqlens_q=cq, cu_seqlens_k=ck)
    dq, dk, dv = attn_bwd(q, k, v, out, lse, dout, causal=True)
    (q8, qs), (k8, ks), (v8, vs) = attn_quantize_fp8_qkv(q, k, v)  # one launch
    out, lse = attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True)
    out, lse = attn_decode_paged(q, k_cache, v_cache, block_table, seq_lens)
    out, lse = attn_decode_kvcache(q, k_cache, v_cache, block_table, seq_lens, k_new=kn, v_new=vn)
"""
from ._binding import (  # noqa: F401
    ATTN_ERR_BAD_INDEX,
    ATTN_ERR_CUDA,
    ATTN_ERR_INVALID_ARG,
    ATTN_ERR_TIMEOUT,
    ATTN_ERR_UNSUPPORTED,
    ATTN_OK,
    AttnError,
    attn_bwd,
    attn_decode_kvcache,
    attn_decode_kvcache_workspace_size,
    attn_decode_paged,
    attn_decode_paged_noalloc,
    attn_decode_workspace_size,
    attn_quantize_fp8,
    attn_quantize_fp8_qkv,
    attn_fp8_scale_count,
    attn_fwd,
    attn_fwd_fp8,
    attn_get_device_status,
    attn_set_validation,
    attn_status_string,
    build,
    lib,
    lib_path,
)
