"""ctypes binding of libattn (include/attn.h): argument marshalling only."""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

from . import _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_CUDA = -3
ATTN_ERR_TIMEOUT = -4
ATTN_ERR_BAD_INDEX = -5

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class AttnError(RuntimeError):
    """A libattn call returned a non-OK status."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


def build(force: bool = False) -> str:
    """Compile libattn.so in-tree (nvcc, sm_103a)."""
    return _build.build(force=force)


def lib_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"libattn is not built ({path} missing); call "
                                   "exact_io_aware_04_gb300.build() first")
            L = ctypes.CDLL(path)
            P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, P, P, P]
            L.attn_fwd.restype = I
            L.attn_fwd_window.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, P, P, P]
            L.attn_fwd_window.restype = I
            L.attn_decode_paged.argtypes = [P, P, P, P, I, P, P, P, I, I, I, I, I, I, F, I, P, Z, P]
            L.attn_decode_paged.restype = I
            L.attn_decode_workspace_size.argtypes = [I, I, I, I, I, I, I]
            L.attn_decode_workspace_size.restype = Z
            L.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, P, P, P, Z, P]
            L.attn_bwd.restype = I
            L.attn_bwd_workspace_size.argtypes = [I, I, I, I]
            L.attn_bwd_workspace_size.restype = Z
            L.attn_decode_kvcache.argtypes = [P, P, P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, F, I, I, P, Z, P]
            L.attn_decode_kvcache.restype = I
            L.attn_decode_kvcache_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
            L.attn_decode_kvcache_workspace_size.restype = Z
            L.attn_fp8_scale_count.argtypes = [I, I]
            L.attn_fp8_scale_count.restype = Z
            L.attn_quantize_fp8.argtypes = [P, P, P, I, I, I, I, P, P]
            L.attn_quantize_fp8.restype = I
            L.attn_quantize_fp8_qkv.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, P]
            L.attn_quantize_fp8_qkv.restype = I
            L.attn_fwd_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, P, P, P]
            L.attn_fwd_fp8.restype = I
            L.attn_fwd_fp8_window.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, P, P, P]
            L.attn_fwd_fp8_window.restype = I
            L.attn_get_device_status.argtypes = [P]
            L.attn_get_device_status.restype = I
            L.attn_set_validation.argtypes = [I]
            L.attn_set_validation.restype = I
            L.attn_status_string.argtypes = [I]
            L.attn_status_string.restype = ctypes.c_char_p
            L.attn_last_error_message.argtypes = []
            L.attn_last_error_message.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _status_name(status: int) -> str:
    try:
        return lib().attn_status_string(status).decode()
    except Exception:
        return f"status {status}"


def _check(status: int):
    if status != ATTN_OK:
        raise AttnError(status, lib().attn_last_error_message().decode())


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, name: str, dtype):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libattn has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, causal: bool,
             scale: Optional[float] = None, window: Optional[tuple] = None,
             cu_seqlens_q: Optional[torch.Tensor] = None, cu_seqlens_k: Optional[torch.Tensor] = None,
             out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, stream=None):
    """Prefill forward.  Returns (out, lse).

    Dense: q [B, Nq, Hq, d] and k/v [B, Nk, Hkv, d] (or the flattened
    [B*N, H, d] with B given by a 4-D tensor only).  Packed: q [T_q, Hq, d],
    k/v [T_k, Hkv, d] with int32 cu_seqlens_q/k of B+1 entries.
    lse is [B, Hq, Nq] (dense) or [Hq, T_q] (packed), fp32.
    window = (left, right) selects the local band mask (attn_fwd_window);
    -1 leaves a side unbounded."""
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16)
    _need(v, "v", torch.bfloat16)
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    d = int(q.shape[-1])
    Hq, Hkv = int(q.shape[-2]), int(k.shape[-2])
    if cu_seqlens_q is not None or cu_seqlens_k is not None:
        if cu_seqlens_q is None or cu_seqlens_k is None:
            raise ValueError("give both cu_seqlens or neither")
        _need(cu_seqlens_q, "cu_seqlens_q", torch.int32)
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int32)
        if q.dim() != 3 or k.dim() != 3:
            raise ValueError("packed mode takes q [T_q, Hq, d] and k/v [T_k, Hkv, d]")
        B = int(cu_seqlens_q.numel()) - 1
        if int(cu_seqlens_k.numel()) != B + 1:
            raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B+1 entries")
        Nq, Nk = int(q.shape[0]), int(k.shape[0])
        lse_shape = (Hq, Nq)
    else:
        if q.dim() != 4 or k.dim() != 4:
            raise ValueError("dense mode takes q [B, Nq, Hq, d] and k/v [B, Nk, Hkv, d]")
        B, Nq, Nk = int(q.shape[0]), int(q.shape[1]), int(k.shape[1])
        if int(k.shape[0]) != B:
            raise ValueError("q and k must have the same batch size")
        lse_shape = (B, Hq, Nq)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16)
    _need(lse, "lse", torch.float32)
    if out.shape != q.shape or tuple(lse.shape) != tuple(lse_shape):
        raise ValueError("out/lse have the wrong shape")
    if window is None:
        _check(lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                              float(scale), 1 if causal else 0, _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                              _stream_handle(stream)))
    else:
        left, right = (int(x) for x in window)
        _check(lib().attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                                     float(scale), 1 if causal else 0, left, right, _ptr(cu_seqlens_q),
                                     _ptr(cu_seqlens_k), _stream_handle(stream)))
    return out, lse


def attn_fp8_scale_count(B: int, T: int) -> int:
    """Scale entries per head of a per-tile 8-bit tensor of T tokens in B sequences."""
    return int(lib().attn_fp8_scale_count(int(B), int(T)))


def attn_quantize_fp8(x: torch.Tensor, *, cu_seqlens: Optional[torch.Tensor] = None,
                      out: Optional[torch.Tensor] = None, scale: Optional[torch.Tensor] = None, stream=None):
    """Per-tile E4M3 quantization.  Dense: x [B, N, H, d] bf16; packed: x
    [T, H, d] with int32 cu_seqlens [B+1].  Returns (codes uint8 shaped like
    x, scales fp32 [H, attn_fp8_scale_count(B, T)])."""
    _need(x, "x", torch.bfloat16)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        if x.dim() != 3:
            raise ValueError("packed mode takes x [T, H, d]")
        B = int(cu_seqlens.numel()) - 1
        T, H, d = (int(v) for v in x.shape)
        N = T
    else:
        if x.dim() != 4:
            raise ValueError("dense mode takes x [B, N, H, d]")
        B, N, H, d = (int(v) for v in x.shape)
        T = B * N
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.zeros((H, attn_fp8_scale_count(B, T)), dtype=torch.float32, device=x.device)
    _need(out, "out", torch.uint8)
    _need(scale, "scale", torch.float32)
    _check(lib().attn_quantize_fp8(_ptr(x), _ptr(out), _ptr(scale), B, H, N, d, _ptr(cu_seqlens),
                                   _stream_handle(stream)))
    return out, scale


def attn_quantize_fp8_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *,
                          cu_seqlens_q: Optional[torch.Tensor] = None, cu_seqlens_k: Optional[torch.Tensor] = None,
                          out: Optional[tuple] = None, scales: Optional[tuple] = None, stream=None):
    """attn_quantize_fp8 of q, k and v in one launch (bit-identical to three
    calls).  Dense: q [B, Nq, Hq, d], k and v [B, Nk, Hkv, d]; packed: q
    [T_q, Hq, d], k and v [T_k, Hkv, d] with both int32 cu_seqlens.  out and
    scales, if given, are (q8, k8, v8) and (q_scale, k_scale, v_scale).
    Returns ((q8, q_scale), (k8, k_scale), (v8, v_scale))."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16)
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    if (cu_seqlens_q is None) != (cu_seqlens_k is None):
        raise ValueError("give both cu_seqlens or neither")
    if cu_seqlens_q is not None:
        _need(cu_seqlens_q, "cu_seqlens_q", torch.int32)
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int32)
        if q.dim() != 3 or k.dim() != 3:
            raise ValueError("packed mode takes q [T_q, Hq, d] and k, v [T_k, Hkv, d]")
        B = int(cu_seqlens_q.numel()) - 1
        if int(cu_seqlens_k.numel()) - 1 != B:
            raise ValueError("cu_seqlens_q and cu_seqlens_k must describe the same batch")
        Nq, Hq, d = (int(x) for x in q.shape)
        Nk, Hkv = int(k.shape[0]), int(k.shape[1])
        Tq, Tk = Nq, Nk
    else:
        if q.dim() != 4 or k.dim() != 4:
            raise ValueError("dense mode takes q [B, Nq, Hq, d] and k, v [B, Nk, Hkv, d]")
        B, Nq, Hq, d = (int(x) for x in q.shape)
        if int(k.shape[0]) != B:
            raise ValueError("q and k must have the same batch")
        Nk, Hkv = int(k.shape[1]), int(k.shape[2])
        Tq, Tk = B * Nq, B * Nk
    if int(k.shape[-1]) != d:
        raise ValueError("q and k must have the same head_dim")
    if out is None:
        out = tuple(torch.empty(x.shape, dtype=torch.uint8, device=x.device) for x in (q, k, v))
    if scales is None:
        scales = (torch.zeros((Hq, attn_fp8_scale_count(B, Tq)), dtype=torch.float32, device=q.device),
                  torch.zeros((Hkv, attn_fp8_scale_count(B, Tk)), dtype=torch.float32, device=q.device),
                  torch.zeros((Hkv, attn_fp8_scale_count(B, Tk)), dtype=torch.float32, device=q.device))
    for t, n in zip(out, ("q8", "k8", "v8")):
        _need(t, n, torch.uint8)
    for t, n in zip(scales, ("q_scale", "k_scale", "v_scale")):
        _need(t, n, torch.float32)
    _check(lib().attn_quantize_fp8_qkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
                                       _ptr(scales[0]), _ptr(scales[1]), _ptr(scales[2]), B, Hq, Hkv, Nq, Nk, d,
                                       _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _stream_handle(stream)))
    return (out[0], scales[0]), (out[1], scales[1]), (out[2], scales[2])


def attn_fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, v8: torch.Tensor, q_scale: torch.Tensor,
                 k_scale: torch.Tensor, v_scale: torch.Tensor, *, causal: bool, scale: Optional[float] = None,
                 cu_seqlens_q: Optional[torch.Tensor] = None, cu_seqlens_k: Optional[torch.Tensor] = None,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 window: Optional[tuple] = None, stream=None):
    """Prefill forward on per-tile E4M3 q8, k8, v8 (uint8 codes, shaped as
    attn_fwd's q, k, v; d = 64 or 128) with their fp32 tile scales from
    attn_quantize_fp8 or attn_quantize_fp8_qkv.  window = (left, right)
    selects the local band mask (attn_fwd_fp8_window).  Returns (out bf16
    shaped like q8, lse) as attn_fwd."""
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8")):
        _need(t, n, torch.uint8)
    for t, n in ((q_scale, "q_scale"), (k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, n, torch.float32)
    if k8.shape != v8.shape:
        raise ValueError("k8 and v8 must have the same shape")
    d = int(q8.shape[-1])
    Hq, Hkv = int(q8.shape[-2]), int(k8.shape[-2])
    if cu_seqlens_q is not None or cu_seqlens_k is not None:
        if cu_seqlens_q is None or cu_seqlens_k is None:
            raise ValueError("give both cu_seqlens or neither")
        _need(cu_seqlens_q, "cu_seqlens_q", torch.int32)
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int32)
        if q8.dim() != 3 or k8.dim() != 3:
            raise ValueError("packed mode takes q8 [T_q, Hq, d] and k8/v8 [T_k, Hkv, d]")
        B = int(cu_seqlens_q.numel()) - 1
        Nq, Nk = int(q8.shape[0]), int(k8.shape[0])
        lse_shape = (Hq, Nq)
        tq, tk = Nq, Nk
    else:
        if q8.dim() != 4 or k8.dim() != 4:
            raise ValueError("dense mode takes q8 [B, Nq, Hq, d] and k8/v8 [B, Nk, Hkv, d]")
        B, Nq, Nk = int(q8.shape[0]), int(q8.shape[1]), int(k8.shape[1])
        lse_shape = (B, Hq, Nq)
        tq, tk = B * Nq, B * Nk
    if tuple(q_scale.shape) != (Hq, attn_fp8_scale_count(B, tq)) or \
            tuple(k_scale.shape) != (Hkv, attn_fp8_scale_count(B, tk)) or k_scale.shape != v_scale.shape:
        raise ValueError("scales must be [heads, attn_fp8_scale_count(B, T)]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q8.shape, dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q8.device)
    _need(out, "out", torch.bfloat16)
    _need(lse, "lse", torch.float32)
    if window is None:
        _check(lib().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                                  _ptr(out), _ptr(lse), B, Hq, Hkv, Nq, Nk, d, float(scale), 1 if causal else 0,
                                  _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _stream_handle(stream)))
    else:
        left, right = (int(x) for x in window)
        _check(lib().attn_fwd_fp8_window(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale),
                                         _ptr(v_scale), _ptr(out), _ptr(lse), B, Hq, Hkv, Nq, Nk, d, float(scale),
                                         1 if causal else 0, left, right, _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                         _stream_handle(stream)))
    return out, lse


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
             dout: torch.Tensor, *, causal: bool, scale: Optional[float] = None, window: Optional[tuple] = None,
             cu_seqlens_q: Optional[torch.Tensor] = None, cu_seqlens_k: Optional[torch.Tensor] = None,
             dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, stream=None):
    """Backward of attn_fwd: returns (dq, dk, dv) for dout = dL/dout.  q, k, v,
    causal, scale, window and cu_seqlens as given to attn_fwd; out and lse are
    its outputs."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, n, torch.bfloat16)
    _need(lse, "lse", torch.float32)
    if out.shape != q.shape or dout.shape != q.shape or k.shape != v.shape:
        raise ValueError("out and dout must be shaped like q; k like v")
    d = int(q.shape[-1])
    Hq, Hkv = int(q.shape[-2]), int(k.shape[-2])
    if cu_seqlens_q is not None or cu_seqlens_k is not None:
        if cu_seqlens_q is None or cu_seqlens_k is None:
            raise ValueError("give both cu_seqlens or neither")
        _need(cu_seqlens_q, "cu_seqlens_q", torch.int32)
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int32)
        if q.dim() != 3 or k.dim() != 3:
            raise ValueError("packed mode takes q [T_q, Hq, d] and k/v [T_k, Hkv, d]")
        B = int(cu_seqlens_q.numel()) - 1
        Nq, Nk = int(q.shape[0]), int(k.shape[0])
        packed = 1
    else:
        if q.dim() != 4 or k.dim() != 4:
            raise ValueError("dense mode takes q [B, Nq, Hq, d] and k/v [B, Nk, Hkv, d]")
        B, Nq, Nk = int(q.shape[0]), int(q.shape[1]), int(k.shape[1])
        packed = 0
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    left, right = (-1, -1) if window is None else (int(x) for x in window)
    ws_bytes = int(lib().attn_bwd_workspace_size(B, Hq, Nq, packed))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _need(t, n, torch.bfloat16)
    _check(lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                          B, Hq, Hkv, Nq, Nk, d, float(scale), 1 if causal else 0, left, right,
                          _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(workspace),
                          int(workspace.numel() * workspace.element_size()), _stream_handle(stream)))
    return dq, dk, dv


def attn_decode_workspace_size(B: int, Hq: int, Hkv: int, d: int, page_size: int,
                               max_pages_per_seq: int, num_splits: int = 0) -> int:
    return int(lib().attn_decode_workspace_size(B, Hq, Hkv, d, page_size, max_pages_per_seq, num_splits))


def attn_decode_paged(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_table: torch.Tensor, seq_lens: torch.Tensor, *,
                      scale: Optional[float] = None, num_splits: int = 0,
                      out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None):
    """Paged split-KV decode.  q [B, Hq, d]; caches [num_pages, page, Hkv, d];
    block_table int32 [B, max_pages]; seq_lens int32 [B].  Returns (out, lse)
    with out [B, Hq, d] bf16 and lse [B, Hq] fp32.  The workspace (device
    scratch for the per-chunk partials) is allocated here when not given."""
    _need(q, "q", torch.bfloat16)
    _need(k_cache, "k_cache", torch.bfloat16)
    _need(v_cache, "v_cache", torch.bfloat16)
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    if k_cache.shape != v_cache.shape or k_cache.dim() != 4 or q.dim() != 3:
        raise ValueError("q [B, Hq, d]; caches [num_pages, page, Hkv, d]")
    B, Hq, d = (int(x) for x in q.shape)
    num_pages, page, Hkv = int(k_cache.shape[0]), int(k_cache.shape[1]), int(k_cache.shape[2])
    if block_table.dim() != 2 or int(block_table.shape[0]) != B or int(seq_lens.numel()) != B:
        raise ValueError("block_table [B, max_pages] and seq_lens [B] required")
    max_pages = int(block_table.shape[1])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    ws_bytes = attn_decode_workspace_size(B, Hq, Hkv, d, page, max_pages, num_splits)
    if ws_bytes == 0:
        raise AttnError(ATTN_ERR_UNSUPPORTED, "no decode plan for these sizes")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check(lib().attn_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), max_pages,
                                   _ptr(seq_lens), _ptr(out), _ptr(lse), B, Hq, Hkv, d, page, num_pages,
                                   float(scale), int(num_splits), _ptr(workspace),
                                   int(workspace.numel() * workspace.element_size()),
                                   _stream_handle(stream)))
    return out, lse


def attn_decode_kvcache_workspace_size(B: int, Nq: int, Hq: int, Hkv: int, d: int, page_size: int,
                                       max_pages_per_seq: int, num_splits: int = 0) -> int:
    return int(lib().attn_decode_kvcache_workspace_size(B, Nq, Hq, Hkv, d, page_size, max_pages_per_seq,
                                                        num_splits))


def attn_decode_kvcache(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                        block_table: torch.Tensor, seq_lens: torch.Tensor, *,
                        k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
                        causal: bool = True, scale: Optional[float] = None, num_splits: int = 0,
                        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None):
    """Nq new queries per sequence over the paged cache, with the new tokens'
    K/V appended in place first when k_new/v_new are given.  q [B, Nq, Hq, d];
    k_new/v_new [B, Nq, Hkv, d]; caches [num_pages, page, Hkv, d] (written by
    the append); seq_lens int32 [B] counts the tokens after the append.
    Returns (out [B, Nq, Hq, d] bf16, lse [B, Hq, Nq] fp32)."""
    _need(q, "q", torch.bfloat16)
    _need(k_cache, "k_cache", torch.bfloat16)
    _need(v_cache, "v_cache", torch.bfloat16)
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    if (k_new is None) != (v_new is None):
        raise ValueError("give both k_new and v_new or neither")
    if k_cache.shape != v_cache.shape or k_cache.dim() != 4 or q.dim() != 4:
        raise ValueError("q [B, Nq, Hq, d]; caches [num_pages, page, Hkv, d]")
    B, Nq, Hq, d = (int(x) for x in q.shape)
    num_pages, page, Hkv = int(k_cache.shape[0]), int(k_cache.shape[1]), int(k_cache.shape[2])
    if k_new is not None:
        _need(k_new, "k_new", torch.bfloat16)
        _need(v_new, "v_new", torch.bfloat16)
        if tuple(k_new.shape) != (B, Nq, Hkv, d) or k_new.shape != v_new.shape:
            raise ValueError("k_new/v_new must be [B, Nq, Hkv, d]")
    if block_table.dim() != 2 or int(block_table.shape[0]) != B or int(seq_lens.numel()) != B:
        raise ValueError("block_table [B, max_pages] and seq_lens [B] required")
    max_pages = int(block_table.shape[1])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    ws_bytes = attn_decode_kvcache_workspace_size(B, Nq, Hq, Hkv, d, page, max_pages, num_splits)
    if ws_bytes == 0:
        raise AttnError(ATTN_ERR_UNSUPPORTED, "no decode plan for these sizes")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    _check(lib().attn_decode_kvcache(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(block_table), max_pages, _ptr(seq_lens), _ptr(out), _ptr(lse),
                                     B, Nq, Hq, Hkv, d, page, num_pages, float(scale), 1 if causal else 0,
                                     int(num_splits), _ptr(workspace),
                                     int(workspace.numel() * workspace.element_size()), _stream_handle(stream)))
    return out, lse


def attn_get_device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error word."""
    return int(lib().attn_get_device_status(_stream_handle(stream)))


def attn_set_validation(enabled: bool) -> bool:
    return bool(lib().attn_set_validation(1 if enabled else 0))


def attn_decode_paged_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                              block_table: torch.Tensor, seq_lens: torch.Tensor, *,
                              scale: Optional[float] = None, num_splits: int = 0,
                              out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                              stream=None):
    """attn_decode_paged without a workspace: for callers that cannot
    allocate device memory at call time, the library keeps the per-chunk
    partials in its own fixed 32 MiB device array (shared by all calls, so
    calls must not overlap on the GPU).  The call runs with q's device
    current, because the array's address is taken in the current device's
    context.  Returns (out, lse)."""
    L = lib()
    f = L.attn_decode_paged_noalloc
    if f.argtypes is None:
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        f.argtypes = [P, P, P, P, I, P, P, P, I, I, I, I, I, I, F, I, P]
        f.restype = I
    _need(q, "q", torch.bfloat16)
    _need(k_cache, "k_cache", torch.bfloat16)
    _need(v_cache, "v_cache", torch.bfloat16)
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    if k_cache.shape != v_cache.shape or k_cache.dim() != 4 or q.dim() != 3:
        raise ValueError("q [B, Hq, d]; caches [num_pages, page, Hkv, d]")
    B, Hq, d = (int(x) for x in q.shape)
    num_pages, page, Hkv = int(k_cache.shape[0]), int(k_cache.shape[1]), int(k_cache.shape[2])
    if block_table.dim() != 2 or int(block_table.shape[0]) != B or int(seq_lens.numel()) != B:
        raise ValueError("block_table [B, max_pages] and seq_lens [B] required")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (block_table, "block_table"),
                 (seq_lens, "seq_lens")):
        if t.device != q.device:
            raise ValueError(f"{n} is on {t.device}, q on {q.device}")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        _check(f(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), int(block_table.shape[1]),
                 _ptr(seq_lens), _ptr(out), _ptr(lse), B, Hq, Hkv, d, page, num_pages, float(scale),
                 int(num_splits), _stream_handle(stream)))
    return out, lse
