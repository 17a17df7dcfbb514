"""The C ABI without a GPU: the library builds, loads, exports every function
include/attn.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    import exact_io_aware_04_gb300 as la
    la.build()
    return la.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "attn_decode_paged", "attn_decode_workspace_size", "attn_get_device_status",
              "attn_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libattn does not export {name}"


def test_status_strings(lib):
    for code, name in [(0, "ATTN_OK"), (-1, "ATTN_ERR_INVALID_ARG"), (-2, "ATTN_ERR_UNSUPPORTED"),
                       (-3, "ATTN_ERR_CUDA"), (-4, "ATTN_ERR_TIMEOUT"), (-5, "ATTN_ERR_BAD_INDEX")]:
        assert lib.attn_status_string(code).decode() == name


FAKE = ctypes.c_void_p(0x10000)  # 16-byte aligned, never dereferenced by host checks


def fwd(lib, q=FAKE, out=FAKE, B=1, Hq=4, Hkv=2, Nq=8, Nk=8, d=128, scale=0.1, causal=1, cq=None, ck=None):
    return lib.attn_fwd(q, FAKE, FAKE, out, FAKE, B, Hq, Hkv, Nq, Nk, d, scale, causal, cq, ck, None)


def test_fwd_host_rejections(lib):
    assert fwd(lib, q=None) == -1
    assert fwd(lib, Hq=5, Hkv=2) == -1               # Hq % Hkv
    assert fwd(lib, Hq=0) == -1
    assert fwd(lib, Hkv=-1) == -1
    assert fwd(lib, B=-1) == -1
    assert fwd(lib, scale=float("nan")) == -1
    assert fwd(lib, scale=float("inf")) == -1
    assert fwd(lib, scale=0.0) == -1
    assert fwd(lib, causal=2) == -1
    assert fwd(lib, cq=FAKE) == -1                   # only one cu_seqlens
    assert fwd(lib, out=ctypes.c_void_p(0x10008)) == -1  # misaligned
    assert fwd(lib, d=96) == -2                      # unsupported head dim
    assert fwd(lib, d=256) == -2
    assert b"Hq % Hkv" in lib.attn_last_error_message() or True
    assert fwd(lib, B=0) == 0                        # nothing to do
    assert fwd(lib, Nq=0) == 0


def test_fwd_window_host_rejections(lib):
    def w(left, right, Nq=8):
        return lib.attn_fwd_window(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 2, Nq, 8, 128, 0.1, 0, left, right,
                                   None, None, None)
    assert w(-2, 0) == -1
    assert w(0, -7) == -1
    assert w(-1, -1, Nq=0) == 0                      # valid window, nothing to do
    assert w(5, 0, Nq=0) == 0


def dec(lib, ws_bytes=1 << 30, B=2, Hq=8, Hkv=2, d=128, page=16, num_pages=10, max_pages=4, splits=0,
        scale=0.1, ws=ctypes.c_void_p(0x10000), bt=FAKE):
    return lib.attn_decode_paged(FAKE, FAKE, FAKE, bt, max_pages, FAKE, FAKE, FAKE, B, Hq, Hkv, d, page,
                                 num_pages, scale, splits, ws, ws_bytes, None)


def test_decode_host_rejections(lib):
    assert dec(lib, bt=None) == -1
    assert dec(lib, Hq=6, Hkv=4) == -1
    assert dec(lib, num_pages=0) == -1
    assert dec(lib, max_pages=0) == -1
    assert dec(lib, splits=-1) == -1
    assert dec(lib, scale=float("nan")) == -1
    assert dec(lib, ws=ctypes.c_void_p(0x10010)) == -1   # workspace must be 256-byte aligned
    assert dec(lib, ws_bytes=16) == -1                  # too small
    assert dec(lib, page=32) == -2
    assert dec(lib, d=80) == -2
    assert dec(lib, B=0) == 0


def noalloc(lib, q=FAKE, out=FAKE, B=64, Hq=32, Hkv=8, d=128, max_pages=2048, splits=64, scale=0.1):
    f = lib.attn_decode_paged_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, I, P, P, P, I, I, I, I, I, I, F, I, P]
    f.restype = I
    return f(q, FAKE, FAKE, FAKE, max_pages, FAKE, out, FAKE, B, Hq, Hkv, d, 16, 10, scale, splits, None)


def test_decode_noalloc_host_rejections(lib):
    """Argument errors come first, worded as attn_decode_paged words them; the
    fixed-array limit (32 MiB of partials) is checked only after them."""
    assert noalloc(lib, q=None) == -1
    assert b"NULL pointer" in lib.attn_last_error_message()
    assert noalloc(lib, out=ctypes.c_void_p(0x10008)) == -1
    assert b"misaligned" in lib.attn_last_error_message()
    assert noalloc(lib, Hq=30) == -1
    assert b"Hq % Hkv" in lib.attn_last_error_message()
    assert noalloc(lib, d=96) == -2
    # valid arguments whose partials need about 64.5 MiB: rejected by the limit
    assert lib.attn_decode_workspace_size(64, 32, 8, 128, 16, 2048, 64) > (64 << 20)
    assert noalloc(lib) == -1
    assert b"scratch" in lib.attn_last_error_message()
    assert b"smaller nonzero num_splits" in lib.attn_last_error_message()
    assert noalloc(lib, B=0, splits=16) == 0       # fits, nothing to do


def test_fp8_host_rejections(lib):
    def q(x=FAKE, x8=FAKE, sc=FAKE, B=2, H=4, N=256, d=128, cu=None):
        return lib.attn_quantize_fp8(x, x8, sc, B, H, N, d, cu, None)
    assert q(x=None) == -1
    assert q(sc=ctypes.c_void_p(0x10002)) == -1        # scales must be 4-byte aligned
    assert q(x8=ctypes.c_void_p(0x10008)) == -1        # codes must be 16-byte aligned
    assert q(H=0) == -1
    assert q(d=96) == -2
    assert q(B=0) == 0 and q(N=0) == 0                 # nothing to do

    def qkv(q=FAKE, k=FAKE, q8=FAKE, ks=FAKE, B=2, Hq=4, Hkv=2, Nq=256, Nk=256, d=128, cq=None, ck=None):
        return lib.attn_quantize_fp8_qkv(q, k, FAKE, q8, FAKE, FAKE, FAKE, ks, FAKE, B, Hq, Hkv, Nq, Nk, d, cq, ck,
                                         None)
    assert qkv(q=None) == -1 and qkv(q8=None) == -1
    assert qkv(k=None) == -1                           # K needed when keys exist
    assert qkv(k=None, ks=None, Nk=0, B=0) == 0        # no keys: K/V and their scales may be NULL
    assert qkv(ks=ctypes.c_void_p(0x10002)) == -1      # scales must be 4-byte aligned
    assert qkv(k=ctypes.c_void_p(0x10008)) == -1       # tensors must be 16-byte aligned
    assert qkv(cq=FAKE) == -1                          # both cu_seqlens or neither
    assert qkv(Hkv=0) == -1 and qkv(Nq=-1) == -1
    assert qkv(d=96) == -2
    assert qkv(B=0) == 0 and qkv(Nq=0, Nk=0) == 0      # nothing to do

    def f(q8=FAKE, k8=FAKE, ks=FAKE, B=1, Hq=4, Hkv=2, Nq=8, Nk=8, d=128, causal=1, cq=None, ck=None):
        return lib.attn_fwd_fp8(q8, k8, FAKE, FAKE, ks, FAKE, FAKE, FAKE, B, Hq, Hkv, Nq, Nk, d, 0.1, causal, cq,
                                ck, None)
    assert f(q8=None) == -1
    assert f(ks=None) == -1                            # K scales needed when keys exist
    assert f(ks=None, k8=None, Nk=0, B=0) == 0         # no keys: K/V and their scales may be NULL
    assert f(Hq=5) == -1
    assert f(causal=3) == -1
    assert f(cq=FAKE) == -1
    assert f(d=96) == -2                               # the 8-bit forward is built for d = 64 and 128
    assert f(B=0) == 0
    # scale entries: T // 128 + B per head
    assert lib.attn_fp8_scale_count(2, 512) == 6 and lib.attn_fp8_scale_count(16, 8192) == 80
    assert lib.attn_fp8_scale_count(-1, 5) == 0

    def w(left, right, B=1, d=128):
        return lib.attn_fwd_fp8_window(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, 4, 2, 8, 8, d, 0.1, 0,
                                       left, right, None, None, None)
    assert w(-2, 5) == -1 and w(5, -3) == -1          # window sides below -1
    assert w(5, 5, d=96) == -2
    assert w(5, 5, B=0) == 0 and w(-1, -1, B=0) == 0


def bwd(lib, B=1, Hq=4, Hkv=2, Nq=8, Nk=8, d=128, causal=1, wl=-1, wr=-1, ws=ctypes.c_void_p(0x100000),
        ws_bytes=1 << 20, dout=FAKE):
    return lib.attn_bwd(FAKE, FAKE, FAKE, FAKE, dout, FAKE, FAKE, FAKE, FAKE, B, Hq, Hkv, Nq, Nk, d, 0.1, causal,
                        wl, wr, None, None, ws, ws_bytes, None)


def test_bwd_host_rejections(lib):
    assert bwd(lib, dout=None) == -1
    assert bwd(lib, Hq=5) == -1
    assert bwd(lib, causal=3) == -1
    assert bwd(lib, wl=-2) == -1
    assert bwd(lib, ws=None) == -1
    assert bwd(lib, ws=ctypes.c_void_p(0x100010)) == -1      # workspace not 256-byte aligned
    assert bwd(lib, ws_bytes=16, Nq=4096) == -1              # workspace too small
    assert bwd(lib, d=96) == -2
    assert bwd(lib, B=0) == 0
    # per head: 4*ceil(T_q/4) + 4*B + 132 floats, for lse*log2(e) and for D
    assert lib.attn_bwd_workspace_size(4, 16, 4096, 0) == 2 * 16 * (16384 + 16 + 132) * 4
    assert lib.attn_bwd_workspace_size(1, 3, 5, 1) == 3584   # 2*3*(8+4+132)*4 = 3456, rounded to 256
    assert lib.attn_bwd_workspace_size(1, 0, 5, 0) == 0


def kvc(lib, B=2, Nq=4, Hq=8, Hkv=2, causal=1, kn=FAKE, vn=FAKE, ws_bytes=1 << 30):
    return lib.attn_decode_kvcache(FAKE, kn, vn, FAKE, FAKE, FAKE, 4, FAKE, FAKE, FAKE, B, Nq, Hq, Hkv, 128, 16,
                                   10, 0.1, causal, 0, ctypes.c_void_p(0x100000), ws_bytes, None)


def test_decode_kvcache_host_rejections(lib):
    assert kvc(lib, Nq=0) == -1
    assert kvc(lib, kn=None) == -1                    # only one of k_new / v_new
    assert kvc(lib, causal=2) == -1
    assert kvc(lib, Hq=7) == -1                       # Hq % Hkv
    assert kvc(lib, Hq=64, Hkv=2, Nq=5) == -2         # 160 query rows per K/V head
    assert kvc(lib, ws_bytes=16) == -1
    assert kvc(lib, B=0) == 0
    assert kvc(lib, B=0, kn=None, vn=None) == 0
    # the workspace grows with Nq; Nq = 1 matches attn_decode_paged's
    one = lib.attn_decode_kvcache_workspace_size(64, 1, 32, 8, 128, 16, 2048, 0)
    assert one == lib.attn_decode_workspace_size(64, 32, 8, 128, 16, 2048, 0)
    # at least one chunk's partial (d floats) and lse per (sequence, head, query) row
    assert lib.attn_decode_kvcache_workspace_size(64, 4, 32, 8, 128, 16, 2048, 0) >= 64 * 32 * 4 * (128 * 4 + 4)
    assert lib.attn_decode_kvcache_workspace_size(64, 0, 32, 8, 128, 16, 2048, 0) == 0


def test_workspace_size(lib):
    f = lib.attn_decode_workspace_size
    assert f(2, 8, 2, 128, 16, 4, 0) > 0
    assert f(2, 8, 2, 128, 16, 4, 0) % 256 == 0
    assert f(2, 8, 2, 128, 32, 4, 0) == 0          # unsupported page size
    assert f(2, 8, 3, 128, 16, 4, 0) == 0          # Hq % Hkv
    # more splits never needs less room
    assert f(64, 32, 8, 128, 16, 2048, 64) >= f(64, 32, 8, 128, 16, 2048, 8)
    # the paged-decode workload fits in well under a gigabyte of scratch
    assert 0 < f(64, 32, 8, 128, 16, 2048, 0) < (1 << 30)


def test_validation_switch(lib):
    prev = lib.attn_set_validation(1)
    assert lib.attn_set_validation(prev) == 1


def test_python_binding_refuses_cpu_tensors():
    import torch
    import exact_io_aware_04_gb300 as la
    q = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        la.attn_fwd(q, q, q, causal=True)


def test_header_is_plain_c(tmp_path):
    """include/attn.h compiles as C99 with warnings as errors, and a C caller
    of the prefill and decode entry points type-checks against it."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(
        '#include <stddef.h>\n#include "attn.h"\n'
        "attn_status call(const void* q, const void* k, const void* v, void* out, float* lse, void* s,\n"
        "                 const int* bt, const int* lens, void* ws, size_t ws_bytes) {\n"
        "    attn_status st = attn_fwd(q, k, v, out, lse, 2, 32, 8, 1024, 1024, 128, 0.0884f, 1, NULL, NULL, s);\n"
        "    if (st != ATTN_OK) return st;\n"
        "    return attn_decode_paged(q, k, v, bt, 64, lens, out, lse, 2, 32, 8, 128, 16, 1000, 0.0884f, 0,\n"
        "                             ws, ws_bytes, s);\n"
        "}\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I",
                        os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
