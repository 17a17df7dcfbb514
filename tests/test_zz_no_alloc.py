"""attn_decode_paged_noalloc: the decode entry point for callers that cannot
allocate device memory at call time (a plug-in whose host runtime owns all
device allocations, or a loop that must never call cudaMalloc/cudaFree).  It
keeps its per-chunk partials in the library's own fixed 32 MiB device array.

Checked through the C ABI against attn_decode_paged (caller workspace) on two
calls in a row, with the tolerance of the other parity tests; the second call
runs over the first call's leftovers in the shared array.  This file is
collected last so a run that stops at the first failure has run every other
test already; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

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


def noalloc_call(la, d, num_splits=0):
    """Direct C-ABI call of attn_decode_paged_noalloc (no workspace argument)."""
    L = la.lib()
    f = L.attn_decode_paged_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, I, P, P, P, I, I, I, I, I, I, F, I, P]
    f.restype = I
    g = d.to("cuda")
    out = torch.empty_like(g.q)
    lse = torch.empty((d.B, d.Hq), dtype=torch.float32, device="cuda")
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    st = f(ptr(g.q), ptr(g.k_cache), ptr(g.v_cache), ptr(g.block_table), int(g.block_table.shape[1]),
           ptr(g.seq_lens), ptr(out), ptr(lse), d.B, d.Hq, d.Hkv, d.d, d.page_size, d.num_pages, float(d.scale),
           int(num_splits), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out, lse


def reference_call(la, d, num_splits=0):
    g = d.to("cuda")
    return la.attn_decode_paged(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, scale=d.scale,
                                num_splits=num_splits)


def test_noalloc_matches_workspace_entry_point_on_two_calls(la):
    first = workloads.make_decode([4000, 17, 1, 2500, 33, 900], 32, 8, 128, num_pages=900, seed=41,
                                  nan_fill_unused=True)
    second = workloads.make_decode([64, 3000, 15, 1200], 16, 2, 64, num_pages=600, seed=42,
                                   nan_fill_unused=True)
    for d in (first, second):   # two calls in a row through the shared array
        st, out, lse = noalloc_call(la, d)
        assert st == 0, la.lib().attn_last_error_message().decode()
        ref_out, ref_lse = reference_call(la, d)
        torch.cuda.synchronize()
        assert_close(d.name, out.float().cpu().numpy().reshape(-1, d.d), lse.cpu().numpy().reshape(-1),
                     ref_out.double().cpu().numpy().reshape(-1, d.d), ref_lse.double().cpu().numpy().reshape(-1))
        assert torch.isfinite(out.float()).all()


def test_noalloc_rejects_sizes_beyond_its_array(la):
    # the full paged-decode workload's automatic plan needs about 64.5 MiB of scratch
    need = la.attn_decode_workspace_size(64, 32, 8, 128, 16, 2048, 0)
    assert need > (32 << 20)
    d = workloads.make_decode([16] * 64, 32, 8, 128, num_pages=64, seed=3, max_pages=2048)
    st, out, lse = noalloc_call(la, d)
    assert st == la.ATTN_ERR_INVALID_ARG
    assert b"scratch" in la.lib().attn_last_error_message()
    # a coarser page range fits and runs
    st, out, lse = noalloc_call(la, d, num_splits=16)
    assert st == 0
    ref_out, ref_lse = reference_call(la, d, num_splits=16)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
