"""attn_decode_paged_noalloc: the decode entry point for callers that cannot
allocate device memory at call time (a plug-in whose host runtime owns all
device allocations, or a loop that must never call cudaMalloc/cudaFree).  It
keeps its per-chunk partials in the library's own fixed 32 MiB device array.

Checked through the C ABI on two calls in a row, against attn_decode_paged
(caller workspace) and against the fp64 oracle, with the tolerance of the
other parity tests; the second call runs over the first call's leftovers in
the shared array.  Once the library's device code is loaded, a call changes
neither torch's allocated bytes nor the device's free memory.  This file is
collected last so a run that stops at the first failure has run every other
test already; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_close

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def la():
    import exact_io_aware_04_gb300 as m
    m.build()
    torch.cuda.set_device(0)
    yield m
    assert m.attn_get_device_status() == 0


def noalloc_call(la, g, out, lse, num_splits=0):
    """Direct C-ABI call of attn_decode_paged_noalloc (no workspace argument)
    on device-resident inputs g and preallocated out/lse."""
    f = la.lib().attn_decode_paged_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, I, P, P, P, I, I, I, I, I, I, F, I, P]
    f.restype = I
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    return f(ptr(g.q), ptr(g.k_cache), ptr(g.v_cache), ptr(g.block_table), int(g.block_table.shape[1]),
             ptr(g.seq_lens), ptr(out), ptr(lse), g.B, g.Hq, g.Hkv, g.d, g.page_size, g.num_pages, float(g.scale),
             int(num_splits), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def reference_call(la, g, num_splits=0):
    return la.attn_decode_paged(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, scale=g.scale,
                                num_splits=num_splits)


def memory_state():
    torch.cuda.synchronize()
    return torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]


def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls(la):
    first = workloads.make_decode([4000, 17, 1, 2500, 33, 900], 32, 8, 128, num_pages=900, seed=41,
                                  nan_fill_unused=True)
    second = workloads.make_decode([64, 3000, 15, 1200], 16, 2, 64, num_pages=600, seed=42,
                                   nan_fill_unused=True)
    for i, d in enumerate((first, second)):   # two calls in a row through the shared array
        g = d.to("cuda")
        out = torch.empty_like(g.q)
        lse = torch.empty((d.B, d.Hq), dtype=torch.float32, device="cuda")
        before = memory_state()
        st = noalloc_call(la, g, out, lse)
        after = memory_state()
        assert st == 0, la.lib().attn_last_error_message().decode()
        if i == 1:   # the library's device code is loaded by now: nothing is allocated
            assert after == before, (before, after)
        got_o = out.float().cpu().numpy().reshape(-1, d.d)
        got_l = lse.cpu().numpy().reshape(-1)
        ref_out, ref_lse = reference_call(la, g)
        assert_close(d.name + " vs attn_decode_paged", got_o, got_l,
                     ref_out.double().cpu().numpy().reshape(-1, d.d), ref_lse.double().cpu().numpy().reshape(-1))
        o_star, l_star = oracle.decode(d)
        assert_close(d.name + " vs oracle", got_o, got_l, o_star, l_star)


def test_noalloc_python_wrapper(la):
    d = workloads.make_decode([700, 5, 130], 8, 2, 128, num_pages=80, seed=43, nan_fill_unused=True)
    g = d.to("cuda")
    out, lse = la.attn_decode_paged_noalloc(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, scale=d.scale)
    torch.cuda.synchronize()
    o_star, l_star = oracle.decode(d)
    assert_close(d.name, out.float().cpu().numpy().reshape(-1, d.d), lse.cpu().numpy().reshape(-1), o_star, l_star)


def test_noalloc_rejects_sizes_beyond_its_array(la):
    d = workloads.make_decode([16] * 64, 32, 8, 128, num_pages=64, seed=3, max_pages=2048)
    g = d.to("cuda")
    out = torch.empty_like(g.q)
    lse = torch.empty((d.B, d.Hq), dtype=torch.float32, device="cuda")
    # 64 chunks per sequence: 64 * 32 rows * 64 chunks of 129 floats, about 64.5 MiB
    assert la.attn_decode_workspace_size(64, 32, 8, 128, 16, 2048, 64) > 2 * SCRATCH_BYTES
    assert noalloc_call(la, g, out, lse, num_splits=64) == la.ATTN_ERR_INVALID_ARG
    assert b"scratch" in la.lib().attn_last_error_message()
    # eight query heads per K/V head under the automatic plan: also about 64.5 MiB
    wide = workloads.make_decode([16] * 64, 64, 8, 128, num_pages=64, seed=4, max_pages=2048)
    assert la.attn_decode_workspace_size(64, 64, 8, 128, 16, 2048, 0) > 2 * SCRATCH_BYTES
    gw = wide.to("cuda")
    assert noalloc_call(la, gw, torch.empty_like(gw.q), torch.empty((64, 64), dtype=torch.float32,
                                                                      device="cuda")) == la.ATTN_ERR_INVALID_ARG
    # a smaller nonzero num_splits (fewer, longer chunks) fits and runs
    assert la.attn_decode_workspace_size(64, 32, 8, 128, 16, 2048, 16) <= SCRATCH_BYTES
    assert noalloc_call(la, g, out, lse, num_splits=16) == 0
    ref_out, ref_lse = reference_call(la, g, num_splits=16)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    o_star, l_star = oracle.decode(d)
    assert_close(d.name, out.float().cpu().numpy().reshape(-1, d.d), lse.cpu().numpy().reshape(-1), o_star, l_star)
