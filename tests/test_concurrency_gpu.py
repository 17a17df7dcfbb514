"""Calls from several host threads, each on its own stream, at the same time.

A serving process overlaps prefill, decode and training work on separate
streams, often from separate threads.  The library's host state is a
thread-local error message, a mutex-guarded device-info cache and atomic
launch-attribute flags; its kernels share nothing but the device error word.
Four threads each loop over one call (prefill, paged decode, backward, and
the 8-bit path: quantization of q, k, v then the 8-bit forward) on their own
stream, and every result must equal a single-threaded reference bit for bit
(the kernels are deterministic)."""
import threading

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    import exact_io_aware_04_gb300 as m
    m.build()
    torch.cuda.set_device(0)
    yield m
    assert m.attn_get_device_status() == 0


def test_four_threads_four_streams(la):
    p = workloads.make_prefill(2, 16, 4, 700, 900, 128, causal=True, seed=1800).to("cuda")
    q = p.q.view(2, 700, 16, 128)
    k = p.k.view(2, 900, 4, 128)
    v = p.v.view(2, 900, 4, 128)
    g = workloads.randn_bf16(tuple(q.shape), seed=1801).cuda()
    dd = workloads.make_decode([300, 2000, 17, 900, 4096, 1], 32, 8, 128, num_pages=700, seed=1802,
                               nan_fill_unused=True).to("cuda")
    scale = 128 ** -0.5

    def prefill():
        return la.attn_fwd(q, k, v, causal=True, scale=scale)

    def decode():
        return la.attn_decode_paged(dd.q, dd.k_cache, dd.v_cache, dd.block_table, dd.seq_lens)

    out0, lse0 = prefill()

    def backward():
        return la.attn_bwd(q, k, v, out0, lse0, g, causal=True, scale=scale)

    def fp8():
        (q8, qs), (k8, ks), (v8, vs) = la.attn_quantize_fp8_qkv(q, k, v)
        o, l = la.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True, scale=scale)
        return q8, qs, k8, ks, v8, vs, o, l

    calls = {"prefill": prefill, "decode": decode, "backward": backward, "fp8": fp8}
    refs = {name: [t.clone() for t in fn()] for name, fn in calls.items()}
    torch.cuda.synchronize()
    errors = []

    def worker(name):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for it in range(25):
                    got = calls[name]()
                    s.synchronize()
                    for a, b in zip(got, refs[name]):
                        if not torch.equal(a, b):
                            errors.append(f"{name} iteration {it} differs")
                            return
        except Exception as e:   # reported by the main thread
            errors.append(f"{name}: {type(e).__name__}: {e}")

    threads = [threading.Thread(target=worker, args=(n,)) for n in calls]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker did not finish"
    assert not errors, errors
