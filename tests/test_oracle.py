"""Pins for the fp64 oracle: checked against what the pages print and what the
mathematics fixes, never against itself.

Each pin is chosen so that a plausible mistake in the oracle fails it: a wrong
mask corner (keep matrices), a wrong head map (GQA lists), a missing max shift
(shift by +-1000), a wrong normaliser or lse (printed l values), a wrong
sequence offset (varlen vs per-sequence), a wrong page gather (paged vs
gathered-dense), a transposed operand or dropped term (SDPA comparison).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def one_row_problem(scores, values):
    """q = [1, 0], k_j = [s_j, 0] so that q.k_j = s_j exactly (scale 1)."""
    n = len(scores)
    dv = len(values[0])
    d = max(2, dv)
    q = torch.zeros(1, 1, d)
    q[0, 0, 0] = 1.0
    k = torch.zeros(n, 1, d)
    k[:, 0, 0] = torch.tensor(scores)
    v = torch.zeros(n, 1, d)
    v[:, 0, :dv] = torch.tensor(values)
    return bf16(q), bf16(k), bf16(v), d


def run_one_row(scores, values, causal=False):
    q, k, v, d = one_row_problem(scores, values)
    out, lse = oracle.prefill_rows(q, k, v, B=1, Hq=1, Hkv=1, Nq=1, Nk=len(scores), scale=1.0,
                                   causal=causal, rows=[[0, 0, 0]])
    return out[0, : len(values[0])], lse[0]


# ---------------------------------------------------------------------------
# printed worked examples
# ---------------------------------------------------------------------------
def test_two_tile_example_printed_output():
    g = golden("two_tile_example.json")
    out, lse = run_one_row(g["scores"], g["values"])
    tol = 0.5 * 10 ** -g["printed_output_decimals"]
    assert np.abs(out - np.array(g["printed_output"])).max() <= tol


def test_two_tile_example_tile_one_state():
    g = golden("two_tile_example.json")
    t1 = g["tile_one"]
    keys = t1["keys"]
    out, lse = run_one_row([g["scores"][j] for j in keys], [g["values"][j] for j in keys])
    tol = 0.5 * 10 ** -t1["decimals"]
    l1 = math.exp(lse - t1["m"])            # normaliser relative to the tile max
    assert abs(l1 - t1["l"]) <= tol
    u1 = out * l1                           # unnormalised numerator
    assert np.abs(u1 - np.array(t1["u"])).max() <= tol


def test_two_tile_example_merge_of_tiles_equals_full():
    """Merging the two tiles' (O, lse) states reproduces the full row; the
    old state's weight relative to the new max is the printed 0.3679."""
    g = golden("two_tile_example.json")
    o1, l1 = run_one_row(g["scores"][:2], g["values"][:2])
    o2, l2 = run_one_row(g["scores"][2:], g["values"][2:])
    of, lf = run_one_row(g["scores"], g["values"])
    lse = np.logaddexp(l1, l2)
    merged = math.exp(l1 - lse) * o1 + math.exp(l2 - lse) * o2
    assert np.abs(merged - of).max() < 1e-12
    assert abs(lse - lf) < 1e-12
    # tile-one normaliser carried to the new max 3: e^(2-3) * 1.3679
    carried = math.exp(l1 - 3.0)
    assert abs(carried - g["rescale_factor_tile_two"] * g["tile_one"]["l"]) < 1e-4


def test_normaliser_example_lse():
    g = golden("normaliser_example.json")
    out, lse = run_one_row(g["scores"], [[1.0]] * 4)
    tol = 0.5 * 10 ** -g["decimals"]
    assert abs(math.exp(lse - g["final_max"]) - g["l_final"]) <= tol
    _, lse1 = run_one_row(g["blocks"][0], [[1.0]] * 2)
    assert abs(math.exp(lse1 - max(g["blocks"][0])) - g["l_block_one"]) <= tol
    assert abs(math.exp(lse1 - g["final_max"]) - g["l_block_one_rescaled"]) <= tol
    _, lse2 = run_one_row(g["blocks"][1], [[1.0]] * 2)
    assert abs(math.exp(lse2 - g["final_max"]) - g["block_two_contribution"]) <= tol


def test_shift_invariance_large_offsets():
    """Adding the same constant to every score leaves O unchanged and moves
    lse by that constant (+-1000 would overflow exp without the max shift)."""
    g = golden("two_tile_example.json")
    base_out, base_lse = run_one_row(g["scores"], g["values"])
    for shift in (-1000.0, 1000.0):
        n = len(g["scores"])
        q = torch.zeros(1, 1, 3)
        q[0, 0, 0] = 1.0
        q[0, 0, 2] = shift
        k = torch.zeros(n, 1, 3)
        k[:, 0, 0] = torch.tensor(g["scores"])
        k[:, 0, 2] = 1.0
        v = torch.zeros(n, 1, 3)
        v[:, 0, :2] = torch.tensor(g["values"])
        out, lse = oracle.prefill_rows(bf16(q), bf16(k), bf16(v), B=1, Hq=1, Hkv=1, Nq=1, Nk=n,
                                       scale=1.0, causal=False, rows=[[0, 0, 0]])
        assert np.isfinite(out).all()
        assert np.abs(out[0, :2] - base_out).max() < 1e-12
        assert abs(lse[0] - (base_lse + shift)) < 1e-9


def test_empty_rows_and_single_key_rows():
    """Nq > Nk under the bottom-right corner: early rows have no key (zero
    output, lse -inf); the first non-empty row sees key 0 only and returns v_0."""
    q = bf16(torch.randn(5, 1, 4))
    k = bf16(torch.randn(2, 1, 4))
    v = bf16(torch.randn(2, 1, 4))
    rows = [[0, 0, i] for i in range(5)]
    out, lse = oracle.prefill_rows(q, k, v, B=1, Hq=1, Hkv=1, Nq=5, Nk=2, scale=0.5,
                                   causal=True, rows=rows)
    assert (out[:3] == 0).all()
    assert np.isneginf(lse[:3]).all()
    assert np.array_equal(out[3], v[0, 0].double().numpy())
    assert lse[3] == pytest.approx(0.5 * float((q[3, 0].double() * k[0, 0].double()).sum()), abs=1e-12)


# ---------------------------------------------------------------------------
# mask corner and head map, read off the oracle's outputs
# ---------------------------------------------------------------------------
def keep_matrix(nq, nk, causal, window=(-1, -1)):
    """Q = 0, V = identity on keys: O[i, c] > 0 exactly when key c is allowed."""
    d = max(nk, 2)
    q = torch.zeros(nq, 1, d)
    k = torch.zeros(nk, 1, d)
    v = torch.zeros(nk, 1, d)
    for j in range(nk):
        v[j, 0, j] = 1.0
    out, lse = oracle.prefill_rows(bf16(q), bf16(k), bf16(v), B=1, Hq=1, Hkv=1, Nq=nq, Nk=nk,
                                   scale=1.0, causal=causal, rows=[[0, 0, i] for i in range(nq)],
                                   window=window)
    keep = (out[:, :nk] > 0).astype(int)
    # each allowed key carries weight 1/|A_i| exactly; lse = ln|A_i|
    for i in range(nq):
        cnt = keep[i].sum()
        if cnt:
            assert np.allclose(out[i, :nk][keep[i] == 1], 1.0 / cnt, atol=1e-15)
            assert lse[i] == pytest.approx(math.log(cnt), abs=1e-12)
        else:
            assert np.isneginf(lse[i])
    return keep.tolist()


def test_bottom_right_keep_matrices():
    g = golden("causal_keep.json")
    for case in g["bottom_right"]:
        assert keep_matrix(case["q"], case["k"], causal=True) == case["keep"]
    # the oracle does not use the top-left corner
    for case in g["top_left"]:
        assert keep_matrix(case["q"], case["k"], causal=True) != case["keep"]
    assert keep_matrix(2, 5, causal=False) == [[1] * 5] * 2


def test_local_window_special_cases():
    """The local window reduces to masks fixed elsewhere: no window is the full
    matrix, right = 0 alone is the printed bottom-right causal corner, (0, 0)
    keeps only the corner diagonal key, and a window wider than the keys
    changes nothing."""
    g = golden("local_window.json")
    printed = {(c["q"], c["k"]): c["keep"] for c in golden("causal_keep.json")["bottom_right"]}
    for nq, nk in g["shapes"]:
        full = [[1] * nk for _ in range(nq)]
        corner = keep_matrix(nq, nk, causal=True)
        diag = [[int(j == i + nk - nq) for j in range(nk)] for i in range(nq)]
        want = {"full": full, "bottom_right_causal": corner, "diagonal": diag}
        for red in g["reductions"]:
            got = keep_matrix(nq, nk, causal=red["causal"], window=tuple(red["window"]))
            assert got == want[red["equals"]], (nq, nk, red)
        if (nq, nk) in printed:
            assert keep_matrix(nq, nk, causal=False, window=(-1, 0)) == printed[(nq, nk)]
        wide = nq + nk
        assert keep_matrix(nq, nk, causal=False, window=(wide, wide)) == full
        assert keep_matrix(nq, nk, causal=True, window=(wide, wide)) == corner


def test_local_window_sides_compose_and_grow_by_one_key():
    """Each side acts alone: the (left, right) set is the intersection of the
    (left, -1) and (-1, right) sets (and of the causal set when causal), and
    widening one side by one adds exactly the single key just outside it."""
    for nq, nk in [(5, 9), (9, 5), (7, 7), (1, 6)]:
        for left in range(0, 5):
            for right in range(0, 5):
                both = np.array(keep_matrix(nq, nk, False, (left, right)))
                lonly = np.array(keep_matrix(nq, nk, False, (left, -1)))
                ronly = np.array(keep_matrix(nq, nk, False, (-1, right)))
                assert (both == (lonly & ronly)).all()
                caus = np.array(keep_matrix(nq, nk, True, (left, right)))
                assert (caus == (both & np.array(keep_matrix(nq, nk, True)))).all()
                wider_l = np.array(keep_matrix(nq, nk, False, (left + 1, right)))
                wider_r = np.array(keep_matrix(nq, nk, False, (left, right + 1)))
                dl, dr = wider_l - both, wider_r - both
                assert dl.min() >= 0 and dr.min() >= 0
                for i in range(nq):
                    assert dl[i].sum() <= 1 and dr[i].sum() <= 1
                    if dl[i].sum():   # the added key sits just left of the row's leftmost kept key
                        j = int(np.argmax(dl[i]))
                        assert both[i, j + 1: j + 2].tolist() == [1] or not both[i].any()
                        assert not both[i, :j + 1].any()
                    if dr[i].sum():
                        j = int(np.argmax(dr[i]))
                        assert not both[i, j:].any()


def test_gqa_head_map():
    g = golden("gqa_map.json")
    for case in g["cases"]:
        hq, hkv = case["q_heads"], case["kv_heads"]
        nk, d = 3, 2
        q = torch.zeros(1, hq, d)
        k = torch.zeros(nk, hkv, d)
        v = torch.zeros(nk, hkv, d)
        for gh in range(hkv):
            v[:, gh, :] = float(gh + 1)
        out, _ = oracle.prefill_rows(bf16(q), bf16(k), bf16(v), B=1, Hq=hq, Hkv=hkv, Nq=1, Nk=nk,
                                     scale=1.0, causal=False, rows=[[0, h, 0] for h in range(hq)])
        got = [int(round(x)) - 1 for x in out[:, 0]]
        assert got == case["map"]
    for hq, hkv in g["rejected"]:
        with pytest.raises(ValueError):
            oracle.prefill_rows(bf16(torch.zeros(1, max(hq, 1), 2)), bf16(torch.zeros(1, hkv, 2)),
                                bf16(torch.zeros(1, hkv, 2)), B=1, Hq=hq, Hkv=hkv, Nq=1, Nk=1,
                                scale=1.0, causal=False, rows=[[0, 0, 0]])


# ---------------------------------------------------------------------------
# against a library routine: torch SDPA, fp64 MATH backend, explicit mask
# ---------------------------------------------------------------------------
def sdpa_reference(q, k, v, nq, nk, hq, hkv, scale, causal, keep=None):
    """q [nq, hq, d], k/v [nk, hkv, d] -> (out [hq, nq, d], lse [hq, nq]) in fp64.
    keep, when given, is the boolean [nq, nk] mask to use instead of the
    causal corner."""
    from torch.nn.attention import SDPBackend, sdpa_kernel
    import torch.nn.functional as F
    qd = q.double().permute(1, 0, 2)[None]
    kd = k.double().permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)[None]
    vd = v.double().permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)[None]
    if keep is None:
        keep = torch.ones(nq, nk, dtype=torch.bool)
        if causal:
            keep = torch.arange(nk)[None, :] <= torch.arange(nq)[:, None] + nk - nq
    with sdpa_kernel(SDPBackend.MATH):
        out = F.scaled_dot_product_attention(qd, kd, vd, attn_mask=keep, is_causal=False,
                                             dropout_p=0.0, scale=scale)[0]
    scores = (qd @ kd.transpose(-2, -1))[0] * scale
    lse = torch.logsumexp(scores.masked_fill(~keep, -math.inf), dim=-1)
    return out, lse, keep


@pytest.mark.parametrize("nq,nk,hq,hkv,d,causal", [
    (2, 5, 2, 2, 3, True), (5, 2, 2, 2, 3, True), (4, 4, 2, 2, 3, True),
    (7, 13, 6, 2, 8, True), (13, 7, 4, 1, 8, True), (9, 9, 4, 4, 16, False),
    (33, 70, 8, 2, 32, True),
])
def test_matches_sdpa_fp64(nq, nk, hq, hkv, d, causal):
    torch.manual_seed(nq * 100 + nk)
    q, k, v = bf16(torch.randn(nq, hq, d)), bf16(torch.randn(nk, hkv, d)), bf16(torch.randn(nk, hkv, d))
    scale = 1.0 / math.sqrt(d)
    rows = [[0, h, i] for h in range(hq) for i in range(nq)]
    out, lse = oracle.prefill_rows(q, k, v, B=1, Hq=hq, Hkv=hkv, Nq=nq, Nk=nk, scale=scale,
                                   causal=causal, rows=rows)
    ref, ref_lse, keep = sdpa_reference(q, k, v, nq, nk, hq, hkv, scale, causal)
    has_key = keep.any(dim=-1)
    for r, (_, h, i) in enumerate(rows):
        if has_key[i]:
            assert np.abs(out[r] - ref[h, i].numpy()).max() <= 1e-12
            assert abs(lse[r] - float(ref_lse[h, i])) <= 1e-12
        else:
            assert (out[r] == 0).all() and np.isneginf(lse[r])


@pytest.mark.parametrize("nq,nk,left,right,causal", [
    (16, 40, 5, 0, True), (40, 16, 3, 2, False), (33, 33, 8, -1, True), (20, 50, -1, 7, False),
    (24, 24, 0, 0, False), (12, 70, 10, 3, True),
])
def test_local_window_matches_sdpa_fp64_with_band_mask(nq, nk, left, right, causal):
    """Random data through SDPA (fp64 MATH backend) with the keep mask built
    from the page's statement of the window as a boolean band; rows with no
    key return 0 and -inf."""
    torch.manual_seed(nq * 1000 + nk * 7 + left)
    hq, hkv, d = 4, 2, 16
    q, k, v = bf16(torch.randn(nq, hq, d)), bf16(torch.randn(nk, hkv, d)), bf16(torch.randn(nk, hkv, d))
    scale = 1.0 / math.sqrt(d)
    i = torch.arange(nq)[:, None]
    j = torch.arange(nk)[None, :]
    centre = i + nk - nq
    keep = torch.ones(nq, nk, dtype=torch.bool)
    if left >= 0:
        keep &= j >= centre - left
    if right >= 0:
        keep &= j <= centre + right
    if causal:
        keep &= j <= centre
    rows = [[0, h, r] for h in range(hq) for r in range(nq)]
    out, lse = oracle.prefill_rows(q, k, v, B=1, Hq=hq, Hkv=hkv, Nq=nq, Nk=nk, scale=scale,
                                   causal=causal, rows=rows, window=(left, right))
    ref, ref_lse, keep = sdpa_reference(q, k, v, nq, nk, hq, hkv, scale, causal, keep=keep)
    has_key = keep.any(dim=-1)
    for r, (_, h, ii) in enumerate(rows):
        if has_key[ii]:
            assert np.abs(out[r] - ref[h, ii].numpy()).max() <= 1e-12
            assert abs(lse[r] - float(ref_lse[h, ii])) <= 1e-12
        else:
            assert (out[r] == 0).all() and np.isneginf(lse[r])


# ---------------------------------------------------------------------------
# invariants and independent algorithms
# ---------------------------------------------------------------------------
def tiled_online_softmax(q, k, v, scale, block):
    """Independent fp64 tiled forward with the running (m, l, acc) state and
    the exp(m_old - m_new) rescale, written from the recurrence the pages
    describe (no masks; one query block)."""
    m = np.full(q.shape[0], -np.inf)
    l = np.zeros(q.shape[0])
    acc = np.zeros((q.shape[0], v.shape[1]))
    for s0 in range(0, k.shape[0], block):
        s = (q @ k[s0:s0 + block].T) * scale
        m_new = np.maximum(m, s.max(axis=1))
        alpha = np.exp(m - m_new)
        p = np.exp(s - m_new[:, None])
        l = alpha * l + p.sum(axis=1)
        acc = alpha[:, None] * acc + p @ v[s0:s0 + block]
        m = m_new
    return acc / l[:, None], m + np.log(l)


def test_matches_independent_tiled_recurrence_256x64():
    g = golden("paged_gather.json")
    n, d = g["tiled_problem_shape"]
    torch.manual_seed(0)
    q, k, v = bf16(torch.randn(n, 1, d)), bf16(torch.randn(n, 1, d)), bf16(torch.randn(n, 1, d))
    scale = 1.0 / math.sqrt(d)
    out, lse = oracle.prefill_rows(q, k, v, B=1, Hq=1, Hkv=1, Nq=n, Nk=n, scale=scale, causal=False,
                                   rows=[[0, 0, i] for i in range(n)])
    for block in (64, 100, 256):
        t_out, t_lse = tiled_online_softmax(q[:, 0].double().numpy(), k[:, 0].double().numpy(),
                                            v[:, 0].double().numpy(), scale, block)
        # the page reports ~6e-16 between its tiled and dense fp64 versions
        assert np.abs(out - t_out).max() < 100 * g["tiled_vs_reference_max_abs_diff_fp64"]
        assert np.abs(lse - t_lse).max() < 1e-12


def test_lse_merge_of_disjoint_key_sets():
    """Split a row's keys into two disjoint sets: logaddexp of the two lse and
    the exp(lse_s - lse)-weighted outputs equal the full row (the split-KV
    combine identity)."""
    torch.manual_seed(3)
    nq, nk, d = 6, 50, 16
    q, k, v = bf16(torch.randn(nq, 2, d)), bf16(torch.randn(nk, 1, d)), bf16(torch.randn(nk, 1, d))
    rows = [[0, h, i] for h in range(2) for i in range(nq)]
    kw = dict(B=1, Hq=2, Hkv=1, Nq=nq, scale=0.3, causal=False, rows=rows)
    full_o, full_l = oracle.prefill_rows(q, k, v, Nk=nk, **kw)
    for s in (1, 17, 49):
        o1, l1 = oracle.prefill_rows(q, k[:s], v[:s], Nk=s, **kw)
        o2, l2 = oracle.prefill_rows(q, k[s:], v[s:], Nk=nk - s, **kw)
        lse = np.logaddexp(l1, l2)
        merged = np.exp(l1 - lse)[:, None] * o1 + np.exp(l2 - lse)[:, None] * o2
        assert np.abs(merged - full_o).max() < 1e-12
        assert np.abs(lse - full_l).max() < 1e-12


def test_rows_sum_to_one():
    """With V = 1 every nonempty row returns exactly 1 (probabilities sum to 1)."""
    p = workloads.make_varlen([3, 40, 0, 17], [9, 40, 5, 3], 4, 2, 16, causal=True, seed=5)
    v1 = torch.ones_like(p.v)
    rows = oracle.all_rows(p)
    out, lse = oracle.prefill_rows(p.q, p.k, v1, B=p.B, Hq=p.Hq, Hkv=p.Hkv, Nq=p.Nq, Nk=p.Nk,
                                   scale=p.scale, causal=True, rows=rows, cu_q=p.cu_q, cu_k=p.cu_k)
    nonempty = np.isfinite(lse)
    assert nonempty.sum() > 0 and (~nonempty).sum() > 0   # sequence 4 has Nq > Nk
    assert np.abs(out[nonempty] - 1.0).max() < 1e-12
    assert (out[~nonempty] == 0).all()


def test_varlen_offsets_equal_per_sequence_dense():
    """A packed problem gives, row for row, the dense result of each sequence
    alone: a wrong cu_seqlens offset would read another sequence's tokens."""
    ql, kl = [5, 1, 33, 0, 12], [5, 9, 20, 4, 40]
    p = workloads.make_varlen(ql, kl, 4, 2, 8, causal=True, seed=11)
    rows = oracle.all_rows(p)
    out, lse = oracle.prefill(p, rows)
    cq = p.cu_q.tolist()
    ck = p.cu_k.tolist()
    r = 0
    for b in range(p.B):
        nq, nk = ql[b], kl[b]
        if nq == 0:
            continue
        rr = [[0, h, i] for h in range(p.Hq) for i in range(nq)]
        o, l = oracle.prefill_rows(p.q[cq[b]:cq[b + 1]], p.k[ck[b]:ck[b + 1]], p.v[ck[b]:ck[b + 1]],
                                   B=1, Hq=p.Hq, Hkv=p.Hkv, Nq=nq, Nk=nk, scale=p.scale,
                                   causal=True, rows=rr)
        assert np.array_equal(out[r:r + len(rr)], o)
        assert np.array_equal(lse[r:r + len(rr)], l)
        r += len(rr)
    assert r == len(rows)


# ---------------------------------------------------------------------------
# paged decode
# ---------------------------------------------------------------------------
def paged_gather(pool, table, length):
    """Concatenate the listed physical pages and keep the first `length`
    tokens (the toy block-table gather the paged-attention page runs)."""
    return torch.cat([pool[int(b)] for b in table], dim=0)[:length]


def test_paged_gather_example_shape():
    g = golden("paged_gather.json")
    pool = torch.randn(*g["pool_shape"])
    assert list(paged_gather(pool, g["table"], g["length"]).shape) == g["gathered_shape"]


def test_decode_equals_dense_on_gathered_keys():
    p = workloads.make_decode([40, 17, 1, 0, 33], 4, 2, 16, num_pages=14, seed=7,
                              nan_fill_unused=True, max_pages=4)
    out, lse = oracle.decode(p)
    assert np.isfinite(out).all()
    r = 0
    for b in range(p.B):
        L = int(p.seq_lens[b])
        n_pages = -(-L // p.page_size)
        table = p.block_table[b, :n_pages].tolist()
        for h in range(p.Hq):
            if L == 0:
                assert (out[r] == 0).all() and np.isneginf(lse[r])
            else:
                kk = paged_gather(p.k_cache, table, L)  # [L, Hkv, d]
                vv = paged_gather(p.v_cache, table, L)
                o, l = oracle.prefill_rows(p.q[b:b + 1], kk, vv, B=1, Hq=p.Hq, Hkv=p.Hkv, Nq=1, Nk=L,
                                           scale=p.scale, causal=True, rows=[[0, h, 0]])
                assert np.array_equal(out[r], o[0])
                assert lse[r] == l[0]
            r += 1


def test_decode_multi_with_one_query_equals_decode():
    p = workloads.make_decode([40, 17, 1, 0, 33], 4, 2, 16, num_pages=14, seed=8, nan_fill_unused=True,
                              max_pages=4)
    o1, l1 = oracle.decode(p)
    rows = np.asarray([(b, h, 0) for b in range(p.B) for h in range(p.Hq)], dtype=np.int32)
    for causal in (False, True):
        o2, l2 = oracle.decode_multi_rows(p.q[:, None], p.k_cache, p.v_cache, p.block_table, p.seq_lens,
                                          scale=p.scale, causal=causal, rows=rows)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def _paged_one_hot(lens, nq, page):
    """Q = 0 and V one-hot by logical token over a shuffled paged pool."""
    need = [-(-L // page) for L in lens]
    n_pages = sum(need) + 3
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(5)).tolist()
    width = max(lens)
    table = torch.full((len(lens), max(need)), -1, dtype=torch.int32)
    kc = torch.zeros(n_pages, page, 1, width)
    vc = torch.full((n_pages, page, 1, width), float("nan"))
    pos = 0
    for b, L in enumerate(lens):
        for pi in range(need[b]):
            pg = perm[pos]
            pos += 1
            table[b, pi] = pg
            vc[pg] = 0.0
            for s in range(page):
                t = pi * page + s
                if t < L:
                    vc[pg, s, 0, t] = 1.0
    q = torch.zeros(len(lens), nq, 1, width)
    return bf16(q), bf16(kc), bf16(vc), table, torch.tensor(lens, dtype=torch.int32)


def test_decode_multi_printed_keep_matrices():
    """The printed bottom-right keep matrices, read through a paged cache:
    Nq new queries over a sequence of Nk cached keys."""
    g = golden("causal_keep.json")
    for case in g["bottom_right"]:
        nq, nk = case["q"], case["k"]
        q, kc, vc, table, lens = _paged_one_hot([nk], nq, page=2)
        rows = [[0, 0, i] for i in range(nq)]
        out, lse = oracle.decode_multi_rows(q, kc, vc, table, lens, scale=1.0, causal=True, rows=rows)
        keep = (out[:, :nk] > 0).astype(int).tolist()
        assert keep == case["keep"]
        out, _ = oracle.decode_multi_rows(q, kc, vc, table, lens, scale=1.0, causal=False, rows=rows)
        assert (out[:, :nk] > 0).all()


def test_decode_multi_equals_prefill_on_gathered_keys():
    lens = [40, 3, 1, 33, 16]
    nq = 3
    p = workloads.make_decode(lens, 4, 2, 16, num_pages=14, seed=9, nan_fill_unused=True, max_pages=4)
    q = bf16(torch.randn(p.B, nq, p.Hq, p.d, generator=torch.Generator().manual_seed(3)))
    rows = np.asarray([(b, h, i) for b in range(p.B) for h in range(p.Hq) for i in range(nq)], dtype=np.int32)
    for causal in (True, False):
        out, lse = oracle.decode_multi_rows(q, p.k_cache, p.v_cache, p.block_table, p.seq_lens, scale=p.scale,
                                            causal=causal, rows=rows)
        for r, (b, h, i) in enumerate(rows):
            L = lens[b]
            table = p.block_table[b, :-(-L // p.page_size)].tolist()
            kk = paged_gather(p.k_cache, table, L)
            vv = paged_gather(p.v_cache, table, L)
            o, l = oracle.prefill_rows(q[b], kk, vv, B=1, Hq=p.Hq, Hkv=p.Hkv, Nq=nq, Nk=L, scale=p.scale,
                                       causal=causal, rows=[[0, h, i]])
            assert np.array_equal(out[r], o[0]) and (lse[r] == l[0] or (np.isneginf(lse[r]) and np.isneginf(l[0])))


def test_append_kv_gathered_sequence_ends_with_the_new_rows():
    """Independent of the oracle's position arithmetic: after the append, each
    sequence read back with the paged gather of the paged-attention page
    (concatenate the listed pages, keep the first `length` tokens) is its old
    first L - Nq tokens followed by the Nq new rows, L being the length after
    the append.  Sequences whose new positions would start below zero keep
    only the rows that land at positions >= 0."""
    lens = [40, 2, 17, 0, 16, 33]
    nq = 3
    p = workloads.make_decode(lens, 4, 2, 16, num_pages=14, seed=12, max_pages=4)
    g = torch.Generator().manual_seed(6)
    k_new = bf16(torch.randn(p.B, nq, p.Hkv, p.d, generator=g))
    v_new = bf16(torch.randn(p.B, nq, p.Hkv, p.d, generator=g))
    kc, vc = oracle.append_kv(p.k_cache, p.v_cache, p.block_table, p.seq_lens, k_new, v_new)
    for b, L in enumerate(lens):
        if L == 0:
            continue
        table = p.block_table[b, :-(-L // p.page_size)].tolist()
        for after, before, new in ((kc, p.k_cache, k_new), (vc, p.v_cache, v_new)):
            seq = paged_gather(after, table, L)
            old = paged_gather(before, table, L)
            kept = max(L - nq, 0)
            assert torch.equal(seq[:kept], old[:kept])
            assert torch.equal(seq[kept:], new[b, nq - (L - kept):])


def test_decode_after_append_equals_prefill_over_old_keys_then_new_keys():
    """The appended tokens are the newest keys: Nq-query decode over the
    appended cache equals the prefill oracle (bottom-right causal corner)
    over the old gathered keys followed by the new rows."""
    lens = [40, 5, 17, 33]
    nq = 4
    p = workloads.make_decode(lens, 4, 2, 16, num_pages=12, seed=13, max_pages=3)
    g = torch.Generator().manual_seed(7)
    k_new = bf16(torch.randn(p.B, nq, p.Hkv, p.d, generator=g))
    v_new = bf16(torch.randn(p.B, nq, p.Hkv, p.d, generator=g))
    q = bf16(torch.randn(p.B, nq, p.Hq, p.d, generator=g))
    kc, vc = oracle.append_kv(p.k_cache, p.v_cache, p.block_table, p.seq_lens, k_new, v_new)
    rows = np.asarray([(b, h, i) for b in range(p.B) for h in range(p.Hq) for i in range(nq)], dtype=np.int32)
    out, lse = oracle.decode_multi_rows(q, kc, vc, p.block_table, p.seq_lens, scale=p.scale, causal=True,
                                        rows=rows)
    for r, (b, h, i) in enumerate(rows):
        L = lens[b]
        table = p.block_table[b, :-(-L // p.page_size)].tolist()
        kk = torch.cat([paged_gather(p.k_cache, table, L)[:L - nq], k_new[b]])
        vv = torch.cat([paged_gather(p.v_cache, table, L)[:L - nq], v_new[b]])
        o, l = oracle.prefill_rows(q[b], kk, vv, B=1, Hq=p.Hq, Hkv=p.Hkv, Nq=nq, Nk=L, scale=p.scale,
                                   causal=True, rows=[[0, h, i]])
        assert np.array_equal(out[r], o[0]) and lse[r] == l[0]


def test_append_kv_writes_exactly_the_new_positions():
    """Brute force: after the append, position L - Nq + i of sequence b, looked
    up through the block table, holds new row i; every other slot keeps its
    bytes; positions below zero and page ids outside the pool are skipped."""
    lens = [40, 2, 17, 0]
    nq = 3
    p = workloads.make_decode(lens, 4, 2, 16, num_pages=10, seed=10, max_pages=4)
    g = torch.Generator().manual_seed(4)
    k_new = bf16(torch.randn(p.B, nq, p.Hkv, p.d, generator=g))
    v_new = bf16(torch.randn(p.B, nq, p.Hkv, p.d, generator=g))
    bt = p.block_table.clone()
    bt[2, 1] = 10_000    # position 16 of sequence 2 lives in a page outside the pool
    kc, vc = oracle.append_kv(p.k_cache, p.v_cache, bt, p.seq_lens, k_new, v_new)
    written = set()
    for b, L in enumerate(lens):
        for i in range(nq):
            pos = L - nq + i
            if pos < 0:
                continue
            pg = int(bt[b, pos // 16])
            if not 0 <= pg < p.num_pages:
                continue
            written.add((pg, pos % 16))
            assert torch.equal(kc[pg, pos % 16], k_new[b, i]) and torch.equal(vc[pg, pos % 16], v_new[b, i])
    # 3 + 2 (one position of sequence 1 is negative) + 2 (position 16 of sequence 2 is skipped) + 0
    assert len(written) == 7
    mask = torch.ones(p.num_pages, 16, dtype=torch.bool)
    for pg, s in written:
        mask[pg, s] = False
    assert torch.equal(kc[mask], p.k_cache[mask]) and torch.equal(vc[mask], p.v_cache[mask])


def test_thread_count_does_not_change_results():
    p = workloads.make_prefill(2, 4, 2, 37, 70, 16, causal=True, seed=9)
    a = oracle.prefill(p, threads=1)
    b = oracle.prefill(p, threads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------
def _sdpa_grads(p, g, keep):
    """dq, dk, dv of <g, O> through SDPA's fp64 MATH backend with an explicit
    keep mask (one dense sequence, q [nq, hq, d], k/v [nk, hkv, d])."""
    from torch.nn.attention import SDPBackend, sdpa_kernel
    import torch.nn.functional as F
    rep = p.Hq // p.Hkv
    q = p.q.double().permute(1, 0, 2)[None].requires_grad_(True)
    k = p.k.double().permute(1, 0, 2)[None].requires_grad_(True)
    v = p.v.double().permute(1, 0, 2)[None].requires_grad_(True)
    with sdpa_kernel(SDPBackend.MATH):
        out = F.scaled_dot_product_attention(q, k.repeat_interleave(rep, dim=1), v.repeat_interleave(rep, dim=1),
                                             attn_mask=keep, is_causal=False, dropout_p=0.0, scale=p.scale)
    has_key = keep.any(dim=-1)
    gg = g.double().permute(1, 0, 2)[None] * has_key[None, None, :, None]   # SDPA's empty rows are NaN
    out = torch.where(has_key[None, None, :, None], out, torch.zeros_like(out))
    dq, dk, dv = torch.autograd.grad(out, (q, k, v), gg)
    f = lambda x: x[0].permute(1, 0, 2).numpy()
    return f(dq), f(dk), f(dv)


def _keep(nq, nk, causal, window=(-1, -1)):
    i = torch.arange(nq)[:, None]
    j = torch.arange(nk)[None, :]
    c = i + nk - nq
    keep = torch.ones(nq, nk, dtype=torch.bool)
    if causal:
        keep &= j <= c
    if window[0] >= 0:
        keep &= j >= c - window[0]
    if window[1] >= 0:
        keep &= j <= c + window[1]
    return keep


@pytest.mark.parametrize("nq,nk,hq,hkv,d,causal,window", [
    (2, 5, 2, 2, 3, True, (-1, -1)), (5, 2, 2, 2, 3, True, (-1, -1)), (4, 4, 2, 2, 3, True, (-1, -1)),
    (7, 13, 6, 2, 8, True, (-1, -1)), (13, 7, 4, 1, 8, False, (-1, -1)), (20, 33, 4, 2, 16, True, (6, -1)),
    (24, 24, 2, 2, 8, False, (3, 2)),
])
def test_backward_matches_sdpa_autograd_fp64(nq, nk, hq, hkv, d, causal, window):
    p = workloads.make_prefill(1, hq, hkv, nq, nk, d, causal=causal, seed=nq * 31 + nk, window=window)
    g = workloads.randn_bf16((nq, hq, d), seed=nq + 5 * nk)
    dq, dk, dv = oracle.backward(p, g)
    rq, rk, rv = _sdpa_grads(p, g, _keep(nq, nk, causal, window))
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert np.abs(got - ref).max() <= 1e-11 * max(1.0, np.abs(ref).max())


def _exact_grid(shape, gen):
    """Values k/4 in [-2, 2]: every x +- 1/64 and x +- 1/32 is exact in bf16."""
    return (torch.randint(-8, 9, shape, generator=gen).float() / 4).to(torch.bfloat16)


def test_backward_matches_finite_differences():
    """Central differences of L = <G, O> along random directions, Richardson-
    extrapolated from steps 1/64 and 1/32 (the perturbed inputs are exact in
    bf16), against <U, grad>: independent of every backward formula."""
    import dataclasses
    gen = torch.Generator().manual_seed(11)
    nq, nk, hq, hkv, d = 6, 9, 4, 2, 8
    for causal in (True, False):
        p = workloads.make_prefill(1, hq, hkv, nq, nk, d, causal=causal, seed=1)
        p = dataclasses.replace(p, q=_exact_grid(p.q.shape, gen), k=_exact_grid(p.k.shape, gen),
                                v=_exact_grid(p.v.shape, gen), scale=0.5)
        g = _exact_grid(p.q.shape, gen)
        grads = oracle.backward(p, g)
        rows = oracle.all_rows(p)

        def loss(pp):
            o, _ = oracle.prefill(pp, rows)
            gi = g.double().numpy()[rows[:, 2], rows[:, 1]]
            return float((o * gi).sum())

        for which, grad in zip(("q", "k", "v"), grads):
            base = getattr(p, which)
            u = torch.randint(-1, 2, base.shape, generator=gen).float()
            est = []
            for t in (1 / 64, 1 / 32):
                plus = (base.float() + t * u).to(torch.bfloat16)
                minus = (base.float() - t * u).to(torch.bfloat16)
                assert torch.equal(plus.float(), base.float() + t * u)   # exact perturbation
                lp = loss(dataclasses.replace(p, **{which: plus}))
                lm = loss(dataclasses.replace(p, **{which: minus}))
                est.append((lp - lm) / (2 * t))
            fd = (4 * est[0] - est[1]) / 3
            an = float((u.double().numpy() * grad).sum())
            assert abs(fd - an) <= 2e-4 * max(1.0, abs(an)), (causal, which, fd, an)


def test_backward_invariants():
    """Adding c to every value shifts each nonempty row's O by c, so
    sum_j dV_j = sum over nonempty rows of G_i (per K/V head, over its group);
    without a mask, adding c to every key leaves O unchanged, so
    sum_j dK_j = 0; rows with no key pass no gradient."""
    for causal, nq, nk in ((True, 9, 5), (False, 7, 7), (True, 30, 40)):
        p = workloads.make_prefill(1, 4, 2, nq, nk, 16, causal=causal, seed=nq + nk)
        g = workloads.randn_bf16((nq, 4, 16), seed=3)
        dq, dk, dv = oracle.backward(p, g)
        keep = _keep(nq, nk, causal)
        nonempty = keep.any(dim=-1).numpy()
        gd = g.double().numpy()
        for kvh in range(2):
            heads = [kvh * 2, kvh * 2 + 1]
            assert np.allclose(dv[:, kvh].sum(0), gd[nonempty][:, heads].sum((0, 1)), atol=1e-12)
            if not causal:
                assert np.allclose(dk[:, kvh].sum(0), 0.0, atol=1e-12)
        assert (dq[~nonempty] == 0).all()


def test_backward_varlen_equals_per_sequence_dense():
    ql, kl = [5, 0, 17, 9], [7, 4, 17, 30]
    p = workloads.make_varlen(ql, kl, 4, 2, 16, causal=True, seed=77)
    g = workloads.randn_bf16((sum(ql), 4, 16), seed=78)
    dq, dk, dv = oracle.backward(p, g)
    cq = np.cumsum([0] + ql)
    ck = np.cumsum([0] + kl)
    for b in range(len(ql)):
        sub = workloads.make_prefill(1, 4, 2, ql[b], kl[b], 16, causal=True, seed=1)
        import dataclasses
        sub = dataclasses.replace(sub, q=p.q[cq[b]:cq[b + 1]], k=p.k[ck[b]:ck[b + 1]], v=p.v[ck[b]:ck[b + 1]])
        if ql[b] == 0:
            assert (dk[ck[b]:ck[b + 1]] == 0).all() and (dv[ck[b]:ck[b + 1]] == 0).all()
            continue
        sq, sk, sv = oracle.backward(sub, g[cq[b]:cq[b + 1]])
        assert np.array_equal(sq, dq[cq[b]:cq[b + 1]])
        assert np.array_equal(sk, dk[ck[b]:ck[b + 1]]) and np.array_equal(sv, dv[ck[b]:ck[b + 1]])



# ---------------------------------------------------------------------------
# 8-bit (E4M3) per-tile quantization ("FP8 Path and Quantization"; "FlashAttention-3:
# asynchrony and low precision on Hopper")
# ---------------------------------------------------------------------------
def test_e4m3_decoding_matches_torch_on_every_code():
    """torch's float8_e4m3fn (a library routine) decodes all 256 codes."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    for c in range(256):
        got = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), c
    assert oracle.e4m3_value(0x7E) == 448.0 and math.isnan(oracle.e4m3_value(0x7F))


def test_e4m3_rounding_matches_torch_on_every_bf16_value():
    """Round to nearest, ties to even, on every finite bf16 value up to 464
    (torch's cast turns larger ones into NaN; this encoding saturates them to
    448 instead)."""
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).to(torch.float32)
    keep = torch.isfinite(x) & (x.abs() <= 464)
    xs = x[keep]
    ref = xs.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    got = [oracle.e4m3_from_float(v) for v in xs.tolist()]
    assert got == ref
    for v in (465.0, 480.0, 1e6, float("inf")):
        assert oracle.e4m3_from_float(v) == 0x7E and oracle.e4m3_from_float(-v) == 0xFE


def test_quantize_tile_maximum_lands_on_448_and_round_trip_within_half_step():
    """Each tile's largest magnitude becomes the code for +-448, and every
    value comes back within half a step of the E4M3 grid at its own scale:
    |x - x~| <= 2^-4 |x| in the normal range, <= 2^-10 * scale below it."""
    lens = [300, 1, 128, 129, 0, 77]
    p = workloads.make_varlen(lens, lens, 3, 2, 64, causal=True, seed=21)
    spread = torch.logspace(-3, 2, p.q.shape[0])[:, None, None]
    x = (p.q.float() * spread).to(torch.bfloat16)
    codes, scales = oracle.quantize_fp8(x, B=p.B, cu=p.cu_q)
    deq = oracle.dequantize_fp8(codes, scales, B=p.B, cu=p.cu_q)
    xd = x.double().numpy()
    cq = p.cu_q.tolist()
    for b, L in enumerate(lens):
        for t in range(0, L, 128):
            r0, r1 = cq[b] + t, cq[b] + min(L, t + 128)
            tile_codes = codes[r0:r1]
            for h in range(x.shape[1]):
                mags = np.abs([oracle.e4m3_value(c) for c in tile_codes[:, h].reshape(-1)])
                assert mags.max() == 448.0
                sc = float(scales[h, cq[b] // 128 + b + t // 128])
                err = np.abs(xd[r0:r1, h] - deq[r0:r1, h])
                bound = np.maximum(2.0 ** -4 * np.abs(xd[r0:r1, h]), 2.0 ** -10 * sc) * (1 + 1e-6)
                assert (err <= bound).all()


def test_quantize_tiles_start_at_each_sequence_start():
    """An outlier changes the codes of its own tile (128 tokens counted from
    its sequence's first token, one head) and of no other."""
    lens = [200, 70, 260]
    p = workloads.make_varlen(lens, lens, 2, 2, 64, causal=False, seed=22)
    base_codes, base_scales = oracle.quantize_fp8(p.q, B=p.B, cu=p.cu_q)
    cq = p.cu_q.tolist()
    for b, tok in ((0, 130), (1, 3), (2, 255)):
        x = p.q.clone()
        x[cq[b] + tok, 1, 5] = 64.0 * x.float().abs().max()
        codes, scales = oracle.quantize_fp8(x, B=p.B, cu=p.cu_q)
        t = tok // 128
        r0, r1 = cq[b] + 128 * t, cq[b] + min(lens[b], 128 * (t + 1))
        changed = np.argwhere((codes != base_codes).any(axis=2))
        assert len(changed) > 0
        assert ((changed[:, 0] >= r0) & (changed[:, 0] < r1) & (changed[:, 1] == 1)).all()
        diff = np.argwhere(scales != base_scales)
        assert diff.tolist() == [[1, cq[b] // 128 + b + t]]


def test_quantize_zero_tile_and_dense_layout():
    x = bf16(torch.randn(2 * 256, 2, 64, generator=torch.Generator().manual_seed(23)))
    x[256 + 128:] = 0.0          # sequence 1, tile 1: all zero
    codes, scales = oracle.quantize_fp8(x, B=2, N=256)
    assert (codes[256 + 128:] == 0).all()
    assert scales.shape == (2, 512 // 128 + 2)
    # sequence 1 starts at token 256: its tiles are entries 2 + 1 and 2 + 1 + 1; entry 2 is a gap
    assert (scales[:, 4] == 1.0).all() and (scales[:, 2] == 0).all()
    assert (scales[:, [0, 1, 3]] > 0).all()


def test_f64_attention_equals_bf16_attention_on_bf16_values():
    p = workloads.make_varlen([33, 130, 0, 7], [40, 200, 5, 7], 4, 2, 64, causal=True, seed=24)
    rows = oracle.all_rows(p)
    o1, l1 = oracle.prefill(p, rows)
    o2, l2 = oracle.prefill_rows_f64(p.q.double().numpy(), p.k.double().numpy(), p.v.double().numpy(), B=p.B,
                                     Hq=p.Hq, Hkv=p.Hkv, Nq=p.Nq, Nk=p.Nk, scale=p.scale, causal=True, rows=rows,
                                     cu_q=p.cu_q, cu_k=p.cu_k)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_fp8_attention_on_exactly_quantizable_inputs_equals_attention():
    """Inputs that are E4M3 values times a power of two, with a +-448 * 2^k
    element in every tile, quantize exactly (scale 2^k): attention on the
    values they stand for is attention on the inputs themselves."""
    g = torch.Generator().manual_seed(25)
    p = workloads.make_prefill(2, 4, 2, 300, 300, 64, causal=True, seed=26)

    def exact(t, k):
        c = torch.randint(0, 256, t.shape, generator=g, dtype=torch.int32)
        c[(c & 0x7F) == 0x7F] = 0          # no NaN codes
        v = c.to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float32) * 2.0 ** k
        rows = t.shape[0]
        for r0 in range(0, rows, 300):       # one +-448 * 2^k element in every tile of every head
            for tt in range(r0, min(rows, r0 + 300), 128):
                v[tt, :, 0] = 448.0 * 2.0 ** k
        return v.to(torch.bfloat16)
    q, k, v = exact(p.q, -8), exact(p.k, -7), exact(p.v, -2)
    p = workloads.Prefill(p.name, q, k, v, p.B, p.Hq, p.Hkv, p.Nq, p.Nk, p.d, p.scale, p.causal, seed=p.seed)
    rows = oracle.all_rows(p)
    o1, l1 = oracle.prefill(p, rows)
    o2, l2 = oracle.prefill_fp8(p, rows)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
