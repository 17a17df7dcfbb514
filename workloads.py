"""Seeded synthetic inputs for exact attention: the only module shared by the
oracle side and the CUDA side.

It draws numbers and lays them out; it holds none of the attention arithmetic
(no scores, no softmax, no masks).  Every tensor is drawn as fp32 N(0, 1) from
a seeded torch generator and rounded to bf16 (round-to-nearest-even), so the
oracle and the GPU path read identical bytes.

Layouts (token-major "THD", the (batch, sequence, heads, head_dim) order of the
FA2 public call described on "Deep Dive - FlashAttention", section "The public
interface is several kernels"):
  q          [T_q, Hq, d]   bf16      T_q = B*Nq (dense) or cu_seqlens_q[-1]
  k, v       [T_k, Hkv, d]  bf16
  cu_seqlens int32 [B+1]    (varlen only)
Paged decode ("FlashAttention-3 and PagedAttention", section "Block tables and
what the kernel does"):
  q          [B, Hq, d]                 bf16
  k_cache    [num_pages, page, Hkv, d]  bf16 (same for v_cache)
  block_table int32 [B, max_pages]      unused entries -1
  seq_lens   int32 [B]

The five named workloads follow the benchmark configurations of this project:
tiny (B1 H2 N256 d64), MHA causal (B4 H16 N4096 d128), GQA causal
(B2 Hq32 Hkv8 N8192 d128, one K channel x3), varlen chunked prefill
(16 sequences, Nk ~ U[1024, 16384], Nq = min(512, Nk)) and paged split-KV
decode (B64 Hq32 Hkv8 d128, len ~ U[4096, 32768], 16-token pages in a
200k-page pool); beyond those, a sliding-window prefill and a four-query
speculative decode step over the paged cache with an in-place append.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

SEED_BASE = 1000  # workload i uses seed SEED_BASE + i


# --------------------------------------------------------------------------
# primitive draws
# --------------------------------------------------------------------------
def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, seed: int, device="cpu", chunk_elems: int = 1 << 28) -> torch.Tensor:
    """fp32 N(0,1) draws rounded to bf16, generated in chunks to bound the
    fp32 temporary (the decode pools hold billions of elements)."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    g = _gen(seed, device)
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        out[s:e] = torch.randn(e - s, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def randint(low: int, high: int, n: int, seed: int) -> torch.Tensor:
    """n integers uniform in [low, high] inclusive (CPU, int64)."""
    return torch.randint(low, high + 1, (n,), generator=_gen(seed))


# --------------------------------------------------------------------------
# prefill problems
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Prefill:
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    B: int
    Hq: int
    Hkv: int
    Nq: int          # max query length (dense: the length)
    Nk: int          # max key length
    d: int
    scale: float
    causal: bool
    cu_q: Optional[torch.Tensor] = None  # int32 [B+1] or None (dense)
    cu_k: Optional[torch.Tensor] = None
    seed: int = 0
    window: tuple = (-1, -1)   # local window (left, right) in keys, -1 = unbounded

    @property
    def varlen(self) -> bool:
        return self.cu_q is not None

    def seq_lens(self):
        """(Nq_b, Nk_b) per sequence as python ints."""
        if self.cu_q is None:
            return [(self.Nq, self.Nk)] * self.B
        cq = self.cu_q.tolist()
        ck = self.cu_k.tolist()
        return [(cq[b + 1] - cq[b], ck[b + 1] - ck[b]) for b in range(self.B)]

    def to(self, device) -> "Prefill":
        f = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(self, q=f(self.q), k=f(self.k), v=f(self.v),
                                   cu_q=f(self.cu_q), cu_k=f(self.cu_k))


def make_prefill(B, Hq, Hkv, Nq, Nk, d, *, causal, seed, scale=None, name="custom",
                 device="cpu", window=(-1, -1)) -> Prefill:
    """Dense problem: B sequences of Nq queries over Nk keys."""
    q = randn_bf16((B * Nq, Hq, d), seed * 7 + 1, device)
    k = randn_bf16((B * Nk, Hkv, d), seed * 7 + 2, device)
    v = randn_bf16((B * Nk, Hkv, d), seed * 7 + 3, device)
    return Prefill(name, q, k, v, B, Hq, Hkv, Nq, Nk, d,
                   1.0 / math.sqrt(d) if scale is None else scale, causal, seed=seed, window=tuple(window))


def make_varlen(q_lens, k_lens, Hq, Hkv, d, *, causal, seed, scale=None, name="varlen",
                device="cpu", window=(-1, -1)) -> Prefill:
    """Packed problem: sequence b has q_lens[b] queries and k_lens[b] keys."""
    q_lens = [int(x) for x in q_lens]
    k_lens = [int(x) for x in k_lens]
    B = len(q_lens)
    cu_q = torch.tensor([0] + list(_cumsum(q_lens)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(_cumsum(k_lens)), dtype=torch.int32)
    Tq, Tk = int(cu_q[-1]), int(cu_k[-1])
    q = randn_bf16((max(Tq, 1), Hq, d), seed * 7 + 1, device)[:Tq]
    k = randn_bf16((max(Tk, 1), Hkv, d), seed * 7 + 2, device)[:Tk]
    v = randn_bf16((max(Tk, 1), Hkv, d), seed * 7 + 3, device)[:Tk]
    return Prefill(name, q, k, v, B, Hq, Hkv, max(q_lens + [0]), max(k_lens + [0]), d,
                   1.0 / math.sqrt(d) if scale is None else scale, causal,
                   cu_q=cu_q.to(device), cu_k=cu_k.to(device), seed=seed, window=tuple(window))


def _cumsum(xs):
    t = 0
    for x in xs:
        t += x
        yield t


def tiny(causal: bool, device="cpu") -> Prefill:
    """B=1, Hq=Hkv=2, Nq=Nk=256, d=64, scale 1/8."""
    return make_prefill(1, 2, 2, 256, 256, 64, causal=causal, seed=SEED_BASE + 0,
                        scale=1.0 / 8.0, name="tiny_causal" if causal else "tiny", device=device)


def mha_causal(device="cpu") -> Prefill:
    """B=4, Hq=Hkv=16, N=4096, d=128, bottom-right causal."""
    return make_prefill(4, 16, 16, 4096, 4096, 128, causal=True, seed=SEED_BASE + 1,
                        name="mha_causal_b4_h16_n4096_d128", device=device)


def gqa_causal(device="cpu") -> Prefill:
    """B=2, Hq=32, Hkv=8, N=8192, d=128; one seeded K channel multiplied by 3
    after bf16 rounding (exact in bf16), which creates large-logit rows."""
    p = make_prefill(2, 32, 8, 8192, 8192, 128, causal=True, seed=SEED_BASE + 2,
                     name="gqa_causal_b2_hq32_hkv8_n8192_d128", device=device)
    c_star = gqa_hot_channel(p.d)
    p.k[:, :, c_star] = p.k[:, :, c_star] * 3
    return p


def swa_causal(device="cpu") -> Prefill:
    """Sliding-window prefill: B=2, Hq=32, Hkv=8, N=16384, d=128, causal with
    a 4096-key window (window (4095, 0): each query sees itself and the 4095
    keys before it)."""
    return make_prefill(2, 32, 8, 16384, 16384, 128, causal=True, seed=SEED_BASE + 6,
                        name="swa_causal_b2_hq32_hkv8_n16384_w4096_d128", device=device, window=(4095, 0))


def gqa_hot_channel(d: int) -> int:
    return int(randint(0, d - 1, 1, SEED_BASE + 2 + 100)[0])


def varlen_lengths(seed=SEED_BASE + 3, n=16, lo=1024, hi=16384, nq_max=512):
    k_lens = randint(lo, hi, n, seed).tolist()
    q_lens = [min(nq_max, x) for x in k_lens]
    return q_lens, k_lens


def varlen_chunked(device="cpu") -> Prefill:
    """16 sequences, Nk_b ~ U[1024, 16384], Nq_b = min(512, Nk_b), Hq=32,
    Hkv=8, d=128, packed with cu_seqlens, bottom-right causal per sequence."""
    q_lens, k_lens = varlen_lengths()
    return make_varlen(q_lens, k_lens, 32, 8, 128, causal=True, seed=SEED_BASE + 3,
                       name="varlen_chunked_16seq_hq32_hkv8_d128", device=device)


# --------------------------------------------------------------------------
# paged decode problems
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Decode:
    name: str
    q: torch.Tensor            # [B, Hq, d]
    k_cache: torch.Tensor      # [P, page, Hkv, d]
    v_cache: torch.Tensor
    block_table: torch.Tensor  # int32 [B, max_pages]
    seq_lens: torch.Tensor     # int32 [B]
    B: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    num_pages: int
    scale: float
    seed: int = 0

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def to(self, device) -> "Decode":
        f = lambda t: t.to(device)
        return dataclasses.replace(self, q=f(self.q), k_cache=f(self.k_cache), v_cache=f(self.v_cache),
                                   block_table=f(self.block_table), seq_lens=f(self.seq_lens))


def make_decode(seq_lens, Hq, Hkv, d, *, num_pages, seed, page_size=16, max_pages=None,
                scale=None, nan_fill_unused=False, name="decode", device="cpu") -> Decode:
    """Pages of a random permutation of the pool are given to the sequences'
    logical pages in order; table entries past a sequence's last page are -1.
    With nan_fill_unused, every slot that no sequence uses (whole unused pages
    and the tail slots of each sequence's last page) holds NaN."""
    seq_lens = [int(x) for x in seq_lens]
    B = len(seq_lens)
    need = [-(-L // page_size) for L in seq_lens]
    if max_pages is None:
        max_pages = max(need + [1])
    if sum(need) > num_pages:
        raise ValueError("pool too small for the requested lengths")
    perm = torch.randperm(num_pages, generator=_gen(seed * 7 + 4))
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    q = randn_bf16((B, Hq, d), seed * 7 + 1, device)
    kc = randn_bf16((num_pages, page_size, Hkv, d), seed * 7 + 2, device)
    vc = randn_bf16((num_pages, page_size, Hkv, d), seed * 7 + 3, device)
    if nan_fill_unused:
        used = torch.zeros(num_pages, page_size, dtype=torch.bool)
        for b, L in enumerate(seq_lens):
            for t in range(0, need[b]):
                pg = int(table[b, t])
                used[pg, : min(page_size, L - t * page_size)] = True
        unused = (~used).to(device)
        kc[unused] = float("nan")
        vc[unused] = float("nan")
    return Decode(name, q, kc, vc, table.to(device),
                  torch.tensor(seq_lens, dtype=torch.int32, device=device),
                  B, Hq, Hkv, d, page_size, num_pages,
                  1.0 / math.sqrt(d) if scale is None else scale, seed=seed)


def decode_lengths(seed=SEED_BASE + 4, n=64, lo=4096, hi=32768):
    return randint(lo, hi, n, seed).tolist()


def paged_decode_small(device="cpu", nan_fill_unused=False) -> Decode:
    """The paged decode layout at one eighth of the lengths (U[512, 4096]) in a
    25,000-page pool (1.6 GB of K+V): a case small enough for multi-pass
    profiler captures of the same kernel."""
    lens = decode_lengths(seed=SEED_BASE + 5, lo=512, hi=4096)
    return make_decode(lens, 32, 8, 128, num_pages=25_000, seed=SEED_BASE + 5, page_size=16,
                       max_pages=256, nan_fill_unused=nan_fill_unused,
                       name="paged_decode_small_b64_hq32_hkv8_d128", device=device)


def paged_decode(device="cpu", nan_fill_unused=False) -> Decode:
    """B=64, Hq=32, Hkv=8, d=128, len ~ U[4096, 32768], 16-token pages in a
    200,000-page pool (one pool each for K and V), block table [64, 2048]."""
    lens = decode_lengths()
    return make_decode(lens, 32, 8, 128, num_pages=200_000, seed=SEED_BASE + 4, page_size=16,
                       max_pages=2048, nan_fill_unused=nan_fill_unused,
                       name="paged_decode_b64_hq32_hkv8_d128", device=device)


@dataclasses.dataclass
class KVCacheDecode:
    """Nq new queries per sequence over a paged cache, with the new tokens'
    K/V appended in place first (k_new None: no append).  seq_lens counts the
    tokens after the append; query i of sequence b is position
    seq_lens[b] - Nq + i."""
    name: str
    q: torch.Tensor            # [B, Nq, Hq, d]
    k_new: Optional[torch.Tensor]  # [B, Nq, Hkv, d] or None
    v_new: Optional[torch.Tensor]
    k_cache: torch.Tensor      # [P, page, Hkv, d]
    v_cache: torch.Tensor
    block_table: torch.Tensor  # int32 [B, max_pages]
    seq_lens: torch.Tensor     # int32 [B]
    B: int
    Nq: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    num_pages: int
    scale: float
    causal: bool
    seed: int = 0

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def to(self, device) -> "KVCacheDecode":
        f = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(self, q=f(self.q), k_new=f(self.k_new), v_new=f(self.v_new),
                                   k_cache=f(self.k_cache), v_cache=f(self.v_cache),
                                   block_table=f(self.block_table), seq_lens=f(self.seq_lens))


def make_kvcache_decode(seq_lens, Nq, Hq, Hkv, d, *, num_pages, seed, causal=True, append=True, page_size=16,
                        max_pages=None, scale=None, nan_fill_unused=False, name="kvcache_decode",
                        device="cpu") -> KVCacheDecode:
    """The cache and block table of make_decode for the lengths after the
    append.  With append, the slots the new tokens will occupy hold NaN until
    the call writes them, so attending before (or without) the write shows."""
    base = make_decode(seq_lens, Hq, Hkv, d, num_pages=num_pages, seed=seed, page_size=page_size,
                       max_pages=max_pages, scale=scale, nan_fill_unused=nan_fill_unused, name=name,
                       device=device)
    B = base.B
    q = randn_bf16((B, Nq, Hq, d), seed * 7 + 5, device)
    k_new = v_new = None
    if append:
        k_new = randn_bf16((B, Nq, Hkv, d), seed * 7 + 6, device)
        v_new = randn_bf16((B, Nq, Hkv, d), seed * 7 + 7, device)
        table = base.block_table.cpu()
        for b, L in enumerate(int(x) for x in seq_lens):
            for i in range(Nq):
                pos = L - Nq + i
                if pos >= 0:
                    pg = int(table[b, pos // page_size])
                    base.k_cache[pg, pos % page_size] = float("nan")
                    base.v_cache[pg, pos % page_size] = float("nan")
    return KVCacheDecode(name, q, k_new, v_new, base.k_cache, base.v_cache, base.block_table, base.seq_lens,
                         B, Nq, Hq, Hkv, d, page_size, num_pages, base.scale, bool(causal), seed=seed)


def spec_decode(device="cpu", nan_fill_unused=False) -> KVCacheDecode:
    """Speculative-decoding verify step: B=64, Nq=4 new tokens per sequence,
    Hq=32, Hkv=8, d=128, len ~ U[4096, 32768] after the append, causal, 16-token
    pages in a 200,000-page pool, block table [64, 2048]."""
    lens = decode_lengths(seed=SEED_BASE + 7)
    return make_kvcache_decode(lens, 4, 32, 8, 128, num_pages=200_000, seed=SEED_BASE + 7, causal=True,
                               append=True, max_pages=2048, nan_fill_unused=nan_fill_unused,
                               name="spec_decode_b64_nq4_hq32_hkv8_d128", device=device)


def spec_decode_small(device="cpu", nan_fill_unused=False) -> KVCacheDecode:
    """The speculative-decoding layout at one eighth of the lengths (U[512,
    4096]) in a 25,000-page pool (1.6 GB of K+V): a case small enough for
    profiler captures of the same kernels."""
    lens = decode_lengths(seed=SEED_BASE + 8, lo=512, hi=4096)
    return make_kvcache_decode(lens, 4, 32, 8, 128, num_pages=25_000, seed=SEED_BASE + 8, causal=True,
                               append=True, max_pages=256, nan_fill_unused=nan_fill_unused,
                               name="spec_decode_small_b64_nq4_hq32_hkv8_d128", device=device)


# --------------------------------------------------------------------------
# row samples and structured inputs
# --------------------------------------------------------------------------
def sample_rows(n_rows_per_seq, lengths, heads, per_head: int, seed: int, tile: int = 128):
    """Seeded sample of (b, h, i) query rows: for every (sequence, head), the
    first and last rows, rows on both sides of every tile boundary (up to the
    budget), then uniform draws without replacement to reach per_head rows."""
    g = _gen(seed)
    out = []
    for b, nq in enumerate(lengths):
        if nq <= 0:
            continue
        for h in range(heads):
            fixed = [0, nq - 1]
            for t in range(tile, nq, tile):
                fixed += [t - 1, t]
            fixed = sorted(set(fixed))
            if len(fixed) >= per_head or nq <= per_head:
                chosen = fixed[:per_head] if nq > per_head else list(range(nq))
            else:
                rest = torch.randperm(nq, generator=g).tolist()
                s = set(fixed)
                chosen = list(fixed)
                for r in rest:
                    if len(chosen) >= per_head:
                        break
                    if r not in s:
                        s.add(r)
                        chosen.append(r)
            out += [(b, h, i) for i in sorted(chosen)]
    return torch.tensor(out, dtype=torch.int32).reshape(-1, 3)


def one_hot_values(p: Prefill, base: int) -> Prefill:
    """Q = 0 and V one-hot by key index inside the window [base, base+d):
    v[key j of sequence b, kv head g, c] = (g+1) if c == j - base else 0.
    Every allowed key then gets weight 1/|A_i|, so O[i, h, c] = (g(h)+1)/|A_i|
    exactly when key base+c is allowed for row i."""
    q = torch.zeros_like(p.q)
    v = torch.zeros_like(p.v)
    lens = p.seq_lens()
    ck = [0] + list(_cumsum([nk for _, nk in lens]))
    for b, (_, nk) in enumerate(lens):
        for c in range(p.d):
            j = base + c
            if 0 <= j < nk:
                for g in range(p.Hkv):
                    v[ck[b] + j, g, c] = float(g + 1)
    return dataclasses.replace(p, q=q, v=v)


def score_ladder(p: Prefill, levels=(0, 4, 4, 13, 13, 2, 20, 0), block: int = 128) -> Prefill:
    """Scores that step by key block: channel 0 of every query row is +8 (even
    query heads) or -8 (odd query heads), channel 0 of key j is
    levels[(j // block) % len(levels)], and the other channels are N(0, 1)/4
    noise from the problem's own draws.  With scale 1/sqrt(128) a level step
    of 1 moves the score by about one unit of log2, so the even heads see the
    running maximum hold, rise a little (many keys of one block above the
    first block's maximum) and jump (far above it); the odd heads see it
    fall.  All values are exact in bf16."""
    q = (p.q.float() * 0.25).to(torch.bfloat16)
    k = (p.k.float() * 0.25).to(torch.bfloat16)
    sign = torch.tensor([8.0 if h % 2 == 0 else -8.0 for h in range(p.Hq)])
    q[:, :, 0] = sign.to(torch.bfloat16)
    lens = p.seq_lens()
    ck = [0] + list(_cumsum([nk for _, nk in lens]))
    for b, (_, nk) in enumerate(lens):
        lv = torch.tensor([float(levels[(j // block) % len(levels)]) for j in range(nk)])
        k[ck[b]:ck[b] + nk, :, 0] = lv[:, None].to(torch.bfloat16)
    return dataclasses.replace(p, q=q, k=k)
