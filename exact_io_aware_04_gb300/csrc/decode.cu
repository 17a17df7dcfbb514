// decode.cu -- paged split-KV decode of exact attention on sm_103a.
//
// attn_decode_split: one CTA per (chunk of a sequence's pages, sequence, group
// of K/V heads).  A producer warp reads the sequence's block-table entries and
// gathers whole pages with one 5-D TMA copy per page for K and one for V
// (all heads of the group, both halves of d, 128-byte swizzled so that every
// head's 16 tokens form a bank-conflict-free tile).  One consumer warp per
// (K/V head, 16 query heads) keeps the query heads that share the K/V head in
// one 16-row tile, so each gathered K/V row is read from shared memory once
// for all of them ("FlashAttention-3 and PagedAttention", section "How GQA and
// MLA reshape the problem"), and runs the online-softmax recurrence over the
// chunk with mma.sync (bf16 in, fp32 accumulate): the tile is too small for
// the fifth-generation tensor core and the kernel is bound by HBM reads.
// Each chunk writes its normalised partial output and its lse.
//
// attn_decode_combine: weights partial i by exp(lse_i - lse_total) and sums
// ("FlashAttention-3 and PagedAttention", section "Why decode starves the
// GPU").
//
// Several new queries per sequence (Nq > 1, "Deep Dive - FlashAttention",
// sections "Causal 2.1 is the decode gotcha" and "Paged KV is a lookup, not a
// cache manager"): the Nq x group query rows that share a K/V head form the
// consumer tiles (row r = i * group + head-in-group), so the gathered page is
// still read once for all of them; with causal, query i is position
// len - Nq + i and its scores past that position are masked on the last pages.
// append_kv_kernel writes the new tokens' K/V into their cache slots first.
//
// Slots at or beyond the sequence length are excluded by selection (their
// score is replaced by -inf and their V entries by zero before any multiply),
// so NaN bits in unused cache slots cannot reach the output.
#include <cuda_bf16.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kPage = 16;            // tokens per page (the only supported page size)
constexpr int kStageBudget = 196608;  // bytes of shared memory for the page ring
constexpr float kRescaleThreshold = 8.0f;

struct DecodeParams {
    CUtensorMap tm_k;  // 5-D view of the K pool: {64, slot, head, d/64, page}
    CUtensorMap tm_v;
    const __nv_bfloat16* q;  // [B, nq, Hq, d]
    const int* block_table;
    const int* seq_lens;
    float* part_o;     // [B, Hq, nq, max_chunks, d]
    float* part_lse;   // [B, Hq, nq, max_chunks]
    int B, Hq, Hkv, group, num_pages, max_pages;
    int nq, causal;    // queries per sequence; bottom-right causal among them
    int pages_per_chunk, max_chunks, head_groups, heads_per_cta, m_tiles;
    float scale_log2;
    int validate;
    int drop_first_page;  // test hook: CTA (0, 0) skips its first page copy
    int* err;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D = A(16x16 bf16) * B(16x8 bf16) + D, fp32.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Address of 16-byte chunk `ch` (0 .. d/8-1) of token `tok` of head `hh` inside
// one gathered page box laid out [d/64][heads][slot][64] with 128B swizzle.
__device__ __forceinline__ uint32_t box_addr(uint32_t base, int hh, int heads, int tok, int ch) {
    const int line = ((ch >> 3) * heads + hh) * kPage + tok;
    return base + line * 128 + (((ch & 7) ^ (line & 7)) << 4);
}

template <int HD>
__global__ void __launch_bounds__(288, 1) attn_decode_split_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int KB = HD / 16;   // k16 blocks of the score product
    constexpr int NB = HD / 8;    // n8 blocks of the output
    extern __shared__ __align__(1024) uint8_t smem_dyn[];
    __shared__ __align__(8) uint64_t bar_full[8], bar_empty[8];

    // the combine kernel (a programmatic dependent launch) may be placed as
    // soon as every CTA here has started; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int chunk = blockIdx.x;
    // (sequence, head group) units run over grid y and z (y at most 65535;
    // the host keeps B * head_groups below 2^31)
    const int unit = static_cast<int>(blockIdx.z * gridDim.y + blockIdx.y);
    if (unit >= p.B * p.head_groups) return;  // padding of the last z slice
    const int b = unit / p.head_groups;
    const int hg = unit - b * p.head_groups;
    const int cap = p.max_pages * kPage;
    const int len = min(max(__ldg(p.seq_lens + b), 0), cap);
    const int tok0 = chunk * p.pages_per_chunk * kPage;
    if (tok0 >= len) return;  // uniform for the CTA: nothing to do, nothing written
    const int tok1 = min(len, tok0 + p.pages_per_chunk * kPage);
    const int n_pages = (tok1 - tok0 + kPage - 1) / kPage;
    const int page0 = tok0 / kPage;

    const int HG = p.heads_per_cta;
    const uint32_t box_bytes = kPage * HG * HD * 2;
    const uint32_t stage_bytes = 2 * box_bytes;
    const int n_stages = min(8, kStageBudget / static_cast<int>(stage_bytes));
    const uint32_t smem0 = (smem_addr(smem_dyn) + 1023u) & ~1023u;
    const int n_consumers = HG * p.m_tiles;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < n_stages; ++s) {
            mbar_init(smem_addr(&bar_full[s]), 1);
            mbar_init(smem_addr(&bar_empty[s]), n_consumers);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_map(&p.tm_k);
            tma_prefetch_map(&p.tm_v);
        }
        const int* bt = p.block_table + static_cast<size_t>(b) * p.max_pages + page0;
        bool ok = true;
        int issued = 0;
        for (int base = 0; base < n_pages && ok; base += 32) {
            // 32 table entries per round trip, one per lane
            int my_page = 0;
            if (base + lane < n_pages) {
                my_page = __ldg(bt + base + lane);
                if (my_page < 0 || my_page >= p.num_pages) {
                    if (p.validate) record_error(p.err, ATTN_ERR_BAD_INDEX);
                    my_page = -1;  // a TMA box outside the pool reads zeros
                }
            }
            const int cnt = min(32, n_pages - base);
            for (int i = 0; i < cnt; ++i) {
                const int page = __shfl_sync(0xffffffffu, my_page, i);
                if (lane == 0) {
                    const int it = base + i;
                    const int st = it % n_stages;
                    if (it >= n_stages) ok = mbar_wait(smem_addr(&bar_empty[st]), ((it / n_stages) - 1) & 1, p.err);
                    const bool drop = p.drop_first_page && it == 0 && blockIdx.x == 0 && blockIdx.y == 0;
                    if (ok && !drop) {
                        const uint32_t dst = smem0 + st * stage_bytes;
                        mbar_arrive_expect_tx(smem_addr(&bar_full[st]), stage_bytes);
                        tma_load_5d(dst, &p.tm_k, smem_addr(&bar_full[st]), 0, 0, hg * HG, 0, page);
                        tma_load_5d(dst + box_bytes, &p.tm_v, smem_addr(&bar_full[st]), 0, 0, hg * HG, 0, page);
                        ++issued;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
            }
        }
        if (lane == 0) {
            // drain: every issued copy has landed before the CTA may exit
            const int first = p.drop_first_page && blockIdx.x == 0 && blockIdx.y == 0 ? 1 : 0;
            for (int it = max(first, issued + first - n_stages); it < issued + first; ++it)
                mbar_wait(smem_addr(&bar_full[it % n_stages]), (it / n_stages) & 1, p.err);
        }
        __syncwarp();
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int cw = warp - 1;
    if (cw >= n_consumers) return;
    const int hh = cw / p.m_tiles;                  // K/V head inside the group
    const int mt = cw - hh * p.m_tiles;             // 16-row tile of its query rows
    const int g = hg * HG + hh;                     // global K/V head
    const int R = p.group * p.nq;                   // query rows per K/V head
    const int rows = min(16, R - mt * 16);          // real query rows in this tile
    const int r0 = lane >> 2, r1 = r0 + 8;          // accumulator rows of this lane
    const int cq = (lane & 3) * 2;                  // column pair inside an 8-wide block
    // row r of the tile is query i = (16 mt + r) / group of query head g*group + (16 mt + r) % group
    const int i0 = (mt * 16 + r0) / p.group, i1 = (mt * 16 + r1) / p.group;
    const int h_r0 = g * p.group + (mt * 16 + r0 - i0 * p.group);
    const int h_r1 = g * p.group + (mt * 16 + r1 - i1 * p.group);
    // last key each row may see (inclusive): position len - nq + i under causal
    const int lim0 = p.causal ? len - p.nq + i0 : len - 1;
    const int lim1 = p.causal ? len - p.nq + i1 : len - 1;
    const int first_limited = p.causal ? len - p.nq : len;  // pages reaching past this need the row limits

    // Q fragments (A operand), rows >= `rows` are zero
    uint32_t qa[KB][4];
    {
        const __nv_bfloat16* qr0 = p.q + ((static_cast<size_t>(b) * p.nq + i0) * p.Hq + h_r0) * HD;
        const __nv_bfloat16* qr1 = p.q + ((static_cast<size_t>(b) * p.nq + i1) * p.Hq + h_r1) * HD;
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            const int c0 = kb * 16 + cq;
            qa[kb][0] = r0 < rows ? *reinterpret_cast<const uint32_t*>(qr0 + c0) : 0u;
            qa[kb][1] = r1 < rows ? *reinterpret_cast<const uint32_t*>(qr1 + c0) : 0u;
            qa[kb][2] = r0 < rows ? *reinterpret_cast<const uint32_t*>(qr0 + c0 + 8) : 0u;
            qa[kb][3] = r1 < rows ? *reinterpret_cast<const uint32_t*>(qr1 + c0 + 8) : 0u;
        }
    }
    float o[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
    float m_ref[2] = {-INFINITY, -INFINITY};
    float l_part[2] = {0.f, 0.f};
    const float sl2 = p.scale_log2;
    bool ok = true;

    // ldmatrix row addresses: K (non-transposed) and V (transposed) patterns
    const int k_tok = (lane & 7) + ((lane >> 4) << 3);
    const int k_chsel = (lane >> 3) & 1;
    const int v_tok = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int v_chsel = lane >> 4;

    for (int it = 0; it < n_pages; ++it) {
        const int st = it % n_stages;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_full[st]), (it / n_stages) & 1, p.err));
        if (!ok) break;
        const uint32_t kbase = smem0 + st * stage_bytes;
        const uint32_t vbase = kbase + box_bytes;
        const int valid = min(kPage, tok1 - (tok0 + it * kPage));  // tokens of this page in the chunk

        // ---- S = Q K^T for the page's 16 tokens (two n8 tiles)
        float s[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            uint32_t b00, b01, b10, b11;
            ldsm_x4(box_addr(kbase, hh, HG, k_tok, 2 * kb + k_chsel), b00, b01, b10, b11);
            mma_16816(s[0], qa[kb], b00, b01);
            mma_16816(s[1], qa[kb], b10, b11);
        }
        if (valid < kPage) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int t0 = nt * 8 + cq;
                if (t0 >= valid) { s[nt][0] = -INFINITY; s[nt][2] = -INFINITY; }
                if (t0 + 1 >= valid) { s[nt][1] = -INFINITY; s[nt][3] = -INFINITY; }
            }
        }
        const int pt = tok0 + it * kPage;  // position of the page's first token
        if (pt + kPage - 1 > first_limited) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int t0 = pt + nt * 8 + cq;
                if (t0 > lim0) s[nt][0] = -INFINITY;
                if (t0 + 1 > lim0) s[nt][1] = -INFINITY;
                if (t0 > lim1) s[nt][2] = -INFINITY;
                if (t0 + 1 > lim1) s[nt][3] = -INFINITY;
            }
        }
        // ---- row maxima (rows r0, r1), reduced over the 4 lanes of a quad
        float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
        float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float t0 = mx0 * sl2, t1 = mx1 * sl2;
        if (it == 0) {
            m_ref[0] = t0;
            m_ref[1] = t1;
        } else {
            const bool need = (t0 > m_ref[0] + kRescaleThreshold) || (t1 > m_ref[1] + kRescaleThreshold);
            if (__any_sync(0xffffffffu, need)) {
                const float n0 = fmaxf(m_ref[0], t0), n1 = fmaxf(m_ref[1], t1);
                const float a0 = n0 == -INFINITY ? 1.f : fast_exp2(m_ref[0] - n0);
                const float a1 = n1 == -INFINITY ? 1.f : fast_exp2(m_ref[1] - n1);
                m_ref[0] = n0;
                m_ref[1] = n1;
                l_part[0] *= a0;
                l_part[1] *= a1;
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    o[nb][0] *= a0;
                    o[nb][1] *= a0;
                    o[nb][2] *= a1;
                    o[nb][3] *= a1;
                }
            }
        }
        const float u0 = m_ref[0] == -INFINITY ? 0.f : m_ref[0];
        const float u1 = m_ref[1] == -INFINITY ? 0.f : m_ref[1];
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            pr[nt][0] = fast_exp2(fmaf(s[nt][0], sl2, -u0));
            pr[nt][1] = fast_exp2(fmaf(s[nt][1], sl2, -u0));
            pr[nt][2] = fast_exp2(fmaf(s[nt][2], sl2, -u1));
            pr[nt][3] = fast_exp2(fmaf(s[nt][3], sl2, -u1));
            l_part[0] += pr[nt][0] + pr[nt][1];
            l_part[1] += pr[nt][2] + pr[nt][3];
        }
        // P as a bf16 pair hi + lo (lo = the rounding residual of hi): the
        // weights then carry about 16 significant bits, so rows with few keys
        // are not limited by an 8-bit P; two MMAs per fragment cost nothing
        // on this HBM-bound path.
        uint32_t pa[4], pl[4];
        pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
        pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
        pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
        pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float a = pr[c >> 1][(c & 1) * 2], bb = pr[c >> 1][(c & 1) * 2 + 1];
            pl[c] = pack_bf16x2(a - bf16_lo(pa[c]), bb - bf16_hi(pa[c]));
        }

        // ---- O += P V
        // B-fragment token rows of this lane: cq, cq+1 (b0) and 8+cq, 9+cq (b1)
        const uint32_t keep_lo0 = (cq < valid) ? 0x0000FFFFu : 0u;
        const uint32_t keep_hi0 = (cq + 1 < valid) ? 0xFFFF0000u : 0u;
        const uint32_t keep_lo1 = (cq + 8 < valid) ? 0x0000FFFFu : 0u;
        const uint32_t keep_hi1 = (cq + 9 < valid) ? 0xFFFF0000u : 0u;
        const uint32_t keep0 = keep_lo0 | keep_hi0, keep1 = keep_lo1 | keep_hi1;
#pragma unroll
        for (int nb = 0; nb < NB; nb += 2) {
            uint32_t v00, v01, v10, v11;
            ldsm_x4_t(box_addr(vbase, hh, HG, v_tok, nb + v_chsel), v00, v01, v10, v11);
            if (valid < kPage) {
                v00 &= keep0;
                v01 &= keep1;
                v10 &= keep0;
                v11 &= keep1;
            }
            mma_16816(o[nb], pa, v00, v01);
            mma_16816(o[nb + 1], pa, v10, v11);
            mma_16816(o[nb], pl, v00, v01);
            mma_16816(o[nb + 1], pl, v10, v11);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bar_empty[st]));
    }
    if (!ok) return;

    // ---- normalise and write this chunk's partial (O / l, lse)
    float l0 = l_part[0], l1 = l_part[1];
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
    const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const size_t slot0 = ((static_cast<size_t>(b) * p.Hq + h_r0) * p.nq + i0) * p.max_chunks + chunk;
    const size_t slot1 = ((static_cast<size_t>(b) * p.Hq + h_r1) * p.nq + i1) * p.max_chunks + chunk;
    if (r0 < rows) {
        float* dst = p.part_o + slot0 * HD;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
            *reinterpret_cast<float2*>(dst + nb * 8 + cq) = make_float2(o[nb][0] * inv0, o[nb][1] * inv0);
        if ((lane & 3) == 0) p.part_lse[slot0] = l0 > 0.f ? (m_ref[0] + log2f(l0)) * 0.69314718055994531f : -INFINITY;
    }
    if (r1 < rows) {
        float* dst = p.part_o + slot1 * HD;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
            *reinterpret_cast<float2*>(dst + nb * 8 + cq) = make_float2(o[nb][2] * inv1, o[nb][3] * inv1);
        if ((lane & 3) == 0) p.part_lse[slot1] = l1 > 0.f ? (m_ref[1] + log2f(l1)) * 0.69314718055994531f : -INFINITY;
    }
}

struct CombineParams {
    const float* part_o;
    const float* part_lse;
    const int* seq_lens;
    __nv_bfloat16* out;  // [B, nq, Hq, d]
    float* lse;          // [B, Hq, nq]
    int B, Hq, nq, max_pages, pages_per_chunk, max_chunks;
};

// One block of kCombineWarps warps per (sequence, query head, query) row:
// lse = log sum_i exp(lse_i), O = sum_i exp(lse_i - lse) O_i over the chunks
// the sequence actually has.  Warp w takes chunks w, w + kCombineWarps, ...;
// lane l of a warp owns d-elements [l*d/32, (l+1)*d/32) as one vector load per chunk.
// The maximum and the normaliser are reduced across the block first, then
// every warp accumulates its chunks and the warps' sums are added in shared
// memory.  Several warps per row keep enough loads in flight to stream the
// partials at memory speed; the chunks are dealt round-robin to the warps.
constexpr int kCombineWarps = 4;

template <int HD>
__global__ void __launch_bounds__(32 * kCombineWarps) attn_decode_combine_kernel(const CombineParams p) {
    constexpr int V = HD / 32;  // floats per lane
    using Vec = typename std::conditional<V == 4, float4, float2>::type;
    __shared__ float red[kCombineWarps];
    __shared__ float acc_s[kCombineWarps][HD];
    // launched as a programmatic dependent of the split kernel: wait until
    // that grid has completed and its partials are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int row = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = row / (p.Hq * p.nq);
    const int hq = (row - b * p.Hq * p.nq) / p.nq;
    const int qi = row - (b * p.Hq + hq) * p.nq;
    const int len = min(max(__ldg(p.seq_lens + b), 0), p.max_pages * kPage);
    const int chunk_tokens = p.pages_per_chunk * kPage;
    const int n = (len + chunk_tokens - 1) / chunk_tokens;
    const float* lse_s = p.part_lse + static_cast<size_t>(row) * p.max_chunks;
    // row maximum of the chunk lse
    float mx = -INFINITY;
    for (int i = threadIdx.x; i < n; i += 32 * kCombineWarps) mx = fmaxf(mx, __ldg(lse_s + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < kCombineWarps; ++w) mx = fmaxf(mx, red[w]);
    __nv_bfloat16* dst = p.out + ((static_cast<size_t>(b) * p.nq + qi) * p.Hq + hq) * HD;
    if (mx == -INFINITY) {  // no keys: O = 0, lse = -inf
        if (threadIdx.x == 0) p.lse[row] = -INFINITY;
        for (int c = threadIdx.x; c < HD; c += 32 * kCombineWarps) dst[c] = __float2bfloat16_rn(0.f);
        return;
    }
    // normaliser
    float total = 0.f;
    for (int i = threadIdx.x; i < n; i += 32 * kCombineWarps) total += expf(__ldg(lse_s + i) - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    __syncthreads();  // every warp has read red[] above
    if (lane == 0) red[warp] = total;
    __syncthreads();
    total = red[0];
#pragma unroll
    for (int w = 1; w < kCombineWarps; ++w) total += red[w];
    const float lse_tot = mx + logf(total);
    // this warp's chunks, weighted
    float acc[V];
#pragma unroll
    for (int c = 0; c < V; ++c) acc[c] = 0.f;
    const float* po = p.part_o + static_cast<size_t>(row) * p.max_chunks * HD + lane * V;
    // rounds of 32 * kCombineWarps chunks: warp w takes chunks c0 + w + kCombineWarps * k,
    // lane k holding that chunk's weight
    for (int c0 = 0; c0 < n; c0 += 32 * kCombineWarps) {
        const int mine = c0 + warp + kCombineWarps * lane;
        const float li = mine < n ? __ldg(lse_s + mine) : -INFINITY;
        const float wl = li == -INFINITY ? 0.f : expf(li - lse_tot);
        const int m = min(32, (n - c0 - warp + kCombineWarps - 1) / kCombineWarps);  // this warp's chunks
#pragma unroll 8
        for (int k = 0; k < m; ++k) {
            const float w = __shfl_sync(0xffffffffu, wl, k);
            const int ch = c0 + warp + kCombineWarps * k;
            const Vec x = __ldg(reinterpret_cast<const Vec*>(po + static_cast<size_t>(ch) * HD));
            const float* xs = reinterpret_cast<const float*>(&x);
#pragma unroll
            for (int c = 0; c < V; ++c) acc[c] = fmaf(w, xs[c], acc[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < V; ++c) acc_s[warp][lane * V + c] = acc[c];
    __syncthreads();
    for (int c = threadIdx.x; c < HD; c += 32 * kCombineWarps) {
        float s = acc_s[0][c];
#pragma unroll
        for (int w = 1; w < kCombineWarps; ++w) s += acc_s[w][c];
        dst[c] = __float2bfloat16_rn(s);
    }
    if (threadIdx.x == 0) p.lse[row] = lse_tot;
}

// In-place cache append: new row i of sequence b goes to position
// len - nq + i, i.e. slot pos % 16 of page block_table[b][pos / 16].  One
// block per (sequence, new token) copies its [Hkv, d] row with 16-byte stores.
// Positions below zero or past the table, and page ids outside the pool, are
// never written (with validation on they are reported as ATTN_ERR_BAD_INDEX).
__global__ void __launch_bounds__(128) append_kv_kernel(const uint4* k_new, const uint4* v_new, uint4* k_cache,
                                                        uint4* v_cache, const int* block_table, const int* seq_lens,
                                                        int nq, int row_vecs, int max_pages, int num_pages,
                                                        int validate, int* err) {
    const int b = blockIdx.x / nq;
    const int i = blockIdx.x - b * nq;
    const int len = __ldg(seq_lens + b);
    const int pos = len - nq + i;
    bool bad = pos < 0 || pos >= max_pages * kPage;
    int pg = -1;
    if (!bad) {
        pg = __ldg(block_table + static_cast<size_t>(b) * max_pages + pos / kPage);
        bad = pg < 0 || pg >= num_pages;
    }
    if (bad) {
        if (validate && threadIdx.x == 0) record_error(err, ATTN_ERR_BAD_INDEX);
        return;
    }
    const size_t src = static_cast<size_t>(blockIdx.x) * row_vecs;
    const size_t dst = (static_cast<size_t>(pg) * kPage + pos % kPage) * row_vecs;
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) {
        k_cache[dst + c] = __ldg(k_new + src + c);
        v_cache[dst + c] = __ldg(v_new + src + c);
    }
}

// Optional check of seq_lens and of the block-table entries each sequence uses.
__global__ void check_pages_kernel(const int* block_table, const int* seq_lens, int max_pages, int num_pages,
                                   int* err) {
    const int b = blockIdx.x;
    const int len = seq_lens[b];
    if (threadIdx.x == 0 && (len < 0 || len > max_pages * kPage)) record_error(err, ATTN_ERR_BAD_INDEX);
    const int used = (min(max(len, 0), max_pages * kPage) + kPage - 1) / kPage;
    for (int i = threadIdx.x; i < used; i += blockDim.x) {
        const int pg = block_table[static_cast<size_t>(b) * max_pages + i];
        if (pg < 0 || pg >= num_pages) record_error(err, ATTN_ERR_BAD_INDEX);
    }
}

template <int HD>
attn_status launch_typed(const DecodeArgs& a, const DecodePlan& plan, const DeviceInfo& dev, cudaStream_t stream) {
    DecodeParams p;
    memset(&p, 0, sizeof(p));
    const int HG = plan.heads_per_cta;
    const uint64_t dims[5] = {64, static_cast<uint64_t>(kPage), static_cast<uint64_t>(a.Hkv),
                              static_cast<uint64_t>(HD / 64), static_cast<uint64_t>(a.num_pages)};
    const uint64_t strides[4] = {static_cast<uint64_t>(a.Hkv) * HD * 2, static_cast<uint64_t>(HD) * 2, 128,
                                 static_cast<uint64_t>(kPage) * a.Hkv * HD * 2};
    const uint32_t box[5] = {64, static_cast<uint32_t>(kPage), static_cast<uint32_t>(HG),
                             static_cast<uint32_t>(HD / 64), 1};
    attn_status st = encode_tma_bf16(&p.tm_k, a.k_cache, 5, dims, strides, box, true);
    if (st != ATTN_OK) return st;
    st = encode_tma_bf16(&p.tm_v, a.v_cache, 5, dims, strides, box, true);
    if (st != ATTN_OK) return st;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.block_table = a.block_table;
    p.seq_lens = a.seq_lens;
    p.part_o = static_cast<float*>(a.workspace);
    p.part_lse = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + plan.partial_o_bytes);
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.group = a.Hq / a.Hkv;
    p.num_pages = a.num_pages;
    p.max_pages = a.max_pages;
    p.pages_per_chunk = plan.pages_per_chunk;
    p.max_chunks = plan.max_chunks;
    p.head_groups = plan.head_groups;
    p.heads_per_cta = HG;
    p.nq = a.nq;
    p.causal = a.causal ? 1 : 0;
    p.m_tiles = (p.group * a.nq + 15) / 16;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.validate = validation_enabled() ? 1 : 0;
    p.drop_first_page = set_drop_page_load(0);  // consume the one-shot test switch
    p.err = dev.err_word;

    // the split grid: (sequence, head group) units over y and z, checked
    // before anything is launched (the append writes the cache)
    const long long units = static_cast<long long>(a.B) * plan.head_groups;
    const unsigned gy = static_cast<unsigned>(std::min<long long>(std::max<long long>(units, 1), 65535));
    const unsigned gz = static_cast<unsigned>((units + gy - 1) / gy);
    if (gz > 65535 || units > 0x7fffffffLL) {
        set_error_message("attn_decode: %lld (sequence, head group) units exceed the grid", units);
        return ATTN_ERR_UNSUPPORTED;
    }
    if (p.validate)
        check_pages_kernel<<<a.B, 128, 0, stream>>>(a.block_table, a.seq_lens, a.max_pages, a.num_pages,
                                                    dev.err_word);
    if (a.k_new != nullptr) {
        append_kv_kernel<<<a.B * a.nq, 128, 0, stream>>>(
            static_cast<const uint4*>(a.k_new), static_cast<const uint4*>(a.v_new), static_cast<uint4*>(a.k_cache_w),
            static_cast<uint4*>(a.v_cache_w), a.block_table, a.seq_lens, a.nq, a.Hkv * HD / 8, a.max_pages,
            a.num_pages, p.validate, dev.err_word);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) {
            set_error_message("append_kv launch: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
    }
    const int stage_bytes = 2 * kPage * HG * HD * 2;
    const int n_stages = std::min(8, kStageBudget / stage_bytes);
    const int smem = n_stages * stage_bytes + 1024;
    static std::atomic<bool> attr_set[kMaxDevices];  // per instantiation and device
    const bool cached = dev.device >= 0 && dev.device < kMaxDevices;
    if (!cached || !attr_set[dev.device].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(attn_decode_split_kernel<HD>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBudget + 1024);
        if (e != cudaSuccess) {
            set_error_message("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        if (cached) attr_set[dev.device].store(true, std::memory_order_release);
    }
    const int threads = 32 * (1 + HG * p.m_tiles);
    dim3 grid(plan.max_chunks, gy, gz);
    attn_decode_split_kernel<HD><<<grid, threads, smem, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error_message("attn_decode_split launch: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    CombineParams c;
    c.part_o = p.part_o;
    c.part_lse = p.part_lse;
    c.seq_lens = a.seq_lens;
    c.out = static_cast<__nv_bfloat16*>(a.out);
    c.lse = a.lse;
    c.B = a.B;
    c.Hq = a.Hq;
    c.nq = a.nq;
    c.max_pages = a.max_pages;
    c.pages_per_chunk = plan.pages_per_chunk;
    c.max_chunks = plan.max_chunks;
    const int rows = a.B * a.Hq * a.nq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows));
    cfg.blockDim = dim3(32 * kCombineWarps);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, attn_decode_combine_kernel<HD>, c);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error_message("attn_decode_combine launch: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

}  // namespace

namespace {
std::atomic<int> g_drop_page_load{0};
}  // namespace

int set_drop_page_load(int enabled) { return g_drop_page_load.exchange(enabled ? 1 : 0); }

bool make_decode_plan(int B, int nq, int Hq, int Hkv, int d, int page_size, int max_pages, int num_splits,
                      DecodePlan* plan) {
    if (B < 0 || nq <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_pages <= 0 || num_splits < 0) return false;
    if (page_size != kPage || (d != 64 && d != 128)) return false;
    const int group = Hq / Hkv;
    if (static_cast<long long>(group) * nq > 128) return false;
    const int m_tiles = (group * nq + 15) / 16;
    if (m_tiles > 8) return false;
    // largest divisor of Hkv whose page box fits a 32 KB stage half and 8 consumer warps
    int hg = 1;
    for (int c = 1; c <= Hkv; ++c)
        if (Hkv % c == 0 && c * d <= 1024 && c * m_tiles <= 8) hg = c;
    plan->heads_per_cta = hg;
    plan->head_groups = Hkv / hg;
    int ppc;
    if (num_splits > 0) {
        ppc = (max_pages + num_splits - 1) / num_splits;
    } else {
        // about 1216 chunks if every sequence were at its longest (8 per SM of a
        // 152-SM part), a power of two in [4, 256] pages.  Several queries per
        // sequence multiply the partials each chunk writes, so they get fewer,
        // longer chunks: 608 for Nq = 2, 304 from Nq = 4 on (measured best on the
        // 64-sequence 4K-32K-token workloads).
        const long long pages = static_cast<long long>(B > 0 ? B : 1) * plan->head_groups * max_pages;
        long long target = pages / (2432 / (2 * nq < 8 ? 2 * nq : 8));
        ppc = 4;
        while (ppc < 256 && 2LL * ppc <= target) ppc *= 2;
    }
    if (ppc < 1) ppc = 1;
    plan->pages_per_chunk = ppc;
    plan->max_chunks = (max_pages + ppc - 1) / ppc;
    const size_t rows = static_cast<size_t>(B) * Hq * nq * plan->max_chunks;
    plan->partial_o_bytes = (rows * d * sizeof(float) + 255) / 256 * 256;
    plan->partial_lse_bytes = (rows * sizeof(float) + 255) / 256 * 256;
    plan->total_bytes = plan->partial_o_bytes + plan->partial_lse_bytes;
    return true;
}

attn_status launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    DeviceInfo dev;
    attn_status st = current_device_info(&dev);
    if (st != ATTN_OK) return st;
    if (a.d == 128) return launch_typed<128>(a, plan, dev, stream);
    if (a.d == 64) return launch_typed<64>(a, plan, dev, stream);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
