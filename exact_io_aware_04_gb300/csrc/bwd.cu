// bwd.cu -- backward of exact attention on sm_103a, by recomputation.
//
// For a nonempty row i with G = dL/dO ("Deep Dive - FlashAttention", section
// "Backward recomputes tiles on purpose"; "FlashAttention: Part 1", section
// 3.6): P = exp(S - lse) is rebuilt tile by tile from the saved lse,
//   dV = P^T G,  dP = G V^T,  D = rowsum(G o O),  dS = P o (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q,
// and masked probabilities (and their gradients) are zero.  Three kernels:
//
//   attn_bwd_dot_kernel   D = rowsum(G o O) in fp32, d/8 threads per row.
//   attn_bwd_dkdv_kernel  one CTA per (sequence, K/V head, 128-key tile): K_j
//                         and V_j stay in shared memory while the (Q_i, G_i)
//                         tiles of every query head of the group stream past;
//                         per step the tensor core runs S^T = K_j Q_i^T and
//                         dP^T = V_j G_i^T, the softmax warps turn them into
//                         P^T and dS^T (bf16, written back into tensor memory
//                         over the fp32 tiles), and the tensor core
//                         accumulates dV += P^T G_i and dK += dS^T Q_i with
//                         the left operand read from tensor memory.
//   attn_bwd_dq_kernel    one CTA per (sequence, query head, 128-row tile):
//                         Q_i and G_i stay, (K_j, V_j) stream; S = Q_i K_j^T,
//                         dP = G_i V_j^T, dS, and dQ += dS K_j.
//
// Computing dQ in its own pass (three products instead of one more in the
// K/V pass) needs no atomic accumulation, so the result is deterministic, and
// each pass fits its accumulators in the 512 tensor-memory columns of one SM.
// The issue order overlaps the softmax work with the tensor core: in the K/V
// pass the tensor core runs dV(s), S^T(s+1), dK(s), dP^T(s+1) while the
// softmax warps produce P^T(s+1) and dS^T(s+1); in the dQ pass it runs
// S(u+1), dQ(u), dP(u+1).
#include <cuda_bf16.h>
#include <math.h>
#include <string.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;  // rows of every tile (keys or queries)
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 208;  // warpgroups 0 and 1
constexpr int kControlRegs = 88;   // warpgroup 2
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kSoftmaxWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;

// Tiled TMA store shared -> global of one box (bulk-group completion).  The
// writer threads make their shared-memory writes visible to the async proxy
// (fence_proxy_async_shared) and hand over through an mbarrier before one
// thread issues it.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk group has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <int HD>
struct Tile {
    static constexpr int kPanels = HD / 64;
    static constexpr int kPanelBytes = kBM * 128;
    static constexpr int kBytes = kPanels * kPanelBytes;
};

struct BwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;  // 2-D [rows, heads*d] bf16, box 64 x 128, 128B swizzle
    CUtensorMap tm_dq, tm_dk, tm_dv;      // the same layout over the outputs (tiled stores)
    int tma_store;                        // 1 when every output is 16-byte aligned
    const float* lse;                      // dense [B, Hq, Nq]; packed [Hq, T_q]
    // workspace: -lse * log2 e and -D, each [Hq][ws_row] fp32 (negated so
    // that the softmax threads use them in packed fma / add directly);
    // sequence b's rows start at ws_offset(b), so every 128-row tile starts
    // 16-byte aligned
    const float* nlse2;
    const float* ndvec;
    long long ws_row;
    __nv_bfloat16 *dq, *dk, *dv;
    const int *cu_q, *cu_k;
    int B, Hq, Hkv, group, Nq, Nk;
    int win_left, win_right;               // < 0 unbounded; causal is right = 0
    int varlen;
    float scale, scale_log2;
    int* err;
};

struct Seq {
    int q_base, k_base, nq, nk;
};

__device__ __forceinline__ int clampi(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

__device__ __forceinline__ Seq seq_of(const BwdParams& p, int b) {
    Seq s;
    if (p.varlen) {
        const int q0 = clampi(__ldg(p.cu_q + b), 0, p.Nq);
        const int q1 = clampi(__ldg(p.cu_q + b + 1), q0, p.Nq);
        const int k0 = clampi(__ldg(p.cu_k + b), 0, p.Nk);
        const int k1 = clampi(__ldg(p.cu_k + b + 1), k0, p.Nk);
        s.q_base = q0;
        s.nq = q1 - q0;
        s.k_base = k0;
        s.nk = k1 - k0;
    } else {
        s.q_base = b * p.Nq;
        s.nq = p.Nq;
        s.k_base = b * p.Nk;
        s.nk = p.Nk;
    }
    return s;
}

// Allowed keys of local query row i: [key_first, key_last] (inclusive, clamped
// to [-1, nk]); the band of the forward pass.
__device__ __forceinline__ int key_first(long long i, int nq, int nk, int left) {
    if (left < 0) return 0;
    const long long k = i + nk - nq - left;
    return static_cast<int>(k < 0 ? 0 : (k > nk ? nk : k));
}
__device__ __forceinline__ int key_last(long long i, int nq, int nk, int right) {
    if (right < 0) return nk - 1;
    const long long k = i + nk - nq + right;
    return static_cast<int>(k < -1 ? -1 : (k > nk - 1 ? nk - 1 : k));
}
// Query rows that see key j: [row_first, row_last] (inclusive, clamped to [-1, nq]).
__device__ __forceinline__ int row_first(long long j, int nq, int nk, int right) {
    if (right < 0) return 0;
    const long long i = j - (nk - nq) - right;
    return static_cast<int>(i < 0 ? 0 : (i > nq ? nq : i));
}
__device__ __forceinline__ int row_last(long long j, int nq, int nk, int left) {
    if (left < 0) return nq - 1;
    const long long i = j - (nk - nq) + left;
    return static_cast<int>(i < -1 ? -1 : (i > nq - 1 ? nq - 1 : i));
}

__device__ __forceinline__ size_t lse_index(const BwdParams& p, int b, int h, const Seq& s, int i) {
    return p.varlen ? static_cast<size_t>(h) * p.Nq + s.q_base + i
                    : (static_cast<size_t>(b) * p.Hq + h) * p.Nq + i;
}

// First workspace element of sequence b (first query row q_base): 16-byte
// aligned, and far enough from sequence b-1's rows.
__host__ __device__ __forceinline__ long long ws_offset(int b, long long q_base) {
    return 4 * ((q_base + 3) / 4) + 4LL * b;
}
// Row length of one head in the workspace: every sequence's offset plus a full
// 128-row tile past the last row (a multiple of 4 floats).
__host__ __device__ __forceinline__ long long bwd_ws_row(int B, long long t_q) {
    return ws_offset(B, t_q) + kBM + 4;
}

// Sequence b and tile t of item x of the packed-mode list: the tiles of
// sequence b (of `rows_per_tile`-row tiles over its nq or nk rows) come after
// those of sequences 0..b-1.  One warp scans cu_seqlens 32 sequences at a time.
__device__ bool find_tile(const BwdParams& p, int x, bool over_keys, int& b_out, int& t_out) {
    const int lane = threadIdx.x & 31;
    int before = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int n = 0;
        if (b < p.B) {
            const Seq s = seq_of(p, b);
            n = ((over_keys ? s.nk : s.nq) + kBM - 1) / kBM;
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (x < before + total) {
            const unsigned hit = __ballot_sync(0xffffffffu, b < p.B && x < before + incl);
            const int l = __ffs(hit) - 1;
            const int excl = __shfl_sync(0xffffffffu, incl - n, l);
            b_out = b0 + l;
            t_out = x - before - excl;
            return true;
        }
        before += total;
    }
    return false;
}

__device__ __forceinline__ uint32_t bar_at(uint32_t bar0, int idx) { return bar0 + 8u * static_cast<uint32_t>(idx); }

// 64 consecutive fp32 values at shared address `saddr` (16-byte aligned), as 16 vector loads.
__device__ __forceinline__ void lds_64(uint32_t saddr, float* r) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(r[4 * i]), "=f"(r[4 * i + 1]), "=f"(r[4 * i + 2]), "=f"(r[4 * i + 3])
                     : "r"(saddr + 16u * i));
}

// P of 64 columns: p[c] = 2^(x[c] * sc + b[c]), with sc = scale * log2 e and
// b = -lse * log2 e (per column in the K/V pass, one value per row in the dQ
// pass); the argument in packed fp32x2 fma, one ex2 per element.
__device__ __forceinline__ void exp2_scaled_64(const float* x, uint64_t sc2, float* b_then_p) {
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
        float a0, a1;
        f2_unpack(f2_fma(f2_pack(x[c], x[c + 1]), sc2, f2_pack(b_then_p[c], b_then_p[c + 1])), a0, a1);
        b_then_p[c] = fast_exp2(a0);
        b_then_p[c + 1] = fast_exp2(a1);
    }
}
__device__ __forceinline__ void exp2_scaled_64(const float* x, uint64_t sc2, uint64_t b2, float* p) {
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
        float a0, a1;
        f2_unpack(f2_fma(f2_pack(x[c], x[c + 1]), sc2, b2), a0, a1);
        p[c] = fast_exp2(a0);
        p[c + 1] = fast_exp2(a1);
    }
}

// dS of 64 columns as bf16 pairs: ds[c] = p[c] * (dp[c] - D), given nd = -D
// (per column, or one value per row), in packed fp32x2 add and mul.
__device__ __forceinline__ void ds_pack_64(const float* pr, const float* dp, const float* nd, uint32_t* pk) {
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
        float a0, a1;
        f2_unpack(f2_mul(f2_add(f2_pack(dp[c], dp[c + 1]), f2_pack(nd[c], nd[c + 1])), f2_pack(pr[c], pr[c + 1])),
                  a0, a1);
        pk[c >> 1] = pack_bf16x2(a0, a1);
    }
}
__device__ __forceinline__ void ds_pack_64(const float* pr, const float* dp, uint64_t nd2, uint32_t* pk) {
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
        float a0, a1;
        f2_unpack(f2_mul(f2_add(f2_pack(dp[c], dp[c + 1]), nd2), f2_pack(pr[c], pr[c + 1])), a0, a1);
        pk[c >> 1] = pack_bf16x2(a0, a1);
    }
}

// S-type product: D[128 x 128] = A[128 x d] B[128 x d]^T, both K-major tiles.
template <int HD>
__device__ __forceinline__ void issue_nt(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBM, false);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * Tile<HD>::kPanelBytes + (kk & 3) * 32) >> 4);
        mma_smem_smem(tmem_d, a_desc + off, b_desc + off, idesc, kk > 0);
    }
}

// Accumulating product: D[128 x d] (+)= A[128 x 128](tensor memory, bf16) B[128 x d]
// with B a row-major tile (MN-major operand).  A is written by two softmax
// warpgroups, each over 64 of the 128 fp32 columns of a tile: each packs its
// 64 bf16 values into the first 32 of ITS OWN columns (a warpgroup never
// writes columns the other one still reads), so the K elements 64h .. 64h+63
// sit at columns 64h .. 64h+31.
template <int HD>
__device__ __forceinline__ void issue_tn(uint32_t tmem_d, uint32_t tmem_a, uint64_t b_desc, bool first) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, HD, true);
#pragma unroll
    for (int kk = 0; kk < kBM / 16; ++kk)
        mma_tmem_smem(tmem_d, tmem_a + (kk >> 2) * 64 + (kk & 3) * 8,
                      b_desc + static_cast<uint64_t>((kk * 2048) >> 4), idesc, (!first || kk > 0) ? 1u : 0u);
}

// Stores 64 bf16 values (a row segment) from fp32 registers, times `mul`:
// 32-byte stores (whole sectors) when dst is 32-byte aligned, else 16-byte.
__device__ __forceinline__ void store_row64(__nv_bfloat16* dst, const float* x, float mul) {
    if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(x[c + 2 * i] * mul, x[c + 2 * i + 1] * mul);
            st_global_v8(dst + c, w);
        }
        return;
    }
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int c = 0; c < 64; c += 8) {
        uint4 w;
        w.x = pack_bf16x2(x[c + 0] * mul, x[c + 1] * mul);
        w.y = pack_bf16x2(x[c + 2] * mul, x[c + 3] * mul);
        w.z = pack_bf16x2(x[c + 4] * mul, x[c + 5] * mul);
        w.w = pack_bf16x2(x[c + 6] * mul, x[c + 7] * mul);
        d4[c >> 3] = w;
    }
}

// Reads the tensor-memory accumulator of this thread's row, columns
// [col, col + n), and writes it as bf16 (times mul) to dst.
template <int N>
__device__ __forceinline__ void drain_row(uint32_t taddr, __nv_bfloat16* dst, float mul, bool store) {
#pragma unroll 1
    for (int c = 0; c < N; c += 64) {
        float x[64];
        tmem_ld_32cols_f(taddr + c, x);
        tmem_ld_32cols_f(taddr + c + 32, x + 32);
        tmem_ld_wait_f(x);
        tmem_ld_wait_f(x + 32);
        if (store) store_row64(dst + c, x, mul);
    }
}
// The 32-column variant for d = 64 split over two warpgroups.
__device__ __forceinline__ void drain_row32(uint32_t taddr, __nv_bfloat16* dst, float mul, bool store) {
    float x[32];
    tmem_ld_32cols_f(taddr, x);
    tmem_ld_wait_f(x);
    if (store) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
            uint4 w;
            w.x = pack_bf16x2(x[c + 0] * mul, x[c + 1] * mul);
            w.y = pack_bf16x2(x[c + 2] * mul, x[c + 3] * mul);
            w.z = pack_bf16x2(x[c + 4] * mul, x[c + 5] * mul);
            w.w = pack_bf16x2(x[c + 6] * mul, x[c + 7] * mul);
            d4[c >> 3] = w;
        }
    }
}

template <int HD>
__device__ __forceinline__ void drain_half(uint32_t taddr_row, int half, __nv_bfloat16* dst_row, float mul,
                                           bool store) {
    // each warpgroup drains HD/2 columns of its rows
    if (HD == 128) drain_row<64>(taddr_row + half * 64, dst_row + half * 64, mul, store);
    else drain_row32(taddr_row + half * 32, dst_row + half * 32, mul, store);
}

// Rounds this thread's HD/2 accumulator columns (times mul) to bf16 and
// writes them into a 128-row tile staged in shared memory in the layout of
// the 128-byte-swizzled TMA maps: 64-column panels of 128 rows x 128 bytes,
// the 16-byte chunk c of row r at chunk c ^ (r & 7) of its row.
template <int HD>
__device__ __forceinline__ void stage_half(uint32_t taddr_row, int half, uint32_t tile_smem, int r, float mul) {
    constexpr int kCols = HD / 2;
    float x[kCols];
#pragma unroll
    for (int c = 0; c < kCols; c += 32) tmem_ld_32cols_f(taddr_row + half * kCols + c, x + c);
#pragma unroll
    for (int c = 0; c < kCols; c += 32) tmem_ld_wait_f(x + c);
#pragma unroll
    for (int cc = 0; cc < kCols / 8; ++cc) {
        const int col = half * kCols + cc * 8;
        const uint32_t addr = tile_smem + (col >> 6) * Tile<HD>::kPanelBytes + r * 128 +
                              ((((col & 63) >> 3) ^ (r & 7)) << 4);
        const float* v = x + cc * 8;
        sts_v4(addr, pack_bf16x2(v[0] * mul, v[1] * mul), pack_bf16x2(v[2] * mul, v[3] * mul),
               pack_bf16x2(v[4] * mul, v[5] * mul), pack_bf16x2(v[6] * mul, v[7] * mul));
    }
}

// The eight softmax warps have staged whole 128-row tiles: each warp makes
// its writes visible to the async proxy and arrives on `staged` (one phase,
// kSoftmaxWarps arrivals); thread 0 waits for all of them (a bounded wait:
// a warp that left on an error leaves the tiles unstored and the error
// recorded), stores the tiles with TMA panel by panel and waits until the
// copies have read shared memory.
template <int HD>
__device__ __forceinline__ void store_staged(const CUtensorMap* m0, uint32_t src0, const CUtensorMap* m1,
                                             uint32_t src1, int x, int y, uint32_t staged, int* err) {
    fence_proxy_async_shared();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(staged);
    if (threadIdx.x == 0 && mbar_wait(staged, 0, err)) {
#pragma unroll
        for (int pn = 0; pn < Tile<HD>::kPanels; ++pn) {
            tma_store_2d(m0, src0 + pn * Tile<HD>::kPanelBytes, x + pn * 64, y);
            if (m1 != nullptr) tma_store_2d(m1, src1 + pn * Tile<HD>::kPanelBytes, x + pn * 64, y);
        }
        bulk_commit_group();
        bulk_wait_group_read0();
    }
}

// ============================================================================ D = rowsum(G o O)
// Block (x, h) takes kRows consecutive tokens of query head h, d/8 threads
// per token, each with one 16-byte load of O and of G (a token's row of one
// head is contiguous).  Consecutive tokens of one head are consecutive in the
// lse and in the workspace, so those reads and writes are contiguous too.
// Every lane of a warp runs the same iterations (tokens past the end
// contribute nothing), so the shuffle reduction always has the full warp.
// Also writes lse * log2 e, both into the padded workspace layout the K/V
// pass copies tile by tile.
template <int HD>
__global__ void __launch_bounds__(256) attn_bwd_dot_kernel(const BwdParams p, const __nv_bfloat16* o,
                                                           const __nv_bfloat16* g, float* nlse2, float* ndvec,
                                                           long long t_q) {
    constexpr int kTpr = HD / 8;              // threads per token
    constexpr int kRows = 256 / kTpr;         // tokens per block
    // the dK/dV pass is a programmatic dependent of this kernel: its CTAs may
    // be placed once every block here has started (they wait for completion
    // before reading the workspace)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int sub = threadIdx.x % kTpr;
    const int h = blockIdx.y;
    const long long t = static_cast<long long>(blockIdx.x) * kRows + threadIdx.x / kTpr;
    float acc = 0.f;
    if (t < t_q) {
        const long long row = t * p.Hq + h;
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * HD) + sub);
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(g + row * HD) + sub);
        const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a);
        const uint32_t* bw = reinterpret_cast<const uint32_t*>(&b);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc = fmaf(bf16_lo(aw[i]), bf16_lo(bw[i]), acc);
            acc = fmaf(bf16_hi(aw[i]), bf16_hi(bw[i]), acc);
        }
    }
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (t < t_q && sub == 0) {
        const int ti = static_cast<int>(t);
        int b;
        if (!p.varlen) {
            b = ti / p.Nq;
        } else {  // the sequence holding token t: last b with cu_q[b] <= t
            int lo = 0, hi = p.B;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (__ldg(p.cu_q + mid) <= ti) lo = mid; else hi = mid;
            }
            b = lo;
        }
        const Seq s = seq_of(p, b);
        const int i = ti - s.q_base;
        const long long w = static_cast<long long>(h) * p.ws_row + ws_offset(b, s.q_base) + i;
        nlse2[w] = -__ldg(p.lse + lse_index(p, b, h, s, i)) * kLog2e;
        ndvec[w] = -acc;
    }
}

// ============================================================================ dK, dV
template <int HD>
struct KvCfg {
    static constexpr int kStages = 2;
    // Q_i, G_i, then lse * log2 e and D of the tile's rows (2 x 128 fp32, padded to 1 KB)
    static constexpr int kStageBytes = 2 * Tile<HD>::kBytes + 1024;
    // at least 120 KB so that one CTA (holding all 512 tensor-memory columns) runs per SM
    static constexpr int kNeed = 2 * Tile<HD>::kBytes + kStages * kStageBytes + 1024;
    static constexpr int kSmemBytes = kNeed > 120 * 1024 ? kNeed : 120 * 1024;
    // tensor memory columns
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + HD;
};

// barriers of the K/V pass.  A stage's Q_i (with the two vectors) and G_i
// have barriers of their own: S^T(s+1) needs only Q_{s+1}, and G_i is
// released as soon as dV has read it.
enum : int { KV_FULL = 0, KV_Q_FULL = 1, KV_Q_EMPTY = 3, KV_G_FULL = 5, KV_G_EMPTY = 7, KV_S_FULL = 9, KV_DP_FULL,
             KV_P_READY, KV_DS_READY, KV_ACC_FULL, KV_STAGED, KV_COUNT };

struct KvItem {
    int b, g, j;
    Seq s;
    int k0, keys;       // first key of the tile, valid keys in it
    int qt_lo, nqt;     // query tiles [qt_lo, qt_lo + nqt) per query head
    int steps;          // group * nqt
};

__device__ __forceinline__ bool kv_item(const BwdParams& p, KvItem& it) {
    const int x = blockIdx.x;
    it.g = blockIdx.y;
    if (!p.varlen) {
        const int nkt = (p.Nk + kBM - 1) / kBM;
        const int t = x / p.B;
        it.b = x - t * p.B;
        // a bounded right edge gives the first key tiles the most query rows
        it.j = p.win_right >= 0 ? t : nkt - 1 - t;
    } else if (!find_tile(p, x, true, it.b, it.j)) {
        return false;
    }
    it.s = seq_of(p, it.b);
    it.k0 = it.j * kBM;
    it.keys = clampi(it.s.nk - it.k0, 0, kBM);
    it.qt_lo = 0;
    it.nqt = 0;
    if (it.keys > 0 && it.s.nq > 0) {
        const int i_lo = row_first(it.k0, it.s.nq, it.s.nk, p.win_right);
        const int i_hi = row_last(it.k0 + it.keys - 1, it.s.nq, it.s.nk, p.win_left);
        if (i_hi >= i_lo) {
            it.qt_lo = i_lo / kBM;
            it.nqt = i_hi / kBM + 1 - it.qt_lo;
        }
    }
    it.steps = p.group * it.nqt;
    return it.keys > 0;
}

template <int HD>
__device__ __noinline__ void kv_producer(const BwdParams& p, const KvItem& it, uint32_t smem0, uint32_t bar0) {
    using T = Tile<HD>;
    using C = KvCfg<HD>;
    const int lane = threadIdx.x & 31;
    const uint32_t stage0 = smem0 + 2 * T::kBytes;
    bool ok = true;
    if (lane == 0) {
        tma_prefetch_map(&p.tm_q);
        tma_prefetch_map(&p.tm_do);
        mbar_arrive_expect_tx(bar_at(bar0, KV_FULL), 2 * T::kBytes);
#pragma unroll
        for (int pn = 0; pn < T::kPanels; ++pn) {
            tma_load_2d(smem0 + pn * T::kPanelBytes, &p.tm_k, bar_at(bar0, KV_FULL), it.g * HD + pn * 64,
                        it.s.k_base + it.k0);
            tma_load_2d(smem0 + T::kBytes + pn * T::kPanelBytes, &p.tm_v, bar_at(bar0, KV_FULL),
                        it.g * HD + pn * 64, it.s.k_base + it.k0);
        }
    }
    // this pass may start before the D kernel has finished (programmatic
    // dependent launch): the workspace it writes is read from here on
    if (lane == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncwarp();
    for (int s = 0; s < it.steps && ok; ++s) {
        const int st = s % C::kStages;
        const int h = it.g * p.group + s / it.nqt;
        const int qt = it.qt_lo + s % it.nqt;
        const uint32_t base = stage0 + st * C::kStageBytes;
        const uint32_t par = ((s / C::kStages) - 1) & 1;
        // Q_i with -lse*log2e and -D of the tile's rows (rows past the
        // sequence hold other values: every use of them is masked by a select)
        if (s >= C::kStages)
            ok = __shfl_sync(0xffffffffu, lane == 0 ? mbar_wait(bar_at(bar0, KV_Q_EMPTY + st), par, p.err) : true, 0);
        if (!ok) break;
        if (lane == 0) {
            const uint32_t full = bar_at(bar0, KV_Q_FULL + st);
            mbar_arrive_expect_tx(full, T::kBytes + 2 * kBM * 4);
#pragma unroll
            for (int pn = 0; pn < T::kPanels; ++pn)
                tma_load_2d(base + pn * T::kPanelBytes, &p.tm_q, full, h * HD + pn * 64, it.s.q_base + qt * kBM);
            const long long w = static_cast<long long>(h) * p.ws_row + ws_offset(it.b, it.s.q_base) + qt * kBM;
            bulk_load(base + 2 * T::kBytes, p.nlse2 + w, kBM * 4, full);
            bulk_load(base + 2 * T::kBytes + kBM * 4, p.ndvec + w, kBM * 4, full);
        }
        // G_i
        if (s >= C::kStages)
            ok = __shfl_sync(0xffffffffu, lane == 0 ? mbar_wait(bar_at(bar0, KV_G_EMPTY + st), par, p.err) : true, 0);
        if (!ok) break;
        if (lane == 0) {
            const uint32_t full = bar_at(bar0, KV_G_FULL + st);
            mbar_arrive_expect_tx(full, T::kBytes);
#pragma unroll
            for (int pn = 0; pn < T::kPanels; ++pn)
                tma_load_2d(base + T::kBytes + pn * T::kPanelBytes, &p.tm_do, full, h * HD + pn * 64,
                            it.s.q_base + qt * kBM);
        }
    }
    // drain: every copy issued has landed before the CTA may exit (a copy
    // left unissued after an error has no transaction to wait for)
    if (lane == 0) {
        mbar_wait(bar_at(bar0, KV_FULL), 0, p.err);
        for (int s = (it.steps > C::kStages ? it.steps - C::kStages : 0); s < it.steps; ++s) {
            mbar_wait(bar_at(bar0, KV_Q_FULL + s % C::kStages), (s / C::kStages) & 1, p.err);
            mbar_wait(bar_at(bar0, KV_G_FULL + s % C::kStages), (s / C::kStages) & 1, p.err);
        }
    }
    __syncwarp();
}

template <int HD>
__device__ __noinline__ void kv_mma(const BwdParams& p, const KvItem& it, uint32_t smem0, uint32_t bar0,
                                    uint32_t tmem) {
    using T = Tile<HD>;
    using C = KvCfg<HD>;
    const uint32_t stage0 = smem0 + 2 * T::kBytes;
    const uint64_t dk_desc = smem_desc_sw128(smem0, 16, 1024);               // K_j, K-major
    const uint64_t dv_desc = smem_desc_sw128(smem0 + T::kBytes, 16, 1024);   // V_j, K-major
    constexpr uint64_t kStageDesc = C::kStageBytes >> 4;
    const uint64_t dq_k0 = smem_desc_sw128(stage0, 16, 1024);                      // Q_i as the B of S^T
    const uint64_t dg_k0 = smem_desc_sw128(stage0 + T::kBytes, 16, 1024);          // G_i as the B of dP^T
    const uint64_t dg_mn0 = smem_desc_sw128(stage0 + T::kBytes, T::kPanelBytes, 1024);  // G_i row-major B
    const uint64_t dq_mn0 = smem_desc_sw128(stage0, T::kPanelBytes, 1024);               // Q_i row-major B
    const uint32_t t_s = tmem + C::kColS, t_dp = tmem + C::kColDP;
    const uint32_t t_dv = tmem + C::kColDV, t_dk = tmem + C::kColDK;
    bool ok = mbar_wait(bar_at(bar0, KV_FULL), 0, p.err);
    const int n = it.steps;
    if (ok && n > 0) {
        ok = mbar_wait(bar_at(bar0, KV_Q_FULL + 0), 0, p.err);
        if (ok) {
            tc_fence_after_sync();
            issue_nt<HD>(t_s, dk_desc, dq_k0);
            tc_commit(bar_at(bar0, KV_S_FULL));
            ok = mbar_wait(bar_at(bar0, KV_G_FULL + 0), 0, p.err);
        }
        if (ok) {
            tc_fence_after_sync();
            issue_nt<HD>(t_dp, dv_desc, dg_k0);
            tc_commit(bar_at(bar0, KV_DP_FULL));
        }
    }
    for (int s = 0; s < n && ok; ++s) {
        const int st = s % C::kStages;
        ok = mbar_wait(bar_at(bar0, KV_P_READY), s & 1, p.err);
        if (!ok) break;
        tc_fence_after_sync();
        issue_tn<HD>(t_dv, t_s, dg_mn0 + st * kStageDesc, s == 0);  // dV += P^T G_i
        tc_commit(bar_at(bar0, KV_G_EMPTY + st));                     // G_i has no later reader
        const bool more = s + 1 < n;
        const int st1 = (s + 1) % C::kStages;
        const uint32_t par1 = ((s + 1) / C::kStages) & 1;
        if (more) {
            ok = mbar_wait(bar_at(bar0, KV_Q_FULL + st1), par1, p.err);
            if (!ok) break;
            tc_fence_after_sync();
            issue_nt<HD>(t_s, dk_desc, dq_k0 + st1 * kStageDesc);  // S^T(s+1)
            tc_commit(bar_at(bar0, KV_S_FULL));
        }
        ok = mbar_wait(bar_at(bar0, KV_DS_READY), s & 1, p.err);
        if (!ok) break;
        tc_fence_after_sync();
        issue_tn<HD>(t_dk, t_dp, dq_mn0 + st * kStageDesc, s == 0);  // dK += dS^T Q_i
        tc_commit(bar_at(bar0, KV_Q_EMPTY + st));  // Q_i and the stage's vectors
        if (more) {
            ok = mbar_wait(bar_at(bar0, KV_G_FULL + st1), par1, p.err);
            if (!ok) break;
            tc_fence_after_sync();
            issue_nt<HD>(t_dp, dv_desc, dg_k0 + st1 * kStageDesc);  // dP^T(s+1)
            tc_commit(bar_at(bar0, KV_DP_FULL));
        }
    }
    // all products done (or abandoned): the accumulators may be read
    tc_commit(bar_at(bar0, KV_ACC_FULL));
}

template <int HD>
__device__ __noinline__ void kv_softmax(const BwdParams& p, const KvItem& it, uint32_t smem0, uint32_t bar0,
                                        uint32_t tmem) {
    using T = Tile<HD>;
    using C = KvCfg<HD>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int half = warp >> 2;                // query columns [64 half, 64 half + 64)
    const int r = (warp & 3) * 32 + lane;      // key row == tensor-memory lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::kColS, t_dp = tmem + lane_off + C::kColDP;
    const uint32_t stage0 = smem0 + 2 * T::kBytes;
    const int key = it.k0 + r;
    const bool key_valid = r < it.keys;
    // the query rows that see this key (none for rows past the sequence)
    const int qmin = key_valid ? row_first(key, it.s.nq, it.s.nk, p.win_right) : 1;
    const int qmax = key_valid ? row_last(key, it.s.nq, it.s.nk, p.win_left) : 0;
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    bool ok = true;
    for (int s = 0; s < it.steps && ok; ++s) {
        const int st = s % C::kStages;
        const int qt = it.qt_lo + s % it.nqt;
        const int c0 = qt * kBM + half * 64;  // first query of this thread's columns
        const uint32_t vec = stage0 + st * C::kStageBytes + 2 * T::kBytes;  // -lse*log2e [128], then -D [128]
        // acquire the stage's vectors (copied with Q_i; the Q part of the
        // stage is not refilled before this step's dK product), then S^T(s)
        ok = __all_sync(0xffffffffu, mbar_wait(bar_at(bar0, KV_Q_FULL + st), (s / C::kStages) & 1, p.err) &&
                                         mbar_wait(bar_at(bar0, KV_S_FULL), s & 1, p.err));
        if (!ok) break;
        tc_fence_after_sync();
        float x[64];
        tmem_ld_32cols_f(t_s + half * 64, x);
        tmem_ld_32cols_f(t_s + half * 64 + 32, x + 32);
        tmem_ld_wait_f(x);
        tmem_ld_wait_f(x + 32);
        const int lo = qmin - c0, hi = qmax - c0;  // allowed columns [lo, hi]
        float pr[64];
        lds_64(vec + half * 64 * 4, pr);  // -lse*log2e of this thread's 64 query columns
        exp2_scaled_64(x, sc2, pr);       // pr = 2^(s * scale * log2 e - lse * log2 e)
        if (!(lo <= 0 && hi >= 63)) {     // masked columns (the common case has none)
#pragma unroll
            for (int c = 0; c < 64; ++c) pr[c] = (c < lo || c > hi) ? 0.f : pr[c];
        }
        {
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) pk[c >> 1] = pack_bf16x2(pr[c], pr[c + 1]);
            tmem_st_32cols(t_s + half * 64, pk);  // over this warpgroup's own S^T columns
            tmem_st_wait();
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(bar0, KV_P_READY));

        ok = __all_sync(0xffffffffu, mbar_wait(bar_at(bar0, KV_DP_FULL), s & 1, p.err));
        if (!ok) break;
        tc_fence_after_sync();
        tmem_ld_32cols_f(t_dp + half * 64, x);
        tmem_ld_32cols_f(t_dp + half * 64 + 32, x + 32);
        tmem_ld_wait_f(x);
        tmem_ld_wait_f(x + 32);
        {
            float nd[64];
            lds_64(vec + (kBM + half * 64) * 4, nd);  // -D of this thread's 64 query columns
            if (!(lo <= 0 && hi >= 63)) {  // masked columns: -D may be any bits there, dP - D := 0
#pragma unroll
                for (int c = 0; c < 64; ++c) nd[c] = (c < lo || c > hi) ? -x[c] : nd[c];
            }
            uint32_t pk[32];
            ds_pack_64(pr, x, nd, pk);
            tmem_st_32cols(t_dp + half * 64, pk);  // over this warpgroup's own dP^T columns
            tmem_st_wait();
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(bar0, KV_DS_READY));
    }
    // epilogue: dV and dK (times scale) of this key row, HD/2 columns per warpgroup
    __nv_bfloat16* dk_row = p.dk + (static_cast<size_t>(it.s.k_base + key) * p.Hkv + it.g) * HD;
    __nv_bfloat16* dv_row = p.dv + (static_cast<size_t>(it.s.k_base + key) * p.Hkv + it.g) * HD;
    if (it.steps == 0) {  // no query sees these keys: zero gradients
        if (key_valid) {
            uint4* a = reinterpret_cast<uint4*>(dk_row + half * (HD / 2));
            uint4* b = reinterpret_cast<uint4*>(dv_row + half * (HD / 2));
            for (int c = 0; c < HD / 16; ++c) a[c] = b[c] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    ok = __all_sync(0xffffffffu, mbar_wait(bar_at(bar0, KV_ACC_FULL), 0, p.err)) && ok;
    if (!ok) return;
    tc_fence_after_sync();
    if (p.tma_store && it.keys == kBM) {
        // every product has completed, so K_j and V_j are no longer read:
        // dV is staged over K_j and dK over V_j, then stored with TMA
        stage_half<HD>(tmem + lane_off + C::kColDV, half, smem0, r, 1.f);
        stage_half<HD>(tmem + lane_off + C::kColDK, half, smem0 + T::kBytes, r, p.scale);
        store_staged<HD>(&p.tm_dv, smem0, &p.tm_dk, smem0 + T::kBytes, it.g * HD, it.s.k_base + it.k0,
                         bar_at(bar0, KV_STAGED), p.err);
        return;
    }
    drain_half<HD>(tmem + lane_off + C::kColDV, half, dv_row, 1.f, key_valid);
    drain_half<HD>(tmem + lane_off + C::kColDK, half, dk_row, p.scale, key_valid);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem_dyn[];
    __shared__ __align__(8) uint64_t bars[KV_COUNT];
    __shared__ uint32_t tmem_slot;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    KvItem it;
    const bool live = kv_item(p, it);  // uniform over the CTA
    // every CTA (not only those that read the workspace) ends after the D
    // kernel has: work queued behind this pass then sees that kernel done
    if (!live) {
        if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }
    const uint32_t smem0 = (smem_addr(smem_dyn) + 1023u) & ~1023u;
    const uint32_t bar0 = smem_addr(bars);
    if (threadIdx.x == 0) {
        mbar_init(bar_at(bar0, KV_FULL), 1);
        for (int s = 0; s < KvCfg<HD>::kStages; ++s) {
            mbar_init(bar_at(bar0, KV_Q_FULL + s), 1);
            mbar_init(bar_at(bar0, KV_Q_EMPTY + s), 1);
            mbar_init(bar_at(bar0, KV_G_FULL + s), 1);
            mbar_init(bar_at(bar0, KV_G_EMPTY + s), 1);
        }
        mbar_init(bar_at(bar0, KV_S_FULL), 1);
        mbar_init(bar_at(bar0, KV_DP_FULL), 1);
        mbar_init(bar_at(bar0, KV_P_READY), kSoftmaxWarps);
        mbar_init(bar_at(bar0, KV_DS_READY), kSoftmaxWarps);
        mbar_init(bar_at(bar0, KV_ACC_FULL), 1);
        mbar_init(bar_at(bar0, KV_STAGED), kSoftmaxWarps);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(&tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_map(&p.tm_k);
        tma_prefetch_map(&p.tm_v);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    if (warp >= 8) {
        regs_decrease<kControlRegs>();
        if (warp == kProducerWarp) kv_producer<HD>(p, it, smem0, bar0);
        if (warp == kMmaWarp && lane == 0) kv_mma<HD>(p, it, smem0, bar0, tmem);
        __syncwarp();
    } else {
        regs_increase<kSoftmaxRegs>();
        kv_softmax<HD>(p, it, smem0, bar0, tmem);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ============================================================================ dQ
// K_j and V_j stream through rings of their own.  V_j is read by one product
// (dP), K_j by two (S, then dQ a step later), so K gets the deeper ring: the
// load of K_{u+1} is issued about one and a half steps before S(u+1) needs it.
template <int HD>
struct QCfg {
    static constexpr int kKStages = HD == 128 ? 3 : 4;
    static constexpr int kVStages = HD == 128 ? 2 : 4;
    static constexpr int kMaxStages = 4;
    // [Q_i][G_i][K ring][V ring]
    static constexpr int kNeed = (2 + kKStages + kVStages) * Tile<HD>::kBytes + 1024;
    static constexpr int kSmemBytes = kNeed > 120 * 1024 ? kNeed : 120 * 1024;  // one CTA per SM
    // tensor memory: S, dQ, and dP in two buffers (dP(u+1) is computed while
    // dQ(u) still waits for dS(u), which the softmax writes over dP(u))
    static constexpr uint32_t kColS = 0, kColDQ = 256;
    __device__ static constexpr uint32_t col_dp(int u) { return (u & 1) ? 384u : 128u; }
    static_assert(kKStages <= kMaxStages && kVStages <= kMaxStages, "ring barriers");
    static_assert(kNeed <= 227 * 1024 - 256, "shared memory of the dQ pass");
};

// DP_FULL, DS_READY and DQ_DONE come in pairs, one per dP buffer: a barrier
// of one buffer completes its next phase only after every waiter has passed
// the current one (no phase can be skipped).
enum : int { Q_FULL = 0, Q_K_FULL = 1, Q_K_EMPTY = 5, Q_V_FULL = 9, Q_V_EMPTY = 13, Q_S_FULL = 17, Q_DP_FULL = 18,
             Q_S_FREE = 20, Q_DS_READY = 21, Q_DQ_DONE = 23, Q_ACC_FULL = 25, Q_S_DP_DONE = 26, Q_STAGED = 27,
             Q_COUNT };

struct QItem {
    int b, h, i;
    Seq s;
    int q0, rows;   // first row of the tile, valid rows
    int lo, n;      // K/V tiles [lo, lo + n)
};

__device__ __forceinline__ bool q_item(const BwdParams& p, QItem& it) {
    const int x = blockIdx.x;
    it.h = blockIdx.y;
    if (!p.varlen) {
        const int nqt = (p.Nq + kBM - 1) / kBM;
        const int t = x / p.B;
        it.b = x - t * p.B;
        // a bounded right edge gives the last query tiles the most keys
        it.i = p.win_right >= 0 ? nqt - 1 - t : t;
    } else if (!find_tile(p, x, false, it.b, it.i)) {
        return false;
    }
    it.s = seq_of(p, it.b);
    it.q0 = it.i * kBM;
    it.rows = clampi(it.s.nq - it.q0, 0, kBM);
    it.lo = 0;
    it.n = 0;
    if (it.rows > 0 && it.s.nk > 0) {
        const int kmin = key_first(it.q0, it.s.nq, it.s.nk, p.win_left);
        const int kmax = key_last(static_cast<long long>(it.q0) + it.rows - 1, it.s.nq, it.s.nk, p.win_right);
        if (kmax >= kmin) {
            it.lo = kmin / kBM;
            it.n = kmax / kBM + 1 - it.lo;
        }
    }
    return it.rows > 0;
}

template <int HD>
__device__ __noinline__ void q_producer(const BwdParams& p, const QItem& it, uint32_t smem0, uint32_t bar0) {
    using T = Tile<HD>;
    using C = QCfg<HD>;
    const uint32_t kring = smem0 + 2 * T::kBytes;
    const uint32_t vring = kring + C::kKStages * T::kBytes;
    const int g = it.h / p.group;
    bool ok = true;
    mbar_arrive_expect_tx(bar_at(bar0, Q_FULL), 2 * T::kBytes);
#pragma unroll
    for (int pn = 0; pn < T::kPanels; ++pn) {
        tma_load_2d(smem0 + pn * T::kPanelBytes, &p.tm_q, bar_at(bar0, Q_FULL), it.h * HD + pn * 64,
                    it.s.q_base + it.q0);
        tma_load_2d(smem0 + T::kBytes + pn * T::kPanelBytes, &p.tm_do, bar_at(bar0, Q_FULL), it.h * HD + pn * 64,
                    it.s.q_base + it.q0);
    }
    for (int u = 0; u < it.n && ok; ++u) {
        const int y = it.s.k_base + (it.lo + u) * kBM;
        const int ks = u % C::kKStages, vs = u % C::kVStages;
        if (u >= C::kKStages) ok = mbar_wait(bar_at(bar0, Q_K_EMPTY + ks), ((u / C::kKStages) - 1) & 1, p.err);
        if (!ok) break;
        const uint32_t kfull = bar_at(bar0, Q_K_FULL + ks);
        mbar_arrive_expect_tx(kfull, T::kBytes);
#pragma unroll
        for (int pn = 0; pn < T::kPanels; ++pn)
            tma_load_2d(kring + ks * T::kBytes + pn * T::kPanelBytes, &p.tm_k, kfull, g * HD + pn * 64, y);
        if (u >= C::kVStages) ok = mbar_wait(bar_at(bar0, Q_V_EMPTY + vs), ((u / C::kVStages) - 1) & 1, p.err);
        if (!ok) break;
        const uint32_t vfull = bar_at(bar0, Q_V_FULL + vs);
        mbar_arrive_expect_tx(vfull, T::kBytes);
#pragma unroll
        for (int pn = 0; pn < T::kPanels; ++pn)
            tma_load_2d(vring + vs * T::kBytes + pn * T::kPanelBytes, &p.tm_v, vfull, g * HD + pn * 64, y);
    }
    // drain: every copy issued has landed before the CTA may exit (a load
    // left unissued after an error has no transaction to wait for)
    mbar_wait(bar_at(bar0, Q_FULL), 0, p.err);
    for (int u = (it.n > C::kKStages ? it.n - C::kKStages : 0); u < it.n; ++u)
        mbar_wait(bar_at(bar0, Q_K_FULL + u % C::kKStages), (u / C::kKStages) & 1, p.err);
    for (int u = (it.n > C::kVStages ? it.n - C::kVStages : 0); u < it.n; ++u)
        mbar_wait(bar_at(bar0, Q_V_FULL + u % C::kVStages), (u / C::kVStages) & 1, p.err);
}

// Two issuing threads.  Thread 0 computes the products that do not need
// dS: S(u+1) and dP(u+1); thread 1 computes dQ(u) = dS(u) K_u once the
// softmax has written dS(u).  Each thread's barrier waits then overlap the
// other thread's products (a thread's issue is close to synchronous with the
// tensor pipe).  Cross-thread reuse of tensor memory waits for completion:
// dP(u+1) overwrites the buffer that held dS(u-1) only after dQ(u-1) has
// completed (DQ_DONE).
template <int HD>
__device__ __noinline__ void q_mma(const BwdParams& p, const QItem& it, uint32_t smem0, uint32_t bar0,
                                   uint32_t tmem, int role) {
    using T = Tile<HD>;
    using C = QCfg<HD>;
    const uint32_t kring = smem0 + 2 * T::kBytes;
    const uint32_t vring = kring + C::kKStages * T::kBytes;
    constexpr uint64_t kSlotDesc = T::kBytes >> 4;  // descriptor step between ring slots
    const int n = it.n;
    bool ok = true;
    if (role == 0) {
        const uint64_t d_q = smem_desc_sw128(smem0, 16, 1024);              // Q_i, K-major
        const uint64_t d_g = smem_desc_sw128(smem0 + T::kBytes, 16, 1024);  // G_i, K-major
        const uint64_t d_k0 = smem_desc_sw128(kring, 16, 1024);             // K_j as the B of S
        const uint64_t d_v0 = smem_desc_sw128(vring, 16, 1024);             // V_j as the B of dP
        const uint32_t t_s = tmem + C::kColS;
        ok = mbar_wait(bar_at(bar0, Q_FULL), 0, p.err);
        for (int u = 0; u < n && ok; ++u) {  // S(u) and dP(u)
            const int ks = u % C::kKStages, vs = u % C::kVStages;
            ok = (u == 0 || mbar_wait_spin(bar_at(bar0, Q_S_FREE), (u - 1) & 1, p.err)) &&
                 mbar_wait(bar_at(bar0, Q_K_FULL + ks), (u / C::kKStages) & 1, p.err);
            if (!ok) break;
            tc_fence_after_sync();
            issue_nt<HD>(t_s, d_q, d_k0 + ks * kSlotDesc);  // S(u)
            tc_commit(bar_at(bar0, Q_S_FULL));
            // the dP buffer of step u last held dS(u-2)
            ok = (u < 2 || mbar_wait(bar_at(bar0, Q_DQ_DONE + (u & 1)), ((u - 2) >> 1) & 1, p.err)) &&
                 mbar_wait(bar_at(bar0, Q_V_FULL + vs), (u / C::kVStages) & 1, p.err);
            if (!ok) break;
            tc_fence_after_sync();
            issue_nt<HD>(tmem + C::col_dp(u), d_g, d_v0 + vs * kSlotDesc);  // dP(u)
            tc_commit(bar_at(bar0, Q_DP_FULL + (u & 1)));
            tc_commit(bar_at(bar0, Q_V_EMPTY + vs));  // V_j has no other reader
        }
        // drain: this thread's products (and their barrier arrivals) are done before it leaves
        tc_commit(bar_at(bar0, Q_S_DP_DONE));
        mbar_wait(bar_at(bar0, Q_S_DP_DONE), 0, p.err);
    } else {
        const uint64_t d_kmn0 = smem_desc_sw128(kring, T::kPanelBytes, 1024);  // K_j row-major B
        const uint32_t t_dq = tmem + C::kColDQ;
        for (int u = 0; u < n && ok; ++u) {  // dQ(u)
            const int ks = u % C::kKStages;
            ok = mbar_wait_spin(bar_at(bar0, Q_DS_READY + (u & 1)), (u >> 1) & 1, p.err) &&
                 mbar_wait(bar_at(bar0, Q_K_FULL + ks), (u / C::kKStages) & 1, p.err);
            if (!ok) break;
            tc_fence_after_sync();
            issue_tn<HD>(t_dq, tmem + C::col_dp(u), d_kmn0 + ks * kSlotDesc, u == 0);  // dQ += dS K_j
            tc_commit(bar_at(bar0, Q_K_EMPTY + ks));
            tc_commit(bar_at(bar0, Q_DQ_DONE + (u & 1)));
        }
        tc_commit(bar_at(bar0, Q_ACC_FULL));
    }
}

template <int HD>
__device__ __noinline__ void q_softmax(const BwdParams& p, const QItem& it, uint32_t smem0, uint32_t bar0,
                                       uint32_t tmem) {
    using C = QCfg<HD>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int half = warp >> 2;                // key columns [64 half, 64 half + 64)
    const int r = (warp & 3) * 32 + lane;      // query row == tensor-memory lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::kColS;
    const int i = it.q0 + r;
    const bool row_valid = r < it.rows;
    const int nq = it.s.nq, nk = it.s.nk;
    const int kmin = row_valid ? key_first(i, nq, nk, p.win_left) : 1;
    const int kmax = row_valid ? key_last(i, nq, nk, p.win_right) : 0;
    float nl2 = 0.f, nd = 0.f;  // -lse * log2 e and -D of this row
    if (row_valid) {
        const long long w = static_cast<long long>(it.h) * p.ws_row + ws_offset(it.b, it.s.q_base) + i;
        nl2 = __ldg(p.nlse2 + w);
        nd = __ldg(p.ndvec + w);
    }
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    bool ok = true;
    for (int u = 0; u < it.n && ok; ++u) {
        const int k0 = (it.lo + u) * kBM + half * 64;
        ok = __all_sync(0xffffffffu, mbar_wait(bar_at(bar0, Q_S_FULL), u & 1, p.err));
        if (!ok) break;
        tc_fence_after_sync();
        float x[64];
        tmem_ld_32cols_f(t_s + half * 64, x);
        tmem_ld_32cols_f(t_s + half * 64 + 32, x + 32);
        tmem_ld_wait_f(x);
        tmem_ld_wait_f(x + 32);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(bar0, Q_S_FREE));  // S may be overwritten
        const int lo = kmin - k0, hi = kmax - k0;
        float pr[64];
        exp2_scaled_64(x, sc2, f2_pack(nl2, nl2), pr);  // pr = 2^(s * scale * log2 e - lse * log2 e)
        if (!(lo <= 0 && hi >= 63)) {                    // masked columns (the common case has none)
#pragma unroll
            for (int c = 0; c < 64; ++c) pr[c] = (c < lo || c > hi) ? 0.f : pr[c];
        }
        ok = __all_sync(0xffffffffu, mbar_wait(bar_at(bar0, Q_DP_FULL + (u & 1)), (u >> 1) & 1, p.err));
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t t_dp = tmem + lane_off + C::col_dp(u);
        tmem_ld_32cols_f(t_dp + half * 64, x);
        tmem_ld_32cols_f(t_dp + half * 64 + 32, x + 32);
        tmem_ld_wait_f(x);
        tmem_ld_wait_f(x + 32);
        {
            uint32_t pk[32];
            ds_pack_64(pr, x, f2_pack(nd, nd), pk);
            tmem_st_32cols(t_dp + half * 64, pk);  // over this warpgroup's own dP columns
            tmem_st_wait();
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(bar0, Q_DS_READY + (u & 1)));
    }
    __nv_bfloat16* dq_row = p.dq + (static_cast<size_t>(it.s.q_base + i) * p.Hq + it.h) * HD;
    if (it.n == 0) {  // no key: zero gradient
        if (row_valid) {
            uint4* a = reinterpret_cast<uint4*>(dq_row + half * (HD / 2));
            for (int c = 0; c < HD / 16; ++c) a[c] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    ok = __all_sync(0xffffffffu, mbar_wait(bar_at(bar0, Q_ACC_FULL), 0, p.err)) && ok;
    if (!ok) return;
    tc_fence_after_sync();
    if (p.tma_store && it.rows == kBM) {
        // every product has completed, so Q_i is no longer read: dQ is
        // staged over it and stored with TMA
        stage_half<HD>(tmem + lane_off + C::kColDQ, half, smem0, r, p.scale);
        store_staged<HD>(&p.tm_dq, smem0, nullptr, 0, it.h * HD, it.s.q_base + it.q0, bar_at(bar0, Q_STAGED),
                         p.err);
        return;
    }
    drain_half<HD>(tmem + lane_off + C::kColDQ, half, dq_row, p.scale, row_valid);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem_dyn[];
    __shared__ __align__(8) uint64_t bars[Q_COUNT];
    __shared__ uint32_t tmem_slot;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    QItem it;
    if (!q_item(p, it)) return;  // uniform over the CTA
    const uint32_t smem0 = (smem_addr(smem_dyn) + 1023u) & ~1023u;
    const uint32_t bar0 = smem_addr(bars);
    if (threadIdx.x == 0) {
        mbar_init(bar_at(bar0, Q_FULL), 1);
        for (int s = 0; s < QCfg<HD>::kMaxStages; ++s) {
            mbar_init(bar_at(bar0, Q_K_FULL + s), 1);
            mbar_init(bar_at(bar0, Q_K_EMPTY + s), 1);
            mbar_init(bar_at(bar0, Q_V_FULL + s), 1);
            mbar_init(bar_at(bar0, Q_V_EMPTY + s), 1);
        }
        mbar_init(bar_at(bar0, Q_S_FULL), 1);
        mbar_init(bar_at(bar0, Q_DP_FULL + 0), 1);
        mbar_init(bar_at(bar0, Q_DP_FULL + 1), 1);
        mbar_init(bar_at(bar0, Q_S_FREE), kSoftmaxWarps);
        mbar_init(bar_at(bar0, Q_DS_READY + 0), kSoftmaxWarps);
        mbar_init(bar_at(bar0, Q_DS_READY + 1), kSoftmaxWarps);
        mbar_init(bar_at(bar0, Q_DQ_DONE + 0), 1);
        mbar_init(bar_at(bar0, Q_DQ_DONE + 1), 1);
        mbar_init(bar_at(bar0, Q_ACC_FULL), 1);
        mbar_init(bar_at(bar0, Q_S_DP_DONE), 1);
        mbar_init(bar_at(bar0, Q_STAGED), kSoftmaxWarps);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(&tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_map(&p.tm_q);
        tma_prefetch_map(&p.tm_do);
        tma_prefetch_map(&p.tm_k);
        tma_prefetch_map(&p.tm_v);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    if (warp >= 8) {
        regs_decrease<kControlRegs>();
        if (warp == kProducerWarp && lane == 0) q_producer<HD>(p, it, smem0, bar0);
        if ((warp == kMmaWarp || warp == kMmaWarp + 1) && lane == 0) q_mma<HD>(p, it, smem0, bar0, tmem, warp - kMmaWarp);
        __syncwarp();
    } else {
        regs_increase<kSoftmaxRegs>();
        q_softmax<HD>(p, it, smem0, bar0, tmem);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// ============================================================================ host
template <typename K>
attn_status prepare_kernel(K kernel, int smem_bytes, std::atomic<bool>* done) {
    if (done != nullptr && done->load(std::memory_order_acquire)) return ATTN_OK;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) {
        set_error_message("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) {
        set_error_message("cudaFuncGetAttributes: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    if (fa.numRegs * kThreads < 2 * 128 * kSoftmaxRegs + 128 * kControlRegs) {
        set_error_message("attn_bwd kernel built with %d registers/thread; the warpgroup split needs %d",
                          fa.numRegs, kLaunchRegs);
        return ATTN_ERR_UNSUPPORTED;
    }
    if (done != nullptr) done->store(true, std::memory_order_release);
    return ATTN_OK;
}

template <int HD>
attn_status launch_typed(const BwdArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
    BwdParams p;
    memset(&p, 0, sizeof(p));
    const bool varlen = a.cu_q != nullptr;
    const uint64_t t_q = varlen ? static_cast<uint64_t>(a.Nq) : static_cast<uint64_t>(a.B) * a.Nq;
    uint64_t t_k = varlen ? static_cast<uint64_t>(a.Nk) : static_cast<uint64_t>(a.B) * a.Nk;
    const uint32_t box[2] = {64, kBM};
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(a.Hq) * HD, t_q};
        const uint64_t strides[1] = {static_cast<uint64_t>(a.Hq) * HD * 2};
        attn_status st = encode_tma_bf16(&p.tm_q, a.q, 2, dims, strides, box, true);
        if (st == ATTN_OK) st = encode_tma_bf16(&p.tm_do, a.dout, 2, dims, strides, box, true);
        if (st != ATTN_OK) return st;
    }
    {
        const bool no_keys = t_k == 0;
        if (no_keys) t_k = 1;  // never read; a zero extent is not encodable
        const uint64_t dims[2] = {static_cast<uint64_t>(a.Hkv) * HD, t_k};
        const uint64_t strides[1] = {static_cast<uint64_t>(a.Hkv) * HD * 2};
        attn_status st = encode_tma_bf16(&p.tm_k, no_keys ? a.q : a.k, 2, dims, strides, box, true);
        if (st == ATTN_OK) st = encode_tma_bf16(&p.tm_v, no_keys ? a.q : a.v, 2, dims, strides, box, true);
        if (st != ATTN_OK) return st;
    }
    // the outputs as TMA store targets of full tiles (outputs that are not
    // 16-byte aligned keep the per-row stores); with no keys at all the
    // K/V pass has no tile and dQ is all zeros, so nothing is stored by TMA
    const auto aligned16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
    const bool any_keys = (varlen ? static_cast<uint64_t>(a.Nk) : static_cast<uint64_t>(a.B) * a.Nk) > 0;
    if (any_keys && t_q > 0 && aligned16(a.dq) && aligned16(a.dk) && aligned16(a.dv)) {
        const uint64_t dq_dims[2] = {static_cast<uint64_t>(a.Hq) * HD, t_q};
        const uint64_t dq_strides[1] = {static_cast<uint64_t>(a.Hq) * HD * 2};
        const uint64_t dk_dims[2] = {static_cast<uint64_t>(a.Hkv) * HD, t_k};
        const uint64_t dk_strides[1] = {static_cast<uint64_t>(a.Hkv) * HD * 2};
        attn_status st = encode_tma_bf16(&p.tm_dq, a.dq, 2, dq_dims, dq_strides, box, true);
        if (st == ATTN_OK) st = encode_tma_bf16(&p.tm_dk, a.dk, 2, dk_dims, dk_strides, box, true);
        if (st == ATTN_OK) st = encode_tma_bf16(&p.tm_dv, a.dv, 2, dk_dims, dk_strides, box, true);
        if (st != ATTN_OK) return st;
        p.tma_store = 1;
    }
    p.lse = a.lse;
    p.ws_row = bwd_ws_row(a.B, varlen ? a.Nq : static_cast<long long>(a.B) * a.Nq);
    p.nlse2 = static_cast<float*>(a.workspace);
    p.ndvec = static_cast<float*>(a.workspace) + p.ws_row * a.Hq;
    p.dq = static_cast<__nv_bfloat16*>(a.dq);
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.cu_q = a.cu_q;
    p.cu_k = a.cu_k;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.group = a.Hq / a.Hkv;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.win_left = a.win_left < 0 ? -1 : a.win_left;
    p.win_right = a.causal ? 0 : (a.win_right < 0 ? -1 : a.win_right);
    p.varlen = varlen ? 1 : 0;
    p.scale = a.scale;
    p.scale_log2 = a.scale * kLog2e;
    p.err = dev.err_word;

    if (varlen && validation_enabled()) {
        launch_check_cu_seqlens(a.cu_q, a.B, a.Nq, stream);
        launch_check_cu_seqlens(a.cu_k, a.B, a.Nk, stream);
    }
    // D = rowsum(G o O)
    if (t_q > 0) {
        constexpr int kRowsPerBlock = 256 / (HD / 8);
        const dim3 grid(static_cast<unsigned>((t_q + kRowsPerBlock - 1) / kRowsPerBlock), static_cast<unsigned>(a.Hq));
        attn_bwd_dot_kernel<HD><<<grid, 256, 0, stream>>>(p, static_cast<const __nv_bfloat16*>(a.out),
                                                          static_cast<const __nv_bfloat16*>(a.dout),
                                                          const_cast<float*>(p.nlse2), const_cast<float*>(p.ndvec),
                                                          static_cast<long long>(t_q));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) {
            set_error_message("attn_bwd_dot launch: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
    }
    static std::atomic<bool> ready_kv[kMaxDevices], ready_q[kMaxDevices];  // per instantiation and device
    const bool cached = dev.device >= 0 && dev.device < kMaxDevices;
    attn_status st = prepare_kernel(attn_bwd_dkdv_kernel<HD>, KvCfg<HD>::kSmemBytes,
                                    cached ? &ready_kv[dev.device] : nullptr);
    if (st == ATTN_OK)
        st = prepare_kernel(attn_bwd_dq_kernel<HD>, QCfg<HD>::kSmemBytes, cached ? &ready_q[dev.device] : nullptr);
    if (st != ATTN_OK) return st;
    // grids: dense = (tiles x B, heads); packed = an upper bound on the
    // (sequence, tile) entries, the surplus CTAs return at once
    const long long kv_x = varlen ? static_cast<long long>(a.Nk) / kBM + a.B
                                  : static_cast<long long>((a.Nk + kBM - 1) / kBM) * a.B;
    const long long q_x = varlen ? static_cast<long long>(a.Nq) / kBM + a.B
                                 : static_cast<long long>((a.Nq + kBM - 1) / kBM) * a.B;
    if (kv_x > 0x7fffffffLL || q_x > 0x7fffffffLL) {
        set_error_message("attn_bwd: too many tiles");
        return ATTN_ERR_UNSUPPORTED;
    }
    if (kv_x > 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(kv_x), static_cast<unsigned>(a.Hkv));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = KvCfg<HD>::kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = t_q > 0 ? 1 : 0;
        cudaError_t e = cudaLaunchKernelEx(&cfg, attn_bwd_dkdv_kernel<HD>, p);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) {
            set_error_message("attn_bwd_dkdv launch: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
    }
    if (q_x > 0) {
        attn_bwd_dq_kernel<HD><<<dim3(static_cast<unsigned>(q_x), a.Hq), kThreads, QCfg<HD>::kSmemBytes,
                                 stream>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) {
            set_error_message("attn_bwd_dq launch: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
    }
    return ATTN_OK;
}

}  // namespace

size_t bwd_workspace_bytes(int B, int Hq, int Nq, bool varlen) {
    const long long t_q = varlen ? static_cast<long long>(Nq) : static_cast<long long>(B) * Nq;
    return (static_cast<size_t>(2 * Hq) * bwd_ws_row(B, t_q) * sizeof(float) + 255) / 256 * 256;
}

attn_status launch_bwd(const BwdArgs& a, cudaStream_t stream) {
    DeviceInfo dev;
    attn_status st = current_device_info(&dev);
    if (st != ATTN_OK) return st;
    if (a.d == 128) return launch_typed<128>(a, dev, stream);
    if (a.d == 64) return launch_typed<64>(a, dev, stream);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
