// fwd.cu -- prefill forward of exact attention on sm_103a.
//
// One persistent CTA per SM walks a longest-first list of work items.  An item
// is (sequence b, query head h, pair of 128-row query tiles).  Inside a CTA
// the warps specialise:
//   warps 0-3  softmax group 0: owns query tile 0 (one thread per row)
//   warps 4-7  softmax group 1: owns query tile 1
//   warp  8    producer: TMA loads of Q tiles and a ring of K and V tiles
//   warp  9    MMA issuer of query tile 0 (one thread), tensor-memory owner
//   warp  10   MMA issuer of query tile 1 (one thread)
//   warp  11   idle (it completes the third warpgroup)
// The 8-bit forward (E4M3 Q, K, V with per-tile scales; F8 = true) keeps
// this layout; there warps 11 and 8 also widen each 8-bit V tile to f16 for
// the PV product, and the softmax folds the tile scales into its exponent.
// The softmax warpgroups raise their register budget to kSoftmaxRegs and the
// third warpgroup lowers its own to kControlRegs (setmaxnreg).
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [0,128)       S0 = Q0 K^T (fp32); P0 (bf16) overwrites its first 64 columns
//   [128,256)     S1, P1
//   [256,256+d)   O0 accumulator (fp32)
//   [256+d,256+2d) O1
// Per K/V tile j the tensor core runs S = Q K_j^T for both query tiles, the
// softmax groups turn S into P in place, and the tensor core runs O += P V_j
// with P read straight from tensor memory.  The issue order
//     PV0(j), S0(j+1), PV1(j), S1(j+1)
// lets softmax group 0 work while the tensor core serves tile 1 and the other
// way round.  Nothing quadratic ever leaves the SM.
//
// The recurrence is the blockwise merge of "Flash Attention: A Complete
// Architectural Autopsy", part 2 ("The Online Softmax Recurrence"): running
// max m, normaliser l, accumulator O, the old state scaled by exp(m_old-m_new)
// when the max rises, and one division by l at the end ("FlashAttention: Part
// 1", section 3.1).  The rescale is conditional ("FlashAttention-3 and
// PagedAttention", FA4 paragraph): the reference max of a row is only moved
// when the tile max exceeds it by more than 2^8 in the exponent, which keeps O
// and l on one common reference (exact in real arithmetic) while skipping
// almost every rescale.  The mask is a band per sequence: query row i keeps
// keys [i + Nk - Nq - left, i + Nk - Nq + right] inside [0, Nk), a side < 0
// being unbounded ("Deep Dive - FlashAttention", section "Causal 2.1 is the
// decode gotcha", its bottom-right corner and its local-window paragraph);
// causal is right = 0.  Tiles wholly outside the band are never loaded; only
// tiles that cross a band edge or a sequence edge are masked ("FlashAttention:
// Part 1", section 3.5).  The two query tiles of an item stream the union of
// their tile ranges; a tile sits out the slots outside its own range.
#include <cuda_bf16.h>
#include <math.h>
#include <string.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;                     // query rows per tile
constexpr int kBN = 128;                     // keys per K/V tile
constexpr int kPairRows = 2 * kBM;           // query rows per work item
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;     // 65536 / 384, rounded down to a multiple of 8
constexpr int kSoftmaxRegs = 208;    // warpgroups 0 and 1
constexpr int kControlRegs = 88;     // warpgroup 2
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleThreshold = 8.0f;    // log2 units
constexpr int kMaxSortedPairs = 1024;        // packed mode: (seq, pair) entries sorted per CTA
constexpr int kChunks = kThreads;            // packed mode: sequences scanned in this many chunks

// F8: the 8-bit forward (E4M3 Q, K, V with per-tile scales).
template <int HD, bool F8 = false>
struct Cfg {
    // Q and K tiles: 128-byte column panels (64 bf16 or 128 E4M3 values
    // wide, 128-byte swizzle), or for the 8-bit tiles at d = 64 one panel of
    // 64-byte rows (64-byte swizzle)
    static constexpr int kRowBytes = (F8 && HD < 128) ? HD : 128;
    static constexpr int kPanels = F8 ? (HD + 127) / 128 : HD / 64;
    static constexpr int kPanelBytes = kBM * kRowBytes;
    static constexpr int kTileBytes = kPanels * kPanelBytes;
    // the V tile as the PV product reads it: 16-bit values (bf16, or f16
    // converted from E4M3), 64-element (128-byte) panels
    static constexpr int kVPanelBytes = kBM * 128;
    static constexpr int kVBytes = (HD / 64) * kVPanelBytes;
    // K/V ring: slot u of an item holds V_{u-1} and K_u (what one step of
    // the MMA issuer consumes), so each step needs one wait and one release
    static constexpr int kStages = HD == 128 ? 2 : 4;
    static constexpr int kSlotBytes = kTileBytes + kVBytes;  // [K part][V part]
    // 8-bit V tiles land in a ring of their own and are widened into the slot
    // (V_j is loaded with K_j, a slot ahead of its use: three stages keep the
    // producer from waiting on the converter)
    static constexpr int kV8Stages = F8 ? 3 : 0;
    static constexpr int kV8Bytes = F8 ? kBM * HD : 0;
    static constexpr int kSmemBytes = 2 * kTileBytes + kStages * kSlotBytes + kV8Stages * kV8Bytes + 1024;
    static constexpr uint32_t kTmemCols = 512;
    // tensor-memory column of S_t / P_t and of O_t
    __device__ static constexpr uint32_t col_s(int t) { return static_cast<uint32_t>(t) * 128u; }
    __device__ static constexpr uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(t) * HD; }
};

struct FwdParams {
    CUtensorMap tm_q;   // [T_q rows, Hq*d] bf16, box 64 x 128, 128B swizzle
    CUtensorMap tm_k;   // [T_k rows, Hkv*d]
    CUtensorMap tm_v;
    __nv_bfloat16* out;
    float* lse;
    const int* cu_q;
    const int* cu_k;
    int B, Hq, Hkv, group;
    int Nq, Nk;         // dense: per-sequence lengths; packed: total rows
    int win_left, win_right;  // band half-widths in keys, < 0 = unbounded (causal: right = 0)
    int varlen;
    float scale_log2;   // scale * log2(e)
    int* err;
    // 8-bit forward: per-tile scales [heads, n_scale_q / n_scale_k], tile t
    // of sequence b at entry q_base_b / 128 + b + t (k_base_b for K and V)
    const float *q_scale, *k_scale, *v_scale;
    long long n_scale_q, n_scale_k;
};

struct Seq {
    int q_base, k_base, nq, nk;
};

__device__ __forceinline__ int clampi(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

__device__ __forceinline__ Seq seq_of(const FwdParams& p, int b) {
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

// First and last allowed key of local query row i (inclusive; last < first
// means none), clamped to [-1, nk].
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

// K/V tiles [lo, hi) that the query tile starting at local row q_start needs
// (lo == hi == 0 when it needs none).
__device__ __forceinline__ void kv_range(int q_start, int nq, int nk, int left, int right, int& lo, int& hi) {
    lo = hi = 0;
    const int rows = min(nq - q_start, kBM);
    if (rows <= 0 || nk <= 0) return;
    const int kmin = key_first(q_start, nq, nk, left);
    const int kmax = key_last(static_cast<long long>(q_start) + rows - 1, nq, nk, right);
    if (kmax < kmin) return;
    lo = kmin / kBN;
    hi = kmax / kBN + 1;
}

struct Item {
    int b, pair, h;
    Seq s;
    int lo[2], hi[2];  // K/V tile range per query tile
    int n[2];          // hi - lo
    int j0, len;       // the item's stream: K/V tiles [j0, j0 + len)
    int rows[2];       // valid query rows per tile
};

__device__ __forceinline__ void fill_item(const FwdParams& p, Item& it) {
    it.s = seq_of(p, it.b);
    int j1 = 0;
    it.j0 = 0x7fffffff;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int q_start = it.pair * kPairRows + t * kBM;
        it.rows[t] = clampi(it.s.nq - q_start, 0, kBM);
        kv_range(q_start, it.s.nq, it.s.nk, p.win_left, p.win_right, it.lo[t], it.hi[t]);
        it.n[t] = it.hi[t] - it.lo[t];
        if (it.n[t] > 0) {
            it.j0 = min(it.j0, it.lo[t]);
            j1 = max(j1, it.hi[t]);
        }
    }
    if (j1 == 0) it.j0 = 0;
    it.len = j1 - it.j0;
}

// Work list shared by all roles of a CTA (packed mode only).
struct Schedule {
    int n_pairs;                    // total (sequence, pair) entries
    int sorted;                     // 1 if the lists below are valid
    int chunk_prefix[kChunks + 1];  // pairs before each chunk of sequences
    int sb[kMaxSortedPairs];        // sorted: sequence of entry
    int sp[kMaxSortedPairs];        // sorted: pair of entry
    int tmp_b[kMaxSortedPairs];
    int tmp_p[kMaxSortedPairs];
    int tmp_c[kMaxSortedPairs];
};

// Longest-first order of (sequence, pair) entries, built by every CTA from
// cu_seqlens (no host round trip, no global scratch).
__device__ void build_schedule(const FwdParams& p, Schedule& sc) {
    const int tid = threadIdx.x;
    const int per = (p.B + kChunks - 1) / kChunks;
    const int b0 = min(tid * per, p.B), b1 = min(b0 + per, p.B);
    int cnt = 0;
    for (int b = b0; b < b1; ++b) cnt += (seq_of(p, b).nq + kPairRows - 1) / kPairRows;
    sc.chunk_prefix[tid + 1] = cnt;
    __syncthreads();
    if (tid == 0) {
        sc.chunk_prefix[0] = 0;
        for (int c = 0; c < kChunks; ++c) sc.chunk_prefix[c + 1] += sc.chunk_prefix[c];
        sc.n_pairs = sc.chunk_prefix[kChunks];
        sc.sorted = sc.n_pairs <= kMaxSortedPairs;
    }
    __syncthreads();
    if (!sc.sorted) return;
    int pos = sc.chunk_prefix[tid];
    for (int b = b0; b < b1; ++b) {
        const Seq s = seq_of(p, b);
        const int np = (s.nq + kPairRows - 1) / kPairRows;
        for (int pr = 0; pr < np; ++pr, ++pos) {
            sc.tmp_b[pos] = b;
            sc.tmp_p[pos] = pr;
            int lo0, hi0, lo1, hi1;
            kv_range(pr * kPairRows, s.nq, s.nk, p.win_left, p.win_right, lo0, hi0);
            kv_range(pr * kPairRows + kBM, s.nq, s.nk, p.win_left, p.win_right, lo1, hi1);
            sc.tmp_c[pos] = hi1 > lo1 ? max(hi0, hi1) - (hi0 > lo0 ? lo0 : lo1) : hi0 - lo0;
        }
    }
    __syncthreads();
    const int n = sc.n_pairs;
    for (int i = tid; i < n; i += kThreads) {
        const int ci = sc.tmp_c[i];
        int rank = 0;
        for (int j = 0; j < n; ++j) {
            const int cj = sc.tmp_c[j];
            rank += (cj > ci) || (cj == ci && j < i);
        }
        sc.sb[rank] = sc.tmp_b[i];
        sc.sp[rank] = sc.tmp_p[i];
    }
    __syncthreads();
}

// Item k of the CTA-independent longest-first order.
__device__ __forceinline__ void item_at(const FwdParams& p, const Schedule& sc, int k, Item& it) {
    if (!p.varlen) {
        const int per = p.B * p.Hq;
        const int pairs = (p.Nq + kPairRows - 1) / kPairRows;
        const int pi = k / per;
        it.pair = p.win_right >= 0 ? pairs - 1 - pi : pi;  // bounded right edge: later pairs see more keys
        const int rem = k - pi * per;
        it.b = rem / p.Hq;
        it.h = rem - it.b * p.Hq;
    } else {
        const int e = k / p.Hq;
        it.h = k - e * p.Hq;
        if (sc.sorted) {
            it.b = sc.sb[e];
            it.pair = sc.sp[e];
        } else {
            // natural order: find the chunk, then the sequence inside it
            int lo = 0, hi = kChunks;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (sc.chunk_prefix[mid] <= e) lo = mid; else hi = mid;
            }
            const int per = (p.B + kChunks - 1) / kChunks;
            int rem = e - sc.chunk_prefix[lo];
            int b = lo * per;
            for (;; ++b) {
                const int np = (seq_of(p, b).nq + kPairRows - 1) / kPairRows;
                if (rem < np) break;
                rem -= np;
            }
            it.b = b;
            it.pair = rem;
        }
    }
    fill_item(p, it);
}

__device__ __forceinline__ int total_items(const FwdParams& p, const Schedule& sc) {
    if (!p.varlen) return ((p.Nq + kPairRows - 1) / kPairRows) * p.B * p.Hq;
    return sc.n_pairs * p.Hq;
}

// Snake order over the grid: round r visits items r*G + c (r even) or
// r*G + G-1-c (r odd), so the heaviest items are spread across CTAs.
__device__ __forceinline__ int snake(int round, int cta, int grid) {
    return round * grid + ((round & 1) ? grid - 1 - cta : cta);
}

// Shared-memory barrier indices (each barrier is 8 bytes at bar0 + 8*index).
// Per query tile t: q_full+t, q_empty+t, s_full+t, p_ready+t, o_final+t,
// o_empty+t, tok+t (issuer t has issued its MMAs of a ring slot), mma_done+t.
// Per ring slot s: kv_full+s, kv_empty+s (one release from each issuer).
// 8-bit forward only: v8_full+s, v8_empty+s for the S8 8-bit V staging
// slots (each staging slot is freed by both widening warps); kv_full then
// also waits for the two widening warps' arrivals.
template <int S, bool F8 = false, int S8 = 0>
struct BarIdx {
    static constexpr int q_full = 0, q_empty = 2;
    static constexpr int kv_full = 4, kv_empty = 4 + S;
    static constexpr int s_full = 4 + 2 * S, p_ready = s_full + 2, o_final = p_ready + 2, o_empty = o_final + 2;
    static constexpr int tok = o_empty + 2, mma_done = tok + 2;
    static constexpr int v8_full = mma_done + 2, v8_empty = v8_full + S8;
    static constexpr int count = F8 ? v8_empty + S8 : mma_done + 2;
    __device__ static constexpr uint32_t arrivals(int i) {
        return (i >= p_ready && i < p_ready + 2) || (i >= o_empty && i < o_empty + 2) ? 4u
               : (i >= kv_empty && i < kv_empty + S)                                   ? 2u
               : (F8 && i >= kv_full && i < kv_full + S)                               ? 3u
               : (F8 && i >= v8_empty && i < v8_empty + S8)                            ? 2u
                                                                                       : 1u;
    }
};

__device__ __forceinline__ uint32_t bar_at(uint32_t bar0, int idx) { return bar0 + 8u * static_cast<uint32_t>(idx); }

// ---------------------------------------------------------------- producer warp (one thread; bf16)
template <int HD>
__device__ __noinline__ void role_producer(const FwdParams& p, const Schedule& sc, uint32_t smem0, uint32_t bar0,
                                           int n_items) {
    using C = Cfg<HD>;
    using BI = BarIdx<C::kStages>;
    constexpr int S = C::kStages;
    constexpr int kPanelElems = 64;  // bf16 values per 128-byte panel
    const uint32_t ring0 = smem0 + 2 * C::kTileBytes;
    const int grid = gridDim.x, cta = blockIdx.x;
    uint32_t uc = 0, qc[2] = {0, 0};
    bool ok = true;
    Item it;
    for (int r = 0; ok && r * grid < n_items; ++r) {
        const int k = snake(r, cta, grid);
        if (k >= n_items) continue;
        item_at(p, sc, k, it);
        const int n = it.len;
        if (n == 0) continue;
        const int g = it.h / p.group;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (it.n[t] == 0) continue;
            if (qc[t] > 0) ok = mbar_wait(bar_at(bar0, BI::q_empty + t), (qc[t] - 1) & 1, p.err);
            if (!ok) break;
            mbar_arrive_expect_tx(bar_at(bar0, BI::q_full + t), C::kTileBytes);
            const int y = it.s.q_base + it.pair * kPairRows + t * kBM;
#pragma unroll
            for (int pn = 0; pn < C::kPanels; ++pn)
                tma_load_2d(smem0 + t * C::kTileBytes + pn * C::kPanelBytes, &p.tm_q, bar_at(bar0, BI::q_full + t),
                            it.h * HD + pn * kPanelElems, y);
            ++qc[t];
        }
        if (!ok) break;
        // slots u = 0..n: V_{j0+u-1} (u >= 1) and K_{j0+u} (u < n)
        for (int u = 0; u <= n && ok; ++u) {
            const uint32_t st = uc % S;
            if (uc >= S) ok = mbar_wait(bar_at(bar0, BI::kv_empty + st), ((uc / S) - 1) & 1, p.err);
            if (!ok) break;
            const uint32_t slot = ring0 + st * C::kSlotBytes;
            const uint32_t full = bar_at(bar0, BI::kv_full + st);
            mbar_arrive_expect_tx(full, (u < n ? C::kTileBytes : 0) + (u >= 1 ? C::kVBytes : 0));
            if (u < n) {
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_load_2d(slot + pn * C::kPanelBytes, &p.tm_k, full, g * HD + pn * kPanelElems,
                                it.s.k_base + (it.j0 + u) * kBN);
            }
            if (u >= 1) {
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_load_2d(slot + C::kTileBytes + pn * C::kPanelBytes, &p.tm_v, full, g * HD + pn * 64,
                                it.s.k_base + (it.j0 + u - 1) * kBN);
            }
            ++uc;
        }
    }
    // Drain: every load issued must have landed before the CTA exits.
    for (uint32_t i = (uc > S ? uc - S : 0); i < uc; ++i)
        mbar_wait(bar_at(bar0, BI::kv_full + i % S), (i / S) & 1, p.err);
    for (int t = 0; t < 2; ++t)
        if (qc[t] > 0) mbar_wait(bar_at(bar0, BI::q_full + t), (qc[t] - 1) & 1, p.err);
}

// ---------------------------------------------------------------- widening of 8-bit V tiles (8-bit forward)
// Each 8-bit V tile is widened into the 16-bit (f16) layout the PV product
// reads -- E4M3 values are exact in f16 -- so that P can stay a 16-bit
// operand.  The staging tile is [128 keys][128 bytes], 128-byte swizzled by
// TMA; the slot's V part is two [128 keys][64 f16] panels, 128-byte swizzled
// the same way as a TMA-loaded bf16 V tile.  Two warps share the work: warp 11
// (idle in the bf16 kernel) widens key rows 0-63 and the producer warp rows
// 64-127, right after issuing its loads.  Each lane converts 16-byte chunks
// (16 values): eight lanes cover one key row, so each shared-memory request
// touches every bank once.  Lane l converts chunk kc = l % 8 (values 16 kc ..
// 16 kc + 15) of key rows 4 i + l / 8; the rows' swizzle phase (row % 8)
// alternates between two values with i, so the byte offsets are set up once.
// Destination: panel kc / 4, 16-byte chunks 2 (kc % 4) and 2 (kc % 4) + 1.
template <int HD>
struct Widen {
    using C = Cfg<HD, true>;
    uint32_t src_off[2], dst_off[2][2];

    __device__ __forceinline__ explicit Widen(int lane) {
        const int kc = lane & 7, r0 = lane >> 3;
#pragma unroll
        for (int par = 0; par < 2; ++par) {
            const int ph = r0 + 4 * par;  // row % 8 for rows 4 i + r0 with i % 2 == par
            src_off[par] = r0 * 128 + ((kc ^ ph) << 4);
            const uint32_t prow = (kc >> 2) * C::kVPanelBytes + r0 * 128;
            dst_off[par][0] = prow + (((2 * (kc & 3)) ^ ph) << 4);
            dst_off[par][1] = prow + (((2 * (kc & 3) + 1) ^ ph) << 4);
        }
    }

    // Key rows 64 half .. 64 half + 63 of the staged tile at src0 into the
    // slot's V part at dst0; the writes are fenced for the tensor core.
    __device__ __forceinline__ void run(uint32_t src0, uint32_t dst0, int half) const {
#pragma unroll
        for (int i2 = 0; i2 < kBN * HD / 16 / 32 / 2; ++i2) {
            const int i = half * (kBN * HD / 16 / 32 / 2) + i2;
            const int par = i2 & 1;  // i2 and i have the same parity (the half offset is even)
            uint32_t w0, w1, w2, w3;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                         : "r"(src0 + src_off[par] + i * 512)
                         : "memory");
            uint32_t h[8];
            e4m3x4_to_f16x2x2(w0, h[0], h[1]);
            e4m3x4_to_f16x2x2(w1, h[2], h[3]);
            e4m3x4_to_f16x2x2(w2, h[4], h[5]);
            e4m3x4_to_f16x2x2(w3, h[6], h[7]);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst0 + dst_off[par][0] + i * 512),
                         "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst0 + dst_off[par][1] + i * 512),
                         "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7])
                         : "memory");
        }
        fence_proxy_async_smem();
    }
};

// d = 64: the staged E4M3 rows are 64 bytes, unswizzled; the f16 tile is one
// 128-byte-swizzled panel.  Lane l converts code chunk kc = l % 4 (values
// 16 kc .. 16 kc + 15) of key rows 8 i + l / 4 into f16 chunks 2 kc and
// 2 kc + 1 of the same rows; a lane's rows all have the swizzle phase l / 4.
// A warp request reads 512 contiguous bytes (eight rows).
template <>
struct Widen<64> {
    uint32_t src_off, dst_off0, dst_off1;

    __device__ __forceinline__ explicit Widen(int lane) {
        const int kc = lane & 3, r0 = lane >> 2;
        src_off = r0 * 64 + kc * 16;
        dst_off0 = r0 * 128 + (((2 * kc) ^ r0) << 4);
        dst_off1 = r0 * 128 + (((2 * kc + 1) ^ r0) << 4);
    }

    // Key rows 64 half .. 64 half + 63 (row groups 8 half .. 8 half + 7).
    __device__ __forceinline__ void run(uint32_t src0, uint32_t dst0, int half) const {
#pragma unroll
        for (int i2 = 0; i2 < 8; ++i2) {
            const int i = half * 8 + i2;
            uint32_t w0, w1, w2, w3;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                         : "r"(src0 + src_off + i * 512)
                         : "memory");
            uint32_t h[8];
            e4m3x4_to_f16x2x2(w0, h[0], h[1]);
            e4m3x4_to_f16x2x2(w1, h[2], h[3]);
            e4m3x4_to_f16x2x2(w2, h[4], h[5]);
            e4m3x4_to_f16x2x2(w3, h[6], h[7]);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst0 + dst_off0 + i * 1024),
                         "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst0 + dst_off1 + i * 1024),
                         "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7])
                         : "memory");
        }
        fence_proxy_async_smem();
    }
};

// Warp 11: widens key rows 0-63 of every 8-bit V tile.  It walks the same
// items and ring slots as the producer and arrives on the slot's full barrier
// once its half is written; a slot without a V tile (u = 0) gets the arrival
// at once.
template <int HD>
__device__ __noinline__ void role_convert(const FwdParams& p, const Schedule& sc, uint32_t smem0, uint32_t bar0,
                                          int n_items) {
    using C = Cfg<HD, true>;
    using BI = BarIdx<C::kStages, true, C::kV8Stages>;
    constexpr int S = C::kStages;
    const int lane = threadIdx.x & 31;
    const uint32_t ring0 = smem0 + 2 * C::kTileBytes;
    const uint32_t v8_0 = ring0 + S * C::kSlotBytes;
    const int grid = gridDim.x, cta = blockIdx.x;
    const Widen<HD> wd(lane);
    uint32_t uc = 0, vc = 0;
    bool ok = true;
    Item it;
    for (int r = 0; ok && r * grid < n_items; ++r) {
        const int k = snake(r, cta, grid);
        if (k >= n_items) continue;
        item_at(p, sc, k, it);
        const int n = it.len;
        if (n == 0) continue;
        for (int u = 0; u <= n && ok; ++u) {
            const uint32_t st = uc % S;
            if (uc >= S) ok = __all_sync(0xffffffffu, mbar_wait(bar_at(bar0, BI::kv_empty + st), ((uc / S) - 1) & 1, p.err));
            if (!ok) break;
            if (u >= 1) {
                const uint32_t s8 = vc % C::kV8Stages;
                ok = __all_sync(0xffffffffu,
                                mbar_wait(bar_at(bar0, BI::v8_full + s8), (vc / C::kV8Stages) & 1, p.err));
                if (!ok) break;
                wd.run(v8_0 + s8 * C::kV8Bytes, ring0 + st * C::kSlotBytes + C::kTileBytes, 0);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_at(bar0, BI::v8_empty + s8));
                ++vc;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_at(bar0, BI::kv_full + st));
            ++uc;
        }
    }
}

// Producer warp of the 8-bit forward (all 32 lanes): lane 0 issues the TMA
// loads as the bf16 producer does -- the 8-bit V_{j0+u} with K_{j0+u}, a
// slot ahead of the slot it is widened into -- and then the whole warp widens
// key rows 64-127 of the V tile that slot u takes.
template <int HD>
__device__ __noinline__ void role_producer_f8(const FwdParams& p, const Schedule& sc, uint32_t smem0, uint32_t bar0,
                                              int n_items) {
    using C = Cfg<HD, true>;
    using BI = BarIdx<C::kStages, true, C::kV8Stages>;
    constexpr int S = C::kStages;
    const int lane = threadIdx.x & 31;
    const bool leader = lane == 0;
    const uint32_t ring0 = smem0 + 2 * C::kTileBytes;
    const uint32_t v8_0 = ring0 + S * C::kSlotBytes;
    const int grid = gridDim.x, cta = blockIdx.x;
    const Widen<HD> wd(lane);
    uint32_t uc = 0, vc = 0, cc = 0, qc[2] = {0, 0};  // ring slots, V8 loads, V8 tiles widened, Q loads
    bool ok = true;
    Item it;
    for (int r = 0; ok && r * grid < n_items; ++r) {
        const int k = snake(r, cta, grid);
        if (k >= n_items) continue;
        item_at(p, sc, k, it);
        const int n = it.len;
        if (n == 0) continue;
        const int g = it.h / p.group;
        if (leader) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (it.n[t] == 0) continue;
                if (qc[t] > 0) ok = mbar_wait(bar_at(bar0, BI::q_empty + t), (qc[t] - 1) & 1, p.err);
                if (!ok) break;
                mbar_arrive_expect_tx(bar_at(bar0, BI::q_full + t), C::kTileBytes);
                tma_load_2d(smem0 + t * C::kTileBytes, &p.tm_q, bar_at(bar0, BI::q_full + t), it.h * HD,
                            it.s.q_base + it.pair * kPairRows + t * kBM);
                ++qc[t];
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        for (int u = 0; u <= n && ok; ++u) {
            const uint32_t st = uc % S;
            if (uc >= S) ok = __all_sync(0xffffffffu, mbar_wait(bar_at(bar0, BI::kv_empty + st), ((uc / S) - 1) & 1, p.err));
            if (!ok) break;
            const uint32_t slot = ring0 + st * C::kSlotBytes;
            if (leader) {
                const uint32_t full = bar_at(bar0, BI::kv_full + st);
                mbar_arrive_expect_tx(full, u < n ? C::kTileBytes : 0);
                if (u < n) {
                    tma_load_2d(slot, &p.tm_k, full, g * HD, it.s.k_base + (it.j0 + u) * kBN);
                    const uint32_t s8 = vc % C::kV8Stages;
                    if (vc >= C::kV8Stages)
                        ok = mbar_wait(bar_at(bar0, BI::v8_empty + s8), ((vc / C::kV8Stages) - 1) & 1, p.err);
                    if (ok) {
                        const uint32_t v8full = bar_at(bar0, BI::v8_full + s8);
                        mbar_arrive_expect_tx(v8full, C::kV8Bytes);
                        tma_load_2d(v8_0 + s8 * C::kV8Bytes, &p.tm_v, v8full, g * HD,
                                    it.s.k_base + (it.j0 + u) * kBN);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (u < n) ++vc;
            if (u >= 1) {  // rows 64-127 of V_{j0+u-1} into this slot
                const uint32_t s8 = cc % C::kV8Stages;
                ok = __all_sync(0xffffffffu,
                                mbar_wait(bar_at(bar0, BI::v8_full + s8), (cc / C::kV8Stages) & 1, p.err));
                if (!ok) break;
                wd.run(v8_0 + s8 * C::kV8Bytes, slot + C::kTileBytes, 1);
                __syncwarp();
                if (leader) mbar_arrive(bar_at(bar0, BI::v8_empty + s8));
                ++cc;
            }
            __syncwarp();
            if (leader) mbar_arrive(bar_at(bar0, BI::kv_full + st));
            ++uc;
        }
    }
    // Drain: every load issued must have landed before the CTA exits.
    if (leader) {
        for (uint32_t i = (uc > S ? uc - S : 0); i < uc; ++i)
            mbar_wait(bar_at(bar0, BI::kv_full + i % S), (i / S) & 1, p.err);
        for (uint32_t i = (vc > C::kV8Stages ? vc - C::kV8Stages : 0); i < vc; ++i)
            mbar_wait(bar_at(bar0, BI::v8_full + i % C::kV8Stages), (i / C::kV8Stages) & 1, p.err);
        for (int t = 0; t < 2; ++t)
            if (qc[t] > 0) mbar_wait(bar_at(bar0, BI::q_full + t), (qc[t] - 1) & 1, p.err);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- MMA warp (one thread)
// Shared-memory descriptor of a K-major Q or K tile: 128-byte rows with the
// 128-byte swizzle (8-row groups 1024 bytes apart), or, for the 8-bit tiles
// at d = 64, 64-byte rows with the 64-byte swizzle (groups 512 bytes apart).
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t desc = 0;
    desc |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    desc |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    desc |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    desc |= 1ull << 46;  // descriptor version for tcgen05
    desc |= 4ull << 61;  // 64-byte swizzle
    return desc;
}
template <int HD, bool F8>
__device__ __forceinline__ uint64_t qk_desc(uint32_t saddr) {
    if constexpr (Cfg<HD, F8>::kRowBytes == 64) return smem_desc_sw64(saddr, 16, 512);
    else return smem_desc_sw128(saddr, 16, 1024);
}

// Descriptors are built once per kernel; each K-step adds a compile-time
// offset (the 14-bit start-address field never overflows: shared memory is
// below 256 KB).  The tensor pipe's input queue is shallow, so issue is
// close to synchronous with execution: the issuing thread keeps the work
// between MMA groups to the minimum.
template <int HD, bool F8>
__device__ __forceinline__ void issue_s(uint32_t tmem_d, uint64_t q_desc, uint64_t k_desc) {
    using C = Cfg<HD, F8>;
    if constexpr (F8) {
        // E4M3 x E4M3: 32 values (32 bytes) of the head dimension per MMA
        constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kBN);
#pragma unroll
        for (int kk = 0; kk < HD / 32; ++kk) {
            const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::kPanelBytes + (kk & 3) * 32) >> 4);
            mma_f8_smem_smem(tmem_d, q_desc + off, k_desc + off, idesc, kk > 0);
        }
    } else {
        constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
            const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::kPanelBytes + (kk & 3) * 32) >> 4);
            mma_smem_smem(tmem_d, q_desc + off, k_desc + off, idesc, kk > 0);
        }
    }
}

// P (16-bit, tensor memory) x V (16-bit, shared memory): bf16, or f16 in the
// 8-bit forward (P carries the V tile's scale there, V the exact E4M3 values).
template <int HD, bool F8>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t v_desc, bool first) {
    constexpr uint32_t idesc = F8 ? idesc_f16_f32(kBM, HD, true) : idesc_bf16_f32(kBM, HD, true);
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk)
        mma_tmem_smem(tmem_o, tmem_p + kk * 8, v_desc + static_cast<uint64_t>((kk * 2048) >> 4), idesc,
                      (!first || kk > 0) ? 1u : 0u);
}

// Two issuing threads, one per query tile, that take turns slot by slot: a
// thread issues its MMAs of ring slot u only after the other thread has
// issued its MMAs of the preceding turn (the `tok` barriers), so the tensor
// pipe sees the single-issuer order
//     ..., PV0(j), S0(j+1), PV1(j), S1(j+1), PV0(j+1), ...
// while each thread's barrier waits overlap the other thread's MMAs (issue is
// close to synchronous with execution, so a wait in a lone issuer idles the
// tensor pipe).  Slot u of an item holds V_{j-1} and K_j (j = j0 + u):
// issuer t runs PV_t(j-1) and S_t(j) for the tiles inside its own range
// [lo_t, hi_t), then releases the slot.
template <int HD, bool F8>
__device__ __noinline__ void role_mma(const FwdParams& p, const Schedule& sc, uint32_t smem0, uint32_t bar0,
                                      uint32_t tmem, int n_items, int t) {
    using C = Cfg<HD, F8>;
    using BI = BarIdx<C::kStages, F8, C::kV8Stages>;
    constexpr int S = C::kStages;
    const uint32_t ring0 = smem0 + 2 * C::kTileBytes;
    const uint64_t dq = qk_desc<HD, F8>(smem0 + t * C::kTileBytes);
    const uint64_t dk0 = qk_desc<HD, F8>(ring0);                                         // K part of slot 0
    const uint64_t dv0 = smem_desc_sw128(ring0 + C::kTileBytes, C::kVPanelBytes, 1024);  // V part of slot 0
    constexpr uint64_t kSlotDesc = C::kSlotBytes >> 4;  // descriptor step between ring slots
    const uint32_t ts = tmem + C::col_s(t);
    const uint32_t to = tmem + C::col_o(t);
    const uint32_t b_q_full = bar_at(bar0, BI::q_full + t), b_q_empty = bar_at(bar0, BI::q_empty + t);
    const uint32_t b_s_full = bar_at(bar0, BI::s_full + t), b_p_ready = bar_at(bar0, BI::p_ready + t);
    const uint32_t b_o_final = bar_at(bar0, BI::o_final + t), b_o_empty = bar_at(bar0, BI::o_empty + t);
    const uint32_t b_tok_mine = bar_at(bar0, BI::tok + t), b_tok_other = bar_at(bar0, BI::tok + (1 - t));
    const int grid = gridDim.x, cta = blockIdx.x;
    uint32_t uc = 0, qc = 0, pc = 0, oc = 0;
    bool ok = true;
    Item it;
    for (int r = 0; ok && r * grid < n_items; ++r) {
        const int k = snake(r, cta, grid);
        if (k >= n_items) continue;
        item_at(p, sc, k, it);
        const int n = it.len;
        const int nt = t == 0 ? it.n[0] : it.n[1];
        if (n == 0) continue;
        // this tile's range, relative to the stream
        const int ulo = (t == 0 ? it.lo[0] : it.lo[1]) - it.j0, uhi = ulo + nt;
        if (nt > 0) {
            ok = mbar_wait(b_q_full, qc & 1, p.err);
            ++qc;
            if (!ok) break;
        }
        for (int u = 0; u <= n && ok; ++u) {
            const uint32_t st = uc % S;
            const bool pv = u - 1 >= ulo && u - 1 < uhi;
            const bool sm = u >= ulo && u < uhi;
            ok = mbar_wait(bar_at(bar0, BI::kv_full + st), (uc / S) & 1, p.err);
            if (ok && pv) {
                // the softmax's hand-off is the chain's critical link: the bf16
                // kernel's issuer keeps polling for it (measured +4-5%); in the
                // 8-bit kernel the widening warps need issue slots too, so the
                // issuer polls briefly and then sleeps
                ok = F8 ? mbar_wait_poll_then_sleep(b_p_ready, pc & 1, p.err)
                        : mbar_wait_spin(b_p_ready, pc & 1, p.err);
                ++pc;
                if (ok && u - 1 == ulo && oc > 0) ok = mbar_wait(b_o_empty, (oc - 1) & 1, p.err);
            }
            // my turn: issuer 0 follows issuer 1's previous turn, issuer 1 follows issuer 0's turn on this slot
            if (ok && (t == 1 || uc > 0)) ok = mbar_wait(b_tok_other, (t == 1 ? uc : uc - 1) & 1, p.err);
            if (!ok) break;
            if (pv) {
                tc_fence_after_sync();
                issue_pv<HD, F8>(to, ts, dv0 + st * kSlotDesc, u - 1 == ulo);
                if (u == uhi) {
                    tc_commit(b_o_final);
                    ++oc;
                }
            }
            if (sm) {
                issue_s<HD, F8>(ts, dq, dk0 + st * kSlotDesc);
                tc_commit(b_s_full);
                if (u == uhi - 1) tc_commit(b_q_empty);
            }
            if (pv || sm) tc_commit(bar_at(bar0, BI::kv_empty + st));
            else mbar_arrive(bar_at(bar0, BI::kv_empty + st));
            mbar_arrive(b_tok_mine);
            ++uc;
        }
    }
    // Drain: all tensor-core work this thread issued must finish before TMEM is freed.
    tc_commit(bar_at(bar0, BI::mma_done + t));
    mbar_wait(bar_at(bar0, BI::mma_done + t), 0, p.err);
}


// 32 lanes x 32 bits, 128 consecutive columns in one request: thread t of
// the warp receives lane (taddr.lane + t), columns taddr.col .. taddr.col+127.
__device__ __forceinline__ void tmem_ld_128cols_f(uint32_t taddr, float* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
        "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, "
        "%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
        "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, "
        "%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, "
        "%112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127"
        "}, [%128];"
        : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7]),
          "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]), "=f"(r[14]), "=f"(r[15]),
          "=f"(r[16]), "=f"(r[17]), "=f"(r[18]), "=f"(r[19]), "=f"(r[20]), "=f"(r[21]), "=f"(r[22]), "=f"(r[23]),
          "=f"(r[24]), "=f"(r[25]), "=f"(r[26]), "=f"(r[27]), "=f"(r[28]), "=f"(r[29]), "=f"(r[30]), "=f"(r[31]),
          "=f"(r[32]), "=f"(r[33]), "=f"(r[34]), "=f"(r[35]), "=f"(r[36]), "=f"(r[37]), "=f"(r[38]), "=f"(r[39]),
          "=f"(r[40]), "=f"(r[41]), "=f"(r[42]), "=f"(r[43]), "=f"(r[44]), "=f"(r[45]), "=f"(r[46]), "=f"(r[47]),
          "=f"(r[48]), "=f"(r[49]), "=f"(r[50]), "=f"(r[51]), "=f"(r[52]), "=f"(r[53]), "=f"(r[54]), "=f"(r[55]),
          "=f"(r[56]), "=f"(r[57]), "=f"(r[58]), "=f"(r[59]), "=f"(r[60]), "=f"(r[61]), "=f"(r[62]), "=f"(r[63]),
          "=f"(r[64]), "=f"(r[65]), "=f"(r[66]), "=f"(r[67]), "=f"(r[68]), "=f"(r[69]), "=f"(r[70]), "=f"(r[71]),
          "=f"(r[72]), "=f"(r[73]), "=f"(r[74]), "=f"(r[75]), "=f"(r[76]), "=f"(r[77]), "=f"(r[78]), "=f"(r[79]),
          "=f"(r[80]), "=f"(r[81]), "=f"(r[82]), "=f"(r[83]), "=f"(r[84]), "=f"(r[85]), "=f"(r[86]), "=f"(r[87]),
          "=f"(r[88]), "=f"(r[89]), "=f"(r[90]), "=f"(r[91]), "=f"(r[92]), "=f"(r[93]), "=f"(r[94]), "=f"(r[95]),
          "=f"(r[96]), "=f"(r[97]), "=f"(r[98]), "=f"(r[99]), "=f"(r[100]), "=f"(r[101]), "=f"(r[102]), "=f"(r[103]),
          "=f"(r[104]), "=f"(r[105]), "=f"(r[106]), "=f"(r[107]), "=f"(r[108]), "=f"(r[109]), "=f"(r[110]), "=f"(r[111]),
          "=f"(r[112]), "=f"(r[113]), "=f"(r[114]), "=f"(r[115]), "=f"(r[116]), "=f"(r[117]), "=f"(r[118]), "=f"(r[119]),
          "=f"(r[120]), "=f"(r[121]), "=f"(r[122]), "=f"(r[123]), "=f"(r[124]), "=f"(r[125]), "=f"(r[126]), "=f"(r[127])
        : "r"(taddr));
}

// Wait for the request above; the registers are passed through so that no
// use of them can move before the wait.
__device__ __forceinline__ void tmem_ld_wait128_f(float* r) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+f"(r[0]), "+f"(r[1]), "+f"(r[2]), "+f"(r[3]), "+f"(r[4]), "+f"(r[5]), "+f"(r[6]), "+f"(r[7]),
          "+f"(r[8]), "+f"(r[9]), "+f"(r[10]), "+f"(r[11]), "+f"(r[12]), "+f"(r[13]), "+f"(r[14]), "+f"(r[15]),
          "+f"(r[16]), "+f"(r[17]), "+f"(r[18]), "+f"(r[19]), "+f"(r[20]), "+f"(r[21]), "+f"(r[22]), "+f"(r[23]),
          "+f"(r[24]), "+f"(r[25]), "+f"(r[26]), "+f"(r[27]), "+f"(r[28]), "+f"(r[29]), "+f"(r[30]), "+f"(r[31]),
          "+f"(r[32]), "+f"(r[33]), "+f"(r[34]), "+f"(r[35]), "+f"(r[36]), "+f"(r[37]), "+f"(r[38]), "+f"(r[39]),
          "+f"(r[40]), "+f"(r[41]), "+f"(r[42]), "+f"(r[43]), "+f"(r[44]), "+f"(r[45]), "+f"(r[46]), "+f"(r[47]),
          "+f"(r[48]), "+f"(r[49]), "+f"(r[50]), "+f"(r[51]), "+f"(r[52]), "+f"(r[53]), "+f"(r[54]), "+f"(r[55]),
          "+f"(r[56]), "+f"(r[57]), "+f"(r[58]), "+f"(r[59]), "+f"(r[60]), "+f"(r[61]), "+f"(r[62]), "+f"(r[63]),
          "+f"(r[64]), "+f"(r[65]), "+f"(r[66]), "+f"(r[67]), "+f"(r[68]), "+f"(r[69]), "+f"(r[70]), "+f"(r[71]),
          "+f"(r[72]), "+f"(r[73]), "+f"(r[74]), "+f"(r[75]), "+f"(r[76]), "+f"(r[77]), "+f"(r[78]), "+f"(r[79]),
          "+f"(r[80]), "+f"(r[81]), "+f"(r[82]), "+f"(r[83]), "+f"(r[84]), "+f"(r[85]), "+f"(r[86]), "+f"(r[87]),
          "+f"(r[88]), "+f"(r[89]), "+f"(r[90]), "+f"(r[91]), "+f"(r[92]), "+f"(r[93]), "+f"(r[94]), "+f"(r[95]),
          "+f"(r[96]), "+f"(r[97]), "+f"(r[98]), "+f"(r[99]), "+f"(r[100]), "+f"(r[101]), "+f"(r[102]), "+f"(r[103]),
          "+f"(r[104]), "+f"(r[105]), "+f"(r[106]), "+f"(r[107]), "+f"(r[108]), "+f"(r[109]), "+f"(r[110]), "+f"(r[111]),
          "+f"(r[112]), "+f"(r[113]), "+f"(r[114]), "+f"(r[115]), "+f"(r[116]), "+f"(r[117]), "+f"(r[118]), "+f"(r[119]),
          "+f"(r[120]), "+f"(r[121]), "+f"(r[122]), "+f"(r[123]), "+f"(r[124]), "+f"(r[125]), "+f"(r[126]), "+f"(r[127])
        :
        : "memory");
}

// ---------------------------------------------------------------- softmax warpgroups
// 8-bit forward: the scores of tile j are c_j * (Q8 K8_j^T) with
// c_j = scale * log2(e) * s_q * s_k(j) (the tiles' scales), and the values
// are s_v(j) * V8_j.  Each tile's scale ratio r_j = s_v(j) / s_ref (s_ref
// the item's first tile's) is folded into the exponent: the exponent of p
// r_j is t + log2 r_j (t = the score in log2 units), the row's running max
// is taken over those, the softmax writes p * r_j / 2^m (f16, at most 2^8)
// and the PV product adds that times V8_j; the normaliser sums p / 2^m
// (the stored value times 1 / r_j), and the epilogue multiplies by
// s_ref / l.
template <int HD, bool F8>
__device__ __noinline__ void role_softmax(const FwdParams& p, const Schedule& sc, uint32_t bar0, uint32_t tmem,
                                          int n_items, int t) {
    using C = Cfg<HD, F8>;
    using BI = BarIdx<C::kStages, F8, C::kV8Stages>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wq = warp & 3;                 // lane quarter of tensor memory
    const int row_in_tile = wq * 32 + lane;  // == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::col_s(t);
    const uint32_t t_o = tmem + lane_off + C::col_o(t);
    const uint32_t b_s_full = bar_at(bar0, BI::s_full + t), b_p_ready = bar_at(bar0, BI::p_ready + t);
    const uint32_t b_o_final = bar_at(bar0, BI::o_final + t), b_o_empty = bar_at(bar0, BI::o_empty + t);
    const float sl2 = p.scale_log2;
    const int grid = gridDim.x, cta = blockIdx.x;
    uint32_t scnt = 0, ocnt = 0;
    bool ok = true;
    Item it;
    for (int r = 0; ok && r * grid < n_items; ++r) {
        const int k = snake(r, cta, grid);
        if (k >= n_items) continue;
        item_at(p, sc, k, it);
        const int rows_t = t == 0 ? it.rows[0] : it.rows[1];
        if (rows_t == 0) continue;
        const int nt = t == 0 ? it.n[0] : it.n[1];
        const int jlo = t == 0 ? it.lo[0] : it.lo[1];
        const int q_tile0 = it.pair * kPairRows + t * kBM;
        const int q_local = q_tile0 + row_in_tile;
        const bool row_valid = row_in_tile < rows_t;
        const int nq = it.s.nq, nk = it.s.nk;
        // allowed keys of this row; a tile needs masking when it reaches past
        // the first row's last key or before the last row's first key
        const int kmin_row = key_first(q_local, nq, nk, p.win_left);
        const int kmax_row = key_last(q_local, nq, nk, p.win_right);
        const int kmax_first = key_last(q_tile0, nq, nk, p.win_right);
        const int kmin_last = key_first(q_tile0 + kBM - 1, nq, nk, p.win_left);
        float m_ref = -INFINITY;
        float l = 0.f;
        // 8-bit: scale entries of this query tile and of the item's K/V tiles.
        // V tile j's scale enters as lv_j = log2(s_v(j) / s_ref), s_ref the
        // scale of the item's first tile, added to the exponent of every p of
        // the tile.  The row max then tracks p * s_v rather than p, so P (f16)
        // is normalised to the row's largest contribution to O, whatever the
        // spread of the V scales.
        float c_q = sl2, s_ref = 1.f, lg_ref = 0.f;
        const float *ks_row = nullptr, *vs_row = nullptr;
        if constexpr (F8) {
            const int g = it.h / p.group;
            c_q = sl2 * __ldg(p.q_scale + it.h * p.n_scale_q + it.s.q_base / kBM + it.b + it.pair * 2 + t);
            ks_row = p.k_scale + g * p.n_scale_k + it.s.k_base / kBN + it.b;
            vs_row = p.v_scale + g * p.n_scale_k + it.s.k_base / kBN + it.b;
            if (nt > 0) {
                s_ref = __ldg(vs_row + jlo);
                asm("lg2.approx.f32 %0, %1;" : "=f"(lg_ref) : "f"(s_ref));
            }
        }
        for (int j = jlo; j < jlo + nt; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_s_full, scnt & 1, p.err));
            ++scnt;
            if (!ok) break;
            tc_fence_after_sync();
            float x[128];
            tmem_ld_128cols_f(t_s, x);
            // 8-bit: this tile's score coefficient, lv_j and 2^-lv_j.  Ratios
            // beyond 2^+-64 are clamped, which keeps every row sum term
            // 2^(t - m) <= 2^72 and 2^-lv finite.
            float ct = sl2, lv = 0.f, inv_r = 1.f;
            if constexpr (F8) {
                ct = c_q * __ldg(ks_row + j);
                float lg;
                asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(__ldg(vs_row + j)));
                lv = fminf(fmaxf(lg - lg_ref, -64.f), 64.f);
                inv_r = fast_exp2(-lv);
            }
            tmem_ld_wait128_f(x);
            const int k0 = j * kBN;
            if (k0 < kmin_last) {  // crosses the band's left edge (and maybe its right one)
                const int hi_lim = kmax_row - k0;  // columns outside [lo_lim, hi_lim] are masked
                const int lo_lim = kmin_row - k0;
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c > hi_lim || c < lo_lim) x[c] = -INFINITY;
            } else if (k0 + kBN - 1 > kmax_first) {  // crosses the right edge or the sequence end only
                const int hi_lim = kmax_row - k0;
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c > hi_lim) x[c] = -INFINITY;
            }
            // row max of the tile in log2 units: 3-input max over 8 independent chains
            auto row_max2 = [&]() {
                float mc[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) mc[c] = fmaxf(x[c], x[c + 8]);
#pragma unroll
                for (int c = 16; c < 128; c += 16) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) mc[k] = fmax3(mc[k], x[c + k], x[c + 8 + k]);
                }
                const float mx =
                    fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
                return F8 ? mx * ct + lv : mx * ct;
            };
            // p = 2^(s*scale*log2e - m) into tensor memory (bf16; 8-bit
            // forward: p * 2^lv_j as f16): packed FMA for the argument, one
            // ex2 per element, four independent packed partial sums; returns
            // the row sum of the stored values (fp32)
            auto exp_pass = [&](float m) {
                const float m_use = ((m == -INFINITY) ? 0.f : m) - lv;
                const uint64_t sc2 = f2_pack(ct, ct);
                const uint64_t nm2 = f2_pack(-m_use, -m_use);
                uint64_t ls[4] = {0, 0, 0, 0};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        float a, b;
                        f2_unpack(f2_fma(f2_pack(x[h * 64 + c], x[h * 64 + c + 1]), sc2, nm2), a, b);
                        a = fast_exp2(a);
                        b = fast_exp2(b);
                        ls[(c >> 1) & 3] = f2_add(ls[(c >> 1) & 3], f2_pack(a, b));
                        pk[c >> 1] = F8 ? pack_f16x2(a, b) : pack_bf16x2(a, b);
                    }
                    tmem_st_32cols(t_s + h * 32, pk);
                }
                const uint64_t s01 = f2_add(ls[0], ls[1]), s23 = f2_add(ls[2], ls[3]);
                float lo, hi;
                f2_unpack(f2_add(s01, s23), lo, hi);
                return lo + hi;
            };
            float lsum;
            if (j == jlo) {
                m_ref = row_max2();
                lsum = exp_pass(m_ref);
            } else {
                // Fast path: the reference max is kept unless the tile max
                // exceeds it by more than the threshold, i.e. unless some
                // p > 2^8.  p >= 0 and a rounded sum of non-negative terms is
                // at least each term, so a row sum <= 2^8 proves every p of
                // the row within the bound and the max is never needed.  A
                // row with no key yet (reference -inf: every earlier key
                // masked) always looks at the max.
                lsum = exp_pass(m_ref);
                if (__any_sync(0xffffffffu, !(lsum <= 256.f) || m_ref == -INFINITY)) {
                    const float mx2 = row_max2();
                    const bool need = mx2 > m_ref + kRescaleThreshold;
                    if (__any_sync(0xffffffffu, need)) {
                        const float m_new = fmaxf(m_ref, mx2);
                        const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_ref - m_new);
                        l *= alpha;
                        m_ref = m_new;
                        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
                        for (int cc = 0; cc < HD; cc += 32) {
                            float o[32];
                            tmem_ld_32cols_f(t_o + cc, o);
                            tmem_ld_wait_f(o);
#pragma unroll
                            for (int c = 0; c < 32; c += 2) {
                                const uint64_t v = f2_mul(f2_pack(o[c], o[c + 1]), a2);
                                f2_unpack(v, o[c], o[c + 1]);
                            }
                            tmem_st_32cols(t_o + cc, reinterpret_cast<const uint32_t(&)[32]>(o));
                        }
                        tmem_st_wait();  // the first pass's P stores land before they are overwritten
                        lsum = exp_pass(m_ref);
                    }
                }
            }
            l += F8 ? lsum * inv_r : lsum;  // 8-bit: the row sum counts p, not p * 2^lv_j
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_p_ready);
        }
        if (!ok) break;
        // ---- epilogue: O / l -> bf16, lse
        const size_t out_row = static_cast<size_t>(it.s.q_base + q_local) * p.Hq + it.h;
        __nv_bfloat16* dst = p.out + out_row * HD;
        const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;  // rows are 128 or 256 bytes
        if (nt > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_o_final, ocnt & 1, p.err));
            ++ocnt;
            if (!ok) break;
            tc_fence_after_sync();
            const float inv_l = l > 0.f ? (F8 ? s_ref : 1.f) / l : 0.f;
            auto store_chunk = [&](const float* o, int cc) {
                if (row_valid && out32) {  // whole 32-byte sectors
#pragma unroll
                    for (int c = 0; c < 32; c += 16) {
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(o[c + 2 * i] * inv_l, o[c + 2 * i + 1] * inv_l);
                        st_global_v8(dst + cc + c, w);
                    }
                } else if (row_valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(o[c + 0] * inv_l, o[c + 1] * inv_l);
                        w.y = pack_bf16x2(o[c + 2] * inv_l, o[c + 3] * inv_l);
                        w.z = pack_bf16x2(o[c + 4] * inv_l, o[c + 5] * inv_l);
                        w.w = pack_bf16x2(o[c + 6] * inv_l, o[c + 7] * inv_l);
                        d4[c >> 3] = w;
                    }
                }
            };
            if constexpr (F8) {
                // 8-bit kernel: chunk k+1's load is in flight while chunk k is
                // stored, and the accumulator is released once the last
                // chunk is in registers (+1.5% there; the bf16 kernel ran
                // 1-2% slower with it, so it keeps one chunk at a time)
                float o0[32], o1[32];
                tmem_ld_32cols_f(t_o, o0);
                tmem_ld_wait_f(o0);
#pragma unroll
                for (int k = 0; k < HD / 32; k += 2) {
                    tmem_ld_32cols_f(t_o + (k + 1) * 32, o1);
                    store_chunk(o0, k * 32);
                    tmem_ld_wait_f(o1);
                    if (k + 2 < HD / 32) {
                        tmem_ld_32cols_f(t_o + (k + 2) * 32, o0);
                    } else {
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(b_o_empty);
                    }
                    store_chunk(o1, (k + 1) * 32);
                    if (k + 2 < HD / 32) tmem_ld_wait_f(o0);
                }
            } else {
#pragma unroll 1
                for (int cc = 0; cc < HD; cc += 32) {
                    float o[32];
                    tmem_ld_32cols_f(t_o + cc, o);
                    tmem_ld_wait_f(o);
                    store_chunk(o, cc);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(b_o_empty);
            }
        } else if (row_valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
            for (int c = 0; c < HD / 8; ++c) d4[c] = make_uint4(0, 0, 0, 0);
        }
        if (row_valid) {
            float lse_v = -INFINITY;
            if (l > 0.f) {
                float lg;
                asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(l));
                lse_v = (m_ref + lg) * 0.69314718055994531f;
            }
            const size_t li = p.varlen ? static_cast<size_t>(it.h) * p.Nq + it.s.q_base + q_local
                                       : (static_cast<size_t>(it.b) * p.Hq + it.h) * p.Nq + q_local;
            p.lse[li] = lse_v;
        }
    }
}

template <int HD, bool F8>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
    using C = Cfg<HD, F8>;
    using BI = BarIdx<C::kStages, F8, C::kV8Stages>;
    extern __shared__ __align__(1024) uint8_t smem_dyn[];
    __shared__ __align__(8) uint64_t bars[BI::count];
    __shared__ uint32_t tmem_base_slot;
    __shared__ Schedule sched;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t smem0 = (smem_addr(smem_dyn) + 1023u) & ~1023u;
    const uint32_t bar0 = smem_addr(bars);

    if (p.varlen) build_schedule(p, sched);

    if (threadIdx.x == 0) {
        for (int i = 0; i < BI::count; ++i) mbar_init(bar_at(bar0, i), BI::arrivals(i));
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(&tmem_base_slot), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_map(&p.tm_q);
        tma_prefetch_map(&p.tm_k);
        tma_prefetch_map(&p.tm_v);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_slot;
    const int n_items = total_items(p, sched);

    if (warp >= 8) {
        regs_decrease<kControlRegs>();
        if constexpr (F8) {
            if (warp == kProducerWarp) role_producer_f8<HD>(p, sched, smem0, bar0, n_items);
        } else {
            if (warp == kProducerWarp && lane == 0) role_producer<HD>(p, sched, smem0, bar0, n_items);
        }
        if (warp == kMmaWarp && lane == 0) role_mma<HD, F8>(p, sched, smem0, bar0, tmem, n_items, 0);
        if (warp == kMmaWarp + 1 && lane == 0) role_mma<HD, F8>(p, sched, smem0, bar0, tmem, n_items, 1);
        if constexpr (F8) {
            if (warp == kMmaWarp + 2) role_convert<HD>(p, sched, smem0, bar0, n_items);
        }
        __syncwarp();
    } else {
        regs_increase<kSoftmaxRegs>();
        role_softmax<HD, F8>(p, sched, bar0, tmem, n_items, warp >> 2);
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

// Optional check of cu_seqlens: start 0, nondecreasing, end == total.
__global__ void check_cu_seqlens_kernel(const int* cu, int B, int total, int* err) {
    for (int i = threadIdx.x; i <= B; i += blockDim.x) {
        const int v = cu[i];
        bool bad = (i == 0 && v != 0) || (i == B && v != total) || v < 0 || v > total;
        if (i > 0 && v < cu[i - 1]) bad = true;
        if (bad) record_error(err, ATTN_ERR_BAD_INDEX);
    }
}

template <int HD, bool F8>
attn_status launch_typed(const FwdArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
    using C = Cfg<HD, F8>;
    FwdParams p;
    memset(&p, 0, sizeof(p));
    const bool varlen = a.cu_q != nullptr;
    const uint64_t t_q = varlen ? static_cast<uint64_t>(a.Nq) : static_cast<uint64_t>(a.B) * a.Nq;
    // With no keys at all the K/V maps are never used; a zero extent is not
    // encodable, so they get one row.
    uint64_t t_k = varlen ? static_cast<uint64_t>(a.Nk) : static_cast<uint64_t>(a.B) * a.Nk;
    if (t_k == 0) t_k = 1;
    // boxes of 128 bytes x 128 rows (64 bf16 or 128 E4M3 values wide,
    // 128-byte swizzle); the 8-bit tiles at d = 64 are 64 bytes wide (Q and K
    // with the 64-byte swizzle, V staged unswizzled for the widening warps)
    constexpr uint64_t kElem = F8 ? 1 : 2;
    const CUtensorMapDataType dtype = F8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t box[2] = {static_cast<uint32_t>(C::kRowBytes / kElem), kBM};
    const CUtensorMapSwizzle sw_qk = C::kRowBytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    const CUtensorMapSwizzle sw_v = C::kRowBytes == 64 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(a.Hq) * HD, t_q};
        const uint64_t strides[1] = {static_cast<uint64_t>(a.Hq) * HD * kElem};
        attn_status st = encode_tma_swizzle(&p.tm_q, dtype, a.q, 2, dims, strides, box, sw_qk);
        if (st != ATTN_OK) return st;
    }
    {
        // with no keys the maps point at q (one row, never read)
        const uint64_t dims[2] = {static_cast<uint64_t>(a.Hkv) * HD, t_k};
        const uint64_t strides[1] = {static_cast<uint64_t>(a.Hkv) * HD * kElem};
        attn_status st = encode_tma_swizzle(&p.tm_k, dtype, a.k, 2, dims, strides, box, sw_qk);
        if (st != ATTN_OK) return st;
        st = encode_tma_swizzle(&p.tm_v, dtype, a.v, 2, dims, strides, box, sw_v);
        if (st != ATTN_OK) return st;
    }
    if constexpr (F8) {
        p.q_scale = a.q_scale;
        p.k_scale = a.k_scale;
        p.v_scale = a.v_scale;
        p.n_scale_q = fp8_scale_count(a.B, static_cast<long long>(t_q));
        p.n_scale_k = fp8_scale_count(a.B, varlen ? static_cast<long long>(a.Nk) : static_cast<long long>(a.B) * a.Nk);
    }
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.lse = a.lse;
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
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.err = dev.err_word;

    long long items;
    if (varlen)  // upper bound on (sequence, pair) entries times heads
        items = (static_cast<long long>(a.Nq) / kPairRows + a.B) * a.Hq;
    else
        items = static_cast<long long>((a.Nq + kPairRows - 1) / kPairRows) * a.B * a.Hq;
    if (items <= 0) return ATTN_OK;
    const int grid = static_cast<int>(items < dev.sm_count ? items : dev.sm_count);

    if (varlen && validation_enabled()) {
        check_cu_seqlens_kernel<<<1, 256, 0, stream>>>(a.cu_q, a.B, a.Nq, dev.err_word);
        check_cu_seqlens_kernel<<<1, 256, 0, stream>>>(a.cu_k, a.B, a.Nk, dev.err_word);
    }
    static std::atomic<bool> attr_set[kMaxDevices];  // per instantiation and device
    const bool cached = dev.device >= 0 && dev.device < kMaxDevices;
    if (!cached || !attr_set[dev.device].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<HD, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) {
            set_error_message("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, attn_fwd_kernel<HD, F8>);
        if (e != cudaSuccess) {
            set_error_message("cudaFuncGetAttributes: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        // setmaxnreg.inc can only draw on what the launch allocated
        if (fa.numRegs * kThreads < 2 * 128 * kSoftmaxRegs + 128 * kControlRegs) {
            set_error_message("attn_fwd kernel built with %d registers/thread; the warpgroup split needs %d",
                              fa.numRegs, kLaunchRegs);
            return ATTN_ERR_UNSUPPORTED;
        }
        if (cached) attr_set[dev.device].store(true, std::memory_order_release);
    }
    attn_fwd_kernel<HD, F8><<<grid, kThreads, C::kSmemBytes, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error_message("attn_fwd launch: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

}  // namespace

void launch_check_cu_seqlens(const int* cu, int B, int total, cudaStream_t stream) {
    DeviceInfo dev;
    if (current_device_info(&dev) != ATTN_OK) return;
    check_cu_seqlens_kernel<<<1, 256, 0, stream>>>(cu, B, total, dev.err_word);
}

attn_status launch_fwd(const FwdArgs& a, cudaStream_t stream) {
    DeviceInfo dev;
    attn_status st = current_device_info(&dev);
    if (st != ATTN_OK) return st;
    if (a.d == 128) return launch_typed<128, false>(a, dev, stream);
    if (a.d == 64) return launch_typed<64, false>(a, dev, stream);
    return ATTN_ERR_UNSUPPORTED;
}

attn_status launch_fwd_fp8(const FwdArgs& a, cudaStream_t stream) {
    DeviceInfo dev;
    attn_status st = current_device_info(&dev);
    if (st != ATTN_OK) return st;
    if (a.d == 128) return launch_typed<128, true>(a, dev, stream);
    if (a.d == 64) return launch_typed<64, true>(a, dev, stream);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
