// quant.cu -- per-tile 8-bit (E4M3) quantization of bf16 tensors.
//
// "FP8 Path and Quantization" ("Flash Attention: A Complete Architectural
// Autopsy", part 4) quantizes each tile with a scale factor taken from the
// tile's absolute maximum; "FlashAttention-3: asynchrony and low precision on
// Hopper" ("FlashAttention-3 and PagedAttention") calls it block quantization.
// Here a tile is 128 consecutive tokens of one sequence (counted from the
// sequence's first token, the last one possibly shorter) for one head and all
// d channels -- exactly the 128-row tiles the 8-bit forward streams -- so the
// forward folds one scale per tile into its score and value arithmetic.
//
// Per tile, in fp32: amax = max |x|; scale = amax / 448 and inv = 448 / amax
// (IEEE-rounded divisions); code = E4M3(x * inv), the product rounded to fp32
// and then to the nearest E4M3 value (ties to even, saturating at 448).  A
// tile whose amax is below 2^-100 gets scale 1 and zero codes.  The scales of
// head h sit in row h of a [H, T/128 + B] array: tile t of sequence b at
// entry first_token_b / 128 + b + t (the entries never collide, and the ones
// between sequences are never written).
//
// HBM-bound: 2 bytes read and 1 written per value.  One launch covers up to
// three tensors (q, k and v of an attention call).  A unit of work is one
// (scale entry, head) pair, the head varying fastest, so that consecutive
// units cover whole token rows (H * d contiguous values).  The grid is three
// CTAs per SM; each walks the units u = blockIdx.x + k * gridDim.x.  In a
// CTA, one loader thread decodes each unit once (skipping the entries between
// sequences) and brings its 128 x d tile in by one TMA tile copy into a
// shared-memory stage, with the decoded unit beside it; eight consumer
// warps read the tile from shared memory, hand the stage back (one arrival
// per warp), reduce the tile's amax (one barrier over the consumer warps),
// and write the codes, 8 bytes per thread per row chunk.
#include <cuda_bf16.h>
#include <stdint.h>
#include <string.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kRows = 128;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;    // + the loader warp
constexpr int kCtasPerSm = 3;

// Stages per CTA: one 32 KB tile (two at d = 64) and three CTAs per SM.
// Measured on the GQA causal q, k, v (GB/s of 6784 copy bandwidth): 3 x 1
// stage 6590-6650; 3 x 2 stages 6290; 2 x 3 stages 6350; 4 x 1 stage
// 6370-6530; 2 x 1 stage 6020; an L2 prefetch of the tiles beyond the ring
// lost 8-15%.  Fewer tiles in flight per SM, spread over more CTAs, is what
// HBM rewards here.
template <int HD>
struct QCfg {
    static constexpr int kTileBytes = kRows * HD * 2;
    static constexpr int kStages = HD == 128 ? 1 : 2;
    static constexpr int kChunksPerRow = HD / 8;                        // 16-byte chunks (8 values)
    static constexpr int kIters = kRows * kChunksPerRow / kConsumers;   // chunks per consumer thread
    static constexpr int kSmemBytes = kStages * kTileBytes + 128;     // + alignment slack
};

// Sizes in 32 bits: the host rejects more than 2^31 tokens or units.
struct QuantTensor {
    uint8_t* x8;
    float* scale;
    int n_scale;        // scale entries per head
    uint32_t units;     // n_scale * H
    int B, H, N;
    const int* cu;
};

struct QuantParams {
    CUtensorMap tm[kMaxQuantTensors];  // x as [T rows, H*d] bf16, box d x 128 rows, no swizzle
    QuantTensor t[kMaxQuantTensors];
    uint32_t units_total;
    int n_tensors;
    int* err;
};

// First token of sequence b and its length.  Packed offsets are clamped into
// [0, N] (each end no lower than the start), so malformed cu_seqlens cannot
// move any access outside x and x8.
__device__ __forceinline__ void seq_span(const QuantTensor& q, int b, int& first, int& len) {
    if (q.cu) {
        const int a = __ldg(q.cu + b), e = __ldg(q.cu + b + 1);
        first = a < 0 ? 0 : (a > q.N ? q.N : a);
        const int end = e < first ? first : (e > q.N ? q.N : e);
        len = end - first;
    } else {
        first = b * q.N;
        len = q.N;
    }
}

__device__ __forceinline__ int tile_base(const QuantTensor& q, int b) {
    int first, len;
    seq_span(q, b, first, len);
    return first / kRows + b;
}

struct Unit {
    int i;               // tensor
    int h;               // head
    int idx;             // scale entry
    int row0;            // first token row of the tile
    int rows;            // valid rows (0: an entry between sequences)
};

__device__ __forceinline__ Unit unit_at(const QuantParams& p, uint32_t u) {
    Unit un;
    un.i = 0;
    while (un.i + 1 < p.n_tensors && u >= p.t[un.i].units) {
        u -= p.t[un.i].units;
        ++un.i;
    }
    const QuantTensor& q = p.t[un.i];
    un.idx = static_cast<int>(u / static_cast<uint32_t>(q.H));
    un.h = static_cast<int>(u - static_cast<uint32_t>(un.idx) * static_cast<uint32_t>(q.H));
    // the sequence owning scale entry idx: the largest b with tile_base(b) <= idx
    // (tile_base strictly increases with b)
    int lo = 0, hi = q.B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tile_base(q, mid) <= un.idx) lo = mid; else hi = mid;
    }
    int first, len;
    seq_span(q, lo, first, len);
    const int t = un.idx - (first / kRows + lo);
    un.rows = (t < 0 || t >= (len + kRows - 1) / kRows) ? 0 : min(len - t * kRows, kRows);
    un.row0 = first + t * kRows;
    return un;
}

// Barrier 1 over the consumer warps only; returns whether `pred` held in
// every consumer thread.
__device__ __forceinline__ bool consumers_sync_and(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "n"(kConsumers)
        : "memory");
    return r != 0;
}

// Per-half unsigned maximum of two pairs of 16-bit values.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Two fp32 values to two E4M3 codes (round to nearest even, saturating);
// `lo` in bits 0..7.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int HD>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) quantize_fp8_kernel(const __grid_constant__ QuantParams p) {
    using C = QCfg<HD>;
    constexpr int S = C::kStages;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[S], empty_bar[S];
    __shared__ Unit info[S];                 // the unit in each stage (rows < 0: no more units)
    __shared__ uint32_t warp_max[2][kConsumerWarps];
    const uint32_t ring = (smem_addr(smem_raw) + 127u) & ~127u;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 1);
            mbar_init(smem_addr(&empty_bar[s]), kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // Loader: decodes the CTA's units u = blockIdx.x + k * gridDim.x once,
        // skips the entries between sequences, and copies each tile into the
        // next free stage together with its decoded unit.
        if (lane != 0) return;
        for (int i = 0; i < p.n_tensors; ++i) tma_prefetch_map(&p.tm[i]);
        int m = 0;
        bool ok = true;
        for (uint32_t u = blockIdx.x; ok; u += gridDim.x) {
            Unit un;
            if (u < p.units_total) {
                un = unit_at(p, u);
                if (un.rows == 0) continue;
            } else {
                un.rows = -1;
            }
            const int s = m % S;
            if (m >= S) ok = mbar_wait(smem_addr(&empty_bar[s]), ((m / S) - 1) & 1, p.err);
            if (!ok) break;
            info[s] = un;
            if (un.rows < 0) {
                mbar_arrive(smem_addr(&full_bar[s]));   // the end marker carries no copy
                break;
            }
            const uint32_t bar = smem_addr(&full_bar[s]);
            mbar_arrive_expect_tx(bar, C::kTileBytes);
            tma_load_2d(ring + s * C::kTileBytes, &p.tm[un.i], bar, un.h * HD, un.row0);
            ++m;
        }
        // after a timeout, let the copies still in flight land (bounded)
        // before the CTA's shared memory is released
        if (!ok)
            for (int k = m - S > 0 ? m - S : 0; k < m; ++k)
                mbar_wait(smem_addr(&full_bar[k % S]), (k / S) & 1, nullptr);
        return;
    }

    for (int n = 0;; ++n) {
        const int s = n % S;
        const bool got = mbar_wait(smem_addr(&full_bar[s]), (n / S) & 1, p.err);
        const Unit un = info[s];         // meaningful once the wait succeeded
        const int rows = got ? un.rows : 0;   // the end marker (rows < 0) reads nothing
        // chunk k of this thread: row (k * kConsumers + tid) / kChunksPerRow.
        // amax on the bit patterns: for finite non-negative bf16 values the
        // unsigned order of the 16-bit patterns is the numeric order, so the
        // per-half integer maximum of |x| (sign bit cleared) is exact.
        uint32_t w[C::kIters][4];
        uint32_t m2[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < C::kIters; ++k) {
            const int L = k * kConsumers + tid;
            const int r = L / C::kChunksPerRow, c = L % C::kChunksPerRow;
            if (r < rows) {
                const uint32_t a = ring + s * C::kTileBytes + r * (HD * 2) + c * 16;
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(w[k][0]), "=r"(w[k][1]), "=r"(w[k][2]), "=r"(w[k][3])
                             : "r"(a));
            } else {
                w[k][0] = w[k][1] = w[k][2] = w[k][3] = 0u;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) m2[j] = max_u16x2(m2[j], w[k][j] & 0x7fff7fffu);
        }
        // the warp's reads of the stage are done: hand it back to the loader
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
        const uint32_t mm = max_u16x2(max_u16x2(m2[0], m2[1]), max_u16x2(m2[2], m2[3]));
        const uint32_t bits = __reduce_max_sync(0xffffffffu, max(mm & 0xffffu, mm >> 16));
        if (lane == 0) warp_max[n & 1][warp] = bits;
        // the consumer warps only (named barrier 1), once per stage, whether or
        // not a thread's wait succeeded; every exit below is taken by all of
        // them (after a failed wait in any thread, or at the end marker, which
        // all of them then read)
        if (!consumers_sync_and(got)) break;
        if (un.rows < 0) break;
        uint32_t amax_bits = warp_max[n & 1][0];
#pragma unroll
        for (int k = 1; k < kConsumerWarps; ++k) amax_bits = max(amax_bits, warp_max[n & 1][k]);
        const float amax = __uint_as_float(amax_bits << 16);

        const QuantTensor& q = p.t[un.i];
        const bool zero = !(amax >= 0x1p-100f);
        const float inv = zero ? 0.f : __fdiv_rn(448.f, amax);
        if (tid == 0)
            q.scale[static_cast<size_t>(un.h) * static_cast<size_t>(q.n_scale) + un.idx] = zero ? 1.f : __fdiv_rn(amax, 448.f);
#pragma unroll
        for (int k = 0; k < C::kIters; ++k) {
            const int L = k * kConsumers + tid;
            const int r = L / C::kChunksPerRow, c = L % C::kChunksPerRow;
            if (r >= un.rows) continue;
            uint32_t code[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t a = w[k][2 * j], b = w[k][2 * j + 1];
                const uint32_t c01 = e4m3x2(__fmul_rn(bf16_lo(a), inv), __fmul_rn(bf16_hi(a), inv));
                const uint32_t c23 = e4m3x2(__fmul_rn(bf16_lo(b), inv), __fmul_rn(bf16_hi(b), inv));
                code[j] = zero ? 0u : (c01 | (c23 << 16));
            }
            *reinterpret_cast<uint2*>(q.x8 + (static_cast<size_t>(un.row0 + r) * static_cast<size_t>(q.H) + un.h) * HD +
                                      c * 8) = make_uint2(code[0], code[1]);
        }
    }
}

template <int HD>
attn_status launch_impl(const QuantArgs* a, int n, cudaStream_t stream) {
    using C = QCfg<HD>;
    bool any = false;
    for (int i = 0; i < n; ++i) any |= a[i].B > 0 && (a[i].cu ? a[i].N : static_cast<long long>(a[i].B) * a[i].N) > 0;
    if (!any) return ATTN_OK;  // nothing to do: no device call at all
    DeviceInfo dev;
    attn_status st = current_device_info(&dev);
    if (st != ATTN_OK) return st;
    static std::atomic<bool> attr_set[kMaxDevices];
    if (!attr_set[dev.device].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(quantize_fp8_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   C::kSmemBytes);
        if (e != cudaSuccess) {
            set_error_message("attn_quantize_fp8: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        attr_set[dev.device].store(true, std::memory_order_release);
    }
    QuantParams p;
    memset(&p, 0, sizeof(p));
    p.n_tensors = 0;
    p.units_total = 0;
    p.err = dev.err_word;
    for (int i = 0; i < n; ++i) {
        const QuantArgs& x = a[i];
        const long long T = x.cu ? static_cast<long long>(x.N) : static_cast<long long>(x.B) * x.N;
        if (x.B == 0 || T == 0) continue;
        QuantTensor& q = p.t[p.n_tensors];
        q.x8 = static_cast<uint8_t*>(x.x8);
        q.scale = x.scale;
        q.n_scale = static_cast<int>(fp8_scale_count(x.B, T));
        q.units = static_cast<uint32_t>(q.n_scale) * static_cast<uint32_t>(x.H);
        q.B = x.B;
        q.H = x.H;
        q.N = x.N;
        q.cu = x.cu;
        const uint64_t dims[2] = {static_cast<uint64_t>(x.H) * HD, static_cast<uint64_t>(T)};
        const uint64_t strides[1] = {static_cast<uint64_t>(x.H) * HD * 2};
        const uint32_t box[2] = {static_cast<uint32_t>(HD), static_cast<uint32_t>(kRows)};
        st = encode_tma_bf16(&p.tm[p.n_tensors], x.x, 2, dims, strides, box, false);
        if (st != ATTN_OK) return st;
        if (x.cu != nullptr && validation_enabled()) launch_check_cu_seqlens(x.cu, x.B, x.N, stream);
        p.units_total += q.units;
        ++p.n_tensors;
    }
    if (p.n_tensors == 0) return ATTN_OK;
    const uint32_t ctas = static_cast<uint32_t>(dev.sm_count) * kCtasPerSm;
    const dim3 grid(p.units_total < ctas ? p.units_total : ctas);
    quantize_fp8_kernel<HD><<<grid, kThreads, C::kSmemBytes, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error_message("attn_quantize_fp8 launch: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

}  // namespace

attn_status launch_quantize_fp8(const QuantArgs* a, int n, cudaStream_t stream) {
    if (n < 1 || n > kMaxQuantTensors) {
        set_error_message("attn_quantize_fp8: %d tensors in one launch (1..%d)", n, kMaxQuantTensors);
        return ATTN_ERR_INVALID_ARG;
    }
    long long units = 0;
    for (int i = 0; i < n; ++i) {
        if (a[i].d != a[0].d) {
            set_error_message("attn_quantize_fp8: tensors of one launch must share head_dim");
            return ATTN_ERR_INVALID_ARG;
        }
        const long long T = a[i].cu ? static_cast<long long>(a[i].N) : static_cast<long long>(a[i].B) * a[i].N;
        if (T > 0x7fffffffLL) {
            set_error_message("attn_quantize_fp8: more than 2^31 tokens");
            return ATTN_ERR_UNSUPPORTED;
        }
        if (a[i].B > 0 && T > 0) units += fp8_scale_count(a[i].B, T) * a[i].H;
    }
    if (units > 0x7fffffffLL) {
        set_error_message("attn_quantize_fp8: more than 2^31 (tile, head) pairs in one launch");
        return ATTN_ERR_UNSUPPORTED;
    }
    return a[0].d == 128 ? launch_impl<128>(a, n, stream) : launch_impl<64>(a, n, stream);
}

}  // namespace attn
