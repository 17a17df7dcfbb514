// quant.cu -- per-tile 8-bit (E4M3) quantization of a bf16 tensor.
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
// One CTA per (tile, head), the head varying fastest so that the CTAs in
// flight cover whole token rows (H * d contiguous values) rather than one
// head's 2d-byte pieces of many rows: the tile's values are read once into registers
// (lanes sharing rows, so each warp request is whole consecutive rows),
// reduced to the tile's amax through shared memory, and written back as
// codes, 8 bytes per lane per row chunk.  HBM-bound: 2 bytes read and 1
// written per value.
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kRows = 128;

struct QuantParams {
    const __nv_bfloat16* x;
    uint8_t* x8;
    float* scale;
    long long n_scale;  // entries per head
    int B, H, N;
    const int* cu;
};

// First token of sequence b and its length.  Packed offsets are clamped into
// [0, N] (each end no lower than the start), so malformed cu_seqlens cannot
// move any access outside x and x8.
__device__ __forceinline__ void seq_span(const QuantParams& p, int b, long long& first, long long& len) {
    if (p.cu) {
        const long long a = __ldg(p.cu + b), e = __ldg(p.cu + b + 1);
        first = a < 0 ? 0 : (a > p.N ? p.N : a);
        const long long end = e < first ? first : (e > p.N ? p.N : e);
        len = end - first;
    } else {
        first = static_cast<long long>(b) * p.N;
        len = p.N;
    }
}

__device__ __forceinline__ long long tile_base(const QuantParams& p, int b) {
    long long first, len;
    seq_span(p, b, first, len);
    return first / kRows + b;
}

// Two fp32 values to two E4M3 codes (round to nearest even, saturating);
// `lo` in bits 0..7.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int HD>
__global__ void __launch_bounds__(kRows) quantize_fp8_kernel(const __grid_constant__ QuantParams p) {
    // Lanes share rows: a row is HD / 8 sixteen-byte chunks (8 values each),
    // so one warp request covers 32 * 16 / (2 HD) consecutive-in-memory rows'
    // worth of whole chunks; the CTA's 4 warps take interleaved row groups.
    constexpr int kChunksPerRow = HD / 8;
    constexpr int kRowsPerWarp = 32 / kChunksPerRow;     // rows per warp request
    constexpr int kRowsPerIter = 4 * kRowsPerWarp;       // rows per CTA request
    constexpr int kIters = kRows / kRowsPerIter;
    const long long idx = blockIdx.x / p.H;
    const int h = static_cast<int>(blockIdx.x - idx * p.H);
    // the sequence owning scale entry idx: the largest b with tile_base(b) <= idx
    // (tile_base strictly increases with b)
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tile_base(p, mid) <= idx) lo = mid; else hi = mid;
    }
    const int b = lo;
    long long first, len;
    seq_span(p, b, first, len);
    const long long t = idx - (first / kRows + b);
    if (t < 0 || t * kRows >= len) return;  // an entry between sequences
    const int rows = static_cast<int>(len - t * kRows < kRows ? len - t * kRows : kRows);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chunk = lane % kChunksPerRow;
    const int row0 = warp * kRowsPerWarp + lane / kChunksPerRow;  // this lane's row in iteration 0
    const long long tile_row0 = first + t * kRows;

    uint32_t w[kIters][4];
    float amax = 0.f;
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int r = row0 + it * kRowsPerIter;
        if (r < rows) {
            const uint4 v = *reinterpret_cast<const uint4*>(
                p.x + (static_cast<size_t>(tile_row0 + r) * p.H + h) * HD + chunk * 8);
            w[it][0] = v.x;
            w[it][1] = v.y;
            w[it][2] = v.z;
            w[it][3] = v.w;
        } else {
            w[it][0] = w[it][1] = w[it][2] = w[it][3] = 0u;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[it][k])), fabsf(bf16_hi(w[it][k]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float warp_max[kRows / 32];
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(warp_max[0], warp_max[1]), fmaxf(warp_max[2], warp_max[3]));

    const bool zero = !(amax >= 0x1p-100f);
    const float inv = zero ? 0.f : __fdiv_rn(448.f, amax);
    if (threadIdx.x == 0) p.scale[static_cast<size_t>(h) * p.n_scale + idx] = zero ? 1.f : __fdiv_rn(amax, 448.f);
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int r = row0 + it * kRowsPerIter;
        if (r >= rows) continue;
        uint32_t c[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint32_t a = w[it][2 * k], bb = w[it][2 * k + 1];
            const uint32_t c01 = e4m3x2(__fmul_rn(bf16_lo(a), inv), __fmul_rn(bf16_hi(a), inv));
            const uint32_t c23 = e4m3x2(__fmul_rn(bf16_lo(bb), inv), __fmul_rn(bf16_hi(bb), inv));
            c[k] = zero ? 0u : (c01 | (c23 << 16));
        }
        *reinterpret_cast<uint2*>(p.x8 + (static_cast<size_t>(tile_row0 + r) * p.H + h) * HD + chunk * 8) =
            make_uint2(c[0], c[1]);
    }
}

}  // namespace

attn_status launch_quantize_fp8(const QuantArgs& a, cudaStream_t stream) {
    const long long T = a.cu ? static_cast<long long>(a.N) : static_cast<long long>(a.B) * a.N;
    const long long n_scale = fp8_scale_count(a.B, T);
    if (a.B == 0 || T == 0) return ATTN_OK;
    if (n_scale * a.H > 0x7fffffffLL) {
        set_error_message("attn_quantize_fp8: more than 2^31 (tile, head) pairs");
        return ATTN_ERR_UNSUPPORTED;
    }
    QuantParams p;
    p.x = static_cast<const __nv_bfloat16*>(a.x);
    p.x8 = static_cast<uint8_t*>(a.x8);
    p.scale = a.scale;
    p.n_scale = n_scale;
    p.B = a.B;
    p.H = a.H;
    p.N = a.N;
    p.cu = a.cu;
    if (a.cu != nullptr && validation_enabled()) launch_check_cu_seqlens(a.cu, a.B, a.N, stream);
    const dim3 grid(static_cast<unsigned>(n_scale * a.H));
    if (a.d == 128)
        quantize_fp8_kernel<128><<<grid, kRows, 0, stream>>>(p);
    else
        quantize_fp8_kernel<64><<<grid, kRows, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error_message("attn_quantize_fp8 launch: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

}  // namespace attn
