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
// One CTA per (tile, head), one thread per token row: the row's d values are
// read once into registers (whole 32-byte sectors), reduced to the tile's
// amax through shared memory, and written back as d bytes.  HBM-bound: 2 d
// bytes read and d bytes written per element row.
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

// First token of sequence b and its length.
__device__ __forceinline__ void seq_span(const QuantParams& p, int b, long long& first, long long& len) {
    if (p.cu) {
        first = __ldg(p.cu + b);
        len = static_cast<long long>(__ldg(p.cu + b + 1)) - first;
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
    const long long idx = blockIdx.x;
    const int h = blockIdx.y;
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
    const int r = threadIdx.x;
    const bool active = r < rows;
    const long long row = first + t * kRows + r;
    const size_t at = (static_cast<size_t>(row) * p.H + h) * HD;

    constexpr int kWords = HD / 2;  // bf16 pairs per row
    uint32_t w[kWords];
    float amax = 0.f;
    if (active) {
        const uint4* src = reinterpret_cast<const uint4*>(p.x + at);
#pragma unroll
        for (int i = 0; i < HD / 8; ++i) {
            const uint4 v = src[i];
            w[4 * i + 0] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
#pragma unroll
        for (int i = 0; i < kWords; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float warp_max[kRows / 32];
    if ((r & 31) == 0) warp_max[r >> 5] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(warp_max[0], warp_max[1]), fmaxf(warp_max[2], warp_max[3]));

    const bool zero = !(amax >= 0x1p-100f);
    const float inv = zero ? 0.f : __fdiv_rn(448.f, amax);
    if (r == 0) p.scale[static_cast<size_t>(h) * p.n_scale + idx] = zero ? 1.f : __fdiv_rn(amax, 448.f);
    if (!active) return;
    uint4* dst = reinterpret_cast<uint4*>(p.x8 + at);
#pragma unroll
    for (int i = 0; i < HD / 16; ++i) {  // 16 codes per 16-byte store
        uint32_t c[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t a = w[8 * i + 2 * k], bb = w[8 * i + 2 * k + 1];
            const uint32_t c01 = e4m3x2(__fmul_rn(bf16_lo(a), inv), __fmul_rn(bf16_hi(a), inv));
            const uint32_t c23 = e4m3x2(__fmul_rn(bf16_lo(bb), inv), __fmul_rn(bf16_hi(bb), inv));
            c[k] = zero ? 0u : (c01 | (c23 << 16));
        }
        dst[i] = make_uint4(c[0], c[1], c[2], c[3]);
    }
}

}  // namespace

attn_status launch_quantize_fp8(const QuantArgs& a, cudaStream_t stream) {
    const long long T = a.cu ? static_cast<long long>(a.N) : static_cast<long long>(a.B) * a.N;
    const long long n_scale = fp8_scale_count(a.B, T);
    if (a.B == 0 || T == 0) return ATTN_OK;
    if (n_scale > 0x7fffffffLL) {
        set_error_message("attn_quantize_fp8: more than 2^31 tiles");
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
    const dim3 grid(static_cast<unsigned>(n_scale), static_cast<unsigned>(a.H));
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
