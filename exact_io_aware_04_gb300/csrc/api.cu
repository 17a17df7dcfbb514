// api.cu -- the C ABI of libattn: argument checks, per-device state, tensor
// map encoding, and dispatch to the kernels in fwd.cu and decode.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "internal.h"

namespace attn {

// One error word per device (each device that loads the library gets its own
// copy of this variable).
__device__ int g_device_error = 0;

namespace {

thread_local char t_message[512] = "";
std::atomic<int> g_validation{0};

std::mutex g_dev_mu;
bool g_dev_ready[kMaxDevices] = {};
DeviceInfo g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

attn_status fail(attn_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_message, sizeof(t_message), fmt, ap);
    va_end(ap);
    return st;
}

}  // namespace

void set_error_message(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_message, sizeof(t_message), fmt, ap);
    va_end(ap);
}

bool validation_enabled() { return g_validation.load(std::memory_order_relaxed) != 0; }

attn_status current_device_info(DeviceInfo* info) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!g_dev_ready[dev]) {
        DeviceInfo d;
        d.device = dev;
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "multiProcessorCount: %s", cudaGetErrorString(e));
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return fail(ATTN_ERR_UNSUPPORTED, "device %d is sm_%d%d; libattn is built for sm_103a only", dev, major,
                        minor);
        void* addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_device_error);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        d.err_word = static_cast<int*>(addr);
        g_dev[dev] = d;
        g_dev_ready[dev] = true;
    }
    *info = g_dev[dev];
    return ATTN_OK;
}

attn_status encode_tma_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128) {
    return encode_tma(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes, box, swizzle128);
}

attn_status encode_tma(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128) {
    return encode_tma_swizzle(map, dtype, base, rank, dims, strides_bytes, box,
                              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

attn_status encode_tma_swizzle(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                               const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                               CUtensorMapSwizzle swizzle) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    if (!g_encode) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t gdim[5];
    cuuint64_t gstride[4];
    cuuint32_t bdim[5];
    cuuint32_t estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
        if (i + 1 < rank) gstride[i] = strides_bytes[i];
    }
    CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
                          gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d, rank %d)", (int)r, rank);
    return ATTN_OK;
}

// Every check of the paged-decode entry points except those on the
// workspace; fills the chunk plan on success.
attn_status decode_check(const char* fn, const void* q, const void* k_new, const void* v_new, const void* k_cache,
                         const void* v_cache, const int* block_table, int max_pages_per_seq, const int* seq_lens,
                         const void* out, const float* lse, int B, int Nq, int Hq, int Hkv, int d, int page_size,
                         int num_pages, float scale, int causal, int num_splits, DecodePlan* plan) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !lse)
        return fail(ATTN_ERR_INVALID_ARG, "%s: NULL pointer", fn);
    if ((k_new == nullptr) != (v_new == nullptr)) return fail(ATTN_ERR_INVALID_ARG, "%s: give both k_new and v_new or neither", fn);
    if (B < 0 || Nq <= 0 || Hq <= 0 || Hkv <= 0 || num_pages <= 0 || max_pages_per_seq <= 0 || num_splits < 0)
        return fail(ATTN_ERR_INVALID_ARG, "%s: bad size", fn);
    if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "%s: Hq %% Hkv != 0 (%d, %d)", fn, Hq, Hkv);
    if (!isfinite(scale) || !(scale > 0.f)) return fail(ATTN_ERR_INVALID_ARG, "%s: scale must be finite and > 0", fn);
    if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "%s: causal must be 0 or 1", fn);
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(lse) ||
        (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return fail(ATTN_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "%s: head_dim %d (built: 64, 128)", fn, d);
    if (page_size != 16) return fail(ATTN_ERR_UNSUPPORTED, "%s: page_size %d (built: 16)", fn, page_size);
    if (static_cast<long long>(max_pages_per_seq) * page_size > INT32_MAX)
        return fail(ATTN_ERR_UNSUPPORTED, "%s: sequences longer than 2^31 tokens", fn);
    if (static_cast<long long>(Hq / Hkv) * Nq > 128)
        return fail(ATTN_ERR_UNSUPPORTED, "%s: (Hq/Hkv) * Nq = %lld query rows per K/V head (built: up to 128)", fn,
                    static_cast<long long>(Hq / Hkv) * Nq);
    if (!make_decode_plan(B, Nq, Hq, Hkv, d, page_size, max_pages_per_seq, num_splits, plan))
        return fail(ATTN_ERR_UNSUPPORTED, "%s: no plan for Hq/Hkv = %d, Nq = %d", fn, Hq / Hkv, Nq);
    return ATTN_OK;
}

}  // namespace attn

using namespace attn;

extern "C" {

attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
                            int Hkv, int Nq, int Nk, int d, float scale, int causal, int window_left,
                            int window_right, const int* cu_seqlens_q, const int* cu_seqlens_k, void* stream) {
    if (!q || !out || !lse) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: NULL tensor pointer");
    if ((!k || !v) && Nk > 0) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: NULL k/v with keys present");
    if ((cu_seqlens_q == nullptr) != (cu_seqlens_k == nullptr))
        return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: give both cu_seqlens or neither");
    if (B < 0 || Nq < 0 || Nk < 0) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: negative size");
    if (Hq <= 0 || Hkv <= 0) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: head counts must be positive");
    if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: Hq %% Hkv != 0 (%d, %d)", Hq, Hkv);
    if (!isfinite(scale) || !(scale > 0.f)) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: scale must be finite and > 0");
    if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: causal must be 0 or 1");
    if (window_left < -1 || window_right < -1)
        return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: window sides must be >= 0, or -1 for unbounded (%d, %d)",
                    window_left, window_right);
    if (Nk == 0) {  // no keys: K/V are never read (NULL allowed)
        k = q;
        v = q;
    }
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
        return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: tensor pointers must be 16-byte aligned");
    if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd: head_dim %d (built: 64, 128)", d);
    const bool varlen = cu_seqlens_q != nullptr;
    if (!varlen && (static_cast<long long>(B) * Nq > INT32_MAX || static_cast<long long>(B) * Nk > INT32_MAX))
        return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd: more than 2^31 tokens");
    if (B == 0 || Nq == 0) return ATTN_OK;
    FwdArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.lse = lse;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.Nq = Nq;
    a.Nk = Nk;
    a.d = d;
    a.scale = scale;
    a.causal = causal;
    a.win_left = window_left;
    a.win_right = window_right;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.q_scale = a.k_scale = a.v_scale = nullptr;
    return launch_fwd(a, static_cast<cudaStream_t>(stream));
}

attn_status attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nk, int d, float scale, int causal, const int* cu_seqlens_q,
                     const int* cu_seqlens_k, void* stream) {
    return attn_fwd_window(q, k, v, out, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, -1, -1, cu_seqlens_q,
                           cu_seqlens_k, stream);
}

size_t attn_fp8_scale_count(int B, int T) {
    if (B < 0 || T < 0) return 0;
    return static_cast<size_t>(fp8_scale_count(B, T));
}

attn_status attn_quantize_fp8(const void* x, void* x8, float* x_scale, int B, int H, int N, int d,
                              const int* cu_seqlens, void* stream) {
    if (!x || !x8 || !x_scale) return fail(ATTN_ERR_INVALID_ARG, "attn_quantize_fp8: NULL pointer");
    if (B < 0 || H <= 0 || N < 0) return fail(ATTN_ERR_INVALID_ARG, "attn_quantize_fp8: bad size");
    if (!aligned16(x) || !aligned16(x8) || (reinterpret_cast<uintptr_t>(x_scale) & 3u) != 0)
        return fail(ATTN_ERR_INVALID_ARG, "attn_quantize_fp8: misaligned pointer");
    if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "attn_quantize_fp8: head_dim %d (built: 64, 128)", d);
    if (!cu_seqlens && static_cast<long long>(B) * N > INT32_MAX)
        return fail(ATTN_ERR_UNSUPPORTED, "attn_quantize_fp8: more than 2^31 tokens");
    QuantArgs a;
    a.x = x;
    a.x8 = x8;
    a.scale = x_scale;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.cu = cu_seqlens;
    return launch_quantize_fp8(&a, 1, static_cast<cudaStream_t>(stream));
}

attn_status attn_quantize_fp8_qkv(const void* q, const void* k, const void* v, void* q8, void* k8, void* v8,
                                  float* q_scale, float* k_scale, float* v_scale, int B, int Hq, int Hkv, int Nq,
                                  int Nk, int d, const int* cu_seqlens_q, const int* cu_seqlens_k, void* stream) {
    if (!q || !q8 || !q_scale) return fail(ATTN_ERR_INVALID_ARG, "attn_quantize_fp8_qkv: NULL pointer");
    if ((!k || !v || !k8 || !v8 || !k_scale || !v_scale) && Nk > 0)
        return fail(ATTN_ERR_INVALID_ARG, "attn_quantize_fp8_qkv: NULL k/v pointer with keys present");
    if ((cu_seqlens_q == nullptr) != (cu_seqlens_k == nullptr))
        return fail(ATTN_ERR_INVALID_ARG, "attn_quantize_fp8_qkv: give both cu_seqlens or neither");
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0)
        return fail(ATTN_ERR_INVALID_ARG, "attn_quantize_fp8_qkv: bad size");
    if (d != 64 && d != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "attn_quantize_fp8_qkv: head_dim %d (built: 64, 128)", d);
    const bool keys = Nk > 0;
    if (!aligned16(q) || !aligned16(q8) || (reinterpret_cast<uintptr_t>(q_scale) & 3u) != 0 ||
        (keys && (!aligned16(k) || !aligned16(v) || !aligned16(k8) || !aligned16(v8) ||
                  (reinterpret_cast<uintptr_t>(k_scale) & 3u) != 0 || (reinterpret_cast<uintptr_t>(v_scale) & 3u) != 0)))
        return fail(ATTN_ERR_INVALID_ARG, "attn_quantize_fp8_qkv: misaligned pointer");
    if (!cu_seqlens_q && (static_cast<long long>(B) * Nq > INT32_MAX || static_cast<long long>(B) * Nk > INT32_MAX))
        return fail(ATTN_ERR_UNSUPPORTED, "attn_quantize_fp8_qkv: more than 2^31 tokens");
    QuantArgs a[3];
    const void* src[3] = {q, k, v};
    void* dst[3] = {q8, k8, v8};
    float* sc[3] = {q_scale, k_scale, v_scale};
    const int n = keys ? 3 : 1;
    for (int i = 0; i < n; ++i) {
        a[i].x = src[i];
        a[i].x8 = dst[i];
        a[i].scale = sc[i];
        a[i].B = B;
        a[i].H = i == 0 ? Hq : Hkv;
        a[i].N = i == 0 ? Nq : Nk;
        a[i].d = d;
        a[i].cu = i == 0 ? cu_seqlens_q : cu_seqlens_k;
    }
    return launch_quantize_fp8(a, n, static_cast<cudaStream_t>(stream));
}

attn_status attn_fwd_fp8_window(const void* q8, const void* k8, const void* v8, const float* q_scale,
                                const float* k_scale, const float* v_scale, void* out, float* lse, int B, int Hq,
                                int Hkv, int Nq, int Nk, int d, float scale, int causal, int window_left,
                                int window_right, const int* cu_seqlens_q, const int* cu_seqlens_k, void* stream) {
    if (!q8 || !out || !lse || !q_scale) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_fp8: NULL tensor pointer");
    if ((!k8 || !v8 || !k_scale || !v_scale) && Nk > 0)
        return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_fp8: NULL k/v or scales with keys present");
    if ((cu_seqlens_q == nullptr) != (cu_seqlens_k == nullptr))
        return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_fp8: give both cu_seqlens or neither");
    if (B < 0 || Nq < 0 || Nk < 0) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_fp8: negative size");
    if (Hq <= 0 || Hkv <= 0) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_fp8: head counts must be positive");
    if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_fp8: Hq %% Hkv != 0 (%d, %d)", Hq, Hkv);
    if (!isfinite(scale) || !(scale > 0.f))
        return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_fp8: scale must be finite and > 0");
    if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_fp8: causal must be 0 or 1");
    if (window_left < -1 || window_right < -1)
        return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_fp8: window sides must be >= 0, or -1 for unbounded (%d, %d)",
                    window_left, window_right);
    if (Nk == 0) {  // no keys: K/V and their scales are never read
        k8 = v8 = q8;
        k_scale = v_scale = q_scale;
    }
    if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(out) || !aligned16(lse) ||
        (reinterpret_cast<uintptr_t>(q_scale) & 3u) != 0 || (reinterpret_cast<uintptr_t>(k_scale) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(v_scale) & 3u) != 0)
        return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_fp8: misaligned pointer");
    if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd_fp8: head_dim %d (built: 64, 128)", d);
    const bool varlen = cu_seqlens_q != nullptr;
    if (!varlen && (static_cast<long long>(B) * Nq > INT32_MAX || static_cast<long long>(B) * Nk > INT32_MAX))
        return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd_fp8: more than 2^31 tokens");
    if (B == 0 || Nq == 0) return ATTN_OK;
    FwdArgs a;
    a.q = q8;
    a.k = k8;
    a.v = v8;
    a.out = out;
    a.lse = lse;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.Nq = Nq;
    a.Nk = Nk;
    a.d = d;
    a.scale = scale;
    a.causal = causal;
    a.win_left = window_left;
    a.win_right = window_right;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.q_scale = q_scale;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    return launch_fwd_fp8(a, static_cast<cudaStream_t>(stream));
}

attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                         const float* v_scale, void* out, float* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                         float scale, int causal, const int* cu_seqlens_q, const int* cu_seqlens_k, void* stream) {
    return attn_fwd_fp8_window(q8, k8, v8, q_scale, k_scale, v_scale, out, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal,
                               -1, -1, cu_seqlens_q, cu_seqlens_k, stream);
}

size_t attn_bwd_workspace_size(int B, int Hq, int Nq, int packed) {
    if (B < 0 || Hq <= 0 || Nq < 0) return 0;
    return bwd_workspace_bytes(B, Hq, Nq, packed != 0);
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                     int causal, int window_left, int window_right, const int* cu_seqlens_q,
                     const int* cu_seqlens_k, void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !out || !dout || !lse || !dq || !workspace)
        return fail(ATTN_ERR_INVALID_ARG, "attn_bwd: NULL tensor pointer");
    if ((!k || !v || !dk || !dv) && Nk > 0) return fail(ATTN_ERR_INVALID_ARG, "attn_bwd: NULL k/v/dk/dv with keys present");
    if ((cu_seqlens_q == nullptr) != (cu_seqlens_k == nullptr))
        return fail(ATTN_ERR_INVALID_ARG, "attn_bwd: give both cu_seqlens or neither");
    if (B < 0 || Nq < 0 || Nk < 0) return fail(ATTN_ERR_INVALID_ARG, "attn_bwd: negative size");
    if (Hq <= 0 || Hkv <= 0) return fail(ATTN_ERR_INVALID_ARG, "attn_bwd: head counts must be positive");
    if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "attn_bwd: Hq %% Hkv != 0 (%d, %d)", Hq, Hkv);
    if (!isfinite(scale) || !(scale > 0.f)) return fail(ATTN_ERR_INVALID_ARG, "attn_bwd: scale must be finite and > 0");
    if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "attn_bwd: causal must be 0 or 1");
    if (window_left < -1 || window_right < -1)
        return fail(ATTN_ERR_INVALID_ARG, "attn_bwd: window sides must be >= 0, or -1 for unbounded");
    if (Nk == 0) {  // no keys: K/V are never read and dK/dV are empty
        k = v = q;
        dk = dv = dq;
    }
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) || !aligned16(lse) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ATTN_ERR_INVALID_ARG, "attn_bwd: misaligned pointer");
    if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "attn_bwd: head_dim %d (built: 64, 128)", d);
    const bool varlen = cu_seqlens_q != nullptr;
    if (!varlen && (static_cast<long long>(B) * Nq > INT32_MAX || static_cast<long long>(B) * Nk > INT32_MAX))
        return fail(ATTN_ERR_UNSUPPORTED, "attn_bwd: more than 2^31 tokens");
    if (workspace_bytes < bwd_workspace_bytes(B, Hq, Nq, varlen))
        return fail(ATTN_ERR_INVALID_ARG, "attn_bwd: workspace %zu bytes < %zu needed", workspace_bytes,
                    bwd_workspace_bytes(B, Hq, Nq, varlen));
    if (B == 0 || (Nq == 0 && Nk == 0)) return ATTN_OK;
    BwdArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.workspace = workspace;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.Nq = Nq;
    a.Nk = Nk;
    a.d = d;
    a.scale = scale;
    a.causal = causal;
    a.win_left = window_left;
    a.win_right = window_right;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    return launch_bwd(a, static_cast<cudaStream_t>(stream));
}

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int d, int page_size, int max_pages_per_seq,
                                  int num_splits) {
    DecodePlan plan;
    if (!make_decode_plan(B, 1, Hq, Hkv, d, page_size, max_pages_per_seq, num_splits, &plan)) return 0;
    return plan.total_bytes;
}

size_t attn_decode_kvcache_workspace_size(int B, int Nq, int Hq, int Hkv, int d, int page_size,
                                          int max_pages_per_seq, int num_splits) {
    DecodePlan plan;
    if (!make_decode_plan(B, Nq, Hq, Hkv, d, page_size, max_pages_per_seq, num_splits, &plan)) return 0;
    return plan.total_bytes;
}

namespace {

// The checks and the launch shared by the paged-decode entry points.
attn_status decode_call(const char* fn, const void* q, const void* k_new, const void* v_new, void* k_cache,
                        void* v_cache, const int* block_table, int max_pages_per_seq, const int* seq_lens, void* out,
                        float* lse, int B, int Nq, int Hq, int Hkv, int d, int page_size, int num_pages, float scale,
                        int causal, int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
    DecodePlan plan;
    attn_status st = decode_check(fn, q, k_new, v_new, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens,
                                  out, lse, B, Nq, Hq, Hkv, d, page_size, num_pages, scale, causal, num_splits, &plan);
    if (st != ATTN_OK) return st;
    if (!workspace) return fail(ATTN_ERR_INVALID_ARG, "%s: NULL pointer", fn);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ATTN_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    if (workspace_bytes < plan.total_bytes)
        return fail(ATTN_ERR_INVALID_ARG, "%s: workspace %zu bytes < %zu needed", fn, workspace_bytes,
                    plan.total_bytes);
    if (B == 0) return ATTN_OK;
    DecodeArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache_w = k_cache;
    a.v_cache_w = v_cache;
    a.block_table = block_table;
    a.max_pages = max_pages_per_seq;
    a.seq_lens = seq_lens;
    a.out = out;
    a.lse = lse;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.page_size = page_size;
    a.num_pages = num_pages;
    a.nq = Nq;
    a.causal = causal;
    a.scale = scale;
    a.num_splits = num_splits;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return launch_decode(a, plan, static_cast<cudaStream_t>(stream));
}

}  // namespace

attn_status attn_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                              int max_pages_per_seq, const int* seq_lens, void* out, float* lse, int B, int Hq,
                              int Hkv, int d, int page_size, int num_pages, float scale, int num_splits,
                              void* workspace, size_t workspace_bytes, void* stream) {
    // the caches are only read on this path (no append)
    return decode_call("attn_decode_paged", q, nullptr, nullptr, const_cast<void*>(k_cache),
                       const_cast<void*>(v_cache), block_table, max_pages_per_seq, seq_lens, out, lse, B, 1, Hq, Hkv,
                       d, page_size, num_pages, scale, 0, num_splits, workspace, workspace_bytes, stream);
}

attn_status attn_decode_kvcache(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                const int* block_table, int max_pages_per_seq, const int* seq_lens, void* out,
                                float* lse, int B, int Nq, int Hq, int Hkv, int d, int page_size, int num_pages,
                                float scale, int causal, int num_splits, void* workspace, size_t workspace_bytes,
                                void* stream) {
    return decode_call("attn_decode_kvcache", q, k_new, v_new, k_cache, v_cache, block_table, max_pages_per_seq,
                       seq_lens, out, lse, B, Nq, Hq, Hkv, d, page_size, num_pages, scale, causal, num_splits,
                       workspace, workspace_bytes, stream);
}

attn_status attn_get_device_status(void* stream) {
    DeviceInfo dev;
    attn_status st = current_device_info(&dev);
    if (st != ATTN_OK) return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    int word = 0;
    e = cudaMemcpy(&word, dev.err_word, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(e));
    if (word != 0) {
        const int zero = 0;
        e = cudaMemcpy(dev.err_word, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "clearing the device error word: %s", cudaGetErrorString(e));
    }
    return static_cast<attn_status>(word);
}

int attn_set_validation(int enabled) { return g_validation.exchange(enabled ? 1 : 0); }

int attn_test_drop_page_load(int enabled) { return attn::set_drop_page_load(enabled); }

const char* attn_status_string(attn_status status) {
    switch (status) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
        case ATTN_ERR_BAD_INDEX: return "ATTN_ERR_BAD_INDEX";
    }
    return "ATTN_UNKNOWN_STATUS";
}

const char* attn_last_error_message(void) { return t_message; }

}  // extern "C"
