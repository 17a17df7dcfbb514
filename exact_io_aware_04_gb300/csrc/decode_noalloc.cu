// decode_noalloc.cu -- attn_decode_paged_noalloc: the paged split-KV decode of
// decode.cu with its scratch in a fixed array compiled into the library, for
// callers that cannot hand the library a device allocation at call time.
//
// Who needs it: code that runs where device memory is not its own to allocate
// -- a plug-in hosted by a runtime that owns every device allocation and
// exposes no allocator to its plug-ins, or a latency-critical serving loop
// that reserves all its memory up front and must never call cudaMalloc or
// cudaFree afterwards (both can synchronise the device and stall every other
// stream on it).  Such callers still own q, the caches, the block table and
// the outputs; only the per-chunk partial results need a home, and here that
// home is kScratchBytes of device memory that every GPU which loads the
// library holds until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"

namespace attn {
namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB

// Per-chunk partial outputs and lse of the split kernel.  The name is only a
// host-side stand-in in host code; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device does it).
attn_status scratch_on_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error_message("cudaGetDevice: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_error_message("device index %d out of range", dev);
        return ATTN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || p == nullptr) {
            set_error_message("cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                 const int* block_table, int max_pages_per_seq, const int* seq_lens,
                                                 void* out, float* lse, int B, int Hq, int Hkv, int d,
                                                 int page_size, int num_pages, float scale, int num_splits,
                                                 void* stream) {
    // Same plan and checks as attn_decode_paged; the scratch must fit the array.
    DecodePlan plan;
    if (B >= 0 && Hq > 0 && Hkv > 0 && max_pages_per_seq > 0 && num_splits >= 0 &&
        make_decode_plan(B, 1, Hq, Hkv, d, page_size, max_pages_per_seq, num_splits, &plan) &&
        plan.total_bytes > kScratchBytes) {
        set_error_message(
            "attn_decode_paged_noalloc: these sizes need %zu bytes of scratch, more than the library's fixed "
            "%zu; use attn_decode_paged with a caller workspace, or a larger num_splits page range",
            plan.total_bytes, kScratchBytes);
        return ATTN_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    // Argument errors are reported by attn_decode_paged before it touches the
    // scratch; look the array up only for calls that can run.
    if (q && k_cache && v_cache && block_table && seq_lens && out && lse && B > 0) {
        attn_status st = scratch_on_current_device(&scratch);
        if (st != ATTN_OK) return st;
    } else {
        scratch = reinterpret_cast<void*>(uintptr_t(256));  // never dereferenced: the checks reject first
    }
    return attn_decode_paged(q, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens, out, lse, B, Hq, Hkv, d,
                             page_size, num_pages, scale, num_splits, scratch, kScratchBytes, stream);
}
