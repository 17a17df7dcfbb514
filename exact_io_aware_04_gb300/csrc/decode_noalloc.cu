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

#include "internal.h"

namespace attn {
namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB

// Per-chunk partial outputs and lse of the split kernel.  The name is only a
// host-side stand-in in host code; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Device address of the scratch array in the current device's context.  It is
// looked up on every call (a table lookup once the module is loaded), so a
// context that was torn down and rebuilt -- cudaDeviceReset, or recovery from
// a sticky error, which reloads the module -- never sees a stale address.  The
// first call on a device may load the module.
attn_status scratch_on_current_device(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
        set_error_message("cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    *out = p;
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
    // attn_decode_paged's own argument checks come first, so a bad pointer or
    // size gets the same error as there; then the scratch must fit the array.
    DecodePlan plan;
    attn_status st = decode_check("attn_decode_paged_noalloc", q, nullptr, nullptr, k_cache, v_cache, block_table,
                                  max_pages_per_seq, seq_lens, out, lse, B, 1, Hq, Hkv, d, page_size, num_pages,
                                  scale, 0, num_splits, &plan);
    if (st != ATTN_OK) return st;
    if (plan.total_bytes > kScratchBytes) {
        set_error_message(
            "attn_decode_paged_noalloc: these sizes need %zu bytes of scratch, more than the library's fixed "
            "%zu; use attn_decode_paged with a caller workspace, or pass a smaller nonzero num_splits "
            "(fewer, longer chunks)",
            plan.total_bytes, kScratchBytes);
        return ATTN_ERR_INVALID_ARG;
    }
    if (B == 0) return ATTN_OK;
    void* scratch = nullptr;
    st = scratch_on_current_device(&scratch);
    if (st != ATTN_OK) return st;
    return attn_decode_paged(q, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens, out, lse, B, Hq, Hkv, d,
                             page_size, num_pages, scale, num_splits, scratch, kScratchBytes, stream);
}
