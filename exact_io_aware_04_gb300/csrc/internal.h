// internal.h -- host-side plumbing shared by the libattn translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "status.h"

namespace attn {

// Launch attributes (dynamic shared memory) are per device: the launchers
// remember having set them for devices below this index.
constexpr int kMaxDevices = 64;

// Per-device facts the launchers need; cached after the first query.
struct DeviceInfo {
    int device;
    int sm_count;
    int* err_word;  // device address of this device's error word
};

// Fills `info` for the current device.  ATTN_ERR_CUDA on failure.
attn_status current_device_info(DeviceInfo* info);

// Records a printf-style detail message for attn_last_error_message().
void set_error_message(const char* fmt, ...);

// Encodes a tiled TMA descriptor for a bf16 tensor.  dims[0] is the
// contiguous dimension; strides_bytes[i] is the byte stride of dims[i+1].
attn_status encode_tma_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128);
// The same for any element type (8-bit codes use CU_TENSOR_MAP_DATA_TYPE_UINT8).
attn_status encode_tma(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128);
// The same with any swizzle mode (the 8-bit tiles at d = 64 use the 64-byte one).
attn_status encode_tma_swizzle(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                               const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                               CUtensorMapSwizzle swizzle);

bool validation_enabled();
// With validation on: checks packed offsets cu[0..B] (start 0, nondecreasing,
// end == total) on the stream and records ATTN_ERR_BAD_INDEX in the device
// error word if they are malformed.
void launch_check_cu_seqlens(const int* cu, int B, int total, cudaStream_t stream);

// One-shot test switch: the next paged-decode launch drops one page copy.
int set_drop_page_load(int enabled);

// ---- launchers (one per translation unit) ----
struct FwdArgs {
    const void *q, *k, *v;
    void* out;
    float* lse;
    int B, Hq, Hkv, Nq, Nk, d;
    float scale;
    int causal;
    int win_left, win_right;  // local window, < 0 = unbounded
    const int *cu_q, *cu_k;
    // 8-bit forward only (q, k, v then hold E4M3 codes): per-tile scales,
    // [heads, fp8_scale_count(B, T)] each (tile t of sequence b at entry
    // first_token_b / 128 + b + t)
    const float *q_scale, *k_scale, *v_scale;
};
attn_status launch_fwd(const FwdArgs& a, cudaStream_t stream);
attn_status launch_fwd_fp8(const FwdArgs& a, cudaStream_t stream);

// Scale entries per head of a per-tile 8-bit tensor of T tokens in B sequences.
inline long long fp8_scale_count(long long B, long long T) { return T / 128 + B; }

struct QuantArgs {
    const void* x;       // [T, H, d] bf16
    void* x8;            // [T, H, d] E4M3 codes
    float* scale;        // [H, fp8_scale_count(B, T)]
    int B, H, N, d;      // N: tokens per sequence (dense) or T (packed)
    const int* cu;       // int32 [B + 1] or NULL (dense)
};
// Quantizes n (1..kMaxQuantTensors) tensors of the same head_dim in one launch.
constexpr int kMaxQuantTensors = 3;
attn_status launch_quantize_fp8(const QuantArgs* a, int n, cudaStream_t stream);

struct BwdArgs {
    const void *q, *k, *v, *out, *dout;  // out = the forward output O, dout = dL/dO
    const float* lse;                    // the forward lse (natural log)
    void *dq, *dk, *dv;
    void* workspace;                     // D = rowsum(dout o out), fp32 in the lse layout
    int B, Hq, Hkv, Nq, Nk, d;
    float scale;
    int causal;
    int win_left, win_right;
    const int *cu_q, *cu_k;
};
size_t bwd_workspace_bytes(int B, int Hq, int Nq, bool varlen);
attn_status launch_bwd(const BwdArgs& a, cudaStream_t stream);

struct DecodeArgs {
    const void* q;                  // [B, nq, Hq, d]
    const void *k_cache, *v_cache;
    const void *k_new, *v_new;      // [B, nq, Hkv, d] appended before attending, or NULL
    void *k_cache_w, *v_cache_w;    // writable views of the caches (used only with k_new)
    const int* block_table;
    int max_pages;
    const int* seq_lens;
    void* out;
    float* lse;
    int B, Hq, Hkv, d, page_size, num_pages;
    int nq, causal;
    float scale;
    int num_splits;
    void* workspace;
    size_t workspace_bytes;
};

// How attn_decode_paged cuts sequences into chunks.
struct DecodePlan {
    int pages_per_chunk;  // chunk length in pages
    int max_chunks;       // chunks of the longest possible sequence
    int heads_per_cta;    // K/V heads gathered by one CTA
    int head_groups;      // Hkv / heads_per_cta
    size_t partial_o_bytes, partial_lse_bytes, total_bytes;
};
bool make_decode_plan(int B, int nq, int Hq, int Hkv, int d, int page_size, int max_pages, int num_splits,
                      DecodePlan* plan);
attn_status launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream);

// Every argument check of the paged-decode entry points except those on the
// workspace (pointers, sizes, alignment, head_dim, page size, plan); fills
// `plan` on success.  `fn` names the entry point in the error message.
attn_status decode_check(const char* fn, const void* q, const void* k_new, const void* v_new, const void* k_cache,
                         const void* v_cache, const int* block_table, int max_pages_per_seq, const int* seq_lens,
                         const void* out, const float* lse, int B, int Nq, int Hq, int Hkv, int d, int page_size,
                         int num_pages, float scale, int causal, int num_splits, DecodePlan* plan);

}  // namespace attn
