/*
 * attn.h -- libattn: exact scaled dot-product attention on one GB300 GPU
 * (sm_103a), computed by tiling with the online-softmax recurrence.
 *
 * O = softmax(Q K^T * scale + mask) V and the per-row log-sum-exp are
 * produced without ever writing an N x N score or probability matrix to
 * device memory ("Deep Dive - FlashAttention", section "Exact attention
 * without an n x n workspace"; "FlashAttention: Part 1", section 3.1).
 * "Exact" means the same operator in real arithmetic; results differ from an
 * fp64 evaluation only by floating-point rounding (bf16 inputs and outputs,
 * fp32 accumulation), not bit-for-bit ("FlashAttention: Part 1", section 3.2).
 *
 * Conventions shared by every entry point
 *  - Pointers: every tensor pointer is a DEVICE pointer owned by the caller;
 *    the library keeps no reference after the call returns.  The library
 *    allocates no device memory.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *    default stream).  Calls only enqueue work; they never synchronise the
 *    stream, except attn_get_device_status.
 *  - Element types: q, k, v, out, caches are bf16 (IEEE bfloat16, 2 bytes);
 *    lse is fp32; index arrays are int32.  All tensors are dense row-major
 *    with the strides implied by their shapes, and 16-byte aligned.
 *  - Head map: query head h reads K/V head h / (Hq / Hkv), i.e. consecutive
 *    groups of Hq/Hkv query heads share one K/V head ("Deep Dive -
 *    FlashAttention", section "The public interface is several kernels").
 *  - Causal mask: aligned to the bottom-right corner -- query i of a sequence
 *    with Nq queries and Nk keys sees key j iff j <= i + Nk - Nq (same page,
 *    section "Causal 2.1 is the decode gotcha").
 *  - Empty rows: a query row with no allowed key gets O = 0 and lse = -inf
 *    (the page returns zero for an entirely masked row and defines lse only
 *    for nonempty rows; -inf = log 0 is the neutral element of an lse merge).
 *  - lse is the natural-log log-sum-exp of the scaled, masked scores:
 *    lse_i = m_i + ln(l_i) (same page, section "Exact attention without an
 *    n x n workspace").
 *  - Errors: host-side argument checks return a status before any work is
 *    enqueued.  Problems only the device can see (a timed-out pipeline wait,
 *    or, with validation on, a malformed index array) are recorded in a
 *    per-process device error word and reported by attn_get_device_status.
 *    Kernels never trap; they stay inside the buffers the ABI describes even
 *    when index arrays hold garbage (offsets are clamped, gathers of
 *    out-of-range pages read zeros).
 */
#ifndef LIBATTN_ATTN_H
#define LIBATTN_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = -1, /* bad pointer, size or value; nothing enqueued   */
    ATTN_ERR_UNSUPPORTED = -2, /* valid but not built (e.g. head_dim 96)          */
    ATTN_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed               */
    ATTN_ERR_TIMEOUT = -4,     /* a kernel's bounded pipeline wait expired        */
    ATTN_ERR_BAD_INDEX = -5    /* validation found a malformed index array        */
} attn_status;

/*
 * attn_fwd -- prefill forward: O = softmax(Q K^T * scale + mask) V and lse.
 *
 * Operation: for every sequence b, query head h and query row i, the tiled
 * forward pass of "FlashAttention: Part 1", section 3.1 (query tile resident,
 * K/V tiles streamed, running max and normaliser with the exp(m_old - m_new)
 * rescale, one division by the normaliser at the end), with the tile skipping
 * of section 3.5: K/V tiles entirely above the causal boundary are never
 * loaded and only tiles crossing the boundary or a sequence edge are masked.
 *
 * Layout ("THD", the (batch, sequence, heads, head_dim) order of the FA2 call):
 *   q    [T_q, Hq,  d] bf16     out [T_q, Hq, d] bf16 (written)
 *   k, v [T_k, Hkv, d] bf16
 *   dense  (cu_seqlens_q == cu_seqlens_k == NULL): B sequences of exactly Nq
 *          queries and Nk keys; T_q = B*Nq, T_k = B*Nk; sequence b owns query
 *          rows [b*Nq, (b+1)*Nq) and key rows [b*Nk, (b+1)*Nk).
 *          lse [B, Hq, Nq] fp32 (written).
 *   packed (both cu_seqlens given): int32 [B+1] cumulative offsets, starting
 *          at 0, nondecreasing ("Deep Dive - FlashAttention", section "Paged
 *          KV is a lookup, not a cache manager"); sequence b owns query rows
 *          [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key rows
 *          [cu_seqlens_k[b], cu_seqlens_k[b+1]).  In this mode Nq and Nk are
 *          the TOTAL row counts of q and k (T_q = Nq = cu_seqlens_q[B],
 *          T_k = Nk = cu_seqlens_k[B]); per-sequence lengths are read on the
 *          device.  lse [Hq, T_q] fp32 (written).
 *   d (head_dim) in {64, 128}; other values return ATTN_ERR_UNSUPPORTED.
 *   scale: finite and > 0; usually 1/sqrt(d).  causal: 0 or 1 (bottom-right corner,
 *   per sequence).
 * Returns ATTN_OK once the work is enqueued on `stream`.
 * k and v may be NULL only when Nk == 0 (no keys: every row is empty).
 * Rejects (ATTN_ERR_INVALID_ARG): NULL q/out/lse (or k/v with Nk > 0), exactly one cu_seqlens
 * NULL, B < 0, Hq <= 0, Hkv <= 0, Hq % Hkv != 0, Nq < 0, Nk < 0, scale not
 * finite, a pointer not 16-byte aligned.  B == 0 or Nq == 0 enqueues nothing.
 */
attn_status attn_fwd(const void *q, const void *k, const void *v,
                     void *out, float *lse,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d,
                     float scale, int causal,
                     const int *cu_seqlens_q, const int *cu_seqlens_k,
                     void *stream);

/*
 * attn_fwd_window -- attn_fwd with a local (sliding-window) band mask.
 *
 * Operation: as attn_fwd, with the mask of "Deep Dive - FlashAttention",
 * section "Causal 2.1 is the decode gotcha", paragraph on local attention:
 * query row i of a sequence with Nq_b queries and Nk_b keys keeps keys
 *     i + Nk_b - Nq_b - window_left  <=  j  <=  i + Nk_b - Nq_b + window_right
 * inside [0, Nk_b); a side of -1 is unbounded; with causal = 1 the causal
 * corner restricts the set further (which makes window_right irrelevant).
 * K/V tiles that no row of a query tile keeps are never loaded ("FlashAttention:
 * Part 1", section 3.5, applied to both band edges), so the cost follows the
 * band's width rather than Nk.  window_left = window_right = -1 is attn_fwd.
 * Layout, ownership and every other rule: as attn_fwd.
 * Rejects (ATTN_ERR_INVALID_ARG) in addition: window_left or window_right < -1.
 */
attn_status attn_fwd_window(const void *q, const void *k, const void *v,
                            void *out, float *lse,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d,
                            float scale, int causal, int window_left, int window_right,
                            const int *cu_seqlens_q, const int *cu_seqlens_k,
                            void *stream);

/*
 * attn_fp8_scale_count -- scale entries per head of a per-tile 8-bit tensor
 * holding T tokens in B sequences: T / 128 + B (integer division).  Tile t of
 * sequence b (its tokens [first_b + 128 t, first_b + 128 (t + 1)), cut at the
 * sequence end) has entry first_b / 128 + b + t, first_b being the
 * sequence's first token; entries between sequences are never used.  0 for
 * B < 0 or T < 0.  Pure host arithmetic.
 */
size_t attn_fp8_scale_count(int B, int T);

/*
 * attn_quantize_fp8 -- per-tile 8-bit (E4M3) quantization of a bf16 tensor
 * for attn_fwd_fp8.
 *
 * Operation: the per-tile quantization of "FP8 Path and Quantization" ("Flash
 * Attention: A Complete Architectural Autopsy", part 4) -- the block
 * quantization of "FlashAttention-3: asynchrony and low precision on Hopper"
 * ("FlashAttention-3 and PagedAttention"): each tile gets a scale factor from
 * its absolute maximum.  A tile is 128 consecutive tokens of one sequence
 * (counted from its first token) for one head and all d channels.  In fp32:
 *     amax = max |x| over the tile,  scale = amax / 448,  inv = 448 / amax,
 *     code = E4M3(x * inv)  (round to nearest even, saturating at 448),
 * so x is represented as E4M3(code) * scale.  A tile with amax < 2^-100 gets
 * scale 1 and zero codes.  E4M3: 1 sign, 4 exponent (bias 7) and 3 mantissa
 * bits, subnormals, no infinities, largest finite 448.  Inputs must be
 * finite.
 *
 * Layout:
 *   x        [T, H, d] bf16 (read); T = B * N (cu_seqlens NULL: sequence b
 *            owns tokens [b N, (b+1) N)) or cu_seqlens[B] (packed: int32
 *            [B+1], nondecreasing from 0, N = T)
 *   x8       [T, H, d] E4M3 codes, one byte each (written)
 *   x_scale  [H, attn_fp8_scale_count(B, T)] fp32 (tile entries written,
 *            entries between sequences untouched)
 *   d in {64, 128}.
 * Rejects (ATTN_ERR_INVALID_ARG): NULL pointers, B < 0, H <= 0, N < 0, x or
 * x8 not 16-byte aligned, x_scale not 4-byte aligned.  B == 0 or T == 0
 * enqueues nothing.
 */
attn_status attn_quantize_fp8(const void *x, void *x8, float *x_scale,
                              int B, int H, int N, int d,
                              const int *cu_seqlens, void *stream);

/*
 * attn_quantize_fp8_qkv -- attn_quantize_fp8 of q, k and v in one launch.
 *
 * Operation: exactly three attn_quantize_fp8 calls -- q with (B, Hq, Nq,
 * cu_seqlens_q), k and v with (B, Hkv, Nk, cu_seqlens_k) -- with
 * bit-identical codes and scales; one kernel launch does all three, which
 * saves the launch gaps and the thin tails of the two smaller tensors.  This
 * is the preparation attn_fwd_fp8 needs ("FP8 Path and Quantization": Q, K
 * and V are quantized per tile).
 *
 * Layout: q [T_q, Hq, d], k and v [T_k, Hkv, d] bf16; q8, k8, v8 the E4M3
 * codes shaped alike; q_scale [Hq, attn_fp8_scale_count(B, T_q)], k_scale
 * and v_scale [Hkv, attn_fp8_scale_count(B, T_k)] fp32.  T and the
 * cu_seqlens as attn_fwd_fp8 (dense: T = B * N; packed: give both
 * cu_seqlens, Nq and Nk the totals).  d in {64, 128}.
 * Rejects (ATTN_ERR_INVALID_ARG): NULL pointers (k, v, k8, v8, k_scale and
 * v_scale may be NULL only when Nk == 0), only one cu_seqlens given, B < 0,
 * head counts <= 0, Nq < 0, Nk < 0, tensors or codes not 16-byte aligned,
 * scales not 4-byte aligned.  Nk == 0 quantizes q alone.
 */
attn_status attn_quantize_fp8_qkv(const void *q, const void *k, const void *v,
                                  void *q8, void *k8, void *v8,
                                  float *q_scale, float *k_scale, float *v_scale,
                                  int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                  const int *cu_seqlens_q, const int *cu_seqlens_k,
                                  void *stream);

/*
 * attn_fwd_fp8 -- prefill forward on per-tile 8-bit (E4M3) Q, K, V.
 *
 * Operation: attn_fwd (bottom-right causal corner, GQA, dense or packed) on
 * the values q8, k8, v8 stand for -- E4M3(code) * the code's tile scale, as
 * attn_quantize_fp8 writes them.  Following "FP8 Path and Quantization" (the
 * score computed from 8-bit operands, then turned back into fp32 for the
 * softmax) and "FlashAttention-3: asynchrony and low precision on Hopper":
 * S = Q8 K8^T is an 8-bit tensor-core product with fp32 accumulation, and
 * the tile scales are folded into the exponent's coefficient.  The
 * probabilities stay 16-bit (f16, with the V tile's scale ratio folded in)
 * and the PV product reads the V tile widened exactly to f16: an 8-bit P
 * would add a relative error of up to 2^-4 per weight.  The output is bf16
 * and lse fp32, exactly as attn_fwd.
 *
 * Layout: q8 [T_q, Hq, d], k8 and v8 [T_k, Hkv, d], E4M3 codes; q_scale
 * [Hq, attn_fp8_scale_count(B, T_q)], k_scale and v_scale [Hkv,
 * attn_fp8_scale_count(B, T_k)], fp32, tiles as attn_quantize_fp8 cuts them
 * (from the same B, N or cu_seqlens).  out, lse, B, Hq, Hkv, Nq, Nk, scale,
 * causal and the cu_seqlens as attn_fwd.  d in {64, 128} (others:
 * ATTN_ERR_UNSUPPORTED).
 * Rejects (ATTN_ERR_INVALID_ARG): attn_fwd's cases, NULL or misaligned
 * (4-byte) scale pointers.  k8, v8, k_scale, v_scale may be NULL only when
 * Nk == 0.
 */
attn_status attn_fwd_fp8(const void *q8, const void *k8, const void *v8,
                         const float *q_scale, const float *k_scale, const float *v_scale,
                         void *out, float *lse,
                         int B, int Hq, int Hkv, int Nq, int Nk, int d,
                         float scale, int causal,
                         const int *cu_seqlens_q, const int *cu_seqlens_k,
                         void *stream);

/*
 * attn_fwd_fp8_window -- attn_fwd_fp8 with attn_fwd_window's local band mask
 * (window_left, window_right; -1 = unbounded side; causal = 1 keeps the
 * causal corner).  K/V tiles outside every row's band are never loaded.
 * window_left = window_right = -1 is attn_fwd_fp8.  Everything else: as
 * attn_fwd_fp8.
 * Rejects (ATTN_ERR_INVALID_ARG) in addition: window_left or window_right < -1.
 */
attn_status attn_fwd_fp8_window(const void *q8, const void *k8, const void *v8,
                                const float *q_scale, const float *k_scale, const float *v_scale,
                                void *out, float *lse,
                                int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                float scale, int causal, int window_left, int window_right,
                                const int *cu_seqlens_q, const int *cu_seqlens_k,
                                void *stream);

/*
 * attn_bwd -- gradients dQ, dK, dV of a loss L through attn_fwd /
 * attn_fwd_window, given G = dL/dO, by recomputation.
 *
 * Operation: "Deep Dive - FlashAttention", section "Backward recomputes tiles
 * on purpose", and "FlashAttention: Part 1", section 3.6.  The forward saved
 * only O and lse; each probability tile is rebuilt as P = exp(S - lse) with
 * the forward's mask, and for every nonempty row
 *     dV = P^T G,   dP = G V^T,   D = rowsum(G o O),   dS = P o (dP - D),
 *     dQ = scale * dS K,   dK = scale * dS^T Q,
 * masked probabilities and their gradients being zero.  With grouped heads
 * the K/V gradients of a K/V head are summed over its Hq / Hkv query heads.
 * Three kernels: D, then dK/dV with K/V tiles resident, then dQ with query
 * tiles resident (no atomic accumulation: the result is deterministic).
 *
 * Arguments: q, k, v, B, Hq, Hkv, Nq, Nk, d, scale, causal, window_left,
 * window_right, cu_seqlens_q, cu_seqlens_k exactly as given to the forward
 * call; out and lse are the forward's outputs; dout = G, laid out like out.
 *   dq [T_q, Hq, d], dk and dv [T_k, Hkv, d], bf16 (written; every row is
 *   written, rows no query attends get 0).
 *   workspace: caller-owned device scratch of attn_bwd_workspace_size(B, Hq,
 *   Nq, packed) bytes, 256-byte aligned; it holds D and lse * log2(e) (fp32)
 *   between the kernels, needs no initialisation and is meaningless afterwards.
 * k, v, dk, dv may be NULL only when Nk == 0.
 * Rejects (ATTN_ERR_INVALID_ARG): the forward's cases, NULL out/dout/dq/
 * workspace, a workspace that is too small or not 256-byte aligned.
 */
attn_status attn_bwd(const void *q, const void *k, const void *v,
                     const void *out, const void *dout, const float *lse,
                     void *dq, void *dk, void *dv,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d,
                     float scale, int causal, int window_left, int window_right,
                     const int *cu_seqlens_q, const int *cu_seqlens_k,
                     void *workspace, size_t workspace_bytes,
                     void *stream);

/*
 * attn_bwd_workspace_size -- bytes of scratch attn_bwd needs: lse * log2(e)
 * and D for every query row and head, each per head in a row of
 * 4*ceil(T_q/4) + 4*B + 132 floats (every sequence's rows start 16-byte
 * aligned so that 128-row tiles are copied in one transfer), rounded up to 256
 * bytes; T_q = B * Nq (packed = 0) or Nq (packed = 1, Nq the total query
 * rows).  0 for invalid arguments.  Pure host arithmetic.
 */
size_t attn_bwd_workspace_size(int B, int Hq, int Nq, int packed);

/*
 * attn_decode_paged -- one new query per sequence over a paged K/V cache,
 * split along the keys (split-KV) with a log-sum-exp combine.
 *
 * Operation: "FlashAttention-3 and PagedAttention", sections "Block tables
 * and what the kernel does" (logical token t of sequence b lives in physical
 * page block_table[b][t / page_size] at slot t % page_size) and "Why decode
 * starves the GPU" (the keys of each sequence are cut into chunks processed
 * in parallel, each chunk emits a partial output and its lse, and a second
 * kernel weights partial i by exp(lse_i - lse_total)).  The single query is
 * the last position, so under the bottom-right rule it sees all seq_lens[b]
 * keys; there is no causal flag.  The query heads that share a K/V head are
 * packed into one tile so each gathered K/V row is read once for all of them.
 *
 * Layout:
 *   q        [B, Hq, d] bf16              out [B, Hq, d] bf16 (written)
 *   k_cache, v_cache [num_pages, page_size, Hkv, d] bf16
 *   block_table int32 [B, max_pages_per_seq]; only the first
 *            ceil(seq_lens[b] / page_size) entries of row b are read (others
 *            may hold anything, e.g. -1).
 *   seq_lens int32 [B], 0 <= seq_lens[b] <= max_pages_per_seq * page_size
 *            (larger values are clamped; a sequence of length 0 yields O = 0,
 *            lse = -inf).
 *   lse      [B, Hq] fp32 (written).
 * Slots past seq_lens[b] in a sequence's last page, and pages no sequence
 * uses, may hold any bits including NaN: they are excluded by selection, not
 * by multiplying with a zero weight.
 *   d in {64, 128}; page_size == 16 (others: ATTN_ERR_UNSUPPORTED).
 *   num_splits: 0 = automatic chunking (a fixed number of pages per chunk,
 *            derived from B, Hkv and max_pages_per_seq only); N > 0 = every
 *            sequence is cut into N equal page ranges.
 *   workspace: caller-owned device scratch of at least
 *            attn_decode_workspace_size(...) bytes (same B, Hq, Hkv, d,
 *            page_size, max_pages_per_seq, num_splits), 256-byte aligned.  It
 *            holds the per-chunk partial outputs and lse between the split and
 *            the combine kernels; its contents need no initialisation and are
 *            meaningless afterwards.  Two calls that overlap on the GPU must
 *            not share a workspace.
 * Rejects (ATTN_ERR_INVALID_ARG): NULL pointers, B < 0, head counts <= 0,
 * Hq % Hkv != 0, num_pages <= 0, max_pages_per_seq <= 0, num_splits < 0,
 * scale not finite, workspace_bytes too small, misaligned pointers.
 */
attn_status attn_decode_paged(const void *q,
                              const void *k_cache, const void *v_cache,
                              const int *block_table, int max_pages_per_seq,
                              const int *seq_lens,
                              void *out, float *lse,
                              int B, int Hq, int Hkv, int d, int page_size, int num_pages,
                              float scale, int num_splits,
                              void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * attn_decode_workspace_size -- bytes of device scratch attn_decode_paged
 * needs for these sizes (0 when the arguments are invalid).  Pure host
 * arithmetic; needs no GPU.
 */
size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int d, int page_size,
                                  int max_pages_per_seq, int num_splits);

/*
 * attn_decode_paged_noalloc -- attn_decode_paged for callers that cannot
 * allocate device memory when they call (no counterpart in the pages this
 * library follows; it exists for integration only).
 *
 * Some callers cannot give the library a workspace: a plug-in whose host
 * runtime owns every device allocation and offers it no allocator, or a
 * serving loop that reserves its memory once and may not call cudaMalloc or
 * cudaFree afterwards (those calls can synchronise the whole device).  This
 * entry point takes the same arguments as attn_decode_paged minus the
 * workspace and keeps the per-chunk partial results in a fixed 32 MiB array
 * compiled into the library; every GPU that loads the library holds that
 * array until the process exits.  It allocates nothing.
 *
 *  - Limit: the scratch that attn_decode_workspace_size reports for the same
 *    sizes must be at most 32 MiB (33554432 bytes); larger sizes return
 *    ATTN_ERR_INVALID_ARG with a message.  A smaller nonzero num_splits
 *    (fewer, longer chunks per sequence) shrinks the requirement.
 *  - Argument errors are checked first and reported exactly as
 *    attn_decode_paged reports them; the size limit is checked after them.
 *  - Every call looks up the array's device address in the current device's
 *    context (cudaGetSymbolAddress); the first call on a device may load the
 *    library's device code there, so make that first call before any stream
 *    capture begins.
 *  - All calls share the one array and it keeps the last call's contents
 *    (nothing in it needs to start at zero).  Calls that overlap on the GPU
 *    -- on different streams, or from different threads -- race on it: order
 *    them on one stream or with events.
 * Everything else (layouts, errors, the result) is as for attn_decode_paged.
 */
attn_status attn_decode_paged_noalloc(const void *q,
                                      const void *k_cache, const void *v_cache,
                                      const int *block_table, int max_pages_per_seq,
                                      const int *seq_lens,
                                      void *out, float *lse,
                                      int B, int Hq, int Hkv, int d, int page_size, int num_pages,
                                      float scale, int num_splits,
                                      void *stream);

/*
 * attn_decode_kvcache -- Nq new queries per sequence over the paged K/V cache,
 * optionally appending the new tokens' K/V to the cache in place first.
 *
 * Operation: attn_decode_paged's split-KV pass and combine, generalised to
 * several queries per sequence ("Deep Dive - FlashAttention", section "Paged
 * KV is a lookup, not a cache manager": the call may update the cache in
 * place; section "Causal 2.1 is the decode gotcha": the bottom-right corner).
 * seq_lens[b] counts the sequence's tokens INCLUDING the Nq new ones; query i
 * is position seq_lens[b] - Nq + i.  With causal = 1 it sees keys
 * j <= seq_lens[b] - Nq + i (the bottom-right rule with Nq queries and
 * seq_lens[b] keys); with causal = 0 it sees all seq_lens[b] keys.  The Nq
 * queries of the query heads that share a K/V head are packed into the same
 * tiles, so each gathered page is read once for all of them.
 * Append (k_new and v_new not NULL): before any score is computed, new row i
 * of sequence b is written to position seq_lens[b] - Nq + i, i.e. slot
 * pos % page_size of page block_table[b][pos / page_size].  The caller
 * reserves those pages in the block table beforehand.  Positions below zero,
 * positions past the table and page ids outside [0, num_pages) are never
 * written (with validation on they are reported as ATTN_ERR_BAD_INDEX).  Two
 * sequences whose new positions map to the same slot race: the result is one
 * of the writes, unspecified which.
 *
 * Layout:
 *   q        [B, Nq, Hq, d] bf16          out [B, Nq, Hq, d] bf16 (written)
 *   k_new, v_new [B, Nq, Hkv, d] bf16, or both NULL (no append)
 *   k_cache, v_cache [num_pages, page_size, Hkv, d] bf16 (written by the append)
 *   block_table, seq_lens, page_size, num_splits: as attn_decode_paged
 *   lse      [B, Hq, Nq] fp32 (written)
 *   workspace: at least attn_decode_kvcache_workspace_size(...) bytes,
 *            256-byte aligned, otherwise as attn_decode_paged.
 * Nq = 1 with no append computes what attn_decode_paged computes.
 * Rejects (ATTN_ERR_INVALID_ARG): attn_decode_paged's cases, Nq <= 0, exactly
 * one of k_new/v_new NULL, causal not 0 or 1.  (Hq / Hkv) * Nq > 128 returns
 * ATTN_ERR_UNSUPPORTED.
 */
attn_status attn_decode_kvcache(const void *q, const void *k_new, const void *v_new,
                                void *k_cache, void *v_cache,
                                const int *block_table, int max_pages_per_seq,
                                const int *seq_lens,
                                void *out, float *lse,
                                int B, int Nq, int Hq, int Hkv, int d, int page_size, int num_pages,
                                float scale, int causal, int num_splits,
                                void *workspace, size_t workspace_bytes,
                                void *stream);

/*
 * attn_decode_kvcache_workspace_size -- bytes of device scratch
 * attn_decode_kvcache needs for these sizes (0 when the arguments are
 * invalid).  Pure host arithmetic; needs no GPU.
 */
size_t attn_decode_kvcache_workspace_size(int B, int Nq, int Hq, int Hkv, int d, int page_size,
                                          int max_pages_per_seq, int num_splits);

/*
 * attn_get_device_status -- synchronises `stream`, then reads and clears the
 * device error word of the current device: ATTN_OK, ATTN_ERR_TIMEOUT or
 * ATTN_ERR_BAD_INDEX (the first error recorded since the last read), or
 * ATTN_ERR_CUDA when the synchronisation itself failed.
 */
attn_status attn_get_device_status(void *stream);

/*
 * attn_set_validation -- process-wide switch (default 0 = off).  When on,
 * kernels check cu_seqlens (start 0, nondecreasing, end == Nq/Nk), block-table
 * entries of the pages a sequence uses (0 <= page < num_pages) and seq_lens
 * (<= max_pages_per_seq * page_size), and record ATTN_ERR_BAD_INDEX in the
 * device error word.  Off, the same inputs are clamped silently.
 * Returns the previous setting.
 */
int attn_set_validation(int enabled);

/*
 * attn_test_drop_page_load -- test hook for the failure path (not for
 * production use).  When called with 1, the next attn_decode_paged launch
 * makes one CTA (chunk 0 of sequence 0) skip its first page copy, so the
 * consumer warps' bounded wait for that page expires: the kernel records
 * ATTN_ERR_TIMEOUT in the device error word and returns instead of hanging;
 * the outputs of that sequence are undefined.  The switch clears itself after
 * one launch.  Returns the previous setting.
 */
int attn_test_drop_page_load(int enabled);

/* attn_status_string -- static, human-readable name of a status code. */
const char *attn_status_string(attn_status status);

/* attn_last_error_message -- detail of the last host-side failure on this
 * thread (static storage, valid until the next call on the thread). */
const char *attn_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBATTN_ATTN_H */
