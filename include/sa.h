/*
 * sa.h -- C ABI of the GB300 (sm_103a) top-k sparse attention library.
 *
 * Operations of the DeepSeek V4 sparse-attention path:
 *
 *  1. o = sparse_attn(q, kv, attn_sink, topk_idxs, softmax_scale)
 *     "DeepSeek V4 源码剖析, 第5章 sparse_attn 与 FlashMLA": §5.1 (argument
 *     shapes and dtypes, -1 marks an invalid slot, softmax_scale =
 *     head_dim^-0.5), §5.2 (per query token and head: gather K indexed kv
 *     rows, logits = scale * q.k, -inf on invalid slots, append the head's
 *     sink logit, softmax, weighted sum of the gathered rows -- the sink's
 *     weight is dropped; V is the same row as K), §5.5 (online softmax over
 *     64-row tiles, sink added once to the denominator, the log-sum-exp form
 *     of the sink for split-KV combine).
 *
 *  2. The bit-packed top-k mask: vLLM PR 52217 page ("Sparse MLA mask
 *     向量化 128-bit 加载", `_topk_mask_shape`, `_build_topk_mask`, the two
 *     alignment tests) and vLLM PR 48770 page (masked MHA for sparse-MLA
 *     prefill: `dense_mask_mod` reads bit kv&31 of word kv>>5, LSB first;
 *     `offset_dense_mask_mod` reads key_start from the last word of row 0).
 *
 *  3. The mask's consumer -- attention over the keys a mask row admits
 *     (the same PR 48770 page) -- and its chunked form: windows of query
 *     rows under the 64 MiB global-mask cap of that page, each row built
 *     only up to its live key end (vLLM PR 56628 page).
 *
 *  4. sparse_attn over an FP8 kv cache in the V4 row format (the same
 *     chapter, §5.3 and §5.6).
 *
 * Conventions for every entry point:
 *   - Tensors are dense, row-major (C order), in DEVICE memory of the current
 *     CUDA device unless stated otherwise.  The caller owns every buffer,
 *     workspace included; the library allocates no device memory and keeps no
 *     per-call state (the one exception, sa_sparse_attn_fwd_static_ws, uses
 *     a workspace array compiled into the library).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  A call returns once its kernels are enqueued.
 *   - Arguments are validated on the host before anything is launched; on any
 *     error nothing is launched and no output byte is written.
 *   - Index VALUES are data, not arguments: an index outside [0, T) (or
 *     [0, max_key_len) for the mask) is treated as an invalid slot and never
 *     dereferenced.
 *   - No entry point throws or aborts.
 */
#ifndef SA_H_
#define SA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers (same underlying type). */
typedef struct CUstream_st *sa_stream_t;

typedef enum {
    SA_OK = 0,
    SA_ERR_INVALID_ARG = 1,        /* NULL pointer, negative size, non-finite scale */
    SA_ERR_SHAPE = 2,              /* a size combination the kernels do not support */
    SA_ERR_ALIGNMENT = 3,          /* a tensor that must start on 16 bytes does not */
    SA_ERR_WORKSPACE = 4,          /* workspace smaller than the size query returned */
    SA_ERR_UNSUPPORTED_DEVICE = 5, /* current device is not compute capability 10.3 */
    SA_ERR_CUDA = 6                /* a CUDA runtime call or launch failed */
} sa_status;

/* Human-readable name of a status code (static storage, never NULL). */
const char *sa_status_string(sa_status status);

/* ------------------------------------------------------------------------ */
/* sparse_attn                                                              */
/* ------------------------------------------------------------------------ */

/* Number of KV splits the library picks for this problem on the current
 * device (1 = no split).  Depends only on the sizes and the device's SM
 * count, never on index values, so a captured CUDA graph keeps its grid.
 * Returns 0 on invalid sizes. */
int sa_sparse_attn_num_splits(int64_t B, int64_t S, int64_t H, int64_t D, int64_t K);

/* Workspace bytes sa_sparse_attn_fwd_splits needs for `num_splits` splits
 * (num_splits <= 0 means the library's choice, as above).  Holds one float32
 * partial output [B*S, splits, H, D] and one float32 log-sum-exp
 * [B*S, splits, H]; 0 when no split is made. */
size_t sa_sparse_attn_workspace_size(int64_t B, int64_t S, int64_t H, int64_t D, int64_t K,
                                     int num_splits);

/* Kernels one sa_sparse_attn_fwd_splits call with these sizes enqueues on the
 * current device: 1 when every token's splits fit one thread-block cluster
 * (splits x head-dim halves <= 8 CTAs) and are combined inside the main
 * kernel, 2 when a separate combine kernel follows.  Host-only; 0 on invalid
 * sizes, B*S == 0, or a device this library does not support.  The pages have
 * no counterpart of this query: it describes this library's launch plan, for
 * callers that budget launches (CUDA graphs, launch-count accounting). */
int sa_sparse_attn_launch_count(int64_t B, int64_t S, int64_t H, int64_t D, int64_t K, int num_splits);

/* o[b,s,h,:] = sum_j w_j * kv[b, topk_idxs[b,s,j], :] with
 *   x_j = softmax_scale * <q[b,s,h,:], kv[b, topk_idxs[b,s,j], :]>  (slot j valid),
 *   w   = softmax([x_0 .. x_{K-1}, attn_sink[h]])[0..K-1],
 * invalid slots (index < 0 or >= T) contributing weight 0.  A token with no
 * valid slot yields o = 0; attn_sink[h] = +inf yields o = 0; -inf is plain
 * softmax attention.
 *
 *   q          bf16  [B,S,H,D]   16-byte aligned
 *   kv         bf16  [B,T,D]     16-byte aligned (shared by all heads: MQA)
 *   attn_sink  fp32  [H]
 *   topk_idxs  int32 [B,S,K]
 *   o          bf16  [B,S,H,D]   16-byte aligned, may not alias the inputs
 *   workspace  >= sa_sparse_attn_workspace_size(B,S,H,D,K,0) bytes, 256-byte
 *              aligned; may be NULL when that size is 0.
 * Supported sizes: 1 <= H <= 128, D in {64, 128, 256, 512}, K >= 1,
 * B*S >= 0 (0 launches nothing), T >= 1, B*T < 2^31, B*S*H < 2^31.
 * Computes in bf16 x bf16 -> fp32 on the tensor cores (tcgen05), softmax in
 * fp32, probabilities rounded to bf16 before P.V, output rounded to bf16. */
sa_status sa_sparse_attn_fwd(const void *q, const void *kv, const float *attn_sink,
                             const int32_t *topk_idxs, float softmax_scale, void *o, int64_t B,
                             int64_t S, int64_t H, int64_t D, int64_t T, int64_t K,
                             void *workspace, size_t workspace_bytes, sa_stream_t stream);

/* Same as sa_sparse_attn_fwd with an explicit split count (1..64; <= 0 picks
 * as sa_sparse_attn_num_splits).  The result does not depend on the split
 * count beyond fp32 rounding. */
sa_status sa_sparse_attn_fwd_splits(const void *q, const void *kv, const float *attn_sink,
                                    const int32_t *topk_idxs, float softmax_scale, void *o,
                                    int64_t B, int64_t S, int64_t H, int64_t D, int64_t T,
                                    int64_t K, int num_splits, void *workspace,
                                    size_t workspace_bytes, sa_stream_t stream);

/* sa_sparse_attn_fwd_splits with a per-token valid-prefix length:
 *   topk_length  int32 [B,S] in device memory, 4-byte aligned, or NULL.
 * Slot j of token (b,s) counts only if j < clamp(topk_length[b,s], 0, K)
 * (and, as always, its index is in [0, T)); slots at or past the length are
 * invalid whatever their index, so callers need not pad the tail with -1.
 * NULL behaves as sa_sparse_attn_fwd_splits.  This is the "top-k length
 * differs per sequence" variant of the FlashMLA kernels ("DeepSeek V4
 * 源码剖析, 第5章", §5.3); the extra second KV source those kernels also
 * accept is not supported.  Other arguments, workspace and errors as in
 * sa_sparse_attn_fwd_splits. */
sa_status sa_sparse_attn_fwd_topk_length(const void *q, const void *kv, const float *attn_sink,
                                         const int32_t *topk_idxs, const int32_t *topk_length,
                                         float softmax_scale, void *o, int64_t B, int64_t S, int64_t H,
                                         int64_t D, int64_t T, int64_t K, int num_splits, void *workspace,
                                         size_t workspace_bytes, sa_stream_t stream);

/* sa_sparse_attn_fwd_topk_length over an FP8 kv cache, D = 512 (the V4 /
 * FlashMLA "MODEL1" cache: "DeepSeek V4 源码剖析, 第5章", §5.3 head dims
 * 448 + 64, quantisation tiles of 64, 8 scales a token, V with the RoPE
 * dims; §5.6 codes dequantised where they are gathered).
 *   kv_fp8  uint8 [B, T, 584] device, 16-byte aligned; row t of request b:
 *           bytes [0, 448)   dims 0..447 as FP8 E4M3 codes (OCP: bias 7,
 *                            subnormals, 0x7F/0xFF NaN, max 448),
 *           bytes [448, 576) dims 448..511 as bf16, little-endian,
 *           bytes [576, 583) one E8M0 scale per 64-dim tile of the codes,
 *                            2^(byte - 127) (255 = NaN); byte 583 unused.
 *   value of dim d < 448 = e4m3(code) * scale[d / 64]; the rows are widened
 *   to bf16 on chip (exact unless a value falls below bf16's range) and the
 *   attention is then that of sa_sparse_attn_fwd_topk_length with D = 512.
 * q and o are bf16 [B,S,H,512]; workspace as sa_sparse_attn_workspace_size
 * (B,S,H,512,K,num_splits).  Errors as sa_sparse_attn_fwd_topk_length. */
sa_status sa_sparse_attn_fwd_fp8(const void *q, const uint8_t *kv_fp8, const float *attn_sink,
                                 const int32_t *topk_idxs, const int32_t *topk_length, float softmax_scale,
                                 void *o, int64_t B, int64_t S, int64_t H, int64_t T, int64_t K, int num_splits,
                                 void *workspace, size_t workspace_bytes, sa_stream_t stream);

/* sparse_attn over two kv sources ("DeepSeek V4 源码剖析, 第5章" §5.6: the
 * SM100 decode kernel keeps separate tensor maps extra_kv_nope /
 * extra_kv_rope beside kv_nope / kv_rope; §5.13: extra_topk_length beside
 * topk_length among the scheduler metadata's inputs).  The pages do not give
 * the addressing; reading taken here: the extra source extra_kv [B, T2, D]
 * (bf16, device, 16-byte aligned, in the main kv's format) has its own slot
 * list extra_topk_idxs [B, S, K2] (int32, -1 or any index outside [0, T2) =
 * invalid) and optional per-token length extra_topk_length [B, S] (NULL:
 * every extra slot may count; same clamping as topk_length).  A token
 * attends over its K main slots followed by its K2 extra slots in ONE
 * softmax, with the sink counted once, so the result equals
 * sa_sparse_attn_fwd_topk_length over the concatenated rows and slot lists.
 * K >= 0, K2 >= 0, K + K2 >= 1; with K = 0, kv and topk_idxs may be NULL,
 * with K2 = 0 the extra arguments may be NULL.  Splits, workspace and launch
 * count are those of K + K2 slots: size the workspace with
 * sa_sparse_attn_workspace_size(B, S, H, D, K + K2, num_splits).  Errors as
 * sa_sparse_attn_fwd_topk_length; also SA_ERR_SHAPE when
 * B*T (rounded up to even) + B*T2 >= 2^31. */
sa_status sa_sparse_attn_fwd_extra(const void *q, const void *kv, const float *attn_sink, const int32_t *topk_idxs,
                                   const int32_t *topk_length, const void *extra_kv, const int32_t *extra_topk_idxs,
                                   const int32_t *extra_topk_length, float softmax_scale, void *o, int64_t B,
                                   int64_t S, int64_t H, int64_t D, int64_t T, int64_t K, int64_t T2, int64_t K2,
                                   int num_splits, void *workspace, size_t workspace_bytes, sa_stream_t stream);

/* The same over FP8 kv caches (both sources in the 584-byte row format of
 * sa_sparse_attn_fwd_fp8), D = 512. */
sa_status sa_sparse_attn_fwd_fp8_extra(const void *q, const uint8_t *kv_fp8, const float *attn_sink,
                                       const int32_t *topk_idxs, const int32_t *topk_length,
                                       const uint8_t *extra_kv_fp8, const int32_t *extra_topk_idxs,
                                       const int32_t *extra_topk_length, float softmax_scale, void *o, int64_t B,
                                       int64_t S, int64_t H, int64_t T, int64_t K, int64_t T2, int64_t K2,
                                       int num_splits, void *workspace, size_t workspace_bytes,
                                       sa_stream_t stream);

/* Kernels one sa_sparse_attn_fwd_fp8 call enqueues (1 or 2); 0 on
 * unsupported sizes. */
int sa_sparse_attn_fp8_launch_count(int64_t B, int64_t S, int64_t H, int64_t K, int num_splits);

/* Allocation-free variant of sa_sparse_attn_fwd_splits, for callers that
 * cannot supply device memory: a plain C host program with no device
 * allocator, or a serving loop that plans all memory up front and must not
 * call cudaMalloc on its hot path (it can block and can fail under memory
 * pressure).  The split-KV workspace is a 32 MiB array inside the library
 * (held on every GPU that uses the library, until the process exits); the
 * caller passes only inputs and outputs, with the same meaning, layout and
 * validation as sa_sparse_attn_fwd_splits.  Returns SA_ERR_WORKSPACE when
 * the planned workspace exceeds 32 MiB.  The first call on a device looks
 * up the array's address (make it before any stream capture).  All calls on
 * a device share the array: calls that overlap on the GPU race and must be
 * serialised by the caller.  The pages have no counterpart of this entry
 * point; it exists for callers that cannot allocate. */
sa_status sa_sparse_attn_fwd_static_ws(const void *q, const void *kv, const float *attn_sink,
                                       const int32_t *topk_idxs, float softmax_scale, void *o,
                                       int64_t B, int64_t S, int64_t H, int64_t D, int64_t T,
                                       int64_t K, int num_splits, sa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* bit-packed top-k mask                                                    */
/* ------------------------------------------------------------------------ */

/* Host-only.  out_shape = (batch, rows, words) with
 *   tile_m = 128 if max_query_len <= 128 else 256,
 *   rows   = ceil(max_query_len / tile_m) * tile_m,
 *   words  = round_up(ceil(max_key_len / 32) + (reserve ? 1 : 0), 4),
 * so every row is a whole number of 16-byte vectors (vLLM PR 52217 page,
 * `_topk_mask_shape`).  SA_ERR_INVALID_ARG on negative sizes or NULL. */
sa_status sa_topk_mask_shape(int64_t batch, int64_t max_query_len, int64_t max_key_len,
                             int reserve_key_starts_word, int64_t out_shape[3]);

/* Scatters each request's top-k rows into the mask.
 *   topk        int32 [topk_rows, K]: rows cu_q_lens[b] .. cu_q_lens[b+1]-1
 *               belong to request b (query q of b is row cu_q_lens[b] + q)
 *   cu_q_lens   int32 [B+1] prefix sums of the per-request query counts
 *   key_starts  int32 [B] or NULL (NULL: no reserved word)
 *   mask        uint32 [mask_shape], 16-byte aligned; mask_shape must equal
 *               sa_topk_mask_shape(B, max_q_len, max_key_len, key_starts!=NULL)
 *   mask_shape  HOST array of 3 int64.
 * For each live row (b, q) with q < min(q_len_b, max_q_len) and source row
 * < topk_rows: words [0, ceil(max_key_len/32)) are overwritten with the OR of
 * (1u << (k & 31)) into word k >> 5 over the row's indices with
 * 0 <= k < max_key_len.  If key_starts != NULL, word words-1 of row (b, 0)
 * receives key_starts[b] (bit pattern) for every b.  Nothing else is written:
 * padding words and rows past each request's query count keep their contents. */
sa_status sa_build_topk_mask(const int32_t *topk, int64_t topk_rows, const int32_t *cu_q_lens,
                             int64_t B, int64_t max_q_len, int64_t max_key_len, int64_t K,
                             const int32_t *key_starts, uint32_t *mask,
                             const int64_t mask_shape[3], sa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* consumer of the mask: dense attention over the admitted keys              */
/* ------------------------------------------------------------------------ */

/* Workspace bytes for sa_masked_dense_attn_fwd with these sizes and split
 * count (<= 0: the planned count); 0 when one split needs none or the sizes
 * are unsupported.  The splits divide the T keys of each query. */
size_t sa_masked_dense_attn_workspace_size(int64_t B, int64_t S, int64_t H, int64_t D, int64_t T,
                                           int num_splits);

/* Kernels one sa_masked_dense_attn_fwd call enqueues (1 or 2), 0 on
 * unsupported sizes. */
int sa_masked_dense_attn_launch_count(int64_t B, int64_t S, int64_t H, int64_t D, int64_t T,
                                      int num_splits);

/* Attention of every query token over the keys its mask row admits: the
 * consumer side of the bit-packed mask (`dense_mask_mod` and, with
 * key_start_word = 1, `offset_dense_mask_mod` on the vLLM PR 48770 page;
 * the 16-byte row contract of the PR 52217 page).
 *   q, kv, attn_sink, o, B, S, H, D, T, softmax_scale: as in
 *               sa_sparse_attn_fwd (kv[b] holds the T keys of request b).
 *   mask        uint32 [B, mask_rows, mask_words] device, 16-byte aligned,
 *               mask_words a multiple of 4 (the layout sa_topk_mask_shape
 *               gives), mask_rows >= S.  Query s of request b reads row
 *               mask[b, s, :].
 *   key_start_word  0: key t tests bit t; 1: key t tests bit t + ks_b where
 *               ks_b = (int32) mask[b, 0, mask_words - 1], the reserved word
 *               sa_build_topk_mask writes (T keys of a context chunk that
 *               starts at absolute position ks_b).
 * Key t of request b is admitted iff 0 <= p < 32 * (mask_words -
 * key_start_word) and bit p & 31 of word p >> 5 of the row is set, p = t
 * (+ ks_b): with key_start_word the last word of every row is the reserved
 * column and admits nothing.  Padding words past the builder's live words
 * are read as key bits if p reaches them (T + ks_b past the max_key_len the
 * mask was built for); the window form's key_ends bounds them.  The result
 * is sa_sparse_attn_fwd's with the admitted keys as the token's slot list.
 * kv must hold finite values: for D <= 256 the G = 128 / H query tokens of
 * a group share dense key tiles, and the keys a row does not admit enter
 * its P.V with weight 0.
 * num_splits: 1..64 key ranges per token (<= 0: planned); workspace as in
 * sa_sparse_attn_fwd_splits, sized by sa_masked_dense_attn_workspace_size.
 * Errors as sa_sparse_attn_fwd_splits, plus SA_ERR_SHAPE for mask_rows < S,
 * mask_words < 1 or not a multiple of 4, and SA_ERR_ALIGNMENT for a mask
 * that is not 16-byte aligned. */
sa_status sa_masked_dense_attn_fwd(const void *q, const void *kv, const float *attn_sink,
                                   const uint32_t *mask, int64_t mask_rows, int64_t mask_words,
                                   int key_start_word, float softmax_scale, void *o, int64_t B, int64_t S,
                                   int64_t H, int64_t D, int64_t T, int num_splits, void *workspace,
                                   size_t workspace_bytes, sa_stream_t stream);

/* Builds one window of the mask: row i of `mask` is query q0 + i of each
 * request (i < q_rows), so a mask larger than a memory budget can be built
 * and consumed a window at a time (the chunked fallback above the 64 MiB
 * global-mask cap, vLLM PR 48770 page).  key_ends: int32 [B] device or NULL;
 * request b's rows get only the words below its live key end
 * min(max(key_ends[b], 0), max_key_len) written, and indices at or past it are
 * dropped -- the build stops at each row's live end (vLLM PR 56628 page), so
 * its cost follows the live context, not the mask width.  mask_shape must
 * equal sa_topk_mask_shape(B, q_rows, max_key_len, key_starts != NULL); the
 * reserved key_start word goes to row 0 of each request.  Everything not
 * written keeps its contents.  Other arguments and errors as
 * sa_build_topk_mask, which is this call with q0 = 0, q_rows = max_q_len and
 * key_ends = NULL. */
sa_status sa_build_topk_mask_window(const int32_t *topk, int64_t topk_rows, const int32_t *cu_q_lens, int64_t B,
                                    int64_t q0, int64_t q_rows, int64_t max_key_len, int64_t K,
                                    const int32_t *key_starts, const int32_t *key_ends, uint32_t *mask,
                                    const int64_t mask_shape[3], sa_stream_t stream);

/* sa_masked_dense_attn_fwd for the query rows q0 .. q0 + S - 1 of each
 * request: q and o are [B, S_total, H, D] (S_total >= q0 + S), mask row s is
 * query q0 + s (a window from sa_build_topk_mask_window), and key_ends (int32
 * [B] device, or NULL) admits no key whose mask position (t, plus key_start
 * with key_start_word) is at or past request b's live end.  Workspace as
 * sa_masked_dense_attn_workspace_size(B, S, H, D, T, num_splits).  Errors as
 * sa_masked_dense_attn_fwd, plus SA_ERR_SHAPE for q0 + S > S_total. */
sa_status sa_masked_dense_attn_fwd_window(const void *q, const void *kv, const float *attn_sink,
                                          const uint32_t *mask, int64_t mask_rows, int64_t mask_words,
                                          int key_start_word, const int32_t *key_ends, float softmax_scale, void *o,
                                          int64_t B, int64_t S_total, int64_t q0, int64_t S, int64_t H, int64_t D,
                                          int64_t T, int num_splits, void *workspace, size_t workspace_bytes,
                                          sa_stream_t stream);

/* Host-only.  Query rows per window so that one window's mask,
 * sa_topk_mask_shape(batch, rows, max_key_len, reserve) words of 4 bytes,
 * fits cap_bytes (<= 0: 64 MiB, the pages' global-mask cap): max_query_len
 * when the whole mask fits, else the largest multiple of 256 (or 128) that
 * fits; 0 if not even 128 rows fit. */
int64_t sa_topk_mask_chunk_rows(int64_t batch, int64_t max_query_len, int64_t max_key_len,
                                int reserve_key_starts_word, int64_t cap_bytes);

/* Attention of every query over the keys its top-k row selects, through the
 * bit-packed mask: for each window of sa_topk_mask_chunk_rows(...) query
 * rows, sa_build_topk_mask_window into mask_buf, then
 * sa_masked_dense_attn_fwd_window, all enqueued on `stream`.  One window
 * when the whole mask fits cap_bytes (the global mask), several otherwise
 * (the chunked fallback).  q, o: bf16 [B, max_q_len, H, D]; kv: bf16
 * [B, T, D], key t of kv[b] at mask position t + key_starts[b] (0 without
 * key_starts); topk, cu_q_lens, key_starts, key_ends as in
 * sa_build_topk_mask_window.  mask_buf: device, 16-byte aligned, at least
 * one window's mask; workspace: sa_topk_masked_attn_workspace_size bytes.
 * Rows q >= q_len_b of o are left unspecified.  Returns SA_ERR_SHAPE when no
 * window fits the cap, SA_ERR_WORKSPACE when mask_buf or the workspace is too
 * small, else the first error of the calls it makes. */
sa_status sa_topk_masked_attn_fwd(const void *q, const void *kv, const float *attn_sink, const int32_t *topk,
                                  int64_t topk_rows, const int32_t *cu_q_lens, const int32_t *key_starts,
                                  const int32_t *key_ends, float softmax_scale, void *o, int64_t B,
                                  int64_t max_q_len, int64_t H, int64_t D, int64_t T, int64_t max_key_len, int64_t K,
                                  int64_t cap_bytes, uint32_t *mask_buf, size_t mask_buf_bytes, void *workspace,
                                  size_t workspace_bytes, sa_stream_t stream);

/* Workspace bytes sa_topk_masked_attn_fwd needs for these sizes and cap. */
size_t sa_topk_masked_attn_workspace_size(int64_t B, int64_t max_q_len, int64_t H, int64_t D, int64_t T,
                                          int64_t max_key_len, int reserve_key_starts_word, int64_t cap_bytes);

/* ------------------------------------------------------------------------ */
/* diagnostics                                                              */
/* ------------------------------------------------------------------------ */

/* Every mbarrier wait inside the kernels is bounded (about 0.1 s of SM
 * clock); a wait that runs out records a nonzero code in a device-side word
 * and its kernel returns early (its output is then undefined).  Once the word
 * is nonzero, every wait of every kernel on the device gives up within about
 * 1024 polls, so a failing launch drains quickly; the word stays set (and
 * later launches fail fast) until it is cleared here.  This call synchronises
 * the current device, returns that word (0 = no failure since the last
 * clear) and clears it if `clear`.  Returns -1 if the word cannot be read. */
int sa_device_error(int clear);

/* Self-test of that mechanism, without any fault: launches one warp that
 * waits, with the kernels' own bounded-wait routine and a limit of
 * `max_cycles` SM clock cycles (1 .. 2^28, i.e. at most ~0.13 s), on a
 * barrier phase that nothing completes.  Synchronises the current device and
 * returns the code the wait recorded (1 = wait timed out, the expected
 * result), leaving the word clear; -1 on a bad argument or a CUDA error.
 * Any earlier code is cleared first.  The pages have no counterpart of this
 * call: it exists to test failure detection on a shared GPU. */
int sa_selftest_wait_timeout(long long max_cycles);

/* Self-test of the fast drain, without any fault: launches `ctas` CTAs
 * (1 .. 1024) of one waiting warp each.  CTA 0 waits on a barrier phase that
 * nothing completes with a limit of `first_cycles` (1 .. 2^28); every other
 * CTA waits likewise with the kernels' full limit (~0.1 s), and must give up
 * as soon as CTA 0 has recorded its timeout.  Writes the elapsed time of the
 * launch in milliseconds (CUDA events) to *elapsed_ms, synchronises the
 * current device and returns the recorded code (1 = timed out, expected),
 * leaving the word clear; -1 on a bad argument or a CUDA error.  The pages
 * have no counterpart of this call. */
int sa_selftest_wait_drain(int ctas, long long first_cycles, float *elapsed_ms);

/* Random-row gather probe: the rate at which the SMs can pull rows picked at
 * random out of a table in device memory, which bounds the kv gather of
 * sparse_attn ("第5章" §5.6: one kv row per valid slot, from anywhere in the
 * cache).  The pages have no counterpart; the call measures the hardware.
 *   table       device, `rows` rows of `row_bytes` bytes (16-byte aligned,
 *               row_bytes a multiple of 16), 1 <= rows <= 2^31 - 1;
 *   part_bytes  bytes copied from the start of each picked row: a power of
 *               two in [16, 32768], at most row_bytes;
 *   idx         device int32 [ctas * tiles * (32768 / part_bytes)]: the rows,
 *               in the order CTA c copies them (c-major); a value outside
 *               [0, rows) copies row 0;
 *   ctas        1 .. 65535 CTAs of 256 threads, one per SM at most (197 KB of
 *               shared memory each); CTA c copies `tiles` (1 .. 2^20) tiles of
 *               32 KB into shared memory through a six-stage ring and
 *               discards them.
 * Enqueued on `stream`; the caller times it (the bytes moved are
 * ctas * tiles * 32768) and flushes L2 first for an HBM figure.  Returns
 * SA_ERR_INVALID_ARG / SA_ERR_ALIGNMENT on bad arguments before launching,
 * SA_ERR_CUDA if the launch fails.  A wait that runs out sets the device
 * error word (sa_device_error). */
sa_status sa_probe_row_gather(const void *table, int64_t rows, int64_t row_bytes, int64_t part_bytes,
                              const int32_t *idx, int64_t ctas, int64_t tiles, sa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SA_H_ */
