/*
 * CPU ORACLE -- test infrastructure only.
 *
 * A plain, slow, double-precision restatement of what top-k sparse attention
 * and the bit-packed top-k mask compute.  Only the test suite, the smoke check
 * and the CPU-baseline leg of the benchmark may load this library; the product
 * path (the CUDA library) never calls it and shares no code with it.
 *
 * Sources, cited by page title and section:
 *   [V4-5.2]  "DeepSeek V4 源码剖析, 第5章 sparse_attn 与 FlashMLA", §5.2
 *             (interface semantics, per-(b,s,h) pseudocode) and §5.1 (shapes,
 *             -1 marks an invalid slot, softmax_scale = head_dim^-0.5).
 *   [V4-5.5]  same chapter, §5.5: the sink enters the softmax denominator only;
 *             sink = +inf zeroes every real weight, sink = -inf means no sink.
 *   [MASK-SHAPE] vLLM PR 52217 page ("Sparse MLA mask 向量化 128-bit 加载"),
 *             key source excerpt `_topk_mask_shape`, `_build_topk_mask`, and the
 *             two tests (129 keys -> 8 words; bits 0 and 128 in words 0 and 4).
 *   [MASK-BITS] vLLM PR 48770 page (masked MHA for sparse-MLA prefill), source
 *             excerpt `dense_mask_mod` / `offset_dense_mask_mod`: word kv>>5,
 *             bit kv&31, LSB first; the last word of row q=0 holds key_start.
 *   [MASK-CAP] same page, review notes: the global mask grows with batch x
 *             query length x key length, so above a 64 MiB cap the chunked
 *             mask path takes over.
 *   [MASK-END] vLLM PR 56628 page: the strided mask kernel stops at each
 *             row's live end, so its cost follows the live context rather
 *             than the workspace width, and leaves the columns past the end
 *             untouched.
 *   [V4-5.3]  same chapter, §5.3: the MODEL1 (V4) constants of FlashMLA --
 *             head dim 512 = 448 "nope" dims + 64 RoPE dims, FP8 quantisation
 *             tiles of 64 dims, 8 scales per token (7 used), V carries the
 *             RoPE dims too; §5.6: the nope part is stored quantised, the RoPE
 *             part stays bf16, and the kernel dequantises what it gathers.
 *             The same §5.6 lists the SM100 decode kernel's separate tensor
 *             maps for an extra kv source (extra_kv_nope / extra_kv_rope)
 *             beside kv_nope / kv_rope, and §5.13 names an extra_topk_length
 *             beside topk_length among the scheduler metadata's inputs.
 *
 * Readings taken where the pages are silent (each one is tested):
 *   R1 a slot is valid iff 0 <= idx < T (the pages only define -1).
 *   R3 all slots invalid, finite sink -> o = 0 (weights are [0..0, 1]).
 *   R4 sink = +inf -> o = 0.      R6 sink = -inf and no valid slot -> o = 0.
 *   R8 the scale multiplies q.k only; the sink is a raw logit.
 *   R14 live mask words [0, ceil(max_key_len/32)) are cleared then OR-ed;
 *   R15 padding words and rows q >= q_len are never written;
 *   R16 the reserved word of row 0 holds the raw bits of key_starts[b].
 *   R19 a per-token topk_length keeps only the slots j < clamp(len, 0, K).
 *   R21 the mask consumer admits key t iff bit t (+ key_start) of the row is
 *       set, within the row's 32 * W positions; in the offset form the last
 *       word of a row is the reserved key_start column and admits nothing.
 *   R22 FP8 row byte order: 448 E4M3 codes, 64 bf16 RoPE dims, 8 E8M0 scales.
 *   R24 a mask window holds query rows q0.. of each request; a live key end
 *       bounds both the words written and the keys the consumer admits.
 *   R25 a second kv source (extra_kv [B,T2,D], same format) comes with its own
 *       slot list [B,S,K2] and optional per-token length; a token's softmax
 *       runs over its K main slots and its K2 extra slots together (main
 *       first), the sink added once.
 *
 * Inputs are bf16 bit patterns (uint16) as stored on the device; each value
 * is widened exactly to double before any arithmetic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1

static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* FP8 KV rows, [V4-5.3] / [V4-5.6]                                          */
/* ------------------------------------------------------------------------ */
/* Reading R22 (the pages give the parts and their sizes, not their order):
 * one kv row is 584 bytes,
 *   [0, 448)    dims 0..447 as FP8 E4M3 codes (OCP 8-bit floating point:
 *               1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 *               infinities; S.1111.111 is NaN; exponent 0 is subnormal),
 *   [448, 576)  dims 448..511 as bf16, little-endian,
 *   [576, 584)  one scale byte per 64-dim tile of the nope dims (7 used, the
 *               8th is padding), each an E8M0 exponent: 2^(byte - 127), 255 = NaN.
 * value(d) = e4m3(code_d) * 2^(scale[d / 64] - 127) for d < 448, else bf16. */
#define FP8_ROW_BYTES 584
#define FP8_NOPE 448
#define FP8_TILE 64
#define FP8_ROPE_OFF 448
#define FP8_SCALE_OFF 576
#define FP8_DIM 512

double oracle_e4m3_to_double(uint8_t c) {
    const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6); /* subnormal: 0.mmm * 2^(1-7) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

double oracle_e8m0_to_double(uint8_t s) {
    if (s == 255) return NAN;
    return ldexp(1.0, (int)s - 127);
}

/* one 584-byte row -> 512 doubles */
static void fp8_row_decode(const uint8_t *row, double *out) {
    for (int d = 0; d < FP8_NOPE; ++d)
        out[d] = oracle_e4m3_to_double(row[d]) * oracle_e8m0_to_double(row[FP8_SCALE_OFF + d / FP8_TILE]);
    for (int d = FP8_NOPE; d < FP8_DIM; ++d) {
        const uint8_t *p = row + FP8_ROPE_OFF + 2 * (d - FP8_NOPE);
        out[d] = bf16_to_double((uint16_t)(p[0] | (p[1] << 8)));
    }
}

int oracle_decode_kv_fp8(const uint8_t *kv8, int64_t rows, double *out /* [rows, 512] */) {
    if (rows < 0) return ORACLE_EINVAL;
    for (int64_t r = 0; r < rows; ++r) fp8_row_decode(kv8 + r * FP8_ROW_BYTES, out + r * FP8_DIM);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* sparse_attn, [V4-5.2]                                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q, *kv;
    const uint8_t *kv8;    /* FP8 rows of 584 bytes instead of bf16 kv (D = 512), or NULL */
    const float *sink;
    const int32_t *idx;
    const int32_t *topk_len; /* [B*S] valid-prefix length per query token, or NULL */
    /* the extra source (R25): kv2 / kv8_2 [B,T2,.] in the format of the main
     * one, idx2 [B,S,K2], topk_len2 [B*S] or NULL; K2 = 0 without it */
    const uint16_t *kv2;
    const uint8_t *kv8_2;
    const int32_t *idx2;
    const int32_t *topk_len2;
    int64_t T2, K2;
    double scale;
    double *o;
    int64_t B, S, H, D, T, K;
    const int64_t *tokens; /* flat b*S+s token ids to evaluate */
    int64_t ntok;
    int64_t next; /* work counter, guarded by mu */
    pthread_mutex_t mu;
} attn_job;

/* kv row `row` (= b*T + t) of source `src` (0 main, 1 extra) as D doubles,
 * from bf16 or from the FP8 layout */
static void load_kv_row(const attn_job *J, int src, int64_t row, double *out) {
    const uint8_t *k8 = src ? J->kv8_2 : J->kv8;
    if (k8) {
        fp8_row_decode(k8 + row * FP8_ROW_BYTES, out);
        return;
    }
    const uint16_t *kr = (src ? J->kv2 : J->kv) + row * J->D;
    for (int64_t d = 0; d < J->D; ++d) out[d] = bf16_to_double(kr[d]);
}

/* One query token (b, s), every head h:
 *   logits_j = scale * q[b,s,h,:] . kv[b, idx_j, :]   for valid slots j,
 *   a slot j being valid when 0 <= idx_j < T and, if a per-token topk_length
 *   is given, j < min(max(topk_length[b,s], 0), K) (the "topk length per
 *   sequence" variant of the FlashMLA kernels, [V4-5.3]);
 *   -inf for invalid ones; the sink logit attn_sink[h] is appended; softmax
 *   over the K+1 values; o = sum_{j<K} w_j * kv[b, idx_j, :] (the sink's
 *   weight is dropped).  [V4-5.2], [V4-5.5] */
static int64_t clamp_len(const int32_t *lens, int64_t tok, int64_t K) {
    if (lens == NULL) return K;
    int64_t len = lens[tok];
    if (len < 0) len = 0;
    if (len > K) len = K;
    return len;
}

/* One query token (b, s), every head h:
 *   logits_j = scale * q[b,s,h,:] . kv[b, idx_j, :]   for valid slots j,
 *   a slot j being valid when 0 <= idx_j < T and, if a per-token topk_length
 *   is given, j < min(max(topk_length[b,s], 0), K) (the "topk length per
 *   sequence" variant of the FlashMLA kernels, [V4-5.3]);
 *   -inf for invalid ones; the sink logit attn_sink[h] is appended; softmax
 *   over the K+1 values; o = sum_{j<K} w_j * kv[b, idx_j, :] (the sink's
 *   weight is dropped).  [V4-5.2], [V4-5.5]
 * With an extra source (R25) the token's slots are its K main slots followed
 * by its K2 extra slots, slot K + j gathering extra_kv[b, idx2_j, :] under the
 * same validity rule with T2 and the extra length; one softmax covers all
 * K + K2 slots and the sink. */
static void attn_one_token(const attn_job *J, int64_t tok, double *out /* [H,D] */) {
    const int64_t b = tok / J->S, s = tok % J->S;
    const int64_t H = J->H, D = J->D, K = J->K, K2 = J->K2, N = J->K + J->K2;
    const int32_t *idx = J->idx + (b * J->S + s) * K;
    const int32_t *idx2 = K2 > 0 ? J->idx2 + (b * J->S + s) * K2 : NULL;
    const int64_t len = clamp_len(J->topk_len, b * J->S + s, K);
    const int64_t len2 = clamp_len(J->topk_len2, b * J->S + s, K2);
    double *logit = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    char *valid = (char *)malloc((size_t)(N > 0 ? N : 1));
    double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
    /* the gathered rows of the token's valid slots, widened once (shared by
     * every head: kv is one head shared by all query heads) */
    double *krows = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * (size_t)D);
    for (int64_t j = 0; j < N; ++j) {
        const int src = j >= K;
        const int64_t t = src ? idx2[j - K] : idx[j];
        const int64_t Tsrc = src ? J->T2 : J->T;
        valid[j] = (src ? (j - K < len2) : (j < len)) && t >= 0 && t < Tsrc; /* R1, R19 */
        if (valid[j]) load_kv_row(J, src, b * Tsrc + t, krows + j * D);
    }
    for (int64_t h = 0; h < H; ++h) {
        double *orow = out + h * D;
        for (int64_t d = 0; d < D; ++d) orow[d] = 0.0;
        const uint16_t *qh = J->q + ((b * J->S + s) * H + h) * D;
        for (int64_t d = 0; d < D; ++d) qrow[d] = bf16_to_double(qh[d]);
        /* logits of the slots, -inf where the slot is invalid (R1) */
        for (int64_t j = 0; j < N; ++j) {
            if (!valid[j]) {
                logit[j] = -INFINITY;
                continue;
            }
            const double *krow = krows + j * D;
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += qrow[d] * krow[d];
            logit[j] = dot * J->scale; /* R8: scale on q.k only */
        }
        const double sink = (double)J->sink[h];
        /* softmax over [logits..., sink] */
        double m = sink;
        for (int64_t j = 0; j < N; ++j)
            if (logit[j] > m) m = logit[j];
        if (isnan(sink)) { /* R7: NaN propagates */
            for (int64_t d = 0; d < D; ++d) orow[d] = NAN;
            continue;
        }
        if (m == INFINITY && sink == INFINITY) continue; /* R4: o = 0 */
        if (m == -INFINITY) continue;                    /* R6: o = 0 */
        double denom = exp(sink - m);
        for (int64_t j = 0; j < N; ++j) denom += exp(logit[j] - m);
        for (int64_t j = 0; j < N; ++j) {
            if (logit[j] == -INFINITY) continue; /* weight exactly 0 */
            const double w = exp(logit[j] - m) / denom;
            const double *krow = krows + j * D;
            for (int64_t d = 0; d < D; ++d) orow[d] += w * krow[d];
        }
    }
    free(logit);
    free(valid);
    free(qrow);
    free(krows);
}

static void *attn_worker(void *arg) {
    attn_job *J = (attn_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int64_t i = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (i >= J->ntok) break;
        attn_one_token(J, J->tokens[i], J->o + i * J->H * J->D);
    }
    return NULL;
}

static int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

typedef struct {
    const uint16_t *kv2;
    const uint8_t *kv8_2;
    const int32_t *idx2, *len2;
    int64_t T2, K2;
} extra_src;

static int run_attn_job_x(const uint16_t *q, const uint16_t *kv, const uint8_t *kv8, const float *attn_sink,
                          const int32_t *topk_idxs, const int32_t *topk_length, const extra_src *X,
                          double softmax_scale, int64_t B, int64_t S, int64_t H, int64_t D, int64_t T, int64_t K,
                          const int64_t *tokens, int64_t ntok, double *o, int nthreads) {
    if (B < 0 || S < 0 || H <= 0 || D <= 0 || T < 0 || K < 0 || ntok < 0) return ORACLE_EINVAL;
    if (X && (X->K2 < 0 || X->T2 < 0 || (X->K2 > 0 && (X->idx2 == NULL || (X->kv2 == NULL && X->kv8_2 == NULL)))))
        return ORACLE_EINVAL;
    for (int64_t i = 0; i < ntok; ++i)
        if (tokens[i] < 0 || tokens[i] >= B * S) return ORACLE_EINVAL;
    attn_job J;
    J.q = q; J.kv = kv; J.kv8 = kv8; J.sink = attn_sink; J.idx = topk_idxs; J.topk_len = topk_length;
    J.kv2 = X ? X->kv2 : NULL; J.kv8_2 = X ? X->kv8_2 : NULL; J.idx2 = X ? X->idx2 : NULL;
    J.topk_len2 = X ? X->len2 : NULL; J.T2 = X ? X->T2 : 0; J.K2 = X ? X->K2 : 0;
    J.scale = softmax_scale;
    J.o = o; J.B = B; J.S = S; J.H = H; J.D = D; J.T = T; J.K = K;
    J.tokens = tokens; J.ntok = ntok; J.next = 0;
    pthread_mutex_init(&J.mu, NULL);
    int nt = resolve_threads(nthreads);
    if (nt > ntok) nt = ntok > 0 ? (int)ntok : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, attn_worker, &J);
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
    return ORACLE_OK;
}

static int run_attn_job(const uint16_t *q, const uint16_t *kv, const uint8_t *kv8, const float *attn_sink,
                        const int32_t *topk_idxs, const int32_t *topk_length, double softmax_scale, int64_t B,
                        int64_t S, int64_t H, int64_t D, int64_t T, int64_t K, const int64_t *tokens, int64_t ntok,
                        double *o, int nthreads) {
    return run_attn_job_x(q, kv, kv8, attn_sink, topk_idxs, topk_length, NULL, softmax_scale, B, S, H, D, T, K,
                          tokens, ntok, o, nthreads);
}

/* Evaluates the tokens listed in `tokens` (flat b*S+s ids); o is [ntok,H,D].
 * topk_length: [B*S] int32 or NULL (every slot may count). */
int oracle_sparse_attn_tokens_len(const uint16_t *q, const uint16_t *kv, const float *attn_sink,
                                  const int32_t *topk_idxs, const int32_t *topk_length,
                                  double softmax_scale, int64_t B, int64_t S, int64_t H, int64_t D,
                                  int64_t T, int64_t K, const int64_t *tokens, int64_t ntok, double *o,
                                  int nthreads) {
    return run_attn_job(q, kv, NULL, attn_sink, topk_idxs, topk_length, softmax_scale, B, S, H, D, T, K, tokens,
                        ntok, o, nthreads);
}

/* The same attention over an FP8 kv cache (rows of 584 bytes, R22): every
 * gathered row is decoded to its 512 exact values first; q and o keep D = 512. */
int oracle_sparse_attn_fp8_tokens(const uint16_t *q, const uint8_t *kv8, const float *attn_sink,
                                  const int32_t *topk_idxs, const int32_t *topk_length, double softmax_scale,
                                  int64_t B, int64_t S, int64_t H, int64_t T, int64_t K, const int64_t *tokens,
                                  int64_t ntok, double *o, int nthreads) {
    if (kv8 == NULL) return ORACLE_EINVAL;
    return run_attn_job(q, NULL, kv8, attn_sink, topk_idxs, topk_length, softmax_scale, B, S, H, FP8_DIM, T, K,
                        tokens, ntok, o, nthreads);
}

/* With the extra kv source (R25): extra_kv bf16 [B,T2,D] (or, for the FP8
 * variant, 584-byte rows), extra_idxs [B,S,K2], extra_length [B*S] or NULL. */
int oracle_sparse_attn_extra_tokens(const uint16_t *q, const uint16_t *kv, const float *attn_sink,
                                    const int32_t *topk_idxs, const int32_t *topk_length, const uint16_t *extra_kv,
                                    const int32_t *extra_idxs, const int32_t *extra_length, double softmax_scale,
                                    int64_t B, int64_t S, int64_t H, int64_t D, int64_t T, int64_t K, int64_t T2,
                                    int64_t K2, const int64_t *tokens, int64_t ntok, double *o, int nthreads) {
    const extra_src X = {extra_kv, NULL, extra_idxs, extra_length, T2, K2};
    return run_attn_job_x(q, kv, NULL, attn_sink, topk_idxs, topk_length, &X, softmax_scale, B, S, H, D, T, K,
                          tokens, ntok, o, nthreads);
}

int oracle_sparse_attn_fp8_extra_tokens(const uint16_t *q, const uint8_t *kv8, const float *attn_sink,
                                        const int32_t *topk_idxs, const int32_t *topk_length,
                                        const uint8_t *extra_kv8, const int32_t *extra_idxs,
                                        const int32_t *extra_length, double softmax_scale, int64_t B, int64_t S,
                                        int64_t H, int64_t T, int64_t K, int64_t T2, int64_t K2,
                                        const int64_t *tokens, int64_t ntok, double *o, int nthreads) {
    if (kv8 == NULL) return ORACLE_EINVAL;
    const extra_src X = {NULL, extra_kv8, extra_idxs, extra_length, T2, K2};
    return run_attn_job_x(q, NULL, kv8, attn_sink, topk_idxs, topk_length, &X, softmax_scale, B, S, H, FP8_DIM, T,
                          K, tokens, ntok, o, nthreads);
}

int oracle_sparse_attn_tokens(const uint16_t *q, const uint16_t *kv, const float *attn_sink,
                              const int32_t *topk_idxs, double softmax_scale, int64_t B,
                              int64_t S, int64_t H, int64_t D, int64_t T, int64_t K,
                              const int64_t *tokens, int64_t ntok, double *o, int nthreads) {
    return oracle_sparse_attn_tokens_len(q, kv, attn_sink, topk_idxs, NULL, softmax_scale, B, S, H, D, T,
                                         K, tokens, ntok, o, nthreads);
}

/* Every token; o is [B,S,H,D]. */
int oracle_sparse_attn(const uint16_t *q, const uint16_t *kv, const float *attn_sink,
                       const int32_t *topk_idxs, double softmax_scale, int64_t B, int64_t S,
                       int64_t H, int64_t D, int64_t T, int64_t K, double *o, int nthreads) {
    int64_t n = B * S;
    int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    for (int64_t i = 0; i < n; ++i) tok[i] = i;
    int rc = oracle_sparse_attn_tokens(q, kv, attn_sink, topk_idxs, softmax_scale, B, S, H, D,
                                       T, K, tok, n, o, nthreads);
    free(tok);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Dense attention under a bit-packed key mask (the consumer side of the     */
/* mask, [MASK-BITS]): key t of kv[b] is admitted for query (b,s) iff bit    */
/* ((t + key_offset[b]) & 31) of word ((t + key_offset[b]) >> 5) in row      */
/* mask[b, s, :] is set.  Same softmax-with-sink as above over the admitted  */
/* keys.  key_offset may be NULL (all zero, `dense_mask_mod`); a non-NULL    */
/* offset is the chunked-context reading (`offset_dense_mask_mod`), whose    */
/* key start sits in the last word of row 0 (R16): with an offset, the last  */
/* word of every row is that reserved column, never a key word (R21).        */
/* key_ends (or NULL): a key at or past request b's live end key_ends[b]     */
/* (in mask positions, i.e. after the offset) is never admitted (R24).       */
/* ------------------------------------------------------------------------ */
int oracle_masked_dense_attn(const uint16_t *q, const uint16_t *kv, const float *attn_sink,
                             const uint32_t *mask, int64_t mask_rows, int64_t mask_words,
                             const int64_t *key_offset, const int64_t *key_ends, double softmax_scale,
                             int64_t B, int64_t S, int64_t H, int64_t D, int64_t T, double *o) {
    if (B < 0 || S < 0 || H <= 0 || D <= 0 || T < 0 || mask_rows < S || mask_words < 0)
        return ORACLE_EINVAL;
    double *logit = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    for (int64_t b = 0; b < B; ++b) {
        const int64_t off = key_offset ? key_offset[b] : 0;
        const int64_t key_words = key_offset ? mask_words - 1 : mask_words;
        for (int64_t s = 0; s < S; ++s) {
            const uint32_t *row = mask + (b * mask_rows + s) * mask_words;
            for (int64_t h = 0; h < H; ++h) {
                double *orow = o + ((b * S + s) * H + h) * D;
                for (int64_t d = 0; d < D; ++d) orow[d] = 0.0;
                const uint16_t *qh = q + ((b * S + s) * H + h) * D;
                for (int64_t t = 0; t < T; ++t) {
                    int64_t key = t + off;
                    int on = key >= 0 && (key >> 5) < key_words &&
                             (key_ends == NULL || key < key_ends[b]) &&
                             ((row[key >> 5] >> (key & 31)) & 1u);
                    if (!on) {
                        logit[t] = -INFINITY;
                        continue;
                    }
                    const uint16_t *kr = kv + (b * T + t) * D;
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        dot += bf16_to_double(qh[d]) * bf16_to_double(kr[d]);
                    logit[t] = dot * softmax_scale;
                }
                const double sink = (double)attn_sink[h];
                if (isnan(sink)) {
                    for (int64_t d = 0; d < D; ++d) orow[d] = NAN;
                    continue;
                }
                double m = sink;
                for (int64_t t = 0; t < T; ++t)
                    if (logit[t] > m) m = logit[t];
                if (m == INFINITY && sink == INFINITY) continue;
                if (m == -INFINITY) continue;
                double denom = exp(sink - m);
                for (int64_t t = 0; t < T; ++t) denom += exp(logit[t] - m);
                for (int64_t t = 0; t < T; ++t) {
                    if (logit[t] == -INFINITY) continue;
                    const double w = exp(logit[t] - m) / denom;
                    const uint16_t *kr = kv + (b * T + t) * D;
                    for (int64_t d = 0; d < D; ++d) orow[d] += w * bf16_to_double(kr[d]);
                }
            }
        }
    }
    free(logit);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Bit-packed top-k mask, [MASK-SHAPE], [MASK-BITS]                          */
/* ------------------------------------------------------------------------ */

static int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* (batch, padded query rows, words per row):
 *   tile_m = 128 when max_query_len <= 128, else 256;
 *   rows   = ceil(max_query_len / tile_m) * tile_m;
 *   words  = ceil(max_key_len / 32) + reserve, rounded up to a multiple of 4
 *            so every row starts on a 16-byte boundary. */
int oracle_topk_mask_shape(int64_t batch, int64_t max_query_len, int64_t max_key_len,
                           int reserve_key_starts_word, int64_t out_shape[3]) {
    if (batch < 0 || max_query_len < 0 || max_key_len < 0) return ORACLE_EINVAL;
    const int64_t tile_m = max_query_len <= 128 ? 128 : 256;
    const int64_t rows = cdiv64(max_query_len, tile_m) * tile_m;
    int64_t words = cdiv64(max_key_len, 32) + (reserve_key_starts_word ? 1 : 0);
    words = cdiv64(words, 4) * 4;
    out_shape[0] = batch;
    out_shape[1] = rows;
    out_shape[2] = words;
    return ORACLE_OK;
}

/* Writes, bit by bit, the mask of every live row (b, q < q_len_b): word
 * k>>5 of row (b,q) gets bit k&31 for each index k of topk row
 * cu_q_lens[b] + q with 0 <= k < max_key_len (R14).  Live words are cleared
 * first.  When key_starts is non-NULL, word W-1 of row (b, 0) receives the
 * raw bits of key_starts[b] (R16).  Nothing else is written (R15). */
/* A window of the mask (reading R24, the chunked fallback of [MASK-CAP]):
 * row i of `mask` is query q0 + i of each request, for the q_rows queries of
 * the window; key_ends (or NULL) gives each request's live key end, and only
 * the words below min(end, max_key_len) of a live row are written (the
 * strided build that stops at the row's end, [MASK-END]).  Everything else --
 * words past the end, padding words, rows past a request's query count and
 * padding rows -- keeps its contents.  The reserved key_start word goes to
 * row 0 of each request, where the consumer reads it. */
int oracle_build_topk_mask_window(const int32_t *topk, int64_t topk_rows, const int32_t *cu_q_lens,
                                  int64_t B, int64_t q0, int64_t q_rows, int64_t max_key_len, int64_t K,
                                  const int32_t *key_starts, const int32_t *key_ends, uint32_t *mask,
                                  const int64_t mask_shape[3]) {
    int64_t want[3];
    if (q0 < 0 || oracle_topk_mask_shape(B, q_rows, max_key_len, key_starts != NULL, want))
        return ORACLE_EINVAL;
    if (mask_shape[0] != want[0] || mask_shape[1] != want[1] || mask_shape[2] != want[2])
        return ORACLE_EINVAL;
    const int64_t R = want[1], W = want[2];
    for (int64_t b = 0; b < B; ++b) {
        int64_t end = max_key_len;
        if (key_ends != NULL && (int64_t)key_ends[b] < end) end = key_ends[b] < 0 ? 0 : key_ends[b];
        const int64_t live_words = cdiv64(end, 32);
        const int64_t q_len = (int64_t)cu_q_lens[b + 1] - (int64_t)cu_q_lens[b];
        for (int64_t i = 0; i < q_rows; ++i) {
            const int64_t qi = q0 + i;
            if (qi >= q_len) break;
            const int64_t src = (int64_t)cu_q_lens[b] + qi;
            if (src < 0 || src >= topk_rows) continue;
            uint32_t *row = mask + (b * R + i) * W;
            for (int64_t w = 0; w < live_words; ++w) row[w] = 0u;
            for (int64_t j = 0; j < K; ++j) {
                const int64_t k = topk[src * K + j];
                if (k < 0 || k >= end) continue;
                row[k >> 5] |= 1u << (k & 31);
            }
        }
        if (key_starts != NULL && R > 0 && W > 0)
            mask[(b * R + 0) * W + (W - 1)] = (uint32_t)key_starts[b];
    }
    return ORACLE_OK;
}

/* The whole mask: the window of every query, no live ends. */
int oracle_build_topk_mask(const int32_t *topk, int64_t topk_rows, const int32_t *cu_q_lens,
                           int64_t B, int64_t max_q_len, int64_t max_key_len, int64_t K,
                           const int32_t *key_starts, uint32_t *mask,
                           const int64_t mask_shape[3]) {
    return oracle_build_topk_mask_window(topk, topk_rows, cu_q_lens, B, 0, max_q_len, max_key_len, K, key_starts,
                                         NULL, mask, mask_shape);
}
