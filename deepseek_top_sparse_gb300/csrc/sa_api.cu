// C ABI entry points (include/sa.h): host-side validation, planning and
// launch.  Nothing here computes the method; every step of it runs in the
// kernels of the other translation units.
#include <cmath>
#include <mutex>

#include "sa_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Above this size the whole (global) top-k mask is not built at once: it is
// built and consumed one window of query rows at a time (vLLM PR 48770 page,
// review notes: GLOBAL_TOPK_MASK_MAX_BYTES = 64 MiB).
constexpr int64_t kGlobalTopkMaskMaxBytes = int64_t(64) << 20;

struct DeviceInfo {
    int sms = 0;
    int major = 0, minor = 0;
    bool ok = false;
};

DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

sa_status current_device(DeviceInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SA_ERR_CUDA;
    std::call_once(g_dev_once[dev], [dev] {
        cudaDeviceProp p{};
        if (cudaGetDeviceProperties(&p, dev) == cudaSuccess) {
            g_dev[dev].sms = p.multiProcessorCount;
            g_dev[dev].major = p.major;
            g_dev[dev].minor = p.minor;
            g_dev[dev].ok = true;
        }
    });
    if (!g_dev[dev].ok) return SA_ERR_CUDA;
    *out = g_dev[dev];
    // The kernels are built for sm_103a only (tcgen05, TMA).
    if (!(out->major == 10 && out->minor == 3)) return SA_ERR_UNSUPPORTED_DEVICE;
    return SA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool attn_sizes_ok(int64_t B, int64_t S, int64_t H, int64_t D, int64_t K) {
    if (B < 0 || S < 0 || H < 1 || H > 128 || K < 1) return false;
    if (!(D == 64 || D == 128 || D == 256 || D == 512)) return false;
    return true;
}

// Split plan: a function of the sizes and the SM count only (never of index
// values), so a captured graph keeps a fixed grid.  One work unit (token,
// split) occupies one CTA, or a 2-CTA cluster when D = 512; a unit holds at
// most sa::max_unit_slots() slots.  Small batches are split so that the units
// cover the SMs once, keeping at least 3 tiles of 64 slots per split.
int min_splits(int64_t K) {
    const int64_t tiles = cdiv(K, 64);
    return int(cdiv(tiles, sa::max_unit_slots() / 64));
}

int clamp_splits(int64_t K, int ns) {
    const int64_t tiles = cdiv(K, 64);
    if (ns > tiles) ns = int(tiles);
    if (ns < min_splits(K)) ns = min_splits(K);
    if (ns < 1) ns = 1;
    return ns;
}

int plan_splits(int64_t B, int64_t S, int64_t H, int64_t D, int64_t K, int num_sms) {
    (void)H;
    const int64_t ctas_per_unit = D == 512 ? 2 : 1;
    const int64_t ctas = B * S * ctas_per_unit;
    const int64_t tiles = cdiv(K, 64);
    int64_t ns = 1;
    if (ctas > 0 && ctas < num_sms) ns = num_sms / ctas;
    const int64_t cap = tiles / 3 > 1 ? tiles / 3 : 1;
    if (ns > cap) ns = cap;
    if (ns > 64) ns = 64;
    return clamp_splits(K, int(ns));
}

// Split workspace layout: fp32 partial rows [units, splits, rows, D], padded
// to 256 bytes, then fp32 log-sum-exp [units, splits, rows].
size_t partials_bytes(int64_t units, int64_t rows, int64_t D, int splits) {
    const size_t o_bytes = size_t(units) * size_t(splits) * size_t(rows) * size_t(D) * sizeof(float);
    return (o_bytes + 255) / 256 * 256;
}

size_t workspace_bytes_for(int64_t B, int64_t S, int64_t H, int64_t D, int splits) {
    if (splits <= 1) return 0;
    const int64_t units = B * S;
    return partials_bytes(units, H, D, splits) + size_t(units) * size_t(splits) * size_t(H) * sizeof(float);
}

// Points the launch arguments at the two parts of a split workspace.
void carve_workspace(sa::AttnArgs &a, void *workspace, int64_t units, int64_t rows, int64_t D, int splits) {
    if (splits <= 1) return;
    a.ws_o = static_cast<float *>(workspace);
    a.ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + partials_bytes(units, rows, D, splits));
}

}  // namespace

extern "C" {

const char *sa_status_string(sa_status s) {
    switch (s) {
        case SA_OK: return "SA_OK";
        case SA_ERR_INVALID_ARG: return "SA_ERR_INVALID_ARG";
        case SA_ERR_SHAPE: return "SA_ERR_SHAPE";
        case SA_ERR_ALIGNMENT: return "SA_ERR_ALIGNMENT";
        case SA_ERR_WORKSPACE: return "SA_ERR_WORKSPACE";
        case SA_ERR_UNSUPPORTED_DEVICE: return "SA_ERR_UNSUPPORTED_DEVICE";
        case SA_ERR_CUDA: return "SA_ERR_CUDA";
    }
    return "SA_ERR_UNKNOWN";
}

int sa_sparse_attn_num_splits(int64_t B, int64_t S, int64_t H, int64_t D, int64_t K) {
    if (!attn_sizes_ok(B, S, H, D, K)) return 0;
    DeviceInfo dev;
    const sa_status st = current_device(&dev);
    if (st != SA_OK) return 0;
    return plan_splits(B, S, H, D, K, dev.sms);
}

size_t sa_sparse_attn_workspace_size(int64_t B, int64_t S, int64_t H, int64_t D, int64_t K,
                                     int num_splits) {
    if (!attn_sizes_ok(B, S, H, D, K)) return 0;
    int splits = num_splits;
    if (splits <= 0) splits = sa_sparse_attn_num_splits(B, S, H, D, K);
    if (splits <= 0) return 0;
    return workspace_bytes_for(B, S, H, D, clamp_splits(K, splits));
}

int sa_sparse_attn_launch_count(int64_t B, int64_t S, int64_t H, int64_t D, int64_t K, int num_splits) {
    if (!attn_sizes_ok(B, S, H, D, K) || num_splits > 64) return 0;
    if (B * S == 0) return 0;
    DeviceInfo dev;
    if (current_device(&dev) != SA_OK) return 0;
    const int splits = clamp_splits(K, num_splits > 0 ? num_splits : plan_splits(B, S, H, D, K, dev.sms));
    return sa::kernels_per_call(D, splits);
}

namespace {

// A second kv source (its K2 slots join each token's softmax after the K main
// slots); K2 = 0 without one.
struct ExtraSrc {
    const void *kv = nullptr;
    const int32_t *idx = nullptr;
    const int32_t *len = nullptr;
    int64_t T2 = 0, K2 = 0;
};

// Every check of the sparse_attn calls, then the launch(es).  kv (and the
// extra kv) are bf16 rows of D values, or FP8 rows of 584 bytes (D = 512).
sa_status attn_call(const void *q, const void *kv, bool fp8, const float *attn_sink, const int32_t *topk_idxs,
                    const int32_t *topk_length, const ExtraSrc &x, float softmax_scale, void *o, int64_t B,
                    int64_t S, int64_t H, int64_t D, int64_t T, int64_t K, int num_splits, void *workspace,
                    size_t workspace_bytes, sa_stream_t stream) {
    if (B < 0 || S < 0 || H < 0 || D < 0 || T < 0 || K < 0 || x.T2 < 0 || x.K2 < 0) return SA_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale)) return SA_ERR_INVALID_ARG;
    if (num_splits > 64) return SA_ERR_INVALID_ARG;
    const int64_t Kt = K + x.K2;   // slots per token
    if (!attn_sizes_ok(B, S, H, D, Kt) || (K > 0 && T < 1) || (x.K2 > 0 && x.T2 < 1)) return SA_ERR_SHAPE;
    if ((B * T + 1) / 2 * 2 + B * x.T2 >= (int64_t(1) << 31)) return SA_ERR_SHAPE;   // 32-bit row numbers
    if (B * S * H >= (int64_t(1) << 31)) return SA_ERR_SHAPE;   // q rows are 32-bit tensor-map coordinates
    if (B * S == 0) return SA_OK;
    if (!q || !attn_sink || !o || (K > 0 && (!kv || !topk_idxs)) || (x.K2 > 0 && (!x.kv || !x.idx)))
        return SA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(o) || !aligned16(x.kv)) return SA_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(topk_idxs) & 3) || (reinterpret_cast<uintptr_t>(attn_sink) & 3) ||
        (reinterpret_cast<uintptr_t>(topk_length) & 3) || (reinterpret_cast<uintptr_t>(x.idx) & 3) ||
        (reinterpret_cast<uintptr_t>(x.len) & 3))
        return SA_ERR_ALIGNMENT;
    DeviceInfo dev;
    const sa_status st = current_device(&dev);
    if (st != SA_OK) return st;

    const int splits = clamp_splits(Kt, num_splits > 0 ? num_splits : plan_splits(B, S, H, D, Kt, dev.sms));
    const size_t need = workspace_bytes_for(B, S, H, D, splits);
    if (workspace_bytes < need || (need > 0 && workspace == nullptr)) return SA_ERR_WORKSPACE;
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255)) return SA_ERR_ALIGNMENT;

    sa::AttnArgs a{};
    a.q = q; a.kv = kv; a.kv_fp8 = fp8; a.sink = attn_sink; a.idx = topk_idxs; a.topk_len = topk_length;
    a.kv2 = x.kv; a.idx2 = x.idx; a.topk_len2 = x.len; a.T2 = x.T2; a.K2 = x.K2;
    a.scale = softmax_scale; a.o = o;
    a.B = B; a.S = S; a.H = H; a.D = D; a.T = T; a.K = K;
    a.num_splits = splits;
    carve_workspace(a, workspace, B * S, H, D, splits);
    // the main kernel, then (for splits too many for one cluster) the combine
    if (sa::launch_sparse_attn(a, dev.sms, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SA_ERR_CUDA;
    return SA_OK;
}

}  // namespace

sa_status sa_sparse_attn_fwd_topk_length(const void *q, const void *kv, const float *attn_sink,
                                         const int32_t *topk_idxs, const int32_t *topk_length,
                                         float softmax_scale, void *o, int64_t B, int64_t S, int64_t H,
                                         int64_t D, int64_t T, int64_t K, int num_splits, void *workspace,
                                         size_t workspace_bytes, sa_stream_t stream) {
    return attn_call(q, kv, false, attn_sink, topk_idxs, topk_length, ExtraSrc{}, softmax_scale, o, B, S, H, D, T,
                     K, num_splits, workspace, workspace_bytes, stream);
}

sa_status sa_sparse_attn_fwd_extra(const void *q, const void *kv, const float *attn_sink, const int32_t *topk_idxs,
                                   const int32_t *topk_length, const void *extra_kv, const int32_t *extra_topk_idxs,
                                   const int32_t *extra_topk_length, float softmax_scale, void *o, int64_t B,
                                   int64_t S, int64_t H, int64_t D, int64_t T, int64_t K, int64_t T2, int64_t K2,
                                   int num_splits, void *workspace, size_t workspace_bytes, sa_stream_t stream) {
    ExtraSrc x;
    x.kv = extra_kv; x.idx = extra_topk_idxs; x.len = extra_topk_length; x.T2 = T2; x.K2 = K2;
    return attn_call(q, kv, false, attn_sink, topk_idxs, topk_length, x, softmax_scale, o, B, S, H, D, T, K,
                     num_splits, workspace, workspace_bytes, stream);
}

int sa_sparse_attn_fp8_launch_count(int64_t B, int64_t S, int64_t H, int64_t K, int num_splits) {
    if (!attn_sizes_ok(B, S, H, 512, K) || num_splits > 64) return 0;
    if (B * S == 0) return 0;
    DeviceInfo dev;
    if (current_device(&dev) != SA_OK) return 0;
    const int splits = clamp_splits(K, num_splits > 0 ? num_splits : plan_splits(B, S, H, 512, K, dev.sms));
    return sa::kernels_per_call(512, splits, true);
}

sa_status sa_sparse_attn_fwd_fp8(const void *q, const uint8_t *kv_fp8, const float *attn_sink,
                                 const int32_t *topk_idxs, const int32_t *topk_length, float softmax_scale,
                                 void *o, int64_t B, int64_t S, int64_t H, int64_t T, int64_t K, int num_splits,
                                 void *workspace, size_t workspace_bytes, sa_stream_t stream) {
    return attn_call(q, kv_fp8, true, attn_sink, topk_idxs, topk_length, ExtraSrc{}, softmax_scale, o, B, S, H,
                     512, T, K, num_splits, workspace, workspace_bytes, stream);
}

sa_status sa_sparse_attn_fwd_fp8_extra(const void *q, const uint8_t *kv_fp8, const float *attn_sink,
                                       const int32_t *topk_idxs, const int32_t *topk_length,
                                       const uint8_t *extra_kv_fp8, const int32_t *extra_topk_idxs,
                                       const int32_t *extra_topk_length, float softmax_scale, void *o, int64_t B,
                                       int64_t S, int64_t H, int64_t T, int64_t K, int64_t T2, int64_t K2,
                                       int num_splits, void *workspace, size_t workspace_bytes,
                                       sa_stream_t stream) {
    ExtraSrc x;
    x.kv = extra_kv_fp8; x.idx = extra_topk_idxs; x.len = extra_topk_length; x.T2 = T2; x.K2 = K2;
    return attn_call(q, kv_fp8, true, attn_sink, topk_idxs, topk_length, x, softmax_scale, o, B, S, H, 512, T, K,
                     num_splits, workspace, workspace_bytes, stream);
}

sa_status sa_sparse_attn_fwd_splits(const void *q, const void *kv, const float *attn_sink,
                                    const int32_t *topk_idxs, float softmax_scale, void *o,
                                    int64_t B, int64_t S, int64_t H, int64_t D, int64_t T,
                                    int64_t K, int num_splits, void *workspace,
                                    size_t workspace_bytes, sa_stream_t stream) {
    return sa_sparse_attn_fwd_topk_length(q, kv, attn_sink, topk_idxs, nullptr, softmax_scale, o, B, S, H, D, T,
                                          K, num_splits, workspace, workspace_bytes, stream);
}

sa_status sa_sparse_attn_fwd(const void *q, const void *kv, const float *attn_sink,
                             const int32_t *topk_idxs, float softmax_scale, void *o, int64_t B,
                             int64_t S, int64_t H, int64_t D, int64_t T, int64_t K,
                             void *workspace, size_t workspace_bytes, sa_stream_t stream) {
    return sa_sparse_attn_fwd_splits(q, kv, attn_sink, topk_idxs, softmax_scale, o, B, S, H, D, T,
                                     K, 0, workspace, workspace_bytes, stream);
}

namespace {

// Split count of the mask consumer: the packed kernel's plan for D <= 256,
// sparse_attn's (the T keys playing the part of the K slots) for D = 512; 0
// when the sizes cannot be planned.
int masked_splits(int64_t B, int64_t S, int64_t H, int64_t D, int64_t T, int num_splits, int sms) {
    if (sa::masked_dense_packed(D)) return sa::masked_dense_splits(B, S, H, D, T, num_splits, sms);
    return clamp_splits(T, num_splits > 0 ? num_splits : plan_splits(B, S, H, D, T, sms));
}

}  // namespace

size_t sa_masked_dense_attn_workspace_size(int64_t B, int64_t S, int64_t H, int64_t D, int64_t T,
                                           int num_splits) {
    if (!attn_sizes_ok(B, S, H, D, T) || num_splits > 64) return 0;
    DeviceInfo dev{};
    if (num_splits <= 0 && current_device(&dev) != SA_OK) return 0;   // the plan needs the SM count
    const int splits = masked_splits(B, S, H, D, T, num_splits, dev.sms);
    return splits > 0 ? workspace_bytes_for(B, S, H, D, splits) : 0;
}

int sa_masked_dense_attn_launch_count(int64_t B, int64_t S, int64_t H, int64_t D, int64_t T, int num_splits) {
    if (!attn_sizes_ok(B, S, H, D, T) || num_splits > 64) return 0;
    if (B * S == 0) return 0;
    DeviceInfo dev;
    if (current_device(&dev) != SA_OK) return 0;
    const int splits = masked_splits(B, S, H, D, T, num_splits, dev.sms);
    if (splits <= 0) return 0;
    if (sa::masked_dense_packed(D)) return splits > 1 ? 2 : 1;
    return sa::kernels_per_call(D, splits);
}

namespace {

sa_status mask_window(const int32_t *topk, int64_t topk_rows, const int32_t *cu_q_lens, int64_t B, int64_t q0,
                      int64_t q_rows, int64_t max_key_len, int64_t K, const int32_t *key_starts,
                      const int32_t *key_ends, uint32_t *mask, const int64_t mask_shape[3], sa_stream_t stream,
                      bool dry_run);

// The consumer over a window: every check of sa_masked_dense_attn_fwd_window,
// then (unless dry_run) the launch.
sa_status masked_window(const void *q, const void *kv, const float *attn_sink, const uint32_t *mask,
                        int64_t mask_rows, int64_t mask_words, int key_start_word, const int32_t *key_ends,
                        float softmax_scale, void *o, int64_t B, int64_t S_total, int64_t q0, int64_t S, int64_t H,
                        int64_t D, int64_t T, int num_splits, void *workspace, size_t workspace_bytes,
                        sa_stream_t stream, bool dry_run) {
    if (B < 0 || S < 0 || S_total < 0 || q0 < 0 || H < 0 || D < 0 || T < 0 || mask_rows < 0 || mask_words < 0)
        return SA_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale)) return SA_ERR_INVALID_ARG;
    if (num_splits > 64 || (key_start_word != 0 && key_start_word != 1)) return SA_ERR_INVALID_ARG;
    if (!attn_sizes_ok(B, S, H, D, T) || T < 1) return SA_ERR_SHAPE;
    if (q0 + S > S_total) return SA_ERR_SHAPE;
    if (B * T + 256 >= (int64_t(1) << 31)) return SA_ERR_SHAPE;   // 32-bit key-tile coordinates
    if (B * S_total * H >= (int64_t(1) << 31)) return SA_ERR_SHAPE;
    if (mask_rows < S || mask_words < 1 || (mask_words & 3)) return SA_ERR_SHAPE;
    if (B * S == 0) return SA_OK;
    if (!q || !kv || !attn_sink || !mask || !o) return SA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(o) || !aligned16(mask)) return SA_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(attn_sink) & 3) || (reinterpret_cast<uintptr_t>(key_ends) & 3))
        return SA_ERR_ALIGNMENT;
    DeviceInfo dev;
    const sa_status st = current_device(&dev);
    if (st != SA_OK) return st;

    const int splits = masked_splits(B, S, H, D, T, num_splits, dev.sms);
    if (splits <= 0) return SA_ERR_SHAPE;
    const size_t need = workspace_bytes_for(B, S, H, D, splits);
    if (workspace_bytes < need || (need > 0 && workspace == nullptr)) return SA_ERR_WORKSPACE;
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255)) return SA_ERR_ALIGNMENT;
    if (dry_run) return SA_OK;

    sa::AttnArgs a{};
    a.q = q; a.kv = kv; a.sink = attn_sink; a.idx = nullptr; a.topk_len = nullptr;
    a.scale = softmax_scale; a.o = o;
    a.B = B; a.S = S; a.H = H; a.D = D; a.T = T; a.K = T;
    a.io_S = S_total; a.io_s0 = q0;
    a.num_splits = splits;
    a.mask = mask; a.mask_rows = mask_rows; a.mask_words = mask_words; a.key_start_word = key_start_word;
    a.key_ends = key_ends;
    carve_workspace(a, workspace, B * S, H, D, splits);
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = sa::masked_dense_packed(D) ? sa::launch_masked_dense(a, cs)
                                                     : sa::launch_sparse_attn(a, dev.sms, cs);
    return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace

sa_status sa_masked_dense_attn_fwd_window(const void *q, const void *kv, const float *attn_sink,
                                          const uint32_t *mask, int64_t mask_rows, int64_t mask_words,
                                          int key_start_word, const int32_t *key_ends, float softmax_scale, void *o,
                                          int64_t B, int64_t S_total, int64_t q0, int64_t S, int64_t H, int64_t D,
                                          int64_t T, int num_splits, void *workspace, size_t workspace_bytes,
                                          sa_stream_t stream) {
    return masked_window(q, kv, attn_sink, mask, mask_rows, mask_words, key_start_word, key_ends, softmax_scale, o, B,
                         S_total, q0, S, H, D, T, num_splits, workspace, workspace_bytes, stream, false);
}

sa_status sa_masked_dense_attn_fwd(const void *q, const void *kv, const float *attn_sink,
                                   const uint32_t *mask, int64_t mask_rows, int64_t mask_words,
                                   int key_start_word, float softmax_scale, void *o, int64_t B, int64_t S,
                                   int64_t H, int64_t D, int64_t T, int num_splits, void *workspace,
                                   size_t workspace_bytes, sa_stream_t stream) {
    return sa_masked_dense_attn_fwd_window(q, kv, attn_sink, mask, mask_rows, mask_words, key_start_word, nullptr,
                                           softmax_scale, o, B, S, 0, S, H, D, T, num_splits, workspace,
                                           workspace_bytes, stream);
}

int64_t sa_topk_mask_chunk_rows(int64_t batch, int64_t max_query_len, int64_t max_key_len,
                                int reserve_key_starts_word, int64_t cap_bytes) {
    if (batch < 1 || max_query_len < 1 || max_key_len < 0) return 0;
    if (cap_bytes <= 0) cap_bytes = kGlobalTopkMaskMaxBytes;
    auto bytes = [&](int64_t rows) {
        int64_t shp[3];
        sa_topk_mask_shape(batch, rows, max_key_len, reserve_key_starts_word, shp);
        return shp[0] * shp[1] * shp[2] * 4;
    };
    if (bytes(max_query_len) <= cap_bytes) return max_query_len;   // the whole (global) mask
    // windows past 128 rows pad to multiples of 256
    const int64_t per256 = bytes(256);
    int64_t k = per256 > 0 ? cap_bytes / per256 : 0;
    if (k * 256 >= max_query_len) k = (max_query_len - 1) / 256;
    if (k >= 1) return k * 256;
    return bytes(128) <= cap_bytes ? 128 : 0;
}

sa_status sa_topk_masked_attn_fwd(const void *q, const void *kv, const float *attn_sink, const int32_t *topk,
                                  int64_t topk_rows, const int32_t *cu_q_lens, const int32_t *key_starts,
                                  const int32_t *key_ends, float softmax_scale, void *o, int64_t B,
                                  int64_t max_q_len, int64_t H, int64_t D, int64_t T, int64_t max_key_len, int64_t K,
                                  int64_t cap_bytes, uint32_t *mask_buf, size_t mask_buf_bytes, void *workspace,
                                  size_t workspace_bytes, sa_stream_t stream) {
    if (B < 0 || max_q_len < 0 || H < 0 || D < 0 || T < 0 || max_key_len < 0 || K < 0 || topk_rows < 0)
        return SA_ERR_INVALID_ARG;
    if (B * max_q_len == 0) return SA_OK;
    const int64_t qc = sa_topk_mask_chunk_rows(B, max_q_len, max_key_len, key_starts != nullptr, cap_bytes);
    if (qc < 1) return SA_ERR_SHAPE;
    int64_t shp[3];
    sa_topk_mask_shape(B, qc, max_key_len, key_starts != nullptr, shp);
    if (mask_buf == nullptr || mask_buf_bytes < size_t(shp[0] * shp[1] * shp[2] * 4)) return SA_ERR_WORKSPACE;
    const int key_start_word = key_starts != nullptr ? 1 : 0;
    // every window is checked before the first launch (windows differ only
    // in their row count: a full one and the last one)
    for (int pass = 0; pass < 2; ++pass) {
        const bool dry = pass == 0;
        for (int64_t q0 = 0; q0 < max_q_len; q0 += qc) {
            const int64_t rows = max_q_len - q0 < qc ? max_q_len - q0 : qc;
            if (dry && q0 > 0 && q0 + qc < max_q_len) continue;   // same shape as the first window
            int64_t ws[3];
            sa_topk_mask_shape(B, rows, max_key_len, key_starts != nullptr, ws);
            auto build = [&] {
                return mask_window(topk, topk_rows, cu_q_lens, B, q0, rows, max_key_len, K, key_starts, key_ends,
                                   mask_buf, ws, stream, dry);
            };
            auto consume = [&] {
                return masked_window(q, kv, attn_sink, mask_buf, ws[1], ws[2], key_start_word, key_ends,
                                     softmax_scale, o, B, max_q_len, q0, rows, H, D, T, 0, workspace,
                                     workspace_bytes, stream, dry);
            };
            // (the checks: the consumer's first, so that its argument errors
            // are reported before the device is queried; the launches: build
            // then consume)
            sa_status st = dry ? consume() : build();
            if (st != SA_OK) return st;
            st = dry ? build() : consume();
            if (st != SA_OK) return st;
        }
    }
    return SA_OK;
}

size_t sa_topk_masked_attn_workspace_size(int64_t B, int64_t max_q_len, int64_t H, int64_t D, int64_t T,
                                          int64_t max_key_len, int reserve_key_starts_word, int64_t cap_bytes) {
    const int64_t qc = sa_topk_mask_chunk_rows(B, max_q_len, max_key_len, reserve_key_starts_word, cap_bytes);
    if (qc < 1) return 0;
    // every window but the last has qc rows; a short last window may plan more splits
    const int64_t last = max_q_len - (max_q_len - 1) / qc * qc;
    const size_t a = sa_masked_dense_attn_workspace_size(B, qc, H, D, T, 0);
    const size_t b = sa_masked_dense_attn_workspace_size(B, last, H, D, T, 0);
    return a > b ? a : b;
}

sa_status sa_topk_mask_shape(int64_t batch, int64_t max_query_len, int64_t max_key_len,
                             int reserve_key_starts_word, int64_t out_shape[3]) {
    if (out_shape == nullptr || batch < 0 || max_query_len < 0 || max_key_len < 0)
        return SA_ERR_INVALID_ARG;
    const int64_t tile_m = max_query_len <= 128 ? 128 : 256;
    out_shape[0] = batch;
    out_shape[1] = cdiv(max_query_len, tile_m) * tile_m;
    out_shape[2] = cdiv(cdiv(max_key_len, 32) + (reserve_key_starts_word ? 1 : 0), 4) * 4;
    return SA_OK;
}

namespace {

// Every check of sa_build_topk_mask_window, then (unless dry_run) the launch.
sa_status mask_window(const int32_t *topk, int64_t topk_rows, const int32_t *cu_q_lens, int64_t B, int64_t q0,
                      int64_t q_rows, int64_t max_key_len, int64_t K, const int32_t *key_starts,
                      const int32_t *key_ends, uint32_t *mask, const int64_t mask_shape[3], sa_stream_t stream,
                      bool dry_run) {
    if (mask_shape == nullptr || B < 0 || q0 < 0 || q_rows < 0 || max_key_len < 0 || K < 0 || topk_rows < 0)
        return SA_ERR_INVALID_ARG;
    if (max_key_len > INT32_MAX || q0 > INT32_MAX - q_rows) return SA_ERR_SHAPE;
    int64_t want[3];
    sa_status st = sa_topk_mask_shape(B, q_rows, max_key_len, key_starts != nullptr, want);
    if (st != SA_OK) return st;
    if (mask_shape[0] != want[0] || mask_shape[1] != want[1] || mask_shape[2] != want[2])
        return SA_ERR_SHAPE;
    const bool any_rows = B * q_rows > 0 && topk_rows > 0;
    const bool any_ks = key_starts != nullptr && want[1] > 0 && B > 0;
    if (!any_rows && !any_ks) return SA_OK;
    if (mask == nullptr || cu_q_lens == nullptr) return SA_ERR_INVALID_ARG;
    if (any_rows && K > 0 && topk == nullptr) return SA_ERR_INVALID_ARG;
    if (!aligned16(mask)) return SA_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(cu_q_lens) & 3) || (reinterpret_cast<uintptr_t>(topk) & 3) ||
        (reinterpret_cast<uintptr_t>(key_starts) & 3) || (reinterpret_cast<uintptr_t>(key_ends) & 3))
        return SA_ERR_ALIGNMENT;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != SA_OK) return st;
    if (dry_run) return SA_OK;
    sa::MaskArgs a{};
    a.topk = topk; a.topk_rows = topk_rows; a.cu_q_lens = cu_q_lens;
    a.B = B; a.max_q_len = q_rows; a.max_key_len = max_key_len; a.K = K;
    a.key_starts = key_starts; a.mask = mask; a.rows = want[1]; a.words = want[2];
    a.q0 = q0; a.key_ends = key_ends;
    if (!any_rows) a.max_q_len = 0;  // only the reserved words remain to write
    if (sa::launch_build_topk_mask(a, dev.sms, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SA_ERR_CUDA;
    return SA_OK;
}

}  // namespace

sa_status sa_build_topk_mask_window(const int32_t *topk, int64_t topk_rows, const int32_t *cu_q_lens, int64_t B,
                                    int64_t q0, int64_t q_rows, int64_t max_key_len, int64_t K,
                                    const int32_t *key_starts, const int32_t *key_ends, uint32_t *mask,
                                    const int64_t mask_shape[3], sa_stream_t stream) {
    return mask_window(topk, topk_rows, cu_q_lens, B, q0, q_rows, max_key_len, K, key_starts, key_ends, mask,
                       mask_shape, stream, false);
}

sa_status sa_build_topk_mask(const int32_t *topk, int64_t topk_rows, const int32_t *cu_q_lens,
                             int64_t B, int64_t max_q_len, int64_t max_key_len, int64_t K,
                             const int32_t *key_starts, uint32_t *mask,
                             const int64_t mask_shape[3], sa_stream_t stream) {
    return sa_build_topk_mask_window(topk, topk_rows, cu_q_lens, B, 0, max_q_len, max_key_len, K, key_starts,
                                     nullptr, mask, mask_shape, stream);
}

int sa_selftest_wait_timeout(long long max_cycles) {
    if (max_cycles < 1 || max_cycles > (1ll << 28)) return -1;
    DeviceInfo dev;
    if (current_device(&dev) != SA_OK) return -1;
    int before = 0;
    if (sa::read_device_error(&before, true) != cudaSuccess) return -1;   // start from a clear word
    if (sa::launch_wait_timeout_selftest(max_cycles, nullptr) != cudaSuccess) return -1;
    int code = 0;
    if (sa::read_device_error(&code, true) != cudaSuccess) return -1;
    return code;
}

int sa_selftest_wait_drain(int ctas, long long first_cycles, float *elapsed_ms) {
    if (ctas < 1 || ctas > 1024 || first_cycles < 1 || first_cycles > (1ll << 28) || elapsed_ms == nullptr)
        return -1;
    DeviceInfo dev;
    if (current_device(&dev) != SA_OK) return -1;
    int before = 0;
    if (sa::read_device_error(&before, true) != cudaSuccess) return -1;   // start from a clear word
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return -1;
    bool ok = cudaEventRecord(e0, nullptr) == cudaSuccess &&
              sa::launch_wait_drain_selftest(ctas, first_cycles, nullptr) == cudaSuccess &&
              cudaEventRecord(e1, nullptr) == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess &&
              cudaEventElapsedTime(elapsed_ms, e0, e1) == cudaSuccess;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (!ok) return -1;
    int code = 0;
    if (sa::read_device_error(&code, true) != cudaSuccess) return -1;
    return code;
}

sa_status sa_probe_row_gather(const void *table, int64_t rows, int64_t row_bytes, int64_t part_bytes,
                              const int32_t *idx, int64_t ctas, int64_t tiles, sa_stream_t stream) {
    if (table == nullptr || idx == nullptr) return SA_ERR_INVALID_ARG;
    if (rows < 1 || rows > INT32_MAX || ctas < 1 || ctas > 65535 || tiles < 1 || tiles > (1 << 20))
        return SA_ERR_INVALID_ARG;
    if (part_bytes < 16 || part_bytes > 32768 || (part_bytes & (part_bytes - 1)) != 0 || row_bytes < part_bytes ||
        row_bytes % 16 != 0)
        return SA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(table) % 16 != 0) return SA_ERR_ALIGNMENT;
    if (rows > INT64_MAX / row_bytes) return SA_ERR_INVALID_ARG;
    DeviceInfo dev;
    const sa_status st = current_device(&dev);
    if (st != SA_OK) return st;
    int shift = 4;
    while ((int64_t(1) << shift) < part_bytes) ++shift;
    if (sa::launch_row_gather_probe(table, rows, row_bytes, shift, idx, int(ctas), int(tiles),
                                    reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SA_ERR_CUDA;
    return SA_OK;
}

int sa_device_error(int clear) {
    int v = 0;
    if (sa::read_device_error(&v, clear != 0) != cudaSuccess) return -1;
    return v;
}

}  // extern "C"
