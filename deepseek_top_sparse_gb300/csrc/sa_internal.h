// Internal declarations shared by the translation units of libsa.so.
// Not part of the public ABI (see include/sa.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sa.h"

namespace sa {

// Launches kern<<<grid, block, smem, stream>>>(args...) with a programmatic
// dependency on the stream's previous kernel: the launch may proceed while
// that kernel runs, so `kern` executes griddepcontrol.wait (ptx::griddep_wait)
// in every thread before its first global memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Codes written to the device error word (see sa_device_error in sa.h).
enum DeviceError : int {
    kErrNone = 0,
    kErrWaitTimeout = 1,   // an mbarrier wait ran past its iteration limit
    kErrBadPlan = 2,       // a kernel received a launch shape it cannot handle
};

// The device error word lives in attn_tc.cu; every kernel that can fail
// records into it with atomicCAS(0 -> code) so the first failure sticks.
cudaError_t read_device_error(int *value, bool clear);
// Device address of the error word on the current device (for kernels of the
// other translation units, which record into the same word).
cudaError_t device_error_word(int **ptr);
// cuTensorMapEncodeTiled from the driver (nullptr when unavailable), as a
// PFN_cuTensorMapEncodeTiled_v12000.
void *tensor_map_encode_fn();
cudaError_t launch_wait_timeout_selftest(long long max_cycles, cudaStream_t stream);
cudaError_t launch_wait_drain_selftest(int ctas, long long first_cycles, cudaStream_t stream);
// The random-row gather probe (row_gather_probe.cu): `ctas` CTAs, each
// copying `tiles` 32 KB tiles of 1 << part_shift bytes of the rows idx picks.
cudaError_t launch_row_gather_probe(const void *table, int64_t rows, int64_t row_bytes, int part_shift,
                                    const int32_t *idx, int ctas, int tiles, cudaStream_t stream);

// ---- launchers (host side, enqueue only; arguments already validated) ----

struct AttnArgs {
    const void *q;          // bf16 [B,S,H,D]
    const void *kv;         // bf16 [B,T,D], or uint8 [B,T,584] FP8 rows when kv_fp8
    const float *sink;      // [H]
    const int32_t *idx;     // [B,S,K]
    const int32_t *topk_len;  // [B,S] or nullptr
    float scale;
    void *o;                // bf16 [B,S,H,D]
    int64_t B, S, H, D, T, K;
    int num_splits;         // >= 1 (planned over K + K2 slots)
    float *ws_o;            // fp32 [tokens, splits, H, D]   (splits > 1)
    float *ws_lse;          // fp32 [tokens, splits, H]      (splits > 1)
    // bit-mask mode (idx == nullptr, K == T): keys admitted by a packed mask
    const uint32_t *mask = nullptr;   // [B, mask_rows, mask_words]
    int64_t mask_rows = 0, mask_words = 0;
    int key_start_word = 0;           // 1: key offset read from mask[b, 0, mask_words - 1]
    bool kv_fp8 = false;              // kv rows in the FP8 format (D = 512)
    const int32_t *key_ends = nullptr;  // bit-mask mode: [B] live key end per request, or nullptr
    // extra kv source: K2 more slots per token (idx2 [B,S,K2]) over kv2
    // [B,T2,.] in kv's format, with an optional length topk_len2 [B,S]
    const void *kv2 = nullptr;
    const int32_t *idx2 = nullptr;
    const int32_t *topk_len2 = nullptr;
    int64_t T2 = 0, K2 = 0;
    // q / o hold io_S query rows per request and the call covers rows
    // io_s0 .. io_s0 + S - 1 of each (io_S = 0: io_S = S, io_s0 = 0)
    int64_t io_S = 0, io_s0 = 0;
};

// Slots handled by one split (a multiple of the 64-row tile).
int64_t split_slots(int64_t K, int num_splits);
// Largest number of slots one work unit (token, split) may hold.
int max_unit_slots();

cudaError_t launch_sparse_attn(const AttnArgs &a, int num_sms, cudaStream_t stream);
cudaError_t launch_attn_combine(const AttnArgs &a, cudaStream_t stream);
// Kernels one sparse_attn call enqueues on the current device: 1, or 2 when
// the splits are too many to combine inside the main kernel (0 on error).
int kernels_per_call(int64_t D, int num_splits, bool kv_fp8 = false);

// The packed consumer of the mask (D = 64, 128 or 256): G = 128 / H query
// tokens share the 128 MMA rows of a work unit, key tiles are dense.
bool masked_dense_packed(int64_t D);
// Its split count for these sizes (num_splits <= 0: planned), 0 when the key
// range cannot be split into at most 64 units.
int masked_dense_splits(int64_t B, int64_t S, int64_t H, int64_t D, int64_t T, int num_splits, int num_sms);
// The packed consumer, then the combine kernel when a.num_splits > 1 (the
// workspace layout of the sparse_attn splits).
cudaError_t launch_masked_dense(const AttnArgs &a, cudaStream_t stream);

struct MaskArgs {
    const int32_t *topk;
    int64_t topk_rows;
    const int32_t *cu_q_lens;
    int64_t B, max_q_len, max_key_len, K;
    const int32_t *key_starts;
    uint32_t *mask;
    int64_t rows, words;    // mask shape [B, rows, words]
    int64_t q0 = 0;                    // mask row i is query q0 + i of each request
    const int32_t *key_ends = nullptr; // [B] live key end per request, or nullptr
};
cudaError_t launch_build_topk_mask(const MaskArgs &a, int num_sms, cudaStream_t stream);

}  // namespace sa
