// Bit-packed top-k mask builder.
//
// Semantics: vLLM PR 52217 page (`_build_topk_mask`: top-k indices scattered
// into 32-bit words, rows padded to a multiple of 4 words and the padding left
// in place) and vLLM PR 48770 page (`dense_mask_mod`: word kv>>5, bit kv&31,
// LSB first; `offset_dense_mask_mod`: key_start in the last word of row 0).
//
// Design: one CTA builds one mask row at a time in shared memory -- the row
// image is cleared, every index of the row is OR-ed in with a shared-memory
// atomic, and the live words go out with 16-byte stores.  The pages' Triton
// scatter ORs straight into global memory; building in shared memory turns
// K scattered 4-byte global atomics per row into ceil(keys/128) coalesced
// 16-byte stores, so the kernel is bound by the streaming read of the
// indices.  Rows wider than kSmemWordsMax words fall back to global atomics.
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kMaskThreads = 256;
constexpr int64_t kSmemWordsMax = 8192;  // 32 KB row image: up to 262144 keys

__device__ __forceinline__ void or_bit(uint32_t *img, int32_t k, uint32_t key_limit) {
    // (uint32_t)k < key_limit rejects negative and too-large indices at once
    if (static_cast<uint32_t>(k) < key_limit) atomicOr(&img[k >> 5], 1u << (k & 31));
}

__device__ __forceinline__ void scatter_row(const int32_t *__restrict__ row, int64_t K,
                                            uint32_t key_limit, uint32_t *img) {
    const bool vec = (K % 4 == 0) && ((reinterpret_cast<uintptr_t>(row) & 15) == 0);
    if (vec) {
        const int4 *r4 = reinterpret_cast<const int4 *>(row);
        const int64_t n4 = K / 4;
        for (int64_t v = threadIdx.x; v < n4; v += blockDim.x) {
            const int4 x = __ldcs(r4 + v);  // streamed once: evict-first
            or_bit(img, x.x, key_limit);
            or_bit(img, x.y, key_limit);
            or_bit(img, x.z, key_limit);
            or_bit(img, x.w, key_limit);
        }
    } else {
        for (int64_t j = threadIdx.x; j < K; j += blockDim.x) or_bit(img, __ldcs(row + j), key_limit);
    }
}

__global__ void __launch_bounds__(kMaskThreads)
build_topk_mask_kernel(MaskArgs a, int64_t live_words, int smem_path) {
    extern __shared__ __align__(16) uint32_t row_img[];
    const uint32_t key_limit = static_cast<uint32_t>(a.max_key_len);

    // reserved key_start word of row (b, 0), for every request b
    if (a.key_starts != nullptr && a.rows > 0) {
        for (int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; b < a.B;
             b += int64_t(gridDim.x) * blockDim.x)
            a.mask[(b * a.rows) * a.words + (a.words - 1)] = static_cast<uint32_t>(a.key_starts[b]);
    }

    const int64_t n_slots = a.B * a.max_q_len;
    for (int64_t r = blockIdx.x; r < n_slots; r += gridDim.x) {
        // everything below is uniform across the CTA
        const int64_t b = r / a.max_q_len, q = r % a.max_q_len;
        const int64_t c0 = a.cu_q_lens[b], c1 = a.cu_q_lens[b + 1];
        if (q >= c1 - c0) continue;
        const int64_t src = c0 + q;
        if (src < 0 || src >= a.topk_rows) continue;
        const int32_t *row = a.topk + src * a.K;
        uint32_t *dst = a.mask + (b * a.rows + q) * a.words;

        if (smem_path) {
            for (int64_t w = threadIdx.x; w < live_words; w += blockDim.x) row_img[w] = 0u;
            __syncthreads();
            scatter_row(row, a.K, key_limit, row_img);
            __syncthreads();
            const int64_t nvec = live_words / 4;
            uint4 *d4 = reinterpret_cast<uint4 *>(dst);  // rows start on 16 B (words % 4 == 0)
            const uint4 *s4 = reinterpret_cast<const uint4 *>(row_img);
            for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) d4[v] = s4[v];
            for (int64_t w = nvec * 4 + threadIdx.x; w < live_words; w += blockDim.x) dst[w] = row_img[w];
            __syncthreads();  // row_img is reused by the next row
        } else {
            for (int64_t w = threadIdx.x; w < live_words; w += blockDim.x) dst[w] = 0u;
            __syncthreads();  // CTA-scope ordering of the clears before the ORs
            scatter_row(row, a.K, key_limit, dst);
            __syncthreads();
        }
    }
}

}  // namespace

cudaError_t launch_build_topk_mask(const MaskArgs &a, int num_sms, cudaStream_t stream) {
    const int64_t live_words = (a.max_key_len + 31) / 32;
    const int64_t n_slots = a.B * a.max_q_len;
    const bool need_ks = a.key_starts != nullptr && a.rows > 0 && a.B > 0;
    if (n_slots == 0 && !need_ks) return cudaSuccess;
    const int smem_path = live_words <= kSmemWordsMax ? 1 : 0;
    const size_t smem = smem_path ? size_t(((live_words + 3) / 4) * 4) * sizeof(uint32_t) : 0;
    int64_t grid = n_slots;
    const int64_t cap = int64_t(num_sms) * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    build_topk_mask_kernel<<<static_cast<unsigned>(grid), kMaskThreads, smem, stream>>>(a, live_words,
                                                                                       smem_path);
    return cudaGetLastError();
}

}  // namespace sa
