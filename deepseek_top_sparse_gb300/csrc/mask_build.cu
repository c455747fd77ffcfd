// Bit-packed top-k mask builder.
//
// Semantics: vLLM PR 52217 page (`_build_topk_mask`: top-k indices scattered
// into 32-bit words, rows padded to a multiple of 4 words and the padding left
// in place) and vLLM PR 48770 page (`dense_mask_mod`: word kv>>5, bit kv&31,
// LSB first; `offset_dense_mask_mod`: key_start in the last word of row 0).
//
// Design: a row is built in shared memory -- its image is cleared, every
// index of the row is OR-ed in with a shared-memory atomic, and the live words
// go out with 16-byte stores.  The pages' Triton scatter ORs straight into
// global memory; building in shared memory turns K scattered 4-byte global
// atomics per row into ceil(keys/128) coalesced 16-byte stores (on GB300, L2
// atomics measured 4x slower than shared-memory ones for this pattern).
//   * rows of up to kWarpRowWords words: one WARP per row, each warp with its
//     own image, so a CTA has 8 rows in flight and needs no CTA barrier.  The
//     row image is ORed with shared-memory atomics, whose bank conflicts on
//     random words bound the kernel; narrow rows are sized for occupancy (32
//     registers, 8 CTAs per SM), which measured faster than deep per-lane
//     load queues.
//   * wider rows up to kSmemWordsMax words: one CTA per row.
//   * wider still: global atomics straight into the output row.
#include "ptx.cuh"
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kMaskThreads = 256;
constexpr int kMaskWarps = kMaskThreads / 32;
constexpr int64_t kSmemWordsMax = 8192;  // 32 KB row image: up to 262144 keys
constexpr int64_t kWarpRowWords = 2048;  // 8 KB image per warp: up to 65536 keys
// Row images of up to kSmallRowWords words let 8 CTAs of 8 warps share an SM:
// those rows take the 32-register variant with 2 16-byte index loads per lane
// in flight; wider images limit occupancy anyway, so their variant keeps 8
// loads per lane in flight instead.
constexpr int64_t kSmallRowWords = 768;

// Live key end of request b: max_key_len, or its entry of key_ends clamped to
// [0, max_key_len] (the build then stops at that row's end).
__device__ __forceinline__ uint32_t live_end(const int32_t *key_ends, int64_t b, uint32_t max_key) {
    if (key_ends == nullptr) return max_key;
    const int32_t e = key_ends[b];
    return e <= 0 ? 0u : (uint32_t(e) < max_key ? uint32_t(e) : max_key);
}

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
build_topk_mask_kernel(MaskArgs a, int smem_path) {
    ptx::griddep_wait();               // the stream's previous kernel: complete and visible
    ptx::griddep_launch_dependents();
    extern __shared__ __align__(16) uint32_t row_img[];
    const uint32_t max_key = static_cast<uint32_t>(a.max_key_len);

    // reserved key_start word of row (b, 0), for every request b
    if (a.key_starts != nullptr && a.rows > 0) {
        for (int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; b < a.B;
             b += int64_t(gridDim.x) * blockDim.x)
            a.mask[(b * a.rows) * a.words + (a.words - 1)] = static_cast<uint32_t>(a.key_starts[b]);
    }

    const int64_t n_slots = a.B * a.max_q_len;
    for (int64_t r = blockIdx.x; r < n_slots; r += gridDim.x) {
        // everything below is uniform across the CTA
        const int64_t b = r / a.max_q_len, i = r % a.max_q_len, q = a.q0 + i;
        const int64_t c0 = a.cu_q_lens[b], c1 = a.cu_q_lens[b + 1];
        if (q >= c1 - c0) continue;
        const int64_t src = c0 + q;
        if (src < 0 || src >= a.topk_rows) continue;
        const int32_t *row = a.topk + src * a.K;
        uint32_t *dst = a.mask + (b * a.rows + i) * a.words;
        const uint32_t key_limit = live_end(a.key_ends, b, max_key);
        const int64_t live_words = (int64_t(key_limit) + 31) / 32;

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

// Arguments of the warp-per-row path, every count below 2^31 (the host checks)
// so the kernel fits 32 registers and 8 CTAs per SM with no spills.
struct WarpMaskArgs {
    const int32_t *topk;
    const int32_t *cu_q_lens;
    const int32_t *key_starts;
    uint32_t *mask;
    const int32_t *key_ends;   // [B] or nullptr
    int topk_rows, B, max_q_len, K, rows, words, live_words, q0;
    uint32_t key_limit;
};

template <int kLoadsInFlight, int kMinBlocks>
__global__ void __launch_bounds__(kMaskThreads, kMinBlocks)
build_topk_mask_warp_kernel(WarpMaskArgs a) {
    ptx::griddep_wait();               // the stream's previous kernel: complete and visible
    ptx::griddep_launch_dependents();
    extern __shared__ __align__(16) uint32_t images[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int img_words = (a.live_words + 3) / 4 * 4;
    uint32_t *img = images + warp * img_words;

    if (a.key_starts != nullptr && a.rows > 0) {
        for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < a.B; b += gridDim.x * blockDim.x)
            a.mask[(int64_t(b) * a.rows) * a.words + (a.words - 1)] = static_cast<uint32_t>(a.key_starts[b]);
    }

    const int n_slots = a.B * a.max_q_len;
    for (int r = blockIdx.x * kMaskWarps + warp; r < n_slots; r += gridDim.x * kMaskWarps) {
        // everything below is uniform across the warp
        const int b = r / a.max_q_len, i = r - b * a.max_q_len, q = a.q0 + i;
        const int c0 = a.cu_q_lens[b], c1 = a.cu_q_lens[b + 1];
        if (q >= c1 - c0) continue;
        const int64_t src = int64_t(c0) + q;
        if (src < 0 || src >= a.topk_rows) continue;
        const int32_t *row = a.topk + src * a.K;
        uint32_t *dst = a.mask + (int64_t(b) * a.rows + i) * a.words;
        const uint32_t key_limit = live_end(a.key_ends, b, a.key_limit);
        const int live_words = int((key_limit + 31u) / 32u);

        for (int w = lane; w < img_words; w += 32) img[w] = 0u;
        __syncwarp();
        if ((a.K % 4 == 0) && ((reinterpret_cast<uintptr_t>(row) & 15) == 0)) {
            const int4 *r4 = reinterpret_cast<const int4 *>(row);
            const int n4 = a.K / 4;
            for (int base = lane; base < n4; base += 32 * kLoadsInFlight) {
                int4 x[kLoadsInFlight];
#pragma unroll
                for (int u = 0; u < kLoadsInFlight; ++u) {
                    const int v = base + u * 32;
                    x[u] = v < n4 ? __ldcs(r4 + v) : make_int4(-1, -1, -1, -1);
                }
#pragma unroll
                for (int u = 0; u < kLoadsInFlight; ++u) {
                    or_bit(img, x[u].x, key_limit);
                    or_bit(img, x[u].y, key_limit);
                    or_bit(img, x[u].z, key_limit);
                    or_bit(img, x[u].w, key_limit);
                }
            }
        } else {
            for (int j = lane; j < a.K; j += 32) or_bit(img, __ldcs(row + j), key_limit);
        }
        __syncwarp();
        const int nvec = live_words / 4;
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);  // rows start on 16 B (words % 4 == 0)
        const uint4 *s4 = reinterpret_cast<const uint4 *>(img);
        for (int v = lane; v < nvec; v += 32) d4[v] = s4[v];
        for (int w = nvec * 4 + lane; w < live_words; w += 32) dst[w] = img[w];
        __syncwarp();  // the image is reused by the warp's next row
    }
}

}  // namespace

cudaError_t launch_build_topk_mask(const MaskArgs &a, int num_sms, cudaStream_t stream) {
    const int64_t live_words = (a.max_key_len + 31) / 32;
    const int64_t n_slots = a.B * a.max_q_len;
    const bool need_ks = a.key_starts != nullptr && a.rows > 0 && a.B > 0;
    if (n_slots == 0 && !need_ks) return cudaSuccess;
    const int64_t cap = int64_t(num_sms) * 8;
    const int64_t lim31 = int64_t(1) << 31;
    if (live_words <= kWarpRowWords && a.K < lim31 && a.topk_rows < lim31 && n_slots < lim31 &&
        a.B + 1 < lim31 && a.rows < lim31 && a.words < lim31 && a.q0 + a.max_q_len < lim31) {
        WarpMaskArgs w;
        w.topk = a.topk; w.cu_q_lens = a.cu_q_lens; w.key_starts = a.key_starts; w.mask = a.mask;
        w.key_ends = a.key_ends; w.q0 = int(a.q0);
        w.topk_rows = int(a.topk_rows); w.B = int(a.B); w.max_q_len = int(a.max_q_len); w.K = int(a.K);
        w.rows = int(a.rows); w.words = int(a.words); w.live_words = int(live_words);
        w.key_limit = static_cast<uint32_t>(a.max_key_len);
        const size_t smem = size_t(kMaskWarps) * size_t((live_words + 3) / 4 * 4) * sizeof(uint32_t);
        int64_t grid = (n_slots + kMaskWarps - 1) / kMaskWarps;
        if (grid > cap) grid = cap;
        if (grid < 1) grid = 1;
        if (live_words <= kSmallRowWords) {
            const cudaError_t e = launch_pdl(build_topk_mask_warp_kernel<2, 8>, dim3(unsigned(grid)), dim3(kMaskThreads),
                                             smem, stream, w);
            if (e != cudaSuccess) return e;
        } else {
            auto kern = build_topk_mask_warp_kernel<8, 3>;
            if (smem > 48 * 1024) {
                const cudaError_t e =
                    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
                if (e != cudaSuccess) return e;
            }
            const cudaError_t e2 = launch_pdl(kern, dim3(unsigned(grid)), dim3(kMaskThreads), smem, stream, w);
            if (e2 != cudaSuccess) return e2;
        }
        return cudaGetLastError();
    }
    const int smem_path = live_words <= kSmemWordsMax ? 1 : 0;
    const size_t smem = smem_path ? size_t(((live_words + 3) / 4) * 4) * sizeof(uint32_t) : 0;
    int64_t grid = n_slots;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    const cudaError_t e = launch_pdl(build_topk_mask_kernel, dim3(unsigned(grid)), dim3(kMaskThreads), smem, stream, a,
                                     smem_path);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sa
