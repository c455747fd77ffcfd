// First CUDA path for sparse_attn: one warp per (token, head), CUDA cores.
//
// "DeepSeek V4 源码剖析, 第5章" §5.2 (semantics) and §5.5 (online softmax with
// the sink added to the denominator after the loop).  Each lane owns D/32
// contiguous elements of q and of the output row; for every valid slot the
// warp reads the indexed kv row once (coalesced), reduces q.k with shuffles and
// updates the running max / sum / accumulator in base 2.
#include <cuda_bf16.h>

#include "sa_internal.h"

namespace sa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int E>  // elements per lane: D / 32
__global__ void __launch_bounds__(128)
attn_simt_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ kv,
                 const float *__restrict__ sink, const int32_t *__restrict__ idx, float scale_log2,
                 __nv_bfloat16 *__restrict__ o, int64_t S, int64_t H, int64_t T, int64_t K) {
    constexpr int D = 32 * E;
    const int lane = threadIdx.x & 31;
    const int64_t h = int64_t(blockIdx.y) * 4 + (threadIdx.x >> 5);
    const int64_t tok = blockIdx.x;
    if (h >= H) return;
    const int64_t b = tok / S;

    float qf[E], acc[E];
    const __nv_bfloat16 *qrow = q + (tok * H + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qf[e] = __bfloat162float(qrow[e]);
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const int32_t *irow = idx + tok * K;
    const __nv_bfloat16 *kvb = kv + b * T * D;
    for (int64_t j = 0; j < K; ++j) {
        const int32_t t = __ldg(irow + j);
        if (t < 0 || t >= T) continue;  // warp-uniform
        const __nv_bfloat16 *kr = kvb + int64_t(t) * D + lane * E;
        float kf[E];
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            kf[e] = __bfloat162float(kr[e]);
            dot = fmaf(qf[e], kf[e], dot);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float x = dot * scale_log2;
        const float m_new = fmaxf(m, x);
        const float alpha = exp2f(m - m_new);
        const float p = exp2f(x - m_new);
        l = l * alpha + p;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(acc[e], alpha, p * kf[e]);
        m = m_new;
    }
    // sink joins the denominator once, after the loop
    const float s2 = sink[h] * kLog2e;
    float f = 0.f;
    if (!(s2 == INFINITY)) {
        const float M = fmaxf(m, s2);
        if (M != -INFINITY) {
            const float den = l * exp2f(m - M) + exp2f(s2 - M);
            f = exp2f(m - M) / den;
        }
        if (isnan(s2)) f = NAN;
    }
    __nv_bfloat16 *orow = o + (tok * H + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) orow[e] = __float2bfloat16_rn(m == -INFINITY ? 0.f : acc[e] * f);
}

}  // namespace

int64_t split_slots(int64_t K, int num_splits) {
    const int64_t tiles = (K + 63) / 64;
    const int64_t per = (tiles + num_splits - 1) / num_splits;
    return per * 64;
}

cudaError_t launch_sparse_attn(const AttnArgs &a, int num_sms, cudaStream_t stream) {
    (void)num_sms;
    const int64_t tokens = a.B * a.S;
    if (tokens == 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>(tokens), static_cast<unsigned>((a.H + 3) / 4));
    const float sl2 = a.scale * kLog2e;
    auto q = static_cast<const __nv_bfloat16 *>(a.q);
    auto kv = static_cast<const __nv_bfloat16 *>(a.kv);
    auto o = static_cast<__nv_bfloat16 *>(a.o);
    switch (a.D) {
        case 64: attn_simt_kernel<2><<<grid, 128, 0, stream>>>(q, kv, a.sink, a.idx, sl2, o, a.S, a.H, a.T, a.K); break;
        case 128: attn_simt_kernel<4><<<grid, 128, 0, stream>>>(q, kv, a.sink, a.idx, sl2, o, a.S, a.H, a.T, a.K); break;
        case 256: attn_simt_kernel<8><<<grid, 128, 0, stream>>>(q, kv, a.sink, a.idx, sl2, o, a.S, a.H, a.T, a.K); break;
        case 512: attn_simt_kernel<16><<<grid, 128, 0, stream>>>(q, kv, a.sink, a.idx, sl2, o, a.S, a.H, a.T, a.K); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_attn_combine(const AttnArgs &, cudaStream_t) { return cudaSuccess; }

static __device__ int g_device_error = 0;

cudaError_t read_device_error(int *value, bool clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
    if (e != cudaSuccess) return e;
    if (clear) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    }
    return e;
}

}  // namespace sa
