// Random-row gather rate of this GPU.
//
// The kv gather of sparse_attn ("DeepSeek V4 源码剖析, 第5章" §5.6: the
// index-driven gather of kv rows) pulls one row per valid slot from random
// places in an HBM-resident cache.  How fast any gather of that kind can go is
// a property of the memory system, not of the attention kernel: this probe
// measures it so that the kernel's gathered bytes can be read against it as
// well as against the copy bandwidth.  It is not part of the attention path.
//
// One CTA per SM (the caller picks the grid): CTA c streams `tiles` tiles of
// 32 KB, each the first `part` bytes of 32768 / part rows picked by idx, into
// shared memory with 16-byte cp.async from 8 warps, through a 6-stage ring
// (each stage's mbarrier counts every thread's cp.async.mbarrier.arrive.noinc
// and is waited, bounded, before the stage is refilled), and discards them.
// Every CTA waits for its own copies before it exits.
#include "ptx.cuh"
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeStages = 6;
constexpr int kProbeStageBytes = 32768;
constexpr long long kProbeWaitCycles = 200000000ll;   // ~0.1 s at 2 GHz

// Bounded wait: false after kProbeWaitCycles (recording the timeout in the
// library's error word) or as soon as any wait has recorded an error.
__device__ __forceinline__ bool probe_wait(uint32_t bar, uint32_t parity, int *err) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((n & 1023u) == 0) {
            if (*reinterpret_cast<volatile int *>(err) != 0) return false;
            if (clock64() - t0 > kProbeWaitCycles) {
                atomicCAS(err, 0, int(kErrWaitTimeout));
                return false;
            }
        }
    }
}

// part = 1 << part_shift bytes of each row, 16 <= part <= 32768; idx values
// outside [0, rows) read row 0.
__global__ void __launch_bounds__(kProbeThreads, 1)
row_gather_probe_kernel(const uint8_t *__restrict__ table, int64_t row_bytes, int part_shift,
                        const int32_t *__restrict__ idx, int32_t rows, int tiles, int *err) {
    extern __shared__ uint8_t probe_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(probe_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bars[kProbeStages];
    const int tid = threadIdx.x;
    const int chunk_shift = part_shift - 4;                        // 16-byte chunks of a row part
    const int rows_per_tile = kProbeStageBytes >> part_shift;
    if (tid == 0) {
        for (int s = 0; s < kProbeStages; ++s) ptx::mbar_init(ptx::smem_u32(&bars[s]), kProbeThreads);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const int32_t *tix = idx + int64_t(blockIdx.x) * tiles * rows_per_tile;
    for (int t = 0; t < tiles; ++t) {
        const int s = t % kProbeStages;
        const uint32_t bar = ptx::smem_u32(&bars[s]);
        if (t >= kProbeStages && !__all_sync(0xffffffffu, probe_wait(bar, uint32_t(t / kProbeStages - 1) & 1u, err)))
            break;
        const uint32_t stage = ptx::smem_u32(sm + s * kProbeStageBytes);
        const int32_t *trows = tix + int64_t(t) * rows_per_tile;
#pragma unroll 4
        for (int it = tid; it < kProbeStageBytes / 16; it += kProbeThreads) {
            const int r = it >> chunk_shift, ch = it & ((1 << chunk_shift) - 1);
            const int32_t row = trows[r];
            const int64_t rr = (row >= 0 && row < rows) ? row : 0;
            ptx::cp_async_16(stage + uint32_t(it) * 16u, table + rr * row_bytes + (int64_t(ch) << 4), 16u);
        }
        ptx::cp_async_arrive_noinc(bar);
    }
    ptx::cp_async_wait_all();   // nothing of ours lands after the CTA exits
}

}  // namespace

cudaError_t launch_row_gather_probe(const void *table, int64_t rows, int64_t row_bytes, int part_shift,
                                    const int32_t *idx, int ctas, int tiles, cudaStream_t stream) {
    int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    const int smem = kProbeStages * kProbeStageBytes + 1024;
    e = cudaFuncSetAttribute(row_gather_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    row_gather_probe_kernel<<<ctas, kProbeThreads, smem, stream>>>(static_cast<const uint8_t *>(table), row_bytes,
                                                                   part_shift, idx, int32_t(rows), tiles, err);
    return cudaGetLastError();
}

}  // namespace sa
