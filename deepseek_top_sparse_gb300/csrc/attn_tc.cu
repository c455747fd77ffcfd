// sparse_attn on the sm_103a tensor cores (tcgen05 + TMEM).
//
// What it computes: "DeepSeek V4 源码剖析, 第5章" §5.2 -- for each query
// token, gather K indexed rows of the token's kv (-1 = invalid slot), logits =
// scale * q.k for all H heads, softmax together with a per-head sink logit,
// output = weighted sum of the gathered rows (V is the same row as K, the
// sink's weight is dropped).  §5.5: online softmax over 64-row tiles with the
// sink added to the denominator once at the end; with split-KV the sink is
// applied once, in the log-sum-exp combine.
//
// Work unit = (query token, KV split).  One unit runs on CL CTAs (a cluster
// of 2 when D = 512): CTA c owns columns [c*DC, (c+1)*DC) of q, of every
// gathered kv row and of o.  Tiles of 64 slots whose slots are all invalid
// are skipped, so the cost follows the live slots.  Per CTA:
//
//   warps 5.. (gather)  one warp per shared-memory stage; each warp copies the
//                       DC-column slice of its tile's 64 indexed kv rows with
//                       16-byte cp.async (one 512-byte row slice per warp
//                       instruction, invalid slots zero-filled), writing the
//                       128B-swizzled K-major layout the MMAs read;
//   warp 4 (MMA)        S = Q_c K_c^T with Q_c resident in TMEM (A operand
//                       from tensor memory), two S buffers in TMEM; O_c += P V_c
//                       with P and V_c (= the same stage, read MN-major) in
//                       shared memory, O_c resident in TMEM for the whole unit.
//                       Issue is event driven: S of a tile may run up to two
//                       tiles ahead of the P.V that trails it;
//   warps 0..3          one thread per head row (= TMEM lane): the partial
//                       logits of tile a+1 go to the partner CTA (distributed
//                       shared memory) before tile a is finished, so the swap
//                       overlaps the softmax; both CTAs add S_0 + S_1 (fp32
//                       addition commutes: identical logits on both), mask
//                       invalid slots, run the online softmax in base 2 with a
//                       lazily rescaled running max and store P (bf16).
//
// TMEM columns (D = 512, DC = 256): O_c [0,256) fp32, S [256,384) two 64-col
// buffers, Q_c [384,512) bf16 pairs.  Every buffer hand-off is an mbarrier
// phase that is never more than one phase away from its waiter, and every
// wait is bounded by the global timer: a wait that runs out records an error
// code and the kernel drains and returns instead of hanging.
#include <cuda_bf16.h>

#include <mutex>

#include "ptx.cuh"
#include "sa_internal.h"

namespace sa {

static __device__ int g_device_error = 0;

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBN = 64;                 // kv rows per tile (MMA N of S, K of P.V)
constexpr int kM = 128;                 // head rows per MMA (TMEM lanes)
constexpr int kMaxUnitSlots = 2048;     // slots per work unit (host enforces)
constexpr int kMaxUnitTiles = kMaxUnitSlots / kBN;
// Bound on any single wait, in SM clock cycles (~2 s at 2 GHz): far beyond
// any legitimate wait.  clock64 is read only after 1024 unsuccessful polls.
constexpr long long kWaitCycles = 4000000000ll;
constexpr float kRescaleThreshold = 8.f;     // log2 units: P <= 256 before normalising
constexpr int kSoftmaxWarps = 8;              // two per TMEM lane quarter, 32 columns each
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kMmaWarp = kSoftmaxWarps;
constexpr int kFirstGatherWarp = kMmaWarp + 1;
constexpr int kGatherWarps = 2;               // both fill every tile, 32 rows each
// A gather warp publishes tile a once it has issued tile a + kGatherLag
// (kGatherLag + 1 tiles in flight per warp).  The softmax needs S(a+1) to
// finish tile a, so publication may not wait on stage reuse past tile a-2:
// kGatherLag <= stages - 2.
constexpr int kGatherLag = 1;

template <int DC, int CL>
struct Cfg {
    static_assert(DC == 64 || DC == 128 || DC == 256, "per-CTA head-dim slice");
    static constexpr int STAGE_BYTES = kBN * DC * 2;
    static constexpr int NS = 4;                          // kv ring depth
    static_assert(kGatherLag <= NS - 2, "gather publication must not depend on the tile being finished");
    static constexpr int THREADS = (kFirstGatherWarp + kGatherWarps) * 32;
    static constexpr int X_BYTES = kM * kBN * 4;          // 32 KB fp32 partial logits
    static constexpr int OFF_KV = 0;
    static constexpr int OFF_X = OFF_KV + NS * STAGE_BYTES;
    static constexpr int OFF_IDX = OFF_X + (CL == 2 ? 2 * X_BYTES : 0);
    static constexpr int OFF_VALID = OFF_IDX + kMaxUnitSlots * 4;
    static constexpr int OFF_LIST = OFF_VALID + kMaxUnitTiles * 8;
    static constexpr int OFF_RED = OFF_LIST + kMaxUnitTiles * 4 + 16;   // float [3][2][128]
    static constexpr int OFF_BAR = OFF_RED + 3 * 2 * kM * 4;
    // kv_full[NS] kv_empty[NS] s_full s_empty p_full[2] p_empty[2]
    // x_full[2] x_empty[2] o_done q_ready mma_done red_bar l_bar
    static constexpr int NUM_BARS = 2 * NS + 15;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM = OFF_TSLOT + 16 + 1024;    // + slack to align the base to 1 KB
    // TMEM columns: O_c fp32, S fp32 (one tile), P bf16 pairs (two tiles), Q_c bf16 pairs
    static constexpr int O_COL = 0;
    static constexpr int S_COL = DC;
    static constexpr int P_COL = DC + kBN;
    static constexpr int Q_COL = DC + 2 * kBN;
    static constexpr int TMEM_USED = Q_COL + DC / 2;
    static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
    static_assert(TMEM_USED <= 512, "TMEM budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

struct TcParams {
    const __nv_bfloat16 *q;   // [tokens, H, D]
    const __nv_bfloat16 *kv;  // [B, T, D]
    const float *sink;        // [H]
    const int32_t *idx;       // [tokens, K]
    __nv_bfloat16 *o;         // [tokens, H, D]
    float *ws_o;              // [tokens, splits, H, D]
    float *ws_lse;            // [tokens, splits, H]
    int64_t S, H, D, T, K;
    int num_splits;
    int unit_slots;           // slots per split, a multiple of kBN, <= kMaxUnitSlots
    float scale_log2;         // softmax_scale * log2(e)
};

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_device_error, 0, code); }

template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity) {
    auto poll = [&] { return kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity); };
    if (poll()) return true;
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        if (poll()) return true;
        if ((n & 1023u) == 0 && clock64() - t0 > kWaitCycles) {
            record_error(kErrWaitTimeout);
            return false;
        }
    }
}

// warp-uniform bounded wait (the warp leaves together or not at all)
template <bool kCluster = false>
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_bar<kCluster>(bar, parity));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b, float &sum) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    sum += __low2float(v) + __high2float(v);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <int DC, int CL>
__global__ void __launch_bounds__(Cfg<DC, CL>::THREADS, 1)
attn_tc_kernel(const TcParams p) {
    using C = Cfg<DC, CL>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = CL == 2 ? ptx::cluster_ctarank() : 0u;
    const int64_t unit = blockIdx.x / CL;
    const int64_t tok = unit / p.num_splits;
    const int split = int(unit % p.num_splits);
    const int64_t b = tok / p.S;
    const int64_t slot0 = int64_t(split) * p.unit_slots;
    const int64_t left = p.K - slot0;
    const int nslots = left <= 0 ? 0 : int(left < p.unit_slots ? left : p.unit_slots);
    const int ntiles = (nslots + kBN - 1) / kBN;

    int32_t *rowc = reinterpret_cast<int32_t *>(smem + C::OFF_IDX);
    uint64_t *vmask = reinterpret_cast<uint64_t *>(smem + C::OFF_VALID);
    int32_t *act = reinterpret_cast<int32_t *>(smem + C::OFF_LIST);  // act[0..n) tiles, act[kMaxUnitTiles] = n
    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);      // [3][2][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::OFF_TSLOT);
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    auto kv_full = [&](int s) { return bar(s); };
    auto kv_empty = [&](int s) { return bar(C::NS + s); };
    const uint32_t s_full = bar(2 * C::NS);
    const uint32_t s_empty = bar(2 * C::NS + 1);
    auto p_full = [&](int i) { return bar(2 * C::NS + 2 + i); };
    auto p_empty = [&](int i) { return bar(2 * C::NS + 4 + i); };
    auto x_full = [&](int i) { return bar(2 * C::NS + 6 + i); };
    auto x_empty = [&](int i) { return bar(2 * C::NS + 8 + i); };
    const uint32_t o_done = bar(2 * C::NS + 10);
    const uint32_t q_ready = bar(2 * C::NS + 11);
    const uint32_t mma_done = bar(2 * C::NS + 12);
    const uint32_t red_bar = bar(2 * C::NS + 13);
    const uint32_t l_bar = bar(2 * C::NS + 14);

    // ---------------------------------------------------------------- prologue
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_u32(tslot), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < C::NS; ++s) {
            ptx::mbar_init(kv_full(s), 32 * kGatherWarps);
            ptx::mbar_init(kv_empty(s), 1);
        }
        ptx::mbar_init(s_full, 1);
        ptx::mbar_init(s_empty, kSoftmaxThreads);
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(p_full(i), kSoftmaxThreads);
            ptx::mbar_init(p_empty(i), 1);
            ptx::mbar_init(x_full(i), 1);   // + X_BYTES of st.async complete_tx per phase
            ptx::mbar_init(x_empty(i), 1);  // one credit per phase from the partner
        }
        ptx::mbar_init(o_done, 1);
        ptx::mbar_init(q_ready, kSoftmaxThreads);
        ptx::mbar_init(mma_done, 1);
        ptx::mbar_init(red_bar, kSoftmaxThreads);
        ptx::mbar_init(l_bar, kSoftmaxThreads);
        ptx::fence_mbar_init();
    }
    // slot indices -> kv row numbers (-1 = invalid) and a 64-bit validity
    // mask per tile, 32 slots per warp step
    {
        const int32_t *irow = p.idx + tok * p.K + slot0;
        for (int ch = warp; ch < ntiles * 2; ch += C::THREADS / 32) {
            const int j = ch * 32 + lane;
            const int32_t t = j < nslots ? __ldg(irow + j) : -1;
            const bool v = t >= 0 && int64_t(t) < p.T;
            rowc[j] = v ? int32_t(b * p.T + t) : -1;
            const uint32_t m = __ballot_sync(0xffffffffu, v);
            if (lane == 0) reinterpret_cast<uint32_t *>(vmask)[ch] = m;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int n = 0;
        for (int t = 0; t < ntiles; ++t)
            if (vmask[t] != 0) act[n++] = t;
        act[kMaxUnitTiles] = n;
    }
    ptx::tc_fence_before();
    if constexpr (CL == 2) {
        ptx::cluster_sync();  // partner barriers initialised before any remote access
    } else {
        __syncthreads();
    }
    ptx::tc_fence_after();
    const uint32_t tbase = *tslot;
    const int n_act = act[kMaxUnitTiles];

    if (warp >= kFirstGatherWarp) {
        // ------------------------------------------------------------ gather
        // every gather warp copies its share of the rows of every tile; a tile
        // is published (fence + arrive) once the warp has issued kGatherLag
        // more, so kGatherLag + 1 tiles per warp are in flight
        constexpr int CPR = DC / 8;     // 16-byte chunks per row slice
        constexpr int RPI = 32 / CPR;   // rows per warp instruction
        constexpr int RPW = kBN / kGatherWarps;
        const int g = warp - kFirstGatherWarp;
        const int sub = lane / CPR, ch = lane % CPR;
        const uint32_t dst_col = uint32_t(ch >> 3) * (kBN * 128);
        const char *kvb = reinterpret_cast<const char *>(p.kv) + (int64_t(crank) * DC + ch * 8) * 2;
        bool ok = true;
        int a = 0;
        for (; a < n_act; ++a) {
            const int s = a % C::NS, f = a / C::NS;
            if (f >= 1 && !wait_all(kv_empty(s), (f - 1) & 1)) {
                ok = false;
                break;
            }
            const uint32_t stage = ptx::smem_u32(smem + C::OFF_KV + s * C::STAGE_BYTES);
            const int32_t *rc = rowc + act[a] * kBN;
#pragma unroll
            for (int i = 0; i < RPW / RPI; ++i) {
                const int r = g * RPW + i * RPI + sub;
                const int32_t row = rc[r];
                const char *src = kvb + (row >= 0 ? int64_t(row) : 0) * p.D * 2;
                const uint32_t dst = stage + dst_col + uint32_t(r) * 128u + uint32_t((ch & 7) ^ (r & 7)) * 16u;
                ptx::cp_async_16(dst, src, row >= 0 ? 16u : 0u);
            }
            ptx::cp_async_commit();
            if (a >= kGatherLag) {
                asm volatile("cp.async.wait_group %0;" ::"n"(kGatherLag) : "memory");
                ptx::fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
                ptx::mbar_arrive(kv_full((a - kGatherLag) % C::NS));
            }
        }
        ptx::cp_async_wait_all();
        if (ok) {
            ptx::fence_proxy_async_smem();
            for (int k = a - kGatherLag < 0 ? 0 : a - kGatherLag; k < a; ++k) ptx::mbar_arrive(kv_full(k % C::NS));
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(kM, kBN, false);
            constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(kM, DC, true);
            bool ok = wait_bar(q_ready, 0);
            ptx::tc_fence_after();
            int qn = 0, pn = 0;
            uint32_t idle = 0;
            long long t0 = 0;
            while (ok && pn < n_act) {
                bool prog = false;
                // S(q) overwrites the single S buffer once S(q-1) has been read
                if (qn < n_act && qn <= pn + 2 && ptx::mbar_test_wait(kv_full(qn % C::NS), (qn / C::NS) & 1) &&
                    (qn == 0 || ptx::mbar_test_wait(s_empty, (qn - 1) & 1))) {
                    ptx::tc_fence_after();
                    const uint32_t ka = ptx::smem_u32(smem + C::OFF_KV + (qn % C::NS) * C::STAGE_BYTES);
#pragma unroll
                    for (int k = 0; k < DC / 16; ++k) {
                        const uint64_t bd = ptx::sdesc_sw128(ka + (k / 4) * (kBN * 128) + (k % 4) * 32, 16, 1024);
                        ptx::mma_ts(tbase + C::S_COL, tbase + C::Q_COL + k * 8, bd, idesc_qk, k > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(s_full);
                    ++qn;
                    prog = true;
                } else if (pn < qn && ptx::mbar_test_wait(p_full(pn & 1), (pn >> 1) & 1)) {
                    ptx::tc_fence_after();
                    const uint32_t va = ptx::smem_u32(smem + C::OFF_KV + (pn % C::NS) * C::STAGE_BYTES);
                    const uint32_t pa = tbase + C::P_COL + (pn & 1) * (kBN / 2);
#pragma unroll
                    for (int t = 0; t < kBN / 16; ++t) {
                        const uint64_t bd = ptx::sdesc_sw128(va + t * 2048, kBN * 128, 1024);
                        ptx::mma_ts(tbase + C::O_COL, pa + t * 8, bd, idesc_pv, (pn > 0 || t > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(kv_empty(pn % C::NS));
                    ptx::mma_commit(p_empty(pn & 1));
                    ptx::mma_commit(o_done);
                    ++pn;
                    prog = true;
                }
                if (prog) {
                    idle = 0;
                } else if (++idle == 1) {
                    t0 = clock64();
                } else if ((idle & 1023u) == 0 && clock64() - t0 > kWaitCycles) {
                    record_error(kErrWaitTimeout);
                    ok = false;
                }
            }
            ptx::mma_commit(mma_done);
        }
    } else {
        // ------------------------------------------------------------ softmax / epilogue
        // thread = (head row h, column half): columns [32*half, 32*half+32) of
        // every tile and [half*DC/2, (half+1)*DC/2) of q and o
        const int quarter = warp & 3;            // TMEM lanes this warp may access
        const int half = warp >> 2;
        const int h = quarter * 32 + lane;       // head row == TMEM lane
        const uint32_t lane_addr = tbase + (uint32_t(quarter * 32) << 16);
        const bool hv = h < p.H;
        {
            // this thread's half of Q_c into TMEM (bf16 pairs, DC/4 columns)
            constexpr int QW = DC / 4;
            const uint4 *qrow = reinterpret_cast<const uint4 *>(p.q + (tok * p.H + (hv ? h : 0)) * p.D +
                                                                int64_t(crank) * DC + half * (DC / 2));
            if constexpr (QW >= 32) {
#pragma unroll
                for (int c = 0; c < QW / 32; ++c) {
                    uint32_t v[32];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint4 x = hv ? __ldg(qrow + c * 8 + i) : make_uint4(0u, 0u, 0u, 0u);
                        v[4 * i] = x.x;
                        v[4 * i + 1] = x.y;
                        v[4 * i + 2] = x.z;
                        v[4 * i + 3] = x.w;
                    }
                    ptx::tmem_st32(lane_addr + C::Q_COL + half * QW + c * 32, v);
                }
            } else {
                uint32_t v[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 x = hv ? __ldg(qrow + i) : make_uint4(0u, 0u, 0u, 0u);
                    v[4 * i] = x.x;
                    v[4 * i + 1] = x.y;
                    v[4 * i + 2] = x.z;
                    v[4 * i + 3] = x.w;
                }
                ptx::tmem_st16(lane_addr + C::Q_COL + half * QW, v);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(q_ready);
        }

        uint32_t xrow_rem = 0, xfull_rem0 = 0, xfull_rem1 = 0, xempty_rem0 = 0, xempty_rem1 = 0;
        if constexpr (CL == 2) {
            xrow_rem = ptx::map_to_rank(ptx::smem_u32(smem + C::OFF_X + h * 16), crank ^ 1u);
            xfull_rem0 = ptx::map_to_rank(x_full(0), crank ^ 1u);
            xfull_rem1 = ptx::map_to_rank(x_full(1), crank ^ 1u);
            xempty_rem0 = ptx::map_to_rank(x_empty(0), crank ^ 1u);
            xempty_rem1 = ptx::map_to_rank(x_empty(1), crank ^ 1u);
        }
        const uint32_t s_addr = lane_addr + C::S_COL + 32 * half;
        // read this thread's 32 partial logits of tile j (frees the S buffer)
        // and, with a partner, send them to its receive buffer j & 1 as
        // asynchronous stores that complete_tx on the partner's x_full
        auto take = [&](int j, uint32_t (&r)[32]) -> bool {
            if (!wait_all(s_full, j & 1)) return false;
            ptx::tc_fence_after();
            ptx::tmem_ld32(s_addr, r);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            ptx::mbar_arrive(s_empty);
            if constexpr (CL == 2) {
                if (j >= 2 && !wait_all(x_empty(j & 1), ((j >> 1) - 1) & 1)) return false;
                // chunk-major layout [16 chunks][128 rows][16 B]: each warp
                // instruction writes 512 contiguous bytes of the partner's buffer
                const uint32_t row = xrow_rem + uint32_t(j & 1) * C::X_BYTES;
                const uint32_t xb = (j & 1) ? xfull_rem1 : xfull_rem0;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    ptx::st_async_v4(row + uint32_t(8 * half + c) * (kM * 16u), r[4 * c], r[4 * c + 1], r[4 * c + 2],
                                     r[4 * c + 3], xb);
            }
            return true;
        };
        bool ok = true;
        float m_run = -INFINITY, l_run = 0.f;
        uint32_t cur[32], nxt[32];
        if (n_act > 0) ok = take(0, cur);
        int a = 0;
        for (; ok && a < n_act; ++a) {
            const uint32_t vm = uint32_t(vmask[act[a]] >> (32 * half));
            if (a + 1 < n_act && !take(a + 1, nxt)) {
                ok = false;
                break;
            }
            float s[32];
            if constexpr (CL == 2) {
                if (tid == 0) ptx::mbar_arrive_expect_tx(x_full(a & 1), C::X_BYTES);
                if (!wait_all<true>(x_full(a & 1), (a >> 1) & 1)) {
                    ok = false;
                    break;
                }
                const uint8_t *xr = smem + C::OFF_X + (a & 1) * C::X_BYTES + h * 16;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 v = *reinterpret_cast<const float4 *>(xr + (8 * half + c) * (kM * 16));
                    s[4 * c] = __uint_as_float(cur[4 * c]) + v.x;
                    s[4 * c + 1] = __uint_as_float(cur[4 * c + 1]) + v.y;
                    s[4 * c + 2] = __uint_as_float(cur[4 * c + 2]) + v.z;
                    s[4 * c + 3] = __uint_as_float(cur[4 * c + 3]) + v.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(cur[j]);
            }
            float mloc = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                s[j] = ((vm >> j) & 1u) ? s[j] * p.scale_log2 : -INFINITY;
                mloc = fmaxf(mloc, s[j]);
            }
            // row max over both column halves
            red[(a & 1) * 256 + half * 128 + h] = mloc;
            ptx::mbar_arrive(red_bar);
            if (!wait_all(red_bar, a & 1)) {
                ok = false;
                break;
            }
            if constexpr (CL == 2) {
                // every softmax thread has read receive buffer a & 1: return the credit
                if (tid == 0) ptx::mbar_arrive_remote_relaxed((a & 1) ? xempty_rem1 : xempty_rem0);
            }
            const float mx = fmaxf(mloc, red[(a & 1) * 256 + (half ^ 1) * 128 + h]);
            // P buffer a & 1 is free once the P.V of tile a-2 has completed
            if (a >= 2 && !wait_all(p_empty(a & 1), ((a >> 1) - 1) & 1)) {
                ok = false;
                break;
            }
            if (a == 0) {
                m_run = mx;
            } else {
                // lazy rescale: only when the running max grows by more than
                // the threshold; warp-uniform because TMEM access is
                const bool need = mx > m_run + kRescaleThreshold;
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = need ? exp2f(m_run - mx) : 1.f;
                    if (need) {
                        l_run *= alpha;
                        m_run = mx;
                    }
                    if (!wait_all(o_done, (a - 1) & 1)) {  // previous P.V done
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
#pragma unroll 1
                    for (int ch = 0; ch < DC / 64; ++ch) {
                        uint32_t r[32];
                        const uint32_t oc = lane_addr + C::O_COL + half * (DC / 2) + ch * 32;
                        ptx::tmem_ld32(oc, r);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        ptx::tmem_st32(oc, r);
                    }
                }
            }
            // P = 2^(x - m) as bf16 pairs into TMEM (A operand of P.V)
            uint32_t pw[16];
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < 16; ++c) pw[c] = pack_bf16(exp2f(s[2 * c] - m_run), exp2f(s[2 * c + 1] - m_run), lsum);
            ptx::tmem_st16(lane_addr + C::P_COL + (a & 1) * (kBN / 2) + half * 16, pw);
            ptx::tmem_wait_st();
            l_run += lsum;
            ptx::tc_fence_before();
            ptx::mbar_arrive(p_full(a & 1));
#pragma unroll
            for (int j = 0; j < 32; ++j) cur[j] = nxt[j];
        }
        // ------------------------------------------------------------ epilogue
        if (ok) ok = wait_all(mma_done, 0);
        float l_tot = l_run;
        if (ok) {
            red[2 * 256 + half * 128 + h] = l_run;
            ptx::mbar_arrive(l_bar);
            ok = wait_all(l_bar, 0);
            if (ok) l_tot = l_run + red[2 * 256 + (half ^ 1) * 128 + h];
        }
        ptx::tc_fence_after();
        if (ok) {
            if (p.num_splits == 1) {
                const float s2 = hv ? p.sink[h] * kLog2e : 0.f;
                float f = 0.f;
                if (n_act > 0 && s2 != INFINITY) {
                    const float M = fmaxf(m_run, s2);
                    const float e = exp2f(m_run - M);
                    f = e / (l_tot * e + exp2f(s2 - M));
                }
                if (isnan(s2)) f = NAN;
                __nv_bfloat16 *orow = p.o + (tok * p.H + (hv ? h : 0)) * p.D + int64_t(crank) * DC + half * (DC / 2);
#pragma unroll 1
                for (int ch = 0; ch < DC / 64; ++ch) {
                    uint32_t r[32];
                    if (n_act > 0) {
                        ptx::tmem_ld32(lane_addr + C::O_COL + half * (DC / 2) + ch * 32, r);
                        ptx::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = 0u;
                    }
                    if (hv) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + ch * 32);
                        float dummy = 0.f;
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 w;
                            w.x = pack_bf16(__uint_as_float(r[8 * v + 0]) * f, __uint_as_float(r[8 * v + 1]) * f, dummy);
                            w.y = pack_bf16(__uint_as_float(r[8 * v + 2]) * f, __uint_as_float(r[8 * v + 3]) * f, dummy);
                            w.z = pack_bf16(__uint_as_float(r[8 * v + 4]) * f, __uint_as_float(r[8 * v + 5]) * f, dummy);
                            w.w = pack_bf16(__uint_as_float(r[8 * v + 6]) * f, __uint_as_float(r[8 * v + 7]) * f, dummy);
                            dst[v] = w;
                        }
                    }
                }
            } else {
                // split partial: O / l (fp32) and lse = m + log2(l) (base 2)
                const float inv = n_act > 0 ? 1.f / l_tot : 0.f;
                const float lse = n_act > 0 ? m_run + log2f(l_tot) : -INFINITY;
                const int64_t prow_i = (tok * p.num_splits + split) * p.H + (hv ? h : 0);
                float *wrow = p.ws_o + prow_i * p.D + int64_t(crank) * DC + half * (DC / 2);
#pragma unroll 1
                for (int ch = 0; ch < DC / 64; ++ch) {
                    uint32_t r[32];
                    if (n_act > 0) {
                        ptx::tmem_ld32(lane_addr + C::O_COL + half * (DC / 2) + ch * 32, r);
                        ptx::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = 0u;
                    }
                    if (hv) {
                        float4 *dst = reinterpret_cast<float4 *>(wrow + ch * 32);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            dst[v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                                 __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
                    }
                }
                if (hv && crank == 0 && half == 0) p.ws_lse[prow_i] = lse;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        if (lane == 0) wait_bar(mma_done, 0);  // no MMA in flight before TMEM is released
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tbase, C::TMEM_COLS);
    }
    if constexpr (CL == 2) ptx::cluster_sync();  // no remote access outlives the partner
}

// Split-KV combine (§5.5, log-sum-exp form with the sink added exactly once):
//   M = max(max_i lse_i, sink*log2e),  w_i = 2^(lse_i - M),
//   o = sum_i w_i O_i / (sum_i w_i + 2^(sink*log2e - M)).
// One warp per (token, head); each lane owns D/32 contiguous columns.
template <int D>
__global__ void __launch_bounds__(128)
attn_combine_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_lse, const float *__restrict__ sink,
                    __nv_bfloat16 *__restrict__ o, int64_t rows, int64_t H, int ns) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * 4 + (threadIdx.x >> 5);  // tok * H + h
    if (row >= rows) return;
    const int64_t tok = row / H, h = row % H;
    const float *lse = ws_lse + tok * ns * H + h;
    float mx = -INFINITY;
    for (int i = lane; i < ns; i += 32) mx = fmaxf(mx, lse[int64_t(i) * H]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float s2 = sink[h] * kLog2e;
    const float M = fmaxf(mx, s2);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float den = 0.f;
    const bool zero = (s2 == INFINITY) || (M == -INFINITY);
    if (!zero) {
        for (int i = 0; i < ns; ++i) {
            const float li = lse[int64_t(i) * H];
            if (li == -INFINITY) continue;
            const float w = exp2f(li - M);
            den += w;
            const float *src = ws_o + ((tok * ns + i) * H + h) * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; e += 2) {
                const float2 v = *reinterpret_cast<const float2 *>(src + e);
                acc[e] = fmaf(w, v.x, acc[e]);
                acc[e + 1] = fmaf(w, v.y, acc[e + 1]);
            }
        }
        den += exp2f(s2 - M);
    }
    const float f = zero ? 0.f : 1.f / den;
    const float fn = isnan(s2) ? NAN : f;
    __nv_bfloat16 *dst = o + row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2)
        *reinterpret_cast<__nv_bfloat162 *>(dst + e) = __floats2bfloat162_rn(acc[e] * fn, acc[e + 1] * fn);
}

// ---------------------------------------------------------------- host side

constexpr int kMaxDev = 64;

template <int DC, int CL>
cudaError_t launch_tc(const AttnArgs &a, cudaStream_t stream) {
    using C = Cfg<DC, CL>;
    static std::once_flag attr_once[kMaxDev];
    static cudaError_t attr_err[kMaxDev];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::call_once(attr_once[dev], [dev] {
        attr_err[dev] = cudaFuncSetAttribute(attn_tc_kernel<DC, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM);
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];

    TcParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.kv = static_cast<const __nv_bfloat16 *>(a.kv);
    p.sink = a.sink;
    p.idx = a.idx;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.ws_o = a.ws_o;
    p.ws_lse = a.ws_lse;
    p.S = a.S; p.H = a.H; p.D = a.D; p.T = a.T; p.K = a.K;
    p.num_splits = a.num_splits;
    p.unit_slots = int(split_slots(a.K, a.num_splits));
    p.scale_log2 = a.scale * kLog2e;
    if (p.unit_slots > kMaxUnitSlots) return cudaErrorInvalidValue;

    const int64_t ctas = a.B * a.S * a.num_splits * CL;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel<DC, CL>, p);
}

}  // namespace

int64_t split_slots(int64_t K, int num_splits) {
    const int64_t tiles = (K + kBN - 1) / kBN;
    const int64_t per = (tiles + num_splits - 1) / num_splits;
    return per * kBN;
}

int max_unit_slots() { return kMaxUnitSlots; }

cudaError_t launch_sparse_attn(const AttnArgs &a, int num_sms, cudaStream_t stream) {
    (void)num_sms;
    if (a.B * a.S == 0) return cudaSuccess;
    cudaError_t e;
    switch (a.D) {
        case 64: e = launch_tc<64, 1>(a, stream); break;
        case 128: e = launch_tc<128, 1>(a, stream); break;
        case 256: e = launch_tc<256, 1>(a, stream); break;
        case 512: e = launch_tc<256, 2>(a, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_attn_combine(const AttnArgs &a, cudaStream_t stream) {
    const int64_t rows = a.B * a.S * a.H;
    if (rows == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((rows + 3) / 4);
    switch (a.D) {
        case 64: attn_combine_kernel<64><<<grid, 128, 0, stream>>>(a.ws_o, a.ws_lse, a.sink, static_cast<__nv_bfloat16 *>(a.o), rows, a.H, a.num_splits); break;
        case 128: attn_combine_kernel<128><<<grid, 128, 0, stream>>>(a.ws_o, a.ws_lse, a.sink, static_cast<__nv_bfloat16 *>(a.o), rows, a.H, a.num_splits); break;
        case 256: attn_combine_kernel<256><<<grid, 128, 0, stream>>>(a.ws_o, a.ws_lse, a.sink, static_cast<__nv_bfloat16 *>(a.o), rows, a.H, a.num_splits); break;
        case 512: attn_combine_kernel<512><<<grid, 128, 0, stream>>>(a.ws_o, a.ws_lse, a.sink, static_cast<__nv_bfloat16 *>(a.o), rows, a.H, a.num_splits); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

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
