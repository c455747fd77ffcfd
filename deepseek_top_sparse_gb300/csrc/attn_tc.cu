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

// Timeline hooks for performance work: with SA_TRACE defined, CTA 0 records
// clock64() at fixed points of each role into g_sa_trace[role][tile][event];
// otherwise they compile to nothing.
#ifdef SA_TRACE
__device__ long long g_sa_trace[4][64][16];
#define SA_TRACE_POINT(role, tile, ev)                                                              \
    do {                                                                                            \
        if (blockIdx.x == 0 && (tile) >= 0 && (tile) < 64) g_sa_trace[role][tile][ev] = clock64(); \
    } while (0)
#else
#define SA_TRACE_POINT(role, tile, ev) \
    do {                               \
    } while (0)
#endif

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

template <int DC, int CL>
struct Cfg {
    static_assert(DC == 64 || DC == 128 || DC == 256, "per-CTA head-dim slice");
    static constexpr int STAGE_BYTES = kBN * DC * 2;
    static constexpr int NS = CL == 2 ? 5 : 4;            // kv ring depth
    static constexpr int THREADS = (kFirstGatherWarp + kGatherWarps) * 32;
    // partner's partial logits of one tile as block floating point: 16-bit
    // codes [8 chunks][128 rows][16 B] then one fp32 step per (row, half)
    static constexpr int XQ_BYTES = kM * kBN * 2;         // 16 KB
    static constexpr int X_BYTES = XQ_BYTES + 2 * kM * 4; // + 1 KB of steps
    static_assert(X_BYTES % 1024 == 0, "receive buffers keep 1 KB alignment");
    static constexpr int OFF_KV = 0;
    static constexpr int OFF_X = OFF_KV + NS * STAGE_BYTES;
    static constexpr int OFF_IDX = OFF_X + (CL == 2 ? 2 * X_BYTES : 0);
    static constexpr int OFF_VALID = OFF_IDX + kMaxUnitSlots * 4;
    static constexpr int OFF_LIST = OFF_VALID + kMaxUnitTiles * 8;
    static constexpr int OFF_RED = OFF_LIST + kMaxUnitTiles * 4 + 16;   // float [3][2][128]
    static constexpr int OFF_BAR = OFF_RED + 3 * 2 * kM * 4;
    // kv_full[NS] kv_empty[NS] s_full s_empty p_full[2] p_empty[2]
    // x_full[2] x_empty[2] o_done q_ready mma_done red_bar l_bar epi_bar
    static constexpr int NUM_BARS = 2 * NS + 16;
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
    static_assert(NS * STAGE_BYTES >= kM * DC * 4, "the kv ring can stage a full fp32 output tile");
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

// Block floating point for the partner exchange: 32 partial logits become
// 16-bit codes sharing one power-of-two step 2^(e-14), where max|x| < 2^e,
// so |x| / step < 2^14 and the absolute error is at most half a step
// (<= max|x| * 2^-15).  Encoding adds kBfpMagic = 1.5*2^23 + 2^15 to x/step:
// the float's low 16 bits are then (round(x/step) + 2^15), with no integer
// conversion.  Decoding ORs a code into 2^23 and removes 2^23 + 2^15.  A
// non-finite block gets a NaN step, so NaN still propagates.
constexpr float kBfpMagic = 12615680.0f;      // 1.5 * 2^23 + 2^15
constexpr float kBfpDecodeBias = 8421376.0f;  // 2^23 + 2^15

struct BfpStep {
    float step, inv;
};

__device__ __forceinline__ BfpStep bfp_step(float amax) {
    const uint32_t bexp = (__float_as_uint(amax) >> 23) & 0xFFu;   // biased exponent of max|x|
    if (bexp == 0xFFu || amax != amax) return {__uint_as_float(0x7FC00000u), 0.f};  // inf / NaN
    if (bexp < 20u) return {__uint_as_float(6u << 23), __uint_as_float(248u << 23)};  // ~0: 2^-121
    // max|x| < 2^(bexp-126); step = 2^(bexp-126-14): biased exponent bexp-13
    return {__uint_as_float((bexp - 13u) << 23), __uint_as_float((267u - bexp) << 23)};
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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
    const uint32_t epi_bar = bar(2 * C::NS + 15);

    // ---------------------------------------------------------------- prologue
    if (tid == 0) SA_TRACE_POINT(3, 0, 0);
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
        ptx::mbar_init(epi_bar, kSoftmaxThreads);
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
    if (tid == 0) SA_TRACE_POINT(3, 0, 1);

    if (warp >= kFirstGatherWarp) {
        // ------------------------------------------------------------ gather
        // every gather warp copies its share of the rows of every tile; each
        // lane's copies arrive on the stage's mbarrier when they land, so a
        // warp runs ahead into every free stage (up to NS tiles in flight)
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
            if (g == 0 && lane == 0) SA_TRACE_POINT(0, a, 0);
            if (f >= 1 && !wait_all(kv_empty(s), (f - 1) & 1)) {
                ok = false;
                break;
            }
            if (g == 0 && lane == 0) SA_TRACE_POINT(0, a, 1);
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
            ptx::cp_async_arrive_noinc(kv_full(s));
            if (g == 0 && lane == 0) SA_TRACE_POINT(0, a, 2);
        }
        ptx::cp_async_wait_all();   // nothing of ours still lands after the CTA exits
        (void)ok;
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
                    ptx::fence_proxy_async_smem();  // gathered rows (generic-proxy writes) -> MMA reads
                    ptx::tc_fence_after();
                    const uint32_t ka = ptx::smem_u32(smem + C::OFF_KV + (qn % C::NS) * C::STAGE_BYTES);
#pragma unroll
                    for (int k = 0; k < DC / 16; ++k) {
                        const uint64_t bd = ptx::sdesc_sw128(ka + (k / 4) * (kBN * 128) + (k % 4) * 32, 16, 1024);
                        ptx::mma_ts(tbase + C::S_COL, tbase + C::Q_COL + k * 8, bd, idesc_qk, k > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(s_full);
                    SA_TRACE_POINT(1, qn, 0);
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
                    SA_TRACE_POINT(1, pn, 1);
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
            if (tid == 0) SA_TRACE_POINT(2, j, 0);
            if (!wait_all(s_full, j & 1)) return false;
            if (tid == 0) SA_TRACE_POINT(2, j, 1);
            ptx::tc_fence_after();
            ptx::tmem_ld32(s_addr, r);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            ptx::mbar_arrive(s_empty);
            if constexpr (CL == 2) {
                // Both CTAs use the block-floating-point value of BOTH partials,
                // so the two sums (and everything after them) are bit-identical.
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(r[i])));
                const BfpStep st = bfp_step(amax);
                const float step = st.step;
                const float nbias = -kBfpMagic * step;
                uint32_t m[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float y0 = fmaf(__uint_as_float(r[2 * i]), st.inv, kBfpMagic);
                    const float y1 = fmaf(__uint_as_float(r[2 * i + 1]), st.inv, kBfpMagic);
                    m[i] = __byte_perm(__float_as_uint(y0), __float_as_uint(y1), 0x5410);
                    r[2 * i] = __float_as_uint(fmaf(y0, step, nbias));   // own partial, same rounding
                    r[2 * i + 1] = __float_as_uint(fmaf(y1, step, nbias));
                }
                if (j >= 2 && !wait_all(x_empty(j & 1), ((j >> 1) - 1) & 1)) return false;
                if (tid == 0) SA_TRACE_POINT(2, j, 2);
                // chunk-major codes [8 chunks][128 rows][16 B] (each warp
                // instruction writes 512 contiguous bytes), then the steps
                const uint32_t buf = xrow_rem + uint32_t(j & 1) * C::X_BYTES;
                const uint32_t xb = (j & 1) ? xfull_rem1 : xfull_rem0;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    ptx::st_async_v4(buf + uint32_t(4 * half + c) * (kM * 16u), m[4 * c], m[4 * c + 1], m[4 * c + 2],
                                     m[4 * c + 3], xb);
                ptx::st_async_b32(buf - uint32_t(h) * 16u + C::XQ_BYTES + uint32_t(half * kM + h) * 4u,
                                  __float_as_uint(step), xb);
                if (tid == 0) SA_TRACE_POINT(2, j, 3);
            }
            return true;
        };
        bool ok = true;
        const bool pos_scale = p.scale_log2 >= 0.f;
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
                if (tid == 0) SA_TRACE_POINT(2, a, 4);
                if (!wait_all<true>(x_full(a & 1), (a >> 1) & 1)) {
                    ok = false;
                    break;
                }
                if (tid == 0) SA_TRACE_POINT(2, a, 5);
                const uint8_t *xbuf = smem + C::OFF_X + (a & 1) * C::X_BYTES;
                const float step = *reinterpret_cast<const float *>(xbuf + C::XQ_BYTES + (half * kM + h) * 4);
                const float dbias = -kBfpDecodeBias * step;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(xbuf + (4 * half + c) * (kM * 16) + h * 16);
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = 8 * c + 2 * e;
                        const float lo = fmaf(__uint_as_float((w[e] & 0xFFFFu) | 0x4B000000u), step, dbias);
                        const float hi = fmaf(__uint_as_float((w[e] >> 16) | 0x4B000000u), step, dbias);
                        s[i] = __uint_as_float(cur[i]) + lo;
                        s[i + 1] = __uint_as_float(cur[i + 1]) + hi;
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(cur[j]);
            }
            // masked, scaled row max of this half (the scale is applied once,
            // to the max, when it is positive; invalid slots become -inf)
            float mloc = -INFINITY;
            if (vm != 0xFFFFFFFFu) {
#pragma unroll
                for (int j = 0; j < 32; ++j) s[j] = ((vm >> j) & 1u) ? s[j] : -INFINITY;
            }
            if (pos_scale) {
#pragma unroll
                for (int j = 0; j < 32; ++j) mloc = fmaxf(mloc, s[j]);
                mloc *= p.scale_log2;
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) mloc = fmaxf(mloc, s[j] * p.scale_log2);
            }
            // row max over both column halves
            if (tid == 0) SA_TRACE_POINT(2, a, 6);
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
            if (tid == 0) SA_TRACE_POINT(2, a, 7);
            const float mx = fmaxf(mloc, red[(a & 1) * 256 + (half ^ 1) * 128 + h]);
            // P buffer a & 1 is free once the P.V of tile a-2 has completed
            if (a >= 2 && !wait_all(p_empty(a & 1), ((a >> 1) - 1) & 1)) {
                ok = false;
                break;
            }
            if (tid == 0) SA_TRACE_POINT(2, a, 8);
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
            // P = 2^(scale*s - m) as bf16 pairs into TMEM (A operand of P.V);
            // invalid slots hold -inf and give exactly 0
            uint32_t pw[16];
            float lsum = 0.f;
            const float nm = -m_run;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float p0 = ex2_approx(fmaf(s[2 * c], p.scale_log2, nm));
                const float p1 = ex2_approx(fmaf(s[2 * c + 1], p.scale_log2, nm));
                lsum += p0 + p1;
                const __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
                pw[c] = *reinterpret_cast<const uint32_t *>(&v);
            }
            ptx::tmem_st16(lane_addr + C::P_COL + (a & 1) * (kBN / 2) + half * 16, pw);
            ptx::tmem_wait_st();
            if (tid == 0) SA_TRACE_POINT(2, a, 9);
            l_run += lsum;
            ptx::tc_fence_before();
            ptx::mbar_arrive(p_full(a & 1));
            if (tid == 0) SA_TRACE_POINT(2, a, 10);
#pragma unroll
            for (int j = 0; j < 32; ++j) cur[j] = nxt[j];
        }
        // ------------------------------------------------------------ epilogue
        if (tid == 0) SA_TRACE_POINT(3, 0, 2);
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
            // Output rows are staged in shared memory (the kv ring is idle once
            // every MMA has completed) and then written with coalesced 16-byte
            // stores, 512 contiguous bytes per warp instruction.  Staged row h
            // holds this CTA's DC columns; its 16-byte chunk c sits at chunk
            // position c ^ (h & 7), so the per-row writes are conflict-free.
            const bool split_out = p.num_splits > 1;
            float f = 0.f, lse = -INFINITY;
            if (!split_out) {
                const float s2 = hv ? p.sink[h] * kLog2e : 0.f;
                if (n_act > 0 && s2 != INFINITY) {
                    const float M = fmaxf(m_run, s2);
                    const float e = exp2f(m_run - M);
                    f = e / (l_tot * e + exp2f(s2 - M));
                }
                if (isnan(s2)) f = NAN;
            } else if (n_act > 0) {
                // split partial: O / l (fp32) and lse = m + log2(l) (base 2)
                f = 1.f / l_tot;
                lse = m_run + log2f(l_tot);
            }
            const int rb = split_out ? DC * 4 : DC * 2;     // staged row bytes
            uint8_t *stage = smem + C::OFF_KV;
            uint8_t *srow = stage + h * rb;
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
                if (split_out) {
                    const int c0 = (half * (DC / 2) + ch * 32) / 4;   // first 16-byte chunk
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const float4 w = make_float4(__uint_as_float(r[4 * v]) * f, __uint_as_float(r[4 * v + 1]) * f,
                                                     __uint_as_float(r[4 * v + 2]) * f,
                                                     __uint_as_float(r[4 * v + 3]) * f);
                        *reinterpret_cast<float4 *>(srow + (((c0 + v) ^ (h & 7)) * 16)) = w;
                    }
                } else {
                    const int c0 = (half * (DC / 2) + ch * 32) / 8;
                    float dummy = 0.f;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(r[8 * v + 0]) * f, __uint_as_float(r[8 * v + 1]) * f, dummy);
                        w.y = pack_bf16(__uint_as_float(r[8 * v + 2]) * f, __uint_as_float(r[8 * v + 3]) * f, dummy);
                        w.z = pack_bf16(__uint_as_float(r[8 * v + 4]) * f, __uint_as_float(r[8 * v + 5]) * f, dummy);
                        w.w = pack_bf16(__uint_as_float(r[8 * v + 6]) * f, __uint_as_float(r[8 * v + 7]) * f, dummy);
                        *reinterpret_cast<uint4 *>(srow + (((c0 + v) ^ (h & 7)) * 16)) = w;
                    }
                }
            }
            if (split_out && hv && crank == 0 && half == 0)
                p.ws_lse[(tok * p.num_splits + split) * p.H + h] = lse;
            ptx::mbar_arrive(epi_bar);
            ok = wait_all(epi_bar, 0);
            if (ok) {
                // warp w copies rows [16w, 16w + 16)
                const int nch = rb / 16;
                for (int rr = 0; rr < kM / kSoftmaxWarps; ++rr) {
                    const int row = warp * (kM / kSoftmaxWarps) + rr;
                    if (row >= p.H) break;
                    uint8_t *dst = split_out
                        ? reinterpret_cast<uint8_t *>(p.ws_o + ((tok * p.num_splits + split) * p.H + row) * p.D +
                                                      int64_t(crank) * DC)
                        : reinterpret_cast<uint8_t *>(p.o + (tok * p.H + row) * p.D + int64_t(crank) * DC);
                    const uint8_t *src = stage + row * rb;
                    for (int c = lane; c < nch; c += 32)
                        *reinterpret_cast<uint4 *>(dst + c * 16) =
                            *reinterpret_cast<const uint4 *>(src + ((c ^ (row & 7)) * 16));
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    if (tid == 0) SA_TRACE_POINT(3, 0, 3);
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

#ifdef SA_TRACE
}  // namespace sa
extern "C" int sa_trace_read(long long *out) { return (int)cudaMemcpyFromSymbol(out, sa::g_sa_trace, sizeof(sa::g_sa_trace)); }
extern "C" int sa_trace_clear() {
    static long long z[4 * 64 * 16] = {0};
    return (int)cudaMemcpyToSymbol(sa::g_sa_trace, z, sizeof(z));
}
namespace sa {
#endif

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
