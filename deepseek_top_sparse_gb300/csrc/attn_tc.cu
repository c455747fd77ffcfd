// sparse_attn on the sm_103a tensor cores (tcgen05 + TMEM + TMA gather4).
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
// gathered kv row and of o.  Per CTA and per 64-row tile of active slots:
//
//   warp 0 (TMA)     gathers the tile's kv rows, DC columns, into a 3/4-deep
//                    ring of shared-memory stages with cp.async.bulk.tensor
//                    tile::gather4 (4 rows per instruction, 128B swizzle,
//                    invalid slots -> an out-of-range row -> zero fill);
//   warp 1 (MMA)     S_c = Q_c K_c^T with Q_c resident in TMEM (A operand from
//                    tensor memory), S double-buffered in TMEM; then
//                    O_c += P V_c from shared memory (V_c = the same stage read
//                    MN-major), O_c resident in TMEM for the whole unit;
//   warps 2..5       one thread per head row: read S_c from TMEM, swap it
//                    with the partner CTA through distributed shared memory
//                    so both hold S = S_0 + S_1 (fp32 addition commutes, both
//                    CTAs see identical logits), mask invalid slots, online
//                    softmax in base 2 with a lazily rescaled running max,
//                    write P (bf16) to shared memory for the P.V MMA.
//
// TMEM columns (D = 512, DC = 256): O_c [0,256) fp32, S [256,384) two 64-col
// buffers, Q_c [384,512) bf16 pairs.  Every wait is bounded by the global
// timer; a wait that runs out records an error code and the kernel drains and
// returns instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
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
constexpr int kThreads = 192;           // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr int kMaxUnitSlots = 2048;     // slots per work unit (host enforces)
constexpr int kMaxUnitTiles = kMaxUnitSlots / kBN;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr float kRescaleThreshold = 8.f;     // log2 units: P <= 256 before normalising

template <int DC, int CL>
struct Cfg {
    static_assert(DC == 64 || DC == 128 || DC == 256, "per-CTA head-dim slice");
    static constexpr int STAGE_BYTES = kBN * DC * 2;
    static constexpr int NS = CL == 2 ? 3 : 4;            // kv ring depth
    static constexpr int P_BYTES = kM * kBN * 2;          // 16 KB bf16
    static constexpr int X_BYTES = kM * kBN * 4;          // 32 KB fp32 partial logits
    static constexpr int OFF_KV = 0;
    static constexpr int OFF_P = OFF_KV + NS * STAGE_BYTES;
    static constexpr int OFF_X = OFF_P + 2 * P_BYTES;
    static constexpr int OFF_IDX = OFF_X + (CL == 2 ? 2 * X_BYTES : 0);
    static constexpr int OFF_VALID = OFF_IDX + kMaxUnitSlots * 4;
    static constexpr int OFF_BAR = OFF_VALID + kMaxUnitTiles * 8;
    // kv_full[NS] kv_empty[NS] s_full[2] p_full[2] x_full[2] o_done q_ready mma_done
    static constexpr int NUM_BARS = 2 * NS + 9;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM = OFF_TSLOT + 16 + 1024;    // + slack to align the base to 1 KB
    static constexpr int O_COL = 0;
    static constexpr int S_COL = DC;
    static constexpr int Q_COL = DC + 2 * kBN;
    static constexpr int TMEM_USED = Q_COL + DC / 2;
    static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
    static_assert(TMEM_USED <= 512, "TMEM budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

struct TcParams {
    const __nv_bfloat16 *q;   // [tokens, H, D]
    const float *sink;        // [H]
    const int32_t *idx;       // [tokens, K]
    __nv_bfloat16 *o;         // [tokens, H, D]
    float *ws_o;              // [tokens, splits, H, D]
    float *ws_lse;            // [tokens, splits, H]
    int64_t S, H, D, T, K;
    int num_splits;
    int unit_slots;           // slots per split, a multiple of kBN, <= kMaxUnitSlots
    int32_t oob_row;          // B*T: a row coordinate outside the kv tensor map
    float scale_log2;         // softmax_scale * log2(e)
};

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_device_error, 0, code); }

template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity) {
    auto poll = [&] { return kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity); };
    if (poll()) return true;
    const uint64_t t0 = gtimer();
    while (!poll()) {
        if (gtimer() - t0 > kWaitNs) {
            record_error(kErrWaitTimeout);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b, float &sum) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    sum += __low2float(v) + __high2float(v);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <int DC, int CL>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmap, const TcParams p) {
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
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::OFF_TSLOT);
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    auto kv_full = [&](int s) { return bar(s); };
    auto kv_empty = [&](int s) { return bar(C::NS + s); };
    auto s_full = [&](int i) { return bar(2 * C::NS + i); };
    auto p_full = [&](int i) { return bar(2 * C::NS + 2 + i); };
    auto x_full = [&](int i) { return bar(2 * C::NS + 4 + i); };
    const uint32_t o_done = bar(2 * C::NS + 6);
    const uint32_t q_ready = bar(2 * C::NS + 7);
    const uint32_t mma_done = bar(2 * C::NS + 8);

    // ---------------------------------------------------------------- prologue
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tslot), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < C::NS; ++s) {
            ptx::mbar_init(kv_full(s), 1);
            ptx::mbar_init(kv_empty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(s_full(i), 1);
            ptx::mbar_init(p_full(i), 128);
            ptx::mbar_init(x_full(i), 128);
        }
        ptx::mbar_init(o_done, 1);
        ptx::mbar_init(q_ready, 128);
        ptx::mbar_init(mma_done, 1);
        ptx::fence_mbar_init();
    }
    // slot indices -> kv row coordinates (invalid -> out-of-range row) and a
    // 64-bit validity mask per tile, 32 slots per warp step
    {
        const int32_t *irow = p.idx + tok * p.K + slot0;
        for (int ch = warp; ch < ntiles * 2; ch += kThreads / 32) {
            const int j = ch * 32 + lane;
            const int32_t t = j < nslots ? __ldg(irow + j) : -1;
            const bool v = t >= 0 && int64_t(t) < p.T;
            rowc[j] = v ? int32_t(b * p.T + t) : p.oob_row;
            const uint32_t m = __ballot_sync(0xffffffffu, v);
            if (lane == 0) reinterpret_cast<uint32_t *>(vmask)[ch] = m;
        }
    }
    ptx::tc_fence_before();
    if constexpr (CL == 2) {
        ptx::cluster_sync();  // partner barriers initialised before any remote arrive
    } else {
        __syncthreads();
    }
    ptx::tc_fence_after();
    const uint32_t tbase = *tslot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tmap);
            int a = 0;
            for (int t = 0; t < ntiles; ++t) {
                if (vmask[t] == 0) continue;
                const int s = a % C::NS;
                if (a >= C::NS && !wait_bar(kv_empty(s), ((a / C::NS) & 1) ^ 1)) break;
                ptx::mbar_arrive_expect_tx(kv_full(s), C::STAGE_BYTES);
                const uint32_t dst0 = ptx::smem_u32(smem + C::OFF_KV + s * C::STAGE_BYTES);
                const int32_t *rc = rowc + t * kBN;
#pragma unroll 1
                for (int at = 0; at < DC / 64; ++at) {
                    const int32_t col = int32_t(crank) * DC + at * 64;
#pragma unroll 4
                    for (int g = 0; g < kBN / 4; ++g)
                        ptx::tma_gather4(dst0 + at * (kBN * 128) + g * 512, &tmap, col, rc[4 * g], rc[4 * g + 1],
                                         rc[4 * g + 2], rc[4 * g + 3], kv_full(s));
                }
                ++a;
            }
            // drain: the last fill of every stage has landed before teardown
            for (int k = (a > C::NS ? a - C::NS : 0); k < a; ++k) wait_bar(kv_full(k % C::NS), (k / C::NS) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(kM, kBN, false);
            constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(kM, DC, true);
            bool ok = wait_bar(q_ready, 0);
            ptx::tc_fence_after();
            auto issue_pv = [&](int j, int stage) -> bool {
                if (!wait_bar(p_full(j & 1), (j >> 1) & 1)) return false;
                ptx::tc_fence_after();
                const uint32_t pa = ptx::smem_u32(smem + C::OFF_P + (j & 1) * C::P_BYTES);
                const uint32_t va = ptx::smem_u32(smem + C::OFF_KV + stage * C::STAGE_BYTES);
#pragma unroll
                for (int t = 0; t < kBN / 16; ++t) {
                    const uint64_t ad = ptx::sdesc_sw128(pa + t * 32, 16, 1024);
                    const uint64_t bd = ptx::sdesc_sw128(va + t * 2048, kBN * 128, 1024);
                    ptx::mma_ss(tbase + C::O_COL, ad, bd, idesc_pv, (j > 0 || t > 0) ? 1u : 0u);
                }
                ptx::mma_commit(kv_empty(stage));
                ptx::mma_commit(o_done);
                return true;
            };
            int a = 0, prev_stage = 0;
            for (int t = 0; t < ntiles && ok; ++t) {
                if (vmask[t] == 0) continue;
                const int s = a % C::NS;
                if (!wait_bar(kv_full(s), (a / C::NS) & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t ka = ptx::smem_u32(smem + C::OFF_KV + s * C::STAGE_BYTES);
                const uint32_t sd = tbase + C::S_COL + (a & 1) * kBN;
#pragma unroll
                for (int k = 0; k < DC / 16; ++k) {
                    const uint64_t bd = ptx::sdesc_sw128(ka + (k / 4) * (kBN * 128) + (k % 4) * 32, 16, 1024);
                    ptx::mma_ts(sd, tbase + C::Q_COL + k * 8, bd, idesc_qk, k > 0 ? 1u : 0u);
                }
                ptx::mma_commit(s_full(a & 1));
                if (a >= 1 && !issue_pv(a - 1, prev_stage)) {
                    ok = false;
                    break;
                }
                prev_stage = s;
                ++a;
            }
            if (ok && a >= 1) issue_pv(a - 1, prev_stage);
            ptx::mma_commit(mma_done);
        }
    } else {
        // ------------------------------------------------------------ softmax / epilogue
        const int quarter = warp & 3;            // TMEM lanes this warp may access
        const int h = quarter * 32 + lane;       // head row == TMEM lane
        const uint32_t lane_addr = tbase + (uint32_t(quarter * 32) << 16);
        {
            // Q_c into TMEM: 64 bf16 (32 columns) per step
            const bool hv = h < p.H;
            const uint4 *qrow = reinterpret_cast<const uint4 *>(p.q + (tok * p.H + (hv ? h : 0)) * p.D +
                                                                int64_t(crank) * DC);
#pragma unroll 1
            for (int ch = 0; ch < DC / 64; ++ch) {
                uint32_t v[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 x = hv ? __ldg(qrow + ch * 8 + i) : make_uint4(0u, 0u, 0u, 0u);
                    v[4 * i] = x.x;
                    v[4 * i + 1] = x.y;
                    v[4 * i + 2] = x.z;
                    v[4 * i + 3] = x.w;
                }
                ptx::tmem_st32(lane_addr + C::Q_COL + ch * 32, v);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(q_ready);
        }

        uint32_t xloc = 0, xrem = 0, xfull_rem0 = 0, xfull_rem1 = 0;
        if constexpr (CL == 2) {
            xloc = ptx::smem_u32(smem + C::OFF_X);
            xrem = ptx::map_to_rank(xloc, crank ^ 1u);
            xfull_rem0 = ptx::map_to_rank(x_full(0), crank ^ 1u);
            xfull_rem1 = ptx::map_to_rank(x_full(1), crank ^ 1u);
        }
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        int a = 0;
        for (int t = 0; t < ntiles; ++t) {
            const uint64_t vm = vmask[t];
            if (vm == 0) continue;
            if (!__all_sync(0xffffffffu, wait_bar(s_full(a & 1), (a >> 1) & 1))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            float s[kBN];
            {
                uint32_t r0[32], r1[32];
                ptx::tmem_ld32(lane_addr + C::S_COL + (a & 1) * kBN, r0);
                ptx::tmem_ld32(lane_addr + C::S_COL + (a & 1) * kBN + 32, r1);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    s[j] = __uint_as_float(r0[j]);
                    s[32 + j] = __uint_as_float(r1[j]);
                }
            }
            if constexpr (CL == 2) {
                // swap partial logits with the partner CTA (rows of 256 B,
                // 16-byte chunks XOR-swizzled by row to avoid bank conflicts)
                const uint32_t row_off = uint32_t(a & 1) * C::X_BYTES + uint32_t(h) * 256u;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint32_t pos = uint32_t(c ^ (h & 7)) * 16u;
                    ptx::st_cluster_v4(xrem + row_off + pos, __float_as_uint(s[4 * c]), __float_as_uint(s[4 * c + 1]),
                                       __float_as_uint(s[4 * c + 2]), __float_as_uint(s[4 * c + 3]));
                }
                ptx::mbar_arrive_remote((a & 1) ? xfull_rem1 : xfull_rem0);
                if (!__all_sync(0xffffffffu, wait_bar<true>(x_full(a & 1), (a >> 1) & 1))) {
                    ok = false;
                    break;
                }
                const uint8_t *xr = smem + C::OFF_X + row_off;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float4 v = *reinterpret_cast<const float4 *>(xr + (c ^ (h & 7)) * 16);
                    s[4 * c] += v.x;
                    s[4 * c + 1] += v.y;
                    s[4 * c + 2] += v.z;
                    s[4 * c + 3] += v.w;
                }
            }
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < kBN; ++j) {
                s[j] = ((vm >> j) & 1ull) ? s[j] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[j]);
            }
            if (a == 0) {
                m_run = mx;
            } else {
                // lazy rescale: only when the running max grows by more than
                // the threshold; the decision is warp-uniform (TMEM access is)
                const bool need = mx > m_run + kRescaleThreshold;
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = need ? exp2f(m_run - mx) : 1.f;
                    if (need) {
                        l_run *= alpha;
                        m_run = mx;
                    }
                    if (!__all_sync(0xffffffffu, wait_bar(o_done, (a - 1) & 1))) {  // previous P.V done
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
#pragma unroll 1
                    for (int ch = 0; ch < DC / 32; ++ch) {
                        uint32_t r[32];
                        ptx::tmem_ld32(lane_addr + C::O_COL + ch * 32, r);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        ptx::tmem_st32(lane_addr + C::O_COL + ch * 32, r);
                    }
                    ptx::tmem_wait_st();
                }
            }
            // P = 2^(x - m) as bf16 into the K-major, 128B-swizzled P tile
            uint8_t *prow = smem + C::OFF_P + (a & 1) * C::P_BYTES + (h >> 3) * 1024 + (h & 7) * 128;
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint4 w;
                w.x = pack_bf16(exp2f(s[8 * c + 0] - m_run), exp2f(s[8 * c + 1] - m_run), lsum);
                w.y = pack_bf16(exp2f(s[8 * c + 2] - m_run), exp2f(s[8 * c + 3] - m_run), lsum);
                w.z = pack_bf16(exp2f(s[8 * c + 4] - m_run), exp2f(s[8 * c + 5] - m_run), lsum);
                w.w = pack_bf16(exp2f(s[8 * c + 6] - m_run), exp2f(s[8 * c + 7] - m_run), lsum);
                *reinterpret_cast<uint4 *>(prow + ((c ^ (h & 7)) * 16)) = w;
            }
            l_run += lsum;
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(p_full(a & 1));
            ++a;
        }

        // ------------------------------------------------------------ epilogue
        const int n_act = a;
        if (ok) ok = __all_sync(0xffffffffu, wait_bar(mma_done, 0));
        ptx::tc_fence_after();
        if (ok) {
            const bool hv = h < p.H;
            if (p.num_splits == 1) {
                const float s2 = hv ? p.sink[h] * kLog2e : 0.f;
                float f = 0.f;
                if (n_act > 0 && s2 != INFINITY) {
                    const float M = fmaxf(m_run, s2);
                    const float e = exp2f(m_run - M);
                    f = e / (l_run * e + exp2f(s2 - M));
                }
                if (isnan(s2)) f = NAN;
                __nv_bfloat16 *orow = p.o + (tok * p.H + (hv ? h : 0)) * p.D + int64_t(crank) * DC;
#pragma unroll 1
                for (int ch = 0; ch < DC / 32; ++ch) {
                    uint32_t r[32];
                    if (n_act > 0) {
                        ptx::tmem_ld32(lane_addr + C::O_COL + ch * 32, r);
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
                const float inv = n_act > 0 ? 1.f / l_run : 0.f;
                const float lse = n_act > 0 ? m_run + log2f(l_run) : -INFINITY;
                const int64_t prow_i = (tok * p.num_splits + split) * p.H + (hv ? h : 0);
                float *wrow = p.ws_o + prow_i * p.D + int64_t(crank) * DC;
#pragma unroll 1
                for (int ch = 0; ch < DC / 32; ++ch) {
                    uint32_t r[32];
                    if (n_act > 0) {
                        ptx::tmem_ld32(lane_addr + C::O_COL + ch * 32, r);
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
                if (hv && crank == 0) p.ws_lse[prow_i] = lse;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q{};
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// kv viewed as a 2-D bf16 tensor [B*T rows, D columns]; box = 64 columns x 1
// row (the gather4 form), 128-byte swizzle matching the UMMA K-major layout.
cudaError_t encode_kv_map(CUtensorMap *map, const void *kv, int64_t rows, int64_t D) {
    auto enc = get_encode();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t gdim[2] = {cuuint64_t(D), cuuint64_t(rows)};
    cuuint64_t gstride[1] = {cuuint64_t(D) * 2};
    cuuint32_t box[2] = {64, 1};
    cuuint32_t estride[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(kv), gdim, gstride, box,
                           estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

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

    CUtensorMap map;
    e = encode_kv_map(&map, a.kv, a.B * a.T, a.D);
    if (e != cudaSuccess) return e;
    TcParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.sink = a.sink;
    p.idx = a.idx;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.ws_o = a.ws_o;
    p.ws_lse = a.ws_lse;
    p.S = a.S; p.H = a.H; p.D = a.D; p.T = a.T; p.K = a.K;
    p.num_splits = a.num_splits;
    p.unit_slots = int(split_slots(a.K, a.num_splits));
    p.oob_row = int32_t(a.B * a.T);
    p.scale_log2 = a.scale * kLog2e;
    if (p.unit_slots > kMaxUnitSlots) return cudaErrorInvalidValue;

    const int64_t ctas = a.B * a.S * a.num_splits * CL;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel<DC, CL>, map, p);
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
