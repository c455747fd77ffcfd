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
//   warps 9..15 (gather) copy the DC-column slice of each tile's 64 indexed
//                        kv rows with 16-byte cp.async (invalid slots
//                        zero-filled) into the 128B-swizzled K-major stage the
//                        MMAs read (an FP8 kv cache: warps 9-10 bulk-copy each
//                        row's bytes into a staging ring, warps 11-15 widen
//                        them to bf16 in the stage);
//   warp 8 (MMA)         S = Q_c K_c^T with Q_c resident in TMEM, into one of
//                        two S buffers (QK^T runs up to two tiles ahead of
//                        the softmax); O_c += P V_c with P (bf16) in one of two
//                        shared-memory buffers and V_c the same stage read
//                        MN-major; O_c resident in TMEM for the unit;
//   warps 0..7 (softmax) warp w reads the 16 TMEM lanes [16*(w/4), +16) of
//                        lane quarter w%4 (16x256b: a thread holds two head
//                        rows x 16 of the tile's 64 columns, four threads per
//                        row pair, so row maxima are quad shuffles).
//
// With two CTAs a head row's logit is the sum of two partial dot products,
// one per CTA.  Rows are owned by one CTA each: CTA c owns lanes
// [16c, 16c+16) of every quarter.  The "sender" warps of a CTA (the lanes it
// does not own) copy their fp32 partial logits to the owner, exactly; the
// "owner" warps add the partner's partials to their own, run the online
// softmax and write P for their rows into the P buffer; one bulk copy per
// warp puts the same rows into the partner's P buffer, and each row's
// rescale factor goes with them to the partner's sender warps, which apply
// it to the partner's half of O.  So each CTA runs the softmax of half the
// rows, and every logit is the plain fp32 sum of the two MMA partials.
//
// TMEM columns (D = 512, DC = 256): O_c [0,256) fp32, S [256,384) two 64-col
// buffers, Q_c [384,512) bf16 pairs.  Every buffer hand-off is an mbarrier phase that
// is never more than one phase away from its waiter; every mbarrier wait is
// bounded by clock64 and gives up early once any wait of any kernel has
// recorded an error, so a failing launch drains in about one wait bound.
// The cluster barriers of the prologue and teardown are hardware barriers
// that every CTA of the cluster reaches on every path.  The kernel launches with
// a programmatic dependency on the stream's previous kernel: every thread
// waits for it (griddepcontrol.wait) before its first global memory access.
#include <cuda_bf16.h>

#include <cudaTypedefs.h>
#include <mutex>
#include <type_traits>

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
// Bound on any single wait, in SM clock cycles (~0.1 s at 2 GHz): far beyond
// any legitimate wait.  clock64 and the device error word are read only after
// 1024 unsuccessful polls.
constexpr long long kWaitCycles = 200000000ll;
constexpr float kRescaleThreshold = 8.f;     // log2 units: P <= 256 before normalising
constexpr int kSoftmaxWarps = 8;              // two per TMEM lane quarter, 16 lanes each
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kMmaWarp = kSoftmaxWarps;
constexpr int kFirstGatherWarp = kMmaWarp + 1;
// cp.async gather throughput per SM grows with the number of issuing warps
// (each warp keeps a bounded number of copies in flight): 7 gather warps.
constexpr int kGatherWarps = 7;               // all fill every tile, rows interleaved
// 16 warps = 4 warpgroups launched at 128 registers a thread; after the
// prologue the two softmax warpgroups grow to 160 and the MMA + gather
// warpgroups shrink to 96: 256 * 160 + 256 * 96 = 512 * 128.
constexpr int kLaunchRegs = 128;
constexpr int kSoftmaxRegs = 160;
constexpr int kOtherRegs = 96;

// FP8 kv rows (the V4 cache format): 448 dims as E4M3 codes, then 64 RoPE
// dims as bf16, then one E8M0 scale byte per 64-dim tile of the codes (7 used,
// 1 pad): 584 bytes, so a row starts on an 8-byte boundary only.
constexpr int kF8Row = 584;
// FP8 gather: every gather warp bulk-copies raw rows into the staging ring
// (three tiles ahead) and widens the same rows into the kv stages
constexpr int kF8WidenWarps = kGatherWarps;
constexpr int kF8ScaleOff = 576;

template <int DC, int CL, bool F8 = false>
struct Cfg {
    static_assert(DC == 64 || DC == 128 || DC == 256, "per-CTA head-dim slice");
    static_assert(!F8 || (DC == 256 && CL == 2), "FP8 rows only at D = 512 (two 256-column halves)");
    static constexpr int STAGE_BYTES = kBN * DC * 2;
    static constexpr int NS = F8 ? 3 : 5;   // kv ring depth (bf16 stages the MMA reads)
    // partner partial-logit buffers per lane quarter: one for a pair (its
    // owner consumes them at the start of a tile, before the sender can need
    // the buffer again), which leaves room for the fifth bf16 kv stage or the
    // third FP8 staging buffer
    static constexpr int XB = CL == 2 ? 1 : 2;
    // FP8: the raw bytes of a tile land in one of NF staging buffers (one
    // 336-byte row per kv row: this CTA's 256 or 320 bytes of codes / RoPE
    // values at [0, 320), its scale bytes at 320) and are widened to bf16
    // into a kv stage by the gather warps, which copy their own rows NF tiles ahead
    static constexpr int NF = F8 ? 3 : 0;
    static constexpr int STG_ROW = 336;
    static constexpr int STG_SCALE = 320;
    static constexpr int STG_BYTES = kBN * STG_ROW;
    static_assert(STG_SCALE + 16 <= STG_ROW && STG_ROW % 16 == 0,
                  "staging row: 320 data bytes, one 16-byte scale window");
    static constexpr int THREADS = (kFirstGatherWarp + kGatherWarps) * 32;
    static_assert(THREADS == 512, "four warpgroups");
    static_assert(kSoftmaxThreads * kSoftmaxRegs + (THREADS - kSoftmaxThreads) * kOtherRegs == THREADS * kLaunchRegs,
                  "register split equals the launch allocation");
    // P of a tile (bf16, the A operand of P.V): [128 rows][64] in the
    // 128B-swizzled K-major layout (8-row atoms of 1 KB), two buffers.
    static constexpr int P_BYTES = kM * kBN * 2;
    // Partner messages (CL == 2), one buffer per (tile parity b, lane quarter q):
    //   X: the partner's fp32 partial logits of this CTA's 16 rows of the
    //      quarter, [8 chunks][32 lanes][16 B] (chunk k = the four values of
    //      16x256b repetition k);
    //   F: one fp32 rescale factor for each of the partner's 16 rows of the
    //      quarter (its P rows arrive directly in the P buffer).
    static constexpr int XQ = 8 * 32 * 16;
    static constexpr int FQ = 16 * 4;
    static constexpr int OFF_KV = 0;
    static constexpr int OFF_STG = OFF_KV + NS * STAGE_BYTES;
    static constexpr int OFF_P = OFF_STG + NF * STG_BYTES;
    static_assert(OFF_P % 1024 == 0, "P buffers keep the 1 KB swizzle alignment");
    static constexpr int OFF_X = OFF_P + 2 * P_BYTES;
    static constexpr int OFF_F = OFF_X + (CL == 2 ? XB * 4 * XQ : 0);
    static constexpr int OFF_IDX = OFF_F + (CL == 2 ? 2 * 4 * FQ : 0);
    static constexpr int OFF_VALID = OFF_IDX + kMaxUnitSlots * 4;
    static constexpr int OFF_LIST = OFF_VALID + kMaxUnitTiles * 8;
    static constexpr int OFF_STAT = OFF_LIST + kMaxUnitTiles * 4 + 16;  // float2 [128]: (m, l) per row
    static constexpr int OFF_LSE = OFF_STAT + kM * 8;                   // float [8 splits][128]
    static constexpr int OFF_SINK = OFF_LSE + 8 * kM * 4;               // float [128]
    static constexpr int OFF_BAR = OFF_SINK + kM * 4;
    // kv_full[NS] kv_empty[NS] s_full[2] s_empty[2] p_full[2] p_empty[2]
    // o_done[2] q_ready mma_done stat_bar q_smem q_free, then x_full[8]
    // x_empty[8] pm_full[8] ([parity][quarter]); FP8: + stg_full[NF]
    // stg_empty[NF].  The layout is the same in every CTA (p_empty receives
    // multicast arrivals at its offset).
    static constexpr int BAR_X = 2 * NS + 15;
    static constexpr int NUM_BARS = BAR_X + 24 + 2 * NF + 1;   // + rcv_bar
    // Q_c arrives by TMA in the last two kv stages (128 rows x DC bf16 =
    // 2 stages), as DC / 64 boxes of [128 rows][128 B], 128B-swizzled
    static constexpr int OFF_QS = OFF_KV + (NS - 2) * STAGE_BYTES;
    static constexpr int Q_BYTES = kM * DC * 2;
    static_assert(Q_BYTES == 2 * STAGE_BYTES, "Q_c fills two kv stages");
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM = OFF_TSLOT + 16 + 1024;    // + slack to align the base to 1 KB
    // TMEM columns: O_c fp32, two S buffers of one tile (fp32), Q_c bf16 pairs
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
    const __nv_bfloat16 *kv;  // [B, T, D]
    const float *sink;        // [H]
    const int32_t *idx;       // [tokens, K]
    const int32_t *topk_len;  // [tokens] valid-prefix length per token, or nullptr
    // extra kv source: a token's slots are its K1 main slots (idx, kv), then
    // its K2 extra slots (idx2 [tokens, K2], kv2 [B, T2, .], topk_len2 or
    // nullptr); K = K1 + K2.  Extra row t2 of request b is row number
    // BT + b*T2 + t2 in the slot lists (BT = B*T rounded up to even, so a
    // row's parity is that of its index in its own source)
    const void *kv2;
    const int32_t *idx2;
    const int32_t *topk_len2;
    int64_t T2, K1, K2, BT;
    __nv_bfloat16 *o;         // [tokens, H, D]
    float *ws_o;              // [tokens, splits, H, D]
    float *ws_lse;            // [tokens, splits, H]
    int64_t S, H, D, T, K;
    int num_splits;
    int fused;                // 1: the token's splits share a cluster and combine in-kernel
    int unit_slots;           // slots per split, a multiple of kBN, <= kMaxUnitSlots
    float scale_log2;         // softmax_scale * log2(e)
    // Bit-mask mode (mask != nullptr, idx unused, K = T): slot j of a token is
    // key j of its kv, admitted iff bit (j + key_start) of the token's mask
    // row is set; each split compacts its admitted keys into full tiles.
    const uint32_t *mask;     // [B, mask_rows, mask_words]
    int64_t mask_rows, mask_words;
    int key_start_word;       // 1: key_start = mask[b, 0, mask_words - 1] (int32), else 0
    const int32_t *key_ends;  // [B] live key end (mask positions) per request, or nullptr
    // q and o rows: token (b, s) of the call is row b * io_S + io_s0 + s of
    // q and o (a window of io_S query rows per request; io_S = S, io_s0 = 0
    // for a whole batch)
    int64_t io_S, io_s0;
};


__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_device_error, 0, code); }

// Bounded mbarrier wait.  Gives up (and returns false) when the wait has run
// past max_cycles, recording kErrWaitTimeout, or as soon as some wait has
// already recorded an error: once one wait has failed, every later wait of
// every CTA returns within about 1024 polls, so a failing launch drains fast.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, long long max_cycles = kWaitCycles) {
    auto poll = [&] { return kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity); };
    if (poll()) return true;
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        if (poll()) return true;
        if ((n & 1023u) == 0) {
            if (*reinterpret_cast<volatile int *>(&g_device_error) != 0) return false;
            if (clock64() - t0 > max_cycles) {
                record_error(kErrWaitTimeout);
                return false;
            }
        }
    }
}

// warp-uniform bounded wait (the warp leaves together or not at all)
template <bool kCluster = false>
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_bar<kCluster>(bar, parity));
}

constexpr int ptx_log2(int x) { return x <= 1 ? 0 : 1 + ptx_log2(x >> 1); }

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

// (a, b) as a bf16 pair, and the two rounded values added to the packed pair
// of partial sums `acc` (the rounded values are what the MMA accumulates).
__device__ __forceinline__ uint32_t pack_bf16_acc(float a, float b, uint64_t &acc) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    const uint32_t u = *reinterpret_cast<const uint32_t *>(&v);
    acc = ptx::fadd2(acc, ptx::f2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u)));
    return u;
}

// E8M0 scale byte -> 2^(byte - 127) as a float (255 -> NaN; 0 -> 2^-127, a
// subnormal float).
__device__ __forceinline__ float e8m0_scale(uint32_t b) {
    if (b == 255u) return __int_as_float(0x7fc00000);
    return b == 0u ? __int_as_float(0x00400000) : __int_as_float(int(b << 23));
}

// two E4M3 codes (low byte first) -> two bf16 values code * sc, packed low =
// first.  E4M3 -> f16 is exact (cvt.rn.f16x2.e4m3x2), so are f16 -> f32 and
// the power-of-two scale (barring overflow or results below the bf16 range);
// the bf16 rounding is then exact too.
__device__ __forceinline__ uint32_t e4m3x2_scaled_bf16x2(uint32_t codes, float sc) {
    uint32_t h2, out;
    float a, b;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(codes)));
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
        : "=f"(a), "=f"(b) : "r"(h2));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(b * sc), "f"(a * sc));
    return out;
}

// Four E4M3 codes (one word, byte i = code i) -> two bf16x2 words (lo =
// codes 0,1; hi = codes 2,3), each value code * 2^(sbyte - 127), given
// s2 = 2^(sbyte - 7) as bf16 in both halves (sbyte <= 134).  Each code's
// sign goes to bit 15 of a 16-bit lane and its 7 exponent/mantissa bits to
// bits 10..4: read as bf16 the lane then holds exactly code * 2^-120 (for
// zero, subnormal and normal codes alike: bf16 has E4M3's mantissa bits and
// f32's exponent range), and one bf16 multiply by s2, a power of two, makes
// it code * 2^(sbyte - 127) without rounding unless the result leaves bf16's
// normal range.  The NaN codes (S.1111.111) need the exact path.
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t c, uint32_t s2, uint32_t &lo, uint32_t &hi) {
    // byte permutes that sign-extend each code to its 16-bit lane (selector
    // nibbles 8-11 replicate the sign bit of bytes 0-3), then one shift puts
    // the 7 exponent/mantissa bits at 10..4 with a sign copy at bit 15
    // (prmt's generic mode; the __byte_perm intrinsic ignores the sign bit of
    // a selector nibble)
    uint32_t x0, x1;
    asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(x0) : "r"(c));   // [c0, sign(c0), c1, sign(c1)]
    asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(x1) : "r"(c));   // [c2, sign(c2), c3, sign(c3)]
    const uint32_t t0 = (x0 << 4) & 0x87F087F0u;
    const uint32_t t1 = (x1 << 4) & 0x87F087F0u;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(t0), "r"(s2));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(t1), "r"(s2));
}

// nonzero iff one of the four codes is a NaN pattern (low 7 bits all ones)
__device__ __forceinline__ uint32_t e4m3x4_has_nan(uint32_t c) {
    return ((c & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
}

// kPosScale: softmax_scale > 0 (the usual case).  A zero or negative scale
// takes another instantiation whose softmax leaves invalid slots out
// explicitly, so the usual one carries no code for it.
template <int DC, int CL, bool kPosScale, bool kFp8>
__global__ void __launch_bounds__(Cfg<DC, CL, kFp8>::THREADS, 1)
attn_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
               const __grid_constant__ CUtensorMap wmap) {
    using C = Cfg<DC, CL, kFp8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    // Launched with a programmatic dependency on the previous kernel of the
    // stream: that kernel's writes are visible only after this wait, so every
    // thread waits before its first global memory access; the next such
    // launch may begin right away (it waits the same way for this grid).
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // A cluster is one token: its splits x the CL head-dim halves (CL alone
    // when the splits are combined by a separate kernel).  Rank = local split
    // * CL + crank, so the head-dim partner is rank ^ 1.
    const uint32_t rank = (CL == 2 || p.fused) ? ptx::cluster_ctarank() : 0u;
    const uint32_t crank = CL == 2 ? (rank & 1u) : 0u;
    const int64_t unit = blockIdx.x / CL;
    const int64_t tok = unit / p.num_splits;
    const int split = int(unit % p.num_splits);
    const int64_t b = tok / p.S;
    const int64_t iotok = b * p.io_S + p.io_s0 + (tok - b * p.S);   // this token's row of q and o
    const int64_t slot0 = int64_t(split) * p.unit_slots;
    const int64_t left = p.K - slot0;
    const int nslots = left <= 0 ? 0 : int(left < p.unit_slots ? left : p.unit_slots);
    int ntiles = (nslots + kBN - 1) / kBN;

    int32_t *rowc = reinterpret_cast<int32_t *>(smem + C::OFF_IDX);
    uint64_t *vmask = reinterpret_cast<uint64_t *>(smem + C::OFF_VALID);
    int32_t *act = reinterpret_cast<int32_t *>(smem + C::OFF_LIST);  // act[0..n) tiles, act[kMaxUnitTiles] = n
    float2 *stat = reinterpret_cast<float2 *>(smem + C::OFF_STAT);  // (m, l) per head row, after the tiles
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::OFF_TSLOT);
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    auto kv_full = [&](int s) { return bar(s); };
    auto kv_empty = [&](int s) { return bar(C::NS + s); };
    auto s_full = [&](int i) { return bar(2 * C::NS + i); };        // S buffer i written by QK^T
    auto s_empty = [&](int i) { return bar(2 * C::NS + 2 + i); };   // S buffer i read by every softmax warp
    auto p_full = [&](int i) { return bar(2 * C::NS + 4 + i); };    // P buffer i complete, O rows rescaled
    auto p_empty = [&](int i) { return bar(2 * C::NS + 6 + i); };   // P.V of buffer i done (both CTAs of a pair)
    auto o_done = [&](int i) { return bar(2 * C::NS + 8 + i); };    // the P.V of a tile of parity i completed
    const uint32_t q_ready = bar(2 * C::NS + 10);  // Q_c in TMEM
    const uint32_t mma_done = bar(2 * C::NS + 11); // every MMA of the unit completed
    const uint32_t stat_bar = bar(2 * C::NS + 12); // row statistics of every row in place
    const uint32_t q_smem = bar(2 * C::NS + 13);   // Q_c landed in shared memory
    const uint32_t q_free = bar(2 * C::NS + 14);   // Q_c copied to TMEM: its stages are free
    // partner messages, per (tile parity b, lane quarter q)
    auto x_full = [&](int b2, int q) { return bar(C::BAR_X + b2 * 4 + q); };        // partner's partials landed
    auto x_empty = [&](int b2, int q) { return bar(C::BAR_X + 8 + b2 * 4 + q); };   // partner read our partials
    auto pm_full = [&](int b2, int q) { return bar(C::BAR_X + 16 + b2 * 4 + q); };  // partner's P rows + factors landed
    auto stg_full = [&](int f) { return bar(C::BAR_X + 24 + f); };            // FP8: staging f landed
    auto stg_empty = [&](int f) { return bar(C::BAR_X + 24 + C::NF + f); };   // FP8: staging f widened
    const uint32_t rcv_bar = bar(C::BAR_X + 24 + 2 * C::NF);   // in-cluster combine: partials landed

    // ---------------------------------------------------------------- prologue
    // The index list heads the longest dependency chain (index -> kv row ->
    // QK^T), so its loads go out first; every load of a thread is issued
    // before the first is used.
    constexpr int kWarpsAll = C::THREADS / 32;
    constexpr int kSteps = (kMaxUnitSlots / 32 + kWarpsAll - 1) / kWarpsAll;
    int32_t tv[kSteps];
    float *sink_tab = reinterpret_cast<float *>(smem + C::OFF_SINK);
    const float sink_t = tid < p.H ? __ldg(p.sink + tid) : 0.f;   // into sink_tab below
    // slot j of this token counts only below its topk length (clamped to
    // [0, K]); loaded beside the index list, applied when it is converted
    const int32_t len_t = p.topk_len != nullptr ? __ldg(p.topk_len + tok) : int32_t(p.K1);
    const int32_t len2_t = p.topk_len2 != nullptr ? __ldg(p.topk_len2 + tok) : int32_t(p.K2);
    if (p.mask == nullptr) {
#pragma unroll
        for (int u = 0; u < kSteps; ++u) {
            const int j = (u * kWarpsAll + warp) * 32 + lane;
            const int64_t g = slot0 + j;   // slot of the token: main slots, then extra ones
            tv[u] = j >= nslots ? -1 : g < p.K1 ? __ldg(p.idx + tok * p.K1 + g) : __ldg(p.idx2 + tok * p.K2 + (g - p.K1));
        }
    } else {
        // key t is admitted iff bit (t + key_start) & 31 of word
        // (t + key_start) >> 5 of the token's mask row is set; positions
        // outside the row, and with key_start_word the row's last word (the
        // reserved key_start column), admit nothing
        const uint32_t *mrow = p.mask + (b * p.mask_rows + (tok - b * p.S)) * p.mask_words;
        const int64_t key_start =
            p.key_start_word ? int64_t(int32_t(__ldg(p.mask + b * p.mask_rows * p.mask_words + p.mask_words - 1)))
                             : 0;
        const int64_t row_bits = (p.mask_words - p.key_start_word) * 32;
        const int64_t key_end = p.key_ends != nullptr ? int64_t(__ldg(p.key_ends + b)) : row_bits;
        // The unit's mask words (at most 65) read as whole 16-byte vectors of
        // the row and staged in kv stage 0, which the gather fills only after
        // the prologue: vectors w_lo, w_lo + 4, ... cover positions
        // [slot0 + key_start, + nslots); vectors outside the row read as 0.
        uint32_t *mw = reinterpret_cast<uint32_t *>(smem + C::OFF_KV);
        const int64_t p_lo = slot0 + key_start;
        const int64_t w_lo = (p_lo >> 5) & ~int64_t(3);
        const int nvec = nslots > 0 ? int((((p_lo + nslots - 1) >> 5) - w_lo) / 4 + 1) : 0;
        if (tid < nvec) {
            const int64_t w = w_lo + 4 * tid;
            const uint4 v = (w >= 0 && w + 4 <= p.mask_words) ? __ldg(reinterpret_cast<const uint4 *>(mrow + w))
                                                              : make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4 *>(mw)[tid] = v;
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kSteps; ++u) {
            const int j = (u * kWarpsAll + warp) * 32 + lane;
            const int64_t key = slot0 + j + key_start;
            const bool on = j < nslots && key >= 0 && key < row_bits && key < key_end &&
                            ((mw[(key >> 5) - w_lo] >> (key & 31)) & 1u);
            tv[u] = on ? int32_t(slot0 + j) : -1;
        }
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_u32(tslot), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < C::NS; ++s) {
            ptx::mbar_init(kv_full(s), kFp8 ? 32 * kF8WidenWarps : 32 * kGatherWarps);
            ptx::mbar_init(kv_empty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(s_full(i), 1);
            ptx::mbar_init(s_empty(i), kSoftmaxWarps);  // one elected lane per softmax warp
            ptx::mbar_init(p_full(i), kSoftmaxWarps);
            ptx::mbar_init(p_empty(i), CL);             // the P.V commit of each CTA of the pair
            for (int q = 0; q < 4; ++q) {
                ptx::mbar_init(x_full(i, q), 1);    // the owner's expect_tx + XQ bytes from the partner
                ptx::mbar_init(x_empty(i, q), 1);   // one credit from the partner's owner warp
                ptx::mbar_init(pm_full(i, q), 1);   // the sender's expect_tx + P rows and factors
            }
        }
        ptx::mbar_init(o_done(0), 1);
        ptx::mbar_init(o_done(1), 1);
        ptx::mbar_init(q_ready, kSoftmaxThreads);
        ptx::mbar_init(mma_done, 1);
        // owner warps (8, or 4 plus one expect_tx for the partner's 512 bytes)
        ptx::mbar_init(stat_bar, CL == 2 ? 5 : kSoftmaxWarps);
        ptx::mbar_init(q_smem, 1);
        ptx::mbar_init(q_free, kSoftmaxThreads);
        for (int f = 0; f < C::NF; ++f) {
            ptx::mbar_init(stg_full(f), 32 * kF8WidenWarps);
            ptx::mbar_init(stg_empty(f), kF8WidenWarps);
        }
        ptx::mbar_init(rcv_bar, 1);   // thread 0's expect_tx + the bytes of every box
        ptx::fence_mbar_init();
        // Q_c of this unit: DC / 64 boxes of 128 head rows x 64 columns
        ptx::mbar_arrive_expect_tx(q_smem, C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < DC / 64; ++c)
            ptx::tma_load_2d(ptx::smem_u32(smem + C::OFF_QS + c * (kM * 128)), &qmap, int32_t(crank) * DC + c * 64,
                             int32_t(iotok * p.H), q_smem);
    }
    // slot indices -> kv row numbers (-1 = invalid) and a 64-bit validity
    // mask per tile, 32 slots per warp step
    if (p.mask == nullptr) {
#pragma unroll
        for (int u = 0; u < kSteps; ++u) {
            const int ch = u * kWarpsAll + warp;
            if (ch < ntiles * 2) {
                const int j = ch * 32 + lane;
                const int64_t g = slot0 + j;
                const bool main = g < p.K1;
                const bool v = tv[u] >= 0 && (main ? int64_t(tv[u]) < p.T && g < int64_t(len_t)
                                                   : int64_t(tv[u]) < p.T2 && g - p.K1 < int64_t(len2_t));
                rowc[j] = !v ? -1 : main ? int32_t(b * p.T + tv[u]) : int32_t(p.BT + b * p.T2 + tv[u]);
                const uint32_t m = __ballot_sync(0xffffffffu, v);
                if (lane == 0) reinterpret_cast<uint32_t *>(vmask)[ch] = m;
            }
        }
    } else {
        // bit-mask mode: the admitted keys, in key order, packed into the
        // leading slots (a stream compaction over the 32-key chunks); only the
        // last tile can be partial
        static_assert(kSteps * kWarpsAll == kMaxUnitSlots / 32 && kMaxUnitSlots / 32 == 64, "one count per lane pair");
        int *cnt = reinterpret_cast<int *>(stat);  // [64] admitted keys per chunk (scratch until the softmax)
        uint32_t mb[kSteps];
#pragma unroll
        for (int u = 0; u < kSteps; ++u) {
            mb[u] = __ballot_sync(0xffffffffu, tv[u] >= 0);
            if (lane == 0) cnt[u * kWarpsAll + warp] = __popc(mb[u]);
        }
        __syncthreads();
        const int c0 = cnt[lane], c1 = cnt[lane + 32];
        const int total = int(__reduce_add_sync(0xffffffffu, uint32_t(c0 + c1)));
#pragma unroll
        for (int u = 0; u < kSteps; ++u) {
            const int ch = u * kWarpsAll + warp;
            const int base =
                int(__reduce_add_sync(0xffffffffu, uint32_t((lane < ch ? c0 : 0) + (lane + 32 < ch ? c1 : 0))));
            if ((mb[u] >> lane) & 1u)
                rowc[base + __popc(mb[u] & ((1u << lane) - 1u))] = int32_t(b * p.T + tv[u]);
        }
        ntiles = (total + kBN - 1) / kBN;
        if (tid < ntiles * kBN - total) rowc[total + tid] = -1;
        if (tid < ntiles) {
            const int r = total - tid * kBN;
            vmask[tid] = r >= kBN ? ~0ull : ((1ull << r) - 1ull);
        }
    }
    if (tid < kM) sink_tab[tid] = sink_t;
    __syncthreads();
    if (warp == 0) {
        // list of tiles with a valid slot, in order (ntiles <= 32: one warp)
        static_assert(kMaxUnitTiles <= 32, "one lane per tile");
        const bool live = lane < ntiles && vmask[lane] != 0;
        const uint32_t bal = __ballot_sync(0xffffffffu, live);
        if (live) act[__popc(bal & ((1u << lane) - 1u))] = lane;
        if (lane == 0) act[kMaxUnitTiles] = __popc(bal);
    }
    ptx::tc_fence_before();
    __syncthreads();
    // Other CTAs of the cluster must have initialised their barriers and be
    // running before this CTA's first remote access: every thread arrives now
    // and waits only just before its first remote access (the softmax warps)
    // or before the teardown's cluster barrier (the others).
    const bool clustered = CL == 2 || p.fused;
    if (clustered) ptx::cluster_arrive_relaxed();
    ptx::tc_fence_after();
    const uint32_t tbase = *tslot;
    const int n_act = act[kMaxUnitTiles];
    if (warp >= kSoftmaxWarps) {
        // MMA and gather warpgroups: a small register budget
        ptx::setmaxnreg_dec<kOtherRegs>();
        if (warp >= kFirstGatherWarp) {
            if constexpr (kFp8) {
                // ------------------------------------------------- gather, FP8 rows
                // This CTA needs bytes [0, 256) of a row (half 0: codes of dims
                // 0..255) or [256, 576) (half 1: codes of dims 256..447, then the
                // 64 RoPE dims in bf16), plus the scale bytes [576, 584).  A row
                // starts 8 bytes past a 16-byte boundary when its index is odd, so
                // the copies start on the 16-byte boundary at or below the first
                // wanted byte.  In a staging row the wanted bytes then start at
                // `shift` (0 for an even row, 8 for an odd one) and the scale bytes
                // sit at STG_SCALE + shift.  Every gather warp copies the rows it will
                // widen NF tiles ahead, turns the staged rows of the current tile into
                // bf16 in the 128B-swizzled kv stage the MMA reads, and frees the
                // staging buffer; a buffer is refilled once all gather warps freed it.
                const uint8_t *kv8 = reinterpret_cast<const uint8_t *>(p.kv);
                const uint8_t *kv8x = reinterpret_cast<const uint8_t *>(p.kv2);   // extra FP8 rows
                const int base_x = crank == 0 ? 0 : 256;          // first wanted byte of a row
                {
                    // half-warp h of gather warp ww widens rows 2 (ww + W i) + h;
                    // lane u of the half-warp owns 16 dims (16u.. of this half): 16
                    // codes, or for u >= 12 of half 1 the RoPE dims 448 + 16 (u - 12)
                    // as bf16, and stores them as two 16-byte chunks, odd chunk
                    // first in every other 64-dim block so each 8-lane store phase
                    // covers eight distinct bank groups
                    const int ww = warp - kFirstGatherWarp;
                    const int h = lane >> 4, u = lane & 15;
                    constexpr int IT = kBN / (2 * kF8WidenWarps) + (kBN % (2 * kF8WidenWarps) ? 1 : 0);
                    constexpr int CB = 4;                                            // row pairs per load batch
                    const bool rope = crank == 1 && u >= 12;
                    const int sc_idx = crank == 0 ? (u >> 2) : 4 + (u >> 2);         // scale byte of the lane's tile
                    const int off = rope ? 192 + 32 * (u - 12) : 16 * u;             // lane's bytes in a staging row
                    const uint32_t blk = uint32_t(u >> 2);                           // 64-dim block of the stage
                    const uint32_t c_first = 2u * uint32_t(u & 3) + (blk & 1u);      // chunk stored first
                    // the bulk copies of this warp's own rows of tile a into staging a % NF:
                    // lane l < 2 IT copies row 2 (IT-index (l / 2) * kF8WidenWarps + ww) + l % 2,
                    // the row that half-warp l % 2 widens in iteration l / 2.  A valid row's
                    // wanted bytes come by one bulk copy, 16-byte aligned at both ends:
                    // [0, 256) or [-8, 264) for half 0, [256, 576) or [248, 584) for half 1,
                    // the latter with the scale bytes.  The scale bytes of an even row come
                    // by a cp.async that reads only those 8 bytes (a bulk copy of their
                    // 16-byte window would read past the last row); half 0 of an odd row
                    // takes the bulk copy of [568, 584).  Each lane adds its bulk bytes to
                    // the staging barrier before issuing them and arrives (noinc) once its
                    // cp.async has landed; invalid rows are not copied (zeros below).
                    const uint32_t data_even = crank == 0 ? 256u : 320u;   // + 16 for an odd row
                    auto issue_copies = [&](int ta) {
                        const int f = ta % C::NF;
                        const uint32_t stg = ptx::smem_u32(smem + C::OFF_STG + f * C::STG_BYTES);
                        const int r = lane < 2 * IT ? 2 * ((lane >> 1) * kF8WidenWarps + ww) + (lane & 1) : kBN;
                        const int32_t row = r < kBN ? rowc[act[ta] * kBN + r] : -1;
                        if (row >= 0) {
                            // row in its own source (extra rows rebased past the even BT)
                            const bool xr = row >= p.BT;
                            const int64_t rr = xr ? int64_t(row) - p.BT : int64_t(row);
                            const int shift = int(rr & 1) * 8;
                            const uint32_t tx = shift ? data_even + 16u + (crank == 0 ? 16u : 0u) : data_even;
                            ptx::mbar_expect_tx(stg_full(f), tx);
                            const uint8_t *rowp = (xr ? kv8x : kv8) + rr * kF8Row;
                            const uint32_t d = stg + uint32_t(r) * C::STG_ROW;
                            ptx::bulk_load(d, rowp + (base_x - shift), data_even + uint32_t(2 * shift), stg_full(f));
                            if (shift == 0)
                                ptx::cp_async_16(d + uint32_t(C::STG_SCALE), rowp + kF8ScaleOff, 8u);
                            else if (crank == 0)
                                ptx::bulk_load(d + uint32_t(C::STG_SCALE), rowp + (kF8ScaleOff - 8), 16u, stg_full(f));
                        }
                        ptx::cp_async_arrive_noinc(stg_full(f));
                    };
                    static_assert(2 * IT <= 32, "one copied row per lane");
                    for (int ta = 0; ta < C::NF && ta < n_act; ++ta) issue_copies(ta);
                    int a = 0;
                    for (; a < n_act; ++a) {
                        const int s = a % C::NS, fs = a / C::NS, f = a % C::NF;
                        if (!wait_all(stg_full(f), (a / C::NF) & 1)) break;
                        if (fs >= 1 && !wait_all(kv_empty(s), (fs - 1) & 1)) break;
                        // the last two stages hold Q_c until the softmax warps copied it
                        if (a == C::NS - 2 && !wait_all(q_free, 0)) break;
                        const uint8_t *stg = smem + C::OFF_STG + f * C::STG_BYTES;
                        uint8_t *stage = smem + C::OFF_KV + s * C::STAGE_BYTES;
                        const int32_t *rc = rowc + act[a] * kBN;
#pragma unroll
                        for (int i0 = 0; i0 < IT; i0 += CB) {
                            // every load of the batch before the first conversion
                            uint2 v[CB][2], w[CB][2];
                            uint32_t sb[CB];
                            bool inval[CB];
#pragma unroll
                            for (int k = 0; k < CB; ++k) {
                                const int r = 2 * ((i0 + k) * kF8WidenWarps + ww) + h;
                                if (i0 + k >= IT || r >= kBN) break;
                                const int32_t row = rc[r];
                                // as copied (an invalid row was not copied: zeros below)
                                const int shift = row > 0 ? (row & 1) * 8 : 0;
                                inval[k] = row < 0;
                                const uint8_t *srow = stg + r * C::STG_ROW;
                                const uint8_t *src = srow + shift + off;
                                v[k][0] = *reinterpret_cast<const uint2 *>(src);
                                v[k][1] = *reinterpret_cast<const uint2 *>(src + 8);
                                if (rope) {
                                    w[k][0] = *reinterpret_cast<const uint2 *>(src + 16);
                                    w[k][1] = *reinterpret_cast<const uint2 *>(src + 24);
                                }
                                sb[k] = srow[C::STG_SCALE + shift + sc_idx];
                            }
#pragma unroll
                            for (int k = 0; k < CB; ++k) {
                                const int r = 2 * ((i0 + k) * kF8WidenWarps + ww) + h;
                                if (i0 + k >= IT || r >= kBN) break;
                                uint4 o0, o1;   // dims 0-7 and 8-15 of the lane's 16
                                if (rope) {
                                    o0 = make_uint4(v[k][0].x, v[k][0].y, v[k][1].x, v[k][1].y);
                                    o1 = make_uint4(w[k][0].x, w[k][0].y, w[k][1].x, w[k][1].y);
                                } else {
                                    const uint32_t nan = e4m3x4_has_nan(v[k][0].x) | e4m3x4_has_nan(v[k][0].y) |
                                                         e4m3x4_has_nan(v[k][1].x) | e4m3x4_has_nan(v[k][1].y);
                                    if (sb[k] <= 134u && !nan) {
                                        // 2^(sb - 7) as bf16, in both halves
                                        const uint32_t s2 = ((sb[k] + 120u) << 7) * 0x00010001u;
                                        e4m3x4_to_bf16x4(v[k][0].x, s2, o0.x, o0.y);
                                        e4m3x4_to_bf16x4(v[k][0].y, s2, o0.z, o0.w);
                                        e4m3x4_to_bf16x4(v[k][1].x, s2, o1.x, o1.y);
                                        e4m3x4_to_bf16x4(v[k][1].y, s2, o1.z, o1.w);
                                    } else {   // NaN codes or a scale above 2^7: exact conversions
                                        const float sc = e8m0_scale(sb[k]);
                                        o0.x = e4m3x2_scaled_bf16x2(v[k][0].x & 0xffffu, sc);
                                        o0.y = e4m3x2_scaled_bf16x2(v[k][0].x >> 16, sc);
                                        o0.z = e4m3x2_scaled_bf16x2(v[k][0].y & 0xffffu, sc);
                                        o0.w = e4m3x2_scaled_bf16x2(v[k][0].y >> 16, sc);
                                        o1.x = e4m3x2_scaled_bf16x2(v[k][1].x & 0xffffu, sc);
                                        o1.y = e4m3x2_scaled_bf16x2(v[k][1].x >> 16, sc);
                                        o1.z = e4m3x2_scaled_bf16x2(v[k][1].y & 0xffffu, sc);
                                        o1.w = e4m3x2_scaled_bf16x2(v[k][1].y >> 16, sc);
                                    }
                                }
                                if (inval[k]) o0 = o1 = make_uint4(0u, 0u, 0u, 0u);   // an invalid slot's row is 0
                                uint8_t *line = stage + blk * (kBN * 128) + uint32_t(r) * 128u;
                                const uint32_t c0 = c_first, c1 = c_first ^ 1u;   // chunk of dims 0-7 is 2(u&3)
                                const uint4 first = (c0 & 1u) ? o1 : o0, second = (c0 & 1u) ? o0 : o1;
                                *reinterpret_cast<uint4 *>(line + ((c0 ^ uint32_t(r & 7)) << 4)) = first;
                                *reinterpret_cast<uint4 *>(line + ((c1 ^ uint32_t(r & 7)) << 4)) = second;
                            }
                        }
                        ptx::fence_proxy_async_smem();   // generic-proxy stores -> MMA reads
                        ptx::mbar_arrive(kv_full(s));
                        __syncwarp();                    // every lane done with the staging rows ...
                        if (lane == 0) ptx::mbar_arrive(stg_empty(f));   // ... before they are refilled
                        // staging f takes tile a + NF once every gather warp has widened tile a
                        if (a + C::NF < n_act) {
                            if (!wait_all(stg_empty(f), uint32_t(a / C::NF) & 1u)) break;
                            issue_copies(a + C::NF);
                        }
                    }
                    // nothing of ours still lands after the CTA exits: the last fill of
                    // every staging buffer has completed (bounded)
                    const int issued = a + C::NF < n_act ? a + C::NF : n_act;
                    for (int k = issued > C::NF ? issued - C::NF : 0; k < issued; ++k) {
                        const long long t0 = clock64();
                        while (!ptx::mbar_try_wait(stg_full(k % C::NF), uint32_t(k / C::NF) & 1u) &&
                               clock64() - t0 < kWaitCycles) {
                        }
                    }
                }
                ptx::cp_async_wait_all();   // nothing of ours still lands after the CTA exits
            } else {
                // ------------------------------------------------------------ gather
                // every gather warp copies its share of the rows of every tile; each
                // lane's copies arrive on the stage's mbarrier when they land, so a
                // warp runs ahead into every free stage (up to NS tiles in flight)
                constexpr int CPR = DC / 8;     // 16-byte chunks per row slice
                constexpr int RPI = 32 / CPR;   // rows per warp instruction
                constexpr int STEP = RPI * kGatherWarps;
                constexpr int ITERS = (kBN + STEP - 1) / STEP;
                const int g = warp - kFirstGatherWarp;
                const int sub = lane / CPR, ch = lane % CPR;
                const uint32_t dst_col = uint32_t(ch >> 3) * (kBN * 128);
                const char *kvb = reinterpret_cast<const char *>(p.kv) + (int64_t(crank) * DC + ch * 8) * 2;
                // extra rows: the same offset into the extra source, rebased past BT
                const char *kvb2 = p.kv2 == nullptr ? kvb
                                                     : reinterpret_cast<const char *>(p.kv2) +
                                                           (int64_t(crank) * DC + ch * 8 - p.BT * p.D) * 2;
                bool ok = true;
                int a = 0;
                for (; a < n_act; ++a) {
                    const int s = a % C::NS, f = a / C::NS;
                    if (f >= 1 && !wait_all(kv_empty(s), (f - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    // the last two stages hold Q_c until the softmax warps copied it
                    if (a == C::NS - 2 && !wait_all(q_free, 0)) {
                        ok = false;
                        break;
                    }
                    const uint32_t stage = ptx::smem_u32(smem + C::OFF_KV + s * C::STAGE_BYTES);
                    const int32_t *rc = rowc + act[a] * kBN;
                        // unrolled by 2 only: the first tile runs this code cold (the
                    // instruction cache misses of a fully unrolled body cost more
                    // than the loop)
#pragma unroll 2
                    for (int i = 0; i < ITERS; ++i) {
                        const int r = i * STEP + g * RPI + sub;   // warp g: row groups g, g + G, ...
                        if (STEP * ITERS > kBN && r >= kBN) break;
                        const int32_t row = rc[r];
                        const char *src = (row >= p.BT ? kvb2 : kvb) + (row >= 0 ? int64_t(row) : 0) * p.D * 2;
                        const uint32_t dst = stage + dst_col + uint32_t(r) * 128u + uint32_t((ch & 7) ^ (r & 7)) * 16u;
                        ptx::cp_async_16(dst, src, row >= 0 ? 16u : 0u);
                    }
                    ptx::cp_async_arrive_noinc(kv_full(s));
                }
                ptx::cp_async_wait_all();   // nothing of ours still lands after the CTA exits
                (void)ok;
            }
        } else {
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
                    // S(q) goes to buffer q & 1 once every softmax warp has
                    // read S(q-2) from it, and only after P.V(q-3) was issued:
                    // whoever has seen S(q) then knows that P.V(q-3) is
                    // complete (the MMAs of a CTA run in issue order), which
                    // keeps every o_done / p_empty waiter within one phase of
                    // the phase it waits for.  P.V(p) reads P buffer p & 1.
                    if (qn < n_act && qn < pn + 3 && ptx::mbar_test_wait(kv_full(qn % C::NS), (qn / C::NS) & 1) &&
                        (qn < 2 || ptx::mbar_test_wait(s_empty(qn & 1), ((qn >> 1) - 1) & 1))) {
                        ptx::fence_proxy_async_smem();  // gathered rows (generic-proxy writes) -> MMA reads
                        ptx::tc_fence_after();
                        const uint32_t ka = ptx::smem_u32(smem + C::OFF_KV + (qn % C::NS) * C::STAGE_BYTES);
                        const uint32_t sa = tbase + C::S_COL + (qn & 1) * kBN;
    #pragma unroll
                        for (int k = 0; k < DC / 16; ++k) {
                            const uint64_t bd = ptx::sdesc_sw128(ka + (k / 4) * (kBN * 128) + (k % 4) * 32, 16, 1024);
                            ptx::mma_ts(sa, tbase + C::Q_COL + k * 8, bd, idesc_qk, k > 0 ? 1u : 0u);
                        }
                        ptx::mma_commit(s_full(qn & 1));
                        ++qn;
                        prog = true;
                    } else if (pn < qn && ptx::mbar_test_wait(p_full(pn & 1), (pn >> 1) & 1)) {
                        ptx::fence_proxy_async_smem();  // P (generic-proxy writes) -> MMA reads
                        ptx::tc_fence_after();
                        const uint32_t va = ptx::smem_u32(smem + C::OFF_KV + (pn % C::NS) * C::STAGE_BYTES);
                        const uint32_t pa = ptx::smem_u32(smem + C::OFF_P + (pn & 1) * C::P_BYTES);
    #pragma unroll
                        for (int t = 0; t < kBN / 16; ++t) {
                            const uint64_t ad = ptx::sdesc_sw128(pa + t * 32, 16, 1024);
                            const uint64_t bd = ptx::sdesc_sw128(va + t * 2048, kBN * 128, 1024);
                            ptx::mma_ss(tbase + C::O_COL, ad, bd, idesc_pv, (pn > 0 || t > 0) ? 1u : 0u);
                        }
                        ptx::mma_commit(kv_empty(pn % C::NS));
                        ptx::mma_commit(o_done(pn & 1));
                        // P buffer pn & 1 is free here and (with a partner) there
                        if constexpr (CL == 2)
                            ptx::mma_commit_multicast(p_empty(pn & 1), uint16_t((1u << rank) | (1u << (rank ^ 1u))));
                        else
                            ptx::mma_commit(p_empty(pn & 1));
                        ++pn;
                        prog = true;
                    }
                    if (prog) {
                        idle = 0;
                    } else if (++idle == 1) {
                        t0 = clock64();
                    } else if ((idle & 1023u) == 0) {
                        if (*reinterpret_cast<volatile int *>(&g_device_error) != 0) {
                            ok = false;
                        } else if (clock64() - t0 > kWaitCycles) {
                            record_error(kErrWaitTimeout);
                            ok = false;
                        }
                    }
                }
                ptx::mma_commit(mma_done);
            }
        }
        if (clustered) ptx::cluster_wait();
        // back to the launch allocation: the teardown below is common code
        ptx::setmaxnreg_inc<kLaunchRegs>();
    } else {
        ptx::setmaxnreg_inc<kSoftmaxRegs>();
        // ------------------------------------------------------------ softmax / epilogue
        // Q copy and epilogue: thread = (head row h, column half), columns
        // [half*DC/2, (half+1)*DC/2) of q and o; the softmax maps threads
        // to TMEM lanes differently (below)
        const int quarter = warp & 3;            // TMEM lanes this warp may access
        const int half = warp >> 2;
        const int h = quarter * 32 + lane;       // head row == TMEM lane
        const uint32_t lane_addr = tbase + (uint32_t(quarter * 32) << 16);
        const bool hv = h < p.H;
        {
            // this thread's half of Q_c (DC/2 columns of row h) from the TMA
            // boxes into TMEM (bf16 pairs, DC/4 columns).  16-byte unit u of
            // the row sits in box u/8 at unit position (u%8) ^ (h&7).
            constexpr int QW = DC / 4;
            const bool qok = wait_all(q_smem, 0);
            const uint8_t *qs = smem + C::OFF_QS + h * 128;
            auto qunit = [&](int u) -> uint4 {
                if (!hv || !qok) return make_uint4(0u, 0u, 0u, 0u);
                return *reinterpret_cast<const uint4 *>(qs + (u >> 3) * (kM * 128) + (((u & 7) ^ (h & 7)) << 4));
            };
            const int u0 = half * (DC / 16);
            if constexpr (QW >= 32) {
#pragma unroll
                for (int c = 0; c < QW / 32; ++c) {
                    uint32_t v[32];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint4 x = qunit(u0 + c * 8 + i);
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
                    const uint4 x = qunit(u0 + i);
                    v[4 * i] = x.x;
                    v[4 * i + 1] = x.y;
                    v[4 * i + 2] = x.z;
                    v[4 * i + 3] = x.w;
                }
                ptx::tmem_st16(lane_addr + C::Q_COL + half * QW, v);
            }
            ptx::mbar_arrive(q_free);   // the two kv stages holding Q_c may be refilled
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(q_ready);
        }

        // ---------------------------------------------------------- softmax
        // Warp w reads TMEM lanes [16*half, 16*half + 16) of quarter w % 4
        // with the 16x256b shape: for 8-column step k of a tile a thread holds
        // rows rA = g8 and rB = g8 + 8 of those lanes at columns 8k + 2qu and
        // 8k + 2qu + 1 (registers 4k .. 4k+3: rA, rA, rB, rB).  P of the same
        // two columns is one bf16 pair: one 4-byte word of the row in the P
        // buffer (16-byte chunk k, bytes 4qu..4qu+3), which the P.V MMA reads
        // from shared memory as its A operand.
        const int qu = lane & 3, g8 = lane >> 2;
        const uint32_t half_addr = tbase + (uint32_t(quarter * 32 + half * 16) << 16);
        const bool owner = CL == 1 || half == int(crank);
        const float sl2 = p.scale_log2;
        bool ok = true;
        // O rows of this warp's lanes times alA (row rA) and alB (row rB)
        auto rescale_rows = [&](float alA, float alB) {
#pragma unroll 1
            for (int c = 0; c < DC; c += 64) {
                uint32_t r[32];
                ptx::tmem_ld_16x256b_x8(half_addr + C::O_COL + c, r);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    r[4 * k] = __float_as_uint(__uint_as_float(r[4 * k]) * alA);
                    r[4 * k + 1] = __float_as_uint(__uint_as_float(r[4 * k + 1]) * alA);
                    r[4 * k + 2] = __float_as_uint(__uint_as_float(r[4 * k + 2]) * alB);
                    r[4 * k + 3] = __float_as_uint(__uint_as_float(r[4 * k + 3]) * alB);
                }
                ptx::tmem_st_16x256b_x8(half_addr + C::O_COL + c, r);
            }
            ptx::tmem_wait_st();
        };
        // Wait until P.V(j) has completed.  Whoever calls this has seen S of
        // tile j + 1, and QK^T(j+1) is issued after P.V(j-2), so P.V(j-2) is
        // complete: o_done(j & 1) is at the phase of P.V(j) or past it, and a
        // parity wait cannot mistake an older phase for it.
        auto pv_done = [&](int j) -> bool { return wait_all(o_done(j & 1), uint32_t(j >> 1) & 1u); };
        // partner addresses (the same offsets in the other CTA of the pair)
        auto remote = [&](uint32_t local) { return ptx::map_to_rank(local, rank ^ 1u); };
        auto x_buf = [&](int b2) { return ptx::smem_u32(smem + C::OFF_X + (b2 * 4 + quarter) * C::XQ); };
        auto f_buf = [&](int b2) { return ptx::smem_u32(smem + C::OFF_F + (b2 * 4 + quarter) * C::FQ); };
        // this warp's 16 rows of P buffer b2: two 1 KB atoms, rows rA and rA + 8
        // at row g8 of each (row r of an atom at r * 128, its 16-byte chunk c
        // at (c ^ r) * 16)
        const int rowblk = quarter * 32 + half * 16;
        auto p_rows = [&](int b2) { return smem + C::OFF_P + b2 * C::P_BYTES + (rowblk >> 3) * 1024; };
        if (clustered) ptx::cluster_wait();   // before the first remote access
        if (owner) {
            // ------------------------------------------------ owner rows
            float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
            for (int a = 0; a < n_act; ++a) {
                const int sb = a & 1;
                const uint32_t ph = uint32_t(a >> 1) & 1u;
                const int xb = a % C::XB;                          // partner partials buffer
                const uint32_t xph = uint32_t(a / C::XB) & 1u;
                if constexpr (CL == 2) {
                    if (lane == 0) ptx::mbar_arrive_expect_tx(x_full(xb, quarter), C::XQ);
                }
                if (!wait_all(s_full(sb), ph)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                float s[32];
                {
                    uint32_t r[32];
                    ptx::tmem_ld_16x256b_x8(half_addr + C::S_COL + sb * kBN, r);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i2 = 0; i2 < 32; ++i2) s[i2] = __uint_as_float(r[i2]);
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(s_empty(sb));
                if constexpr (CL == 2) {
                    // + the partner's partial logits of the same rows and columns
                    if (!wait_all<true>(x_full(xb, quarter), xph)) {
                        ok = false;
                        break;
                    }
                    const uint8_t *xp = smem + C::OFF_X + (xb * 4 + quarter) * C::XQ + lane * 16;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 v = *reinterpret_cast<const float4 *>(xp + k * 512);
                        s[4 * k] += v.x;
                        s[4 * k + 1] += v.y;
                        s[4 * k + 2] += v.z;
                        s[4 * k + 3] += v.w;
                    }
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive_remote_relaxed(remote(x_empty(xb, quarter)));
                }
                // Row maxima of scale * s over the valid columns.  With a
                // positive scale (the usual case) invalid slots become -inf,
                // the scale is applied once to the maximum, and 2^(scale *
                // -inf - m) gives P = 0 below.  A zero or negative scale would
                // turn -inf into NaN or +inf, so it takes a path that leaves
                // invalid slots out of the maximum and selects P = 0 for them.
                const uint64_t vm = vmask[act[a]];
                const bool full = vm == ~0ull;
                const uint64_t vq = vm >> (2 * qu);   // bit 8k + e: column 8k + 2qu + e
                float mxA = -INFINITY, mxB = -INFINITY;
                if constexpr (kPosScale) {
                    if (!full) {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
#pragma unroll
                            for (int e = 0; e < 2; ++e)
                                if (!((vq >> (8 * k + e)) & 1ull)) s[4 * k + e] = s[4 * k + 2 + e] = -INFINITY;
                    }
                    // 3-input maxima over the 16 values of each row: row A holds
                    // s[4k], s[4k + 1], row B s[4k + 2], s[4k + 3]
                    auto row_max = [&](int o) {
                        const float a0 = ptx::max3(s[o], s[o + 1], s[o + 4]);
                        const float a1 = ptx::max3(s[o + 5], s[o + 8], s[o + 9]);
                        const float a2 = ptx::max3(s[o + 12], s[o + 13], s[o + 16]);
                        const float a3 = ptx::max3(s[o + 17], s[o + 20], s[o + 21]);
                        const float a4 = ptx::max3(s[o + 24], s[o + 25], s[o + 28]);
                        return ptx::max3(ptx::max3(a0, a1, a2), a3, fmaxf(a4, s[o + 29]));
                    };
                    mxA = row_max(0);
                    mxB = row_max(2);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            if ((vq >> (8 * k + e)) & 1ull) {
                                mxA = fmaxf(mxA, s[4 * k + e] * sl2);
                                mxB = fmaxf(mxB, s[4 * k + 2 + e] * sl2);
                            }
                }
                mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
                mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
                mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
                mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
                if constexpr (kPosScale) {
                    mxA *= sl2;
                    mxB *= sl2;
                }
                // lazy rescale: the running maximum moves only when a row's
                // maximum grows by more than the threshold; the factor goes to
                // the partner, which scales its half of the row's O
                float alA = 1.f, alB = 1.f;
                if (a == 0) {
                    mA = mxA;
                    mB = mxB;
                } else {
                    const bool needA = mxA > mA + kRescaleThreshold;
                    const bool needB = mxB > mB + kRescaleThreshold;
                    if (__any_sync(0xffffffffu, needA || needB)) {
                        if (needA) {
                            alA = exp2f(mA - mxA);
                            lA *= alA;
                            mA = mxA;
                        }
                        if (needB) {
                            alB = exp2f(mB - mxB);
                            lB *= alB;
                            mB = mxB;
                        }
                        if (!pv_done(a - 1)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        rescale_rows(alA, alB);
                    }
                }
                // P = 2^(scale*s - m) as bf16 pairs (invalid slots give exactly
                // 0); l sums the rounded values the MMA accumulates
                uint32_t pw[16];
                uint64_t accA = 0ull, accB = 0ull;   // packed pairs of partial sums
                const uint64_t sl22 = ptx::f2(sl2, sl2), nA2 = ptx::f2(-mA, -mA), nB2 = ptx::f2(-mB, -mB);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float z0, z1, z2, z3;
                    ptx::f2_split(ptx::ffma2(ptx::f2(s[4 * k], s[4 * k + 1]), sl22, nA2), z0, z1);
                    ptx::f2_split(ptx::ffma2(ptx::f2(s[4 * k + 2], s[4 * k + 3]), sl22, nB2), z2, z3);
                    float p0 = ex2_approx(z0);
                    float p1 = ex2_approx(z1);
                    float p2 = ex2_approx(z2);
                    float p3 = ex2_approx(z3);
                    if constexpr (!kPosScale) {
                        if (!full) {
                            const bool v0 = (vq >> (8 * k)) & 1ull, v1 = (vq >> (8 * k + 1)) & 1ull;
                            p0 = v0 ? p0 : 0.f;
                            p2 = v0 ? p2 : 0.f;
                            p1 = v1 ? p1 : 0.f;
                            p3 = v1 ? p3 : 0.f;
                        }
                    }
                    pw[2 * k] = pack_bf16_acc(p0, p1, accA);
                    pw[2 * k + 1] = pack_bf16_acc(p2, p3, accB);
                }
                {
                    float a0, a1, b0, b1;
                    ptx::f2_split(accA, a0, a1);
                    ptx::f2_split(accB, b0, b1);
                    lA += a0 + a1;
                    lB += b0 + b1;
                }
                // P of these rows into P buffer sb (free once the P.V of tile
                // a-2 is done in both CTAs of the pair), and with a partner
                // the same rows into its buffer sb, with their rescale factors
                if (a >= 2 && !wait_all(p_empty(sb), uint32_t((a >> 1) - 1) & 1u)) {
                    ok = false;
                    break;
                }
                {
                    // four stmatrix.x4, each the 8x8 blocks (rA, k), (rB, k),
                    // (rA, k+1), (rB, k+1): lane 8i + j addresses row j of
                    // block i, 16-byte chunk k (+1) of the swizzled row
                    const int blk = lane >> 3, jr = lane & 7;
                    const uint32_t row_base = ptx::smem_u32(p_rows(sb)) + uint32_t((blk & 1) * 1024 + jr * 128);
#pragma unroll
                    for (int k = 0; k < 8; k += 2) {
                        const int c = k + (blk >> 1);
                        ptx::stmatrix_x4(row_base + uint32_t(((c ^ jr) & 7) << 4), pw[2 * k], pw[2 * k + 1],
                                         pw[2 * k + 2], pw[2 * k + 3]);
                    }
                }
                if constexpr (CL == 2) {
                    if (qu < 2)
                        ptx::st_async_b32(remote(f_buf(sb)) + uint32_t((qu * 8 + g8) * 4),
                                          __float_as_uint(qu == 0 ? alA : alB), remote(pm_full(sb, quarter)));
                }
                ptx::fence_proxy_async_smem();   // P stores -> MMA and bulk-copy reads
                ptx::tc_fence_before();          // (rescaled O rows -> the next P.V)
                __syncwarp();
                if (lane == 0) {
                    if constexpr (CL == 2) {
                        const uint32_t src = ptx::smem_u32(p_rows(sb));
                        ptx::bulk_copy_to_cluster(remote(src), src, 2048, remote(pm_full(sb, quarter)));
                    }
                    ptx::mbar_arrive(p_full(sb));
                }
            }
            // row statistics (m, l) of these rows, here and at the partner
            lA += __shfl_xor_sync(0xffffffffu, lA, 1);
            lB += __shfl_xor_sync(0xffffffffu, lB, 1);
            lA += __shfl_xor_sync(0xffffffffu, lA, 2);
            lB += __shfl_xor_sync(0xffffffffu, lB, 2);
            if (qu == 0) {
                const int rA = quarter * 32 + half * 16 + g8;
                stat[rA] = make_float2(mA, lA);
                stat[rA + 8] = make_float2(mB, lB);
                if constexpr (CL == 2) {
                    const uint32_t dst = remote(ptx::smem_u32(&stat[rA])), sbar = remote(stat_bar);
                    ptx::st_async_v2(dst, __float_as_uint(mA), __float_as_uint(lA), sbar);
                    ptx::st_async_v2(dst + 64, __float_as_uint(mB), __float_as_uint(lB), sbar);
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(stat_bar);
        } else if constexpr (CL == 2) {
            // ------------------------------------------------ partner rows
            // S of tile j (partner rows) to the partner, one tile ahead
            auto send_s = [&](int j2) -> bool {
                const int jb = j2 & 1;
                if (!wait_all(s_full(jb), uint32_t(j2 >> 1) & 1u)) return false;
                ptx::tc_fence_after();
                uint32_t r[32];
                ptx::tmem_ld_16x256b_x8(half_addr + C::S_COL + jb * kBN, r);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(s_empty(jb));
                const int xj = j2 % C::XB;
                if (j2 >= C::XB && !wait_all(x_empty(xj, quarter), uint32_t((j2 / C::XB) - 1) & 1u)) return false;
                const uint32_t dst = remote(x_buf(xj)) + uint32_t(lane * 16), fbar = remote(x_full(xj, quarter));
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    ptx::st_async_v4(dst + uint32_t(k * 512), r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3], fbar);
                return true;
            };
            if (quarter == 0 && lane == 0) ptx::mbar_arrive_expect_tx(stat_bar, 64 * 8);
            if (n_act > 0) ok = send_s(0);
            for (int a = 0; ok && a < n_act; ++a) {
                if (a + 1 < n_act && !send_s(a + 1)) {
                    ok = false;
                    break;
                }
                // the partner's P rows of tile a (into P buffer a & 1) and
                // their rescale factors, applied to this CTA's half of O
                const int sb = a & 1;
                if (lane == 0) ptx::mbar_arrive_expect_tx(pm_full(sb, quarter), 2048 + C::FQ);
                if (!wait_all<true>(pm_full(sb, quarter), uint32_t(a >> 1) & 1u)) {
                    ok = false;
                    break;
                }
                const float *fa = reinterpret_cast<const float *>(smem + C::OFF_F + (sb * 4 + quarter) * C::FQ);
                const float alA = fa[g8], alB = fa[8 + g8];
                if (__any_sync(0xffffffffu, alA != 1.f || alB != 1.f)) {
                    if (!pv_done(a - 1)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    rescale_rows(alA, alB);
                    ptx::tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(p_full(sb));
            }
        }
        // ------------------------------------------------------------ epilogue
        // every row's (m, l) is in the table once all MMAs have completed;
        // with splits, thread (row h, half 0) publishes the row's
        // log-sum-exp m + log2(l) (base 2; -inf for an empty split): to every
        // split CTA of the token with the same head-dim half (fused), or to
        // the workspace for the combine kernel
        if (ok) ok = wait_all(mma_done, 0);
        if (ok) ok = wait_all<CL == 2>(stat_bar, 0);
        if (ok && p.num_splits > 1 && hv && half == 0) {
            const float2 st = stat[h];
            const float lse = n_act > 0 ? st.x + log2f(st.y) : -INFINITY;
            if (p.fused) {
                const uint32_t slot = ptx::smem_u32(smem + C::OFF_LSE + ((split % 8) * kM + h) * 4);
                for (int s2 = 0; s2 < p.num_splits; ++s2)
                    ptx::st_cluster_b32(ptx::map_to_rank(slot, uint32_t(s2 * CL) + crank), __float_as_uint(lse));
            } else if (crank == 0) {
                p.ws_lse[(tok * p.num_splits + split) * p.H + h] = lse;
            }
        }
        if (!ok) stat[h] = make_float2(NAN, NAN);   // a failed unit writes NaN, never stale data
        ptx::setmaxnreg_dec<kLaunchRegs>();
    }

    // ---------------------------------------------------------------- teardown
    // Output from TMEM by all 16 warps: warp w reads the rows of lane quarter
    // w % 4 (thread = row hr) and column slice w / 4 (DC / 4 columns, in
    // chunks of CC), scales them and writes them into 128B-swizzled staging
    // boxes in the dead kv ring; TMA then stores whole boxes (the H rows of
    // the token by 128 bytes of columns).
    //   one split: o = O * f, f = 2^(m-M) / (l 2^(m-M) + 2^(sink*log2e - M)),
    //     M = max(m, sink*log2e) (§5.5: the sink joins the denominator once,
    //     at the end), bf16;
    //   splits, separate combine: the partial O / l (fp32) to the workspace;
    //   splits combined in the cluster: once every split's log-sum-exp is in
    //     the table, split s scales its O by its final weight w_s / l_s (the
    //     combine kernel's formula), stores the 64-column granules other splits
    //     finish to the workspace and, after a cluster barrier, finishes its
    //     own granules: its weighted O plus the other splits' from L2.
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    {
        constexpr int CW = DC / 4;                        // columns of a warp's slice
        constexpr int CC = CW < 32 ? CW : 32;             // columns per TMEM load
        constexpr int NG = DC / 64;                       // 64-column granules of this CTA
        constexpr int BOX = kM * 128;                     // one staging box: 128 rows x 128 B
        const int q4 = warp & 3, cs = warp >> 2;
        const int hr = q4 * 32 + lane;                    // this thread's row
        const bool rv = hr < p.H;
        const int c_slice = cs * CW;                      // first column of the slice
        const int gran = c_slice / 64;                    // its granule (warp-uniform)
        const uint32_t taddr = tbase + (uint32_t(q4 * 32) << 16) + C::O_COL + c_slice;
        const float2 st = stat[hr];
        const float sink2 = sink_tab[hr] * kLog2e;
        const int ns = p.num_splits;
        const int32_t y_ws = int32_t((tok * ns + split) * p.H);           // workspace rows of this split
        // chunk cc of the slice (fp32; 0 when the unit had no live tile); all
        // 32 lanes load (tcgen05.ld is warp-collective)
        auto load_chunk = [&](int cc, float (&x)[CC]) {
            if (n_act > 0) {
                uint32_t r[CC];
                if constexpr (CC == 32) ptx::tmem_ld32(taddr + cc * CC, r);
                else ptx::tmem_ld16(taddr + cc * CC, r);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int i2 = 0; i2 < CC; ++i2) x[i2] = __uint_as_float(r[i2]);
            } else {
#pragma unroll
                for (int i2 = 0; i2 < CC; ++i2) x[i2] = 0.f;
            }
        };
        // staging box `box` at `base`: row r's 16-byte chunk c at r*128 + ((c ^ (r & 7)) << 4)
        auto box_addr = [&](int base, int box, int chunk) {
            return smem + base + box * BOX + hr * 128 + (((chunk ^ hr) & 7) << 4);
        };
        // columns [c0, c0 + CC) of row hr as fp32 (box = column / 32) or bf16 (box = column / 64)
        auto stage_f32 = [&](int base, int c0, const float (&x)[CC], float f) {
#pragma unroll
            for (int v2 = 0; v2 < CC / 4; ++v2) {
                const int c = c0 + 4 * v2;
                *reinterpret_cast<float4 *>(box_addr(base, c / 32, (c % 32) / 4)) =
                    make_float4(x[4 * v2] * f, x[4 * v2 + 1] * f, x[4 * v2 + 2] * f, x[4 * v2 + 3] * f);
            }
        };
        auto stage_bf16 = [&](int base, int c0, const float (&x)[CC], float f) {
            float dummy = 0.f;
#pragma unroll
            for (int v2 = 0; v2 < CC / 8; ++v2) {
                const int c = c0 + 8 * v2;
                uint4 w;
                w.x = pack_bf16(x[8 * v2] * f, x[8 * v2 + 1] * f, dummy);
                w.y = pack_bf16(x[8 * v2 + 2] * f, x[8 * v2 + 3] * f, dummy);
                w.z = pack_bf16(x[8 * v2 + 4] * f, x[8 * v2 + 5] * f, dummy);
                w.w = pack_bf16(x[8 * v2 + 6] * f, x[8 * v2 + 7] * f, dummy);
                *reinterpret_cast<uint4 *>(box_addr(base, c / 64, (c % 64) / 8)) = w;
            }
        };
        auto publish = [&] {   // generic stores -> TMA reads, all staging written
            ptx::fence_proxy_async_smem();
            __syncthreads();
        };
        // o from the staged bf16 boxes of granules [g0, g1) at `base` (box j:
        // the token's rows by 64 columns, 128B-swizzled), once every thread
        // has staged: 16-byte chunk c of row r goes to thread (r * cpr + c) mod
        // 512, so a warp writes whole rows of this CTA's columns, contiguous in
        // o.  Plain stores let the CTA finish without waiting for a copy engine
        // to read its shared memory.
        auto store_o = [&](int base, int g0, int g1) {
            __syncthreads();
            // (a split finishes 1, 2 or 4 granules: NG is 1, 2 or 4 and the
            // splits share them out as floor(s NG / ns))
            const int cs_shift = 3 + (31 - __clz(g1 - g0));   // log2 of the 16-byte chunks a row
            const int nchunks = p.H << cs_shift;
            __nv_bfloat16 *orow = p.o + int64_t(iotok * p.H) * p.D + int64_t(crank) * DC + 64 * g0;
            for (int i = tid; i < nchunks; i += C::THREADS) {
                const int r = i >> cs_shift, c = i & ((1 << cs_shift) - 1);
                const uint4 v = *reinterpret_cast<const uint4 *>(smem + base + (g0 + (c >> 3)) * BOX + r * 128 +
                                                                (((c & 7) ^ (r & 7)) << 4));
                *reinterpret_cast<uint4 *>(orow + int64_t(r) * p.D + 8 * c) = v;
            }
        };
        const uint32_t sbase = ptx::smem_u32(smem);
        if (ns == 1) {
            float f = 0.f;
            if (n_act > 0 && sink2 != INFINITY) {
                const float M = fmaxf(st.x, sink2);
                const float e = exp2f(st.x - M);
                f = e / (st.y * e + exp2f(sink2 - M));
            }
            if (isnan(sink2) || isnan(st.x)) f = NAN;
#pragma unroll 1
            for (int cc = 0; cc < CW / CC; ++cc) {
                float x[CC];
                load_chunk(cc, x);
                if (rv) stage_bf16(0, c_slice + cc * CC, x, f);
            }
            store_o(0, 0, NG);
        } else if (!p.fused) {
            const float f = n_act > 0 ? 1.f / st.y : 0.f;
#pragma unroll 1
            for (int cc = 0; cc < CW / CC; ++cc) {
                float x[CC];
                load_chunk(cc, x);
                if (rv) stage_f32(0, c_slice + cc * CC, x, f);
            }
            publish();
            if (tid == 0) {
                for (int k = 0; k < 2 * NG; ++k) ptx::tma_store_2d(&wmap, sbase + k * BOX, int32_t(crank) * DC + 32 * k, y_ws);
                ptx::bulk_commit();
                ptx::bulk_wait_read_all();
            }
        } else {
            // Right after its last P.V this split stores the granules other
            // splits finish, as O / l (0 for an empty split), while slower
            // CTAs of the cluster are still in their main loops; one cluster
            // barrier then covers those stores and every split's
            // log-sum-exp in the tables, and the weights are applied on receipt.
            const int gs0 = split * NG / ns, gs1 = (split + 1) * NG / ns;   // this split's granules
            const bool mine = gran >= gs0 && gran < gs1;
            const float inv_l = (n_act > 0 && st.y > 0.f) ? 1.f / st.y : 0.f;
            if (!mine) {
#pragma unroll 1
                for (int cc = 0; cc < CW / CC; ++cc) {
                    float x[CC];
                    load_chunk(cc, x);
                    if (rv) stage_f32(0, c_slice + cc * CC, x, inv_l);
                }
            }
            publish();
            if (tid == 0) {
                for (int k = 0; k < 2 * NG; ++k)
                    if (k / 2 < gs0 || k / 2 >= gs1)
                        ptx::tma_store_2d(&wmap, sbase + k * BOX, int32_t(crank) * DC + 32 * k, y_ws);
                ptx::bulk_commit();
                ptx::bulk_wait_all();              // written, not just read
                ptx::fence_proxy_async_global();   // async-proxy writes before the barrier's release
            }
            float acc[CW];
            if (mine) {
#pragma unroll
                for (int cc = 0; cc < CW / CC; ++cc) {
                    float x[CC];
                    load_chunk(cc, x);
#pragma unroll
                    for (int i2 = 0; i2 < CC; ++i2) acc[cc * CC + i2] = x[i2] * inv_l;
                }
            }
            ptx::cluster_sync();   // every split's partials in the workspace, its log-sum-exp in the tables
            // final weight of every split for row hr (the combine kernel's formula)
            const float *tab = reinterpret_cast<const float *>(smem + C::OFF_LSE);   // [split][row]
            float mx = -INFINITY;
            for (int i2 = 0; i2 < ns; ++i2) mx = fmaxf(mx, tab[i2 * kM + hr]);
            const float M = fmaxf(mx, sink2);
            const bool zero = (sink2 == INFINITY) || (M == -INFINITY);
            float den = 0.f;
            if (!zero) {
                for (int i2 = 0; i2 < ns; ++i2) {
                    const float li = tab[i2 * kM + hr];
                    if (li != -INFINITY) den += exp2f(li - M);
                }
                den += exp2f(sink2 - M);
            }
            const float fn = isnan(sink2) ? NAN : 1.f;
            auto weight = [&](int t) {   // w_t / den (0 for an empty split)
                const float lt = tab[t * kM + hr];
                return (zero || lt == -INFINITY) ? 0.f : exp2f(lt - M) / den;
            };
            if (mine) {
                const float w_own = weight(split);
#pragma unroll
                for (int i2 = 0; i2 < CW; ++i2) acc[i2] *= w_own;
            }
            // the other splits' partials of this split's granules, a round of
            // as many splits as the receive area holds at a time, added to
            // this split's own with their weights
            const int nsub = 2 * (gs1 - gs0);                                // 32-column boxes per split
            const int hbase = (C::OFF_STAT - NG * BOX) / 1024 * 1024;          // bf16 staging, above the receive area
            const int per_round = nsub > 0 ? hbase / (nsub * BOX) : 1;
            bool rok = true;
            int done = 0, round = 0;
            while (nsub > 0 && done < ns - 1) {
                const int cnt = ns - 1 - done < per_round ? ns - 1 - done : per_round;
                if (tid == 0) {
                    ptx::fence_proxy_async_global();   // the barrier's acquire before these async-proxy reads
                    ptx::mbar_arrive_expect_tx(rcv_bar, uint32_t(cnt * nsub) * uint32_t(p.H) * 128u);
                    for (int t2 = 0; t2 < cnt; ++t2) {
                        const int oth = done + t2 < split ? done + t2 : done + t2 + 1;   // t2-th other split
                        for (int k = 0; k < nsub; ++k)
                            ptx::tma_load_2d(sbase + (t2 * nsub + k) * BOX, &wmap, int32_t(crank) * DC + 64 * gs0 + 32 * k,
                                             int32_t((tok * ns + oth) * p.H), rcv_bar);
                    }
                }
                rok = rok && wait_all(rcv_bar, uint32_t(round) & 1u);
                if (mine && rok) {
                    for (int t2 = 0; t2 < cnt; ++t2) {
                        const int oth = done + t2 < split ? done + t2 : done + t2 + 1;
                        const float wt = weight(oth);
#pragma unroll
                        for (int v2 = 0; v2 < CW / 4; ++v2) {
                            const int c = c_slice + 4 * v2;                     // column of this CTA
                            const int k = (c - 64 * gs0) / 32;                  // box among this split's
                            const float4 w4 = *reinterpret_cast<const float4 *>(
                                smem + (t2 * nsub + k) * BOX + hr * 128 + (((((c % 32) / 4) ^ hr) & 7) << 4));
                            acc[4 * v2] = fmaf(wt, w4.x, acc[4 * v2]);
                            acc[4 * v2 + 1] = fmaf(wt, w4.y, acc[4 * v2 + 1]);
                            acc[4 * v2 + 2] = fmaf(wt, w4.z, acc[4 * v2 + 2]);
                            acc[4 * v2 + 3] = fmaf(wt, w4.w, acc[4 * v2 + 3]);
                        }
                    }
                }
                __syncthreads();   // the receive area is read before it is refilled
                done += cnt;
                ++round;
            }
            // the finished granules as bf16, staged above the receive area
            if (mine && rv) {
#pragma unroll
                for (int cc = 0; cc < CW / CC; ++cc) {
                    float x[CC];
#pragma unroll
                    for (int i2 = 0; i2 < CC; ++i2) x[i2] = rok ? acc[cc * CC + i2] * fn : NAN;
                    stage_bf16(hbase, c_slice + cc * CC, x, 1.f);
                }
            }
            if (gs1 > gs0) store_o(hbase, gs0, gs1);
            else __syncthreads();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        if (lane == 0) wait_bar(mma_done, 0);  // no MMA in flight before TMEM is released
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tbase, C::TMEM_COLS);
    }
    if constexpr (CL == 2) {
        if (!p.fused) ptx::cluster_sync();  // no remote access outlives the partner
    }
}

// Split-KV combine (§5.5, log-sum-exp form with the sink added exactly once):
//   M = max(max_i lse_i, sink*log2e),  w_i = 2^(lse_i - M),
//   o = sum_i w_i O_i / (sum_i w_i + 2^(sink*log2e - M)).
// One warp per (token, head); lane l owns the 4-column groups l, l + 32, ...
// so every warp load is 512 contiguous bytes.
template <int D>
__global__ void __launch_bounds__(128)
attn_combine_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_lse, const float *__restrict__ sink,
                    __nv_bfloat16 *__restrict__ o, int64_t rows, int64_t H, int ns, int64_t S, int64_t io_S,
                    int64_t io_s0) {
    ptx::griddep_wait();               // the stream's previous kernel: complete and visible
    ptx::griddep_launch_dependents();
    constexpr int E = D / 32;              // columns per lane
    constexpr int V = E >= 4 ? 4 : 2;      // columns per vector access
    constexpr int G = E / V;               // vectors per lane
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
            const float *src = ws_o + ((tok * ns + i) * H + h) * D + lane * V;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                if constexpr (V == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(src + g * 128);
                    acc[4 * g] = fmaf(w, v.x, acc[4 * g]);
                    acc[4 * g + 1] = fmaf(w, v.y, acc[4 * g + 1]);
                    acc[4 * g + 2] = fmaf(w, v.z, acc[4 * g + 2]);
                    acc[4 * g + 3] = fmaf(w, v.w, acc[4 * g + 3]);
                } else {
                    const float2 v = *reinterpret_cast<const float2 *>(src + g * 64);
                    acc[2 * g] = fmaf(w, v.x, acc[2 * g]);
                    acc[2 * g + 1] = fmaf(w, v.y, acc[2 * g + 1]);
                }
            }
        }
        den += exp2f(s2 - M);
    }
    const float f = zero ? 0.f : 1.f / den;
    const float fn = isnan(s2) ? NAN : f;
    const int64_t bq = tok / S;   // o row of token tok: a window of io_S query rows per request
    __nv_bfloat16 *dst = o + ((bq * io_S + io_s0 + (tok - bq * S)) * H + h) * D + lane * V;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[V * g] * fn, acc[V * g + 1] * fn);
        if constexpr (V == 4) {
            const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[4 * g + 2] * fn, acc[4 * g + 3] * fn);
            *reinterpret_cast<uint2 *>(dst + g * 128) =
                make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
        } else {
            *reinterpret_cast<__nv_bfloat162 *>(dst + g * 64) = lo;
        }
    }
}

// ---------------------------------------------------------------- host side

constexpr int kMaxDev = 64;

constexpr int kMaxFusedCluster = 8;   // portable cluster size

// The CUDA driver API's tensor-map encoder, looked up once through the
// runtime (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        (void)cudaGetLastError();
    });
    return fn;
}

// q viewed as [tokens * H rows][D columns] bf16; boxes of 128 rows x 64
// columns (128 B), 128B-swizzled, rows past the end read as zeros.
cudaError_t encode_q_map(CUtensorMap *m, const AttnArgs &a) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return cudaErrorNotSupported;
    const int64_t io_S = a.io_S > 0 ? a.io_S : a.S;
    cuuint64_t dims[2] = {cuuint64_t(a.D), cuuint64_t(a.B * io_S * a.H)};
    cuuint64_t strides[1] = {cuuint64_t(a.D) * 2};
    cuuint32_t box[2] = {64, cuuint32_t(kM)};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.q), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The kernel's output boxes: the H rows of one token by 128 bytes of
// columns, 128B-swizzled.  o: bf16 [B * io_S * H rows][D] (64 columns a box);
// the split workspace: fp32 [tokens * splits * H rows][D] (32 columns a box).
cudaError_t encode_out_maps(CUtensorMap *omap, CUtensorMap *wmap, const AttnArgs &a) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return cudaErrorNotSupported;
    const int64_t io_S = a.io_S > 0 ? a.io_S : a.S;
    cuuint32_t estr[2] = {1, 1};
    {
        cuuint64_t dims[2] = {cuuint64_t(a.D), cuuint64_t(a.B * io_S * a.H)};
        cuuint64_t strides[1] = {cuuint64_t(a.D) * 2};
        cuuint32_t box[2] = {64, cuuint32_t(a.H)};
        const CUresult r = enc(omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.o, dims, strides, box, estr,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    if (a.num_splits > 1) {
        cuuint64_t dims[2] = {cuuint64_t(a.D), cuuint64_t(a.B * a.S * a.num_splits * a.H)};
        cuuint64_t strides[1] = {cuuint64_t(a.D) * 4};
        cuuint32_t box[2] = {32, cuuint32_t(a.H)};
        const CUresult r = enc(wmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.ws_o, dims, strides, box, estr,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    } else {
        *wmap = CUtensorMap{};   // unused without splits
    }
    return cudaSuccess;
}

// Opt the kernel into its dynamic shared memory once per device.
template <int DC, int CL, bool F8>
cudaError_t prepare_kernel(int dev) {
    using C = Cfg<DC, CL, F8>;
    static std::once_flag attr_once[kMaxDev];
    static cudaError_t attr_err[kMaxDev];
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::call_once(attr_once[dev], [dev] {
        attr_err[dev] = cudaFuncSetAttribute(attn_tc_kernel<DC, CL, true, F8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (attr_err[dev] == cudaSuccess)
            attr_err[dev] = cudaFuncSetAttribute(attn_tc_kernel<DC, CL, false, F8>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        // The warpgroups' setmaxnreg split is drawn from the launch allocation;
        // a build that launched with fewer registers per thread could never
        // satisfy the softmax warpgroups' increase, so it is not launched.
        cudaFuncAttributes fa{};
        for (int k = 0; k < 2 && attr_err[dev] == cudaSuccess; ++k) {
            attr_err[dev] = k == 0 ? cudaFuncGetAttributes(&fa, attn_tc_kernel<DC, CL, true, F8>)
                                   : cudaFuncGetAttributes(&fa, attn_tc_kernel<DC, CL, false, F8>);
            if (attr_err[dev] == cudaSuccess && fa.numRegs < kLaunchRegs) attr_err[dev] = cudaErrorInvalidConfiguration;
        }
    });
    return attr_err[dev];
}

// Whether a token's ns splits are combined inside the kernel: they must fit
// one portable cluster together with their head-dim halves, and such a
// cluster must be placeable on this device (asked once per cluster size).
template <int DC, int CL, bool F8>
bool fused_combine(int dev, int ns) {
    using C = Cfg<DC, CL, F8>;
    static std::once_flag fit_once[kMaxDev][kMaxFusedCluster + 1];
    static bool fits[kMaxDev][kMaxFusedCluster + 1];
    const int cs = CL * ns;
    if (ns < 2 || cs > kMaxFusedCluster || dev < 0 || dev >= kMaxDev) return false;
    if (prepare_kernel<DC, CL, F8>(dev) != cudaSuccess) return false;
    std::call_once(fit_once[dev][cs], [dev, cs] {
        cudaLaunchConfig_t q{};
        q.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
        q.blockDim = dim3(C::THREADS, 1, 1);
        q.dynamicSmemBytes = C::SMEM;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = static_cast<unsigned>(cs);
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        q.attrs = qa;
        q.numAttrs = 1;
        int n = 0;
        const cudaError_t qe = cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<DC, CL, true, F8>, &q);
        fits[dev][cs] = qe == cudaSuccess && n >= 1;
        (void)cudaGetLastError();   // a refused query is not a launch error
    });
    return fits[dev][cs];
}

template <int DC, int CL, bool F8>
cudaError_t launch_tc(const AttnArgs &a, cudaStream_t stream, bool *fused_out) {
    using C = Cfg<DC, CL, F8>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = prepare_kernel<DC, CL, F8>(dev);
    if (e != cudaSuccess) return e;

    TcParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.kv = static_cast<const __nv_bfloat16 *>(a.kv);
    p.sink = a.sink;
    p.idx = a.idx;
    p.topk_len = a.topk_len;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.ws_o = a.ws_o;
    p.ws_lse = a.ws_lse;
    p.S = a.S; p.H = a.H; p.D = a.D; p.T = a.T; p.K = a.K + a.K2;
    p.K1 = a.K; p.K2 = a.K2; p.T2 = a.T2;
    p.kv2 = a.kv2; p.idx2 = a.idx2; p.topk_len2 = a.topk_len2;
    p.BT = (a.B * a.T + 1) / 2 * 2;
    p.num_splits = a.num_splits;
    p.unit_slots = int(split_slots(a.K + a.K2, a.num_splits));
    const int cs_fused = CL * a.num_splits;
    const bool fused = fused_combine<DC, CL, F8>(dev, a.num_splits);
    p.fused = fused ? 1 : 0;
    *fused_out = fused;
    p.scale_log2 = a.scale * kLog2e;
    p.mask = a.mask;
    p.mask_rows = a.mask_rows;
    p.mask_words = a.mask_words;
    p.key_start_word = a.key_start_word;
    p.key_ends = a.key_ends;
    p.io_S = a.io_S > 0 ? a.io_S : a.S;
    p.io_s0 = a.io_s0;
    if (p.unit_slots > kMaxUnitSlots) return cudaErrorInvalidValue;

    const int64_t ctas = a.B * a.S * a.num_splits * CL;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(fused ? cs_fused : CL);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: the kernel waits (griddepcontrol.wait)
    // for the stream's previous kernel before it touches global memory
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    CUtensorMap qmap;
    e = encode_q_map(&qmap, a);
    if (e != cudaSuccess) return e;
    CUtensorMap omap, wmap;
    e = encode_out_maps(&omap, &wmap, a);
    if (e != cudaSuccess) return e;
    return a.scale > 0.f ? cudaLaunchKernelEx(&cfg, attn_tc_kernel<DC, CL, true, F8>, p, qmap, omap, wmap)
                         : cudaLaunchKernelEx(&cfg, attn_tc_kernel<DC, CL, false, F8>, p, qmap, omap, wmap);
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
    bool fused = false;
    if (a.kv_fp8) {
        if (a.D != 512) return cudaErrorInvalidValue;
        e = launch_tc<256, 2, true>(a, stream, &fused);
    } else {
        switch (a.D) {
            case 64: e = launch_tc<64, 1, false>(a, stream, &fused); break;
            case 128: e = launch_tc<128, 1, false>(a, stream, &fused); break;
            case 256: e = launch_tc<256, 1, false>(a, stream, &fused); break;
            case 512: e = launch_tc<256, 2, false>(a, stream, &fused); break;
            default: return cudaErrorInvalidValue;
        }
    }
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.num_splits > 1 && !fused) return launch_attn_combine(a, stream);
    return cudaSuccess;
}

int kernels_per_call(int64_t D, int num_splits, bool kv_fp8) {
    if (num_splits <= 1) return 1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    bool fused = false;
    if (kv_fp8) {
        if (D != 512) return 0;
        fused = fused_combine<256, 2, true>(dev, num_splits);
    } else {
        switch (D) {
            case 64: fused = fused_combine<64, 1, false>(dev, num_splits); break;
            case 128: fused = fused_combine<128, 1, false>(dev, num_splits); break;
            case 256: fused = fused_combine<256, 1, false>(dev, num_splits); break;
            case 512: fused = fused_combine<256, 2, false>(dev, num_splits); break;
            default: return 0;
        }
    }
    return fused ? 1 : 2;
}

cudaError_t launch_attn_combine(const AttnArgs &a, cudaStream_t stream) {
    const int64_t rows = a.B * a.S * a.H;
    const int64_t io_S = a.io_S > 0 ? a.io_S : a.S;   // 0: o holds exactly the call's S rows per request
    if (rows == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((rows + 3) / 4);
    cudaError_t e;
    switch (a.D) {
        case 64: e = launch_pdl(attn_combine_kernel<64>, grid, dim3(128), 0, stream, a.ws_o, a.ws_lse, a.sink, static_cast<__nv_bfloat16 *>(a.o), rows, a.H, a.num_splits, a.S, io_S, a.io_s0); break;
        case 128: e = launch_pdl(attn_combine_kernel<128>, grid, dim3(128), 0, stream, a.ws_o, a.ws_lse, a.sink, static_cast<__nv_bfloat16 *>(a.o), rows, a.H, a.num_splits, a.S, io_S, a.io_s0); break;
        case 256: e = launch_pdl(attn_combine_kernel<256>, grid, dim3(128), 0, stream, a.ws_o, a.ws_lse, a.sink, static_cast<__nv_bfloat16 *>(a.o), rows, a.H, a.num_splits, a.S, io_S, a.io_s0); break;
        case 512: e = launch_pdl(attn_combine_kernel<512>, grid, dim3(128), 0, stream, a.ws_o, a.ws_lse, a.sink, static_cast<__nv_bfloat16 *>(a.o), rows, a.H, a.num_splits, a.S, io_S, a.io_s0); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}


// Self-test of the bounded wait: one warp waits, with the kernel's own wait
// routine and a short cycle limit, on an mbarrier phase that nothing ever
// completes.  The wait must give up, record kErrWaitTimeout and return.
__global__ void wait_timeout_selftest_kernel(long long max_cycles) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    (void)wait_bar(ptx::smem_u32(&bar), 0, max_cycles);
}

cudaError_t launch_wait_timeout_selftest(long long max_cycles, cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(max_cycles);
    return cudaGetLastError();
}

// Self-test of the fast drain: CTA 0 waits with a short limit on a phase
// nothing completes, every other CTA with the full limit; all of them return
// soon after CTA 0 records its timeout (the waits watch the error word).
__global__ void wait_drain_selftest_kernel(long long first_cycles) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    (void)wait_bar(ptx::smem_u32(&bar), 0, blockIdx.x == 0 ? first_cycles : kWaitCycles);
}

cudaError_t launch_wait_drain_selftest(int ctas, long long first_cycles, cudaStream_t stream) {
    wait_drain_selftest_kernel<<<ctas, 32, 0, stream>>>(first_cycles);
    return cudaGetLastError();
}

cudaError_t device_error_word(int **ptr) {
    static std::once_flag once[kMaxDev];
    static int *addr[kMaxDev];
    static cudaError_t err[kMaxDev];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        void *a = nullptr;
        err[dev] = cudaGetSymbolAddress(&a, g_device_error);
        addr[dev] = static_cast<int *>(a);
    });
    *ptr = addr[dev];
    return err[dev];
}

void *tensor_map_encode_fn() { return reinterpret_cast<void *>(tensor_map_encoder()); }

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
