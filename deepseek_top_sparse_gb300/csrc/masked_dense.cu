// The consumer of the bit-packed top-k mask for D <= 256 on the sm_103a
// tensor cores: dense attention of every query token over the keys its mask
// row admits ("dense_mask_mod" / "offset_dense_mask_mod" on the vLLM PR 48770
// page, rows of whole 16-byte vectors on the vLLM PR 52217 page), with the
// softmax and sink of sparse_attn ("DeepSeek V4 源码剖析, 第5章" §5.2, §5.5).
//
// Packing.  kv[b] is shared by every head of request b, so the G = 128 / H
// query tokens of a group share one key tile: the 128 MMA rows are G tokens x
// H heads (row r = token r / H, head r % H) and each row applies its own
// token's mask bits in the softmax.  A work unit is (request, group of G
// consecutive query tokens, key split); a key tile is BN consecutive keys of
// kv[b], loaded whole by TMA -- the keys are dense, nothing is gathered.
//
// Per CTA (one unit, 8 warps):
//   all warps  (prologue) read the group's mask rows over the unit's key range
//              with 16-byte loads and mark, in a shared bitmap, every key tile
//              in which some row admits a key; only those tiles are loaded and
//              computed;
//   warp 4     TMA: Q once (128 rows x D), then the marked key tiles through an
//              NS-stage ring;
//   warp 5     tcgen05.mma: S = Q K^T into one of NB TMEM S buffers (ahead of
//              the softmax), O += P V with P (bf16) read from one of NB TMEM P
//              buffers and V the same stage read MN-major; O stays in TMEM for
//              the unit (warps 6 and 7 only help with the prologue);
//   warps 0..3 softmax, one thread per row (lane quarter = warp): the
//              row's mask words for the tile (prefetched one tile ahead: one
//              aligned vector load when the tile's positions start on a
//              multiple of BN inside the admissible range, else two 16-byte
//              vectors and a funnel shift), masked row maximum, lazy rescale
//              of O (only when the maximum grows by more than 2^8),
//              P = 2^(x - m) into TMEM; then the epilogue (o = O / (l + sink
//              term), bf16, or the split partials for the combine kernel).
//
// Units launch with the query groups last-first (the requests interleaved):
// later queries usually see more keys, so the heaviest units start first.
//
// Every mbarrier wait is bounded by clock64 and gives up early once any wait
// has recorded an error in the library's device error word; before it exits a
// CTA waits (bounded) for its own TMA loads and MMAs.
#include <cuda_bf16.h>

#include <cudaTypedefs.h>
#include <mutex>

#include "ptx.cuh"
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kRows = 128;               // MMA rows (TMEM lanes): G tokens x H heads
constexpr int kThreads = 256;
// D = 64 (two CTAs per SM): launched at 128 registers a thread; after the
// prologue the softmax warpgroup grows to 200 and the other warpgroup shrinks
// to 56: 128 * 200 + 128 * 56 = 256 * 128.
constexpr int kLaunchRegs = 128;
constexpr int kSoftmaxRegs = 200;
constexpr int kOtherRegs = 56;
static_assert(128 * kSoftmaxRegs + 128 * kOtherRegs <= kThreads * kLaunchRegs, "register split");
// setmaxnreg acts on whole warpgroups: every warpgroup of the CTA must be
// complete and execute the same setmaxnreg
static_assert(kThreads % 128 == 0, "whole warpgroups");
constexpr int kMaxTiles = 8192;          // key tiles per work unit (the host enforces it)
constexpr int kBitmapWords = kMaxTiles / 32;
constexpr long long kWaitCycles = 200000000ll;   // ~0.1 s at 2 GHz per wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.f;      // O and l are rescaled once the row maximum grows by more

// D = 64 runs two CTAs per SM (128-key tiles with one S and one P buffer in
// 256 TMEM columns each), so each SM sub-partition interleaves two softmax
// warps; D = 128 (128-key tiles) and 256 (64-key tiles) run one CTA with two
// S and two P buffers.
template <int D>
struct Md {
    static constexpr int CPS = D == 64 ? 2 : 1;      // CTAs per SM
    static constexpr int BN = D <= 128 ? 128 : 64;   // keys per tile
    static constexpr int NB = D == 64 ? 1 : 2;       // S and P buffers
    static constexpr int NCH = D / 64;               // 128-byte column chunks of a row
    static constexpr int NW = BN / 32;               // mask words per tile
    static constexpr int Q_BYTES = kRows * D * 2;
    static constexpr int STAGE = BN * D * 2;
    static constexpr int NS = D == 64 ? 4 : (D == 128 ? 5 : 4);
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_KV = OFF_Q + Q_BYTES;
    static constexpr int OFF_BITS = OFF_KV + NS * STAGE;
    static constexpr int OFF_BAR = OFF_BITS + kBitmapWords * 4;
    // mbarriers
    static constexpr int B_KV_FULL = 0;              // [NS] TMA bytes landed
    static constexpr int B_KV_EMPTY = NS;            // [NS] the P.V that read the stage is done
    static constexpr int B_S_FULL = 2 * NS;          // [2] S buffer written (NB used)
    static constexpr int B_S_EMPTY = 2 * NS + 2;     // [2] S buffer read by the 4 softmax warps
    static constexpr int B_P_FULL = 2 * NS + 4;      // [2] P buffer written by the 4 softmax warps
    static constexpr int B_PV_DONE = 2 * NS + 6;     // [2] the P.V of that P buffer is done
    static constexpr int B_Q = 2 * NS + 8;
    static constexpr int B_MMA_DONE = 2 * NS + 9;
    static constexpr int NUM_BARS = 2 * NS + 10;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM = OFF_TSLOT + 16 + 1024;   // + slack to align the base to 1 KB
    // TMEM columns
    static constexpr int O_COL = 0;
    static constexpr int S_COL = D;                  // NB buffers of BN fp32 columns
    static constexpr int P_COL = D + NB * BN;        // NB buffers of BN / 2 columns (bf16 pairs)
    static constexpr int TMEM_COLS = CPS == 2 ? 256 : 512;
    static_assert(P_COL + NB * BN / 2 <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM * CPS <= 227 * 1024, "shared memory budget");
    static_assert(Q_BYTES % 1024 == 0 && STAGE % 1024 == 0, "1 KB swizzle alignment");
};

struct MdParams {
    const float *sink;          // [H]
    const uint32_t *mask;       // [B, mask_rows, W]
    const int32_t *key_ends;    // [B] live key end (mask position), or nullptr
    __nv_bfloat16 *o;           // [B, io_S, H, D]
    float *ws_o, *ws_lse;       // split partials (ns > 1)
    int *err;                   // the library's device error word
    int64_t mask_rows, W, T;
    int key_start_word;
    int B, S, io_S, io_s0, H, G, groups, ns, tps, nt;
    float scale_log2;
};

__device__ __forceinline__ void record_error(int *err, int code) { atomicCAS(err, 0, code); }

// Bounded wait: false after kWaitCycles (recording the timeout) or as soon as
// any wait has recorded an error.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, int *err) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((n & 1023u) == 0) {
            if (*reinterpret_cast<volatile int *>(err) != 0) return false;
            if (clock64() - t0 > kWaitCycles) {
                record_error(err, kErrWaitTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, int *err) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, err));
}

// Bounded wait that ignores the error word: a CTA's drain of its own copies.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!ptx::mbar_try_wait(bar, parity) && clock64() - t0 < kWaitCycles) {
    }
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// The marked key tiles of the unit in ascending order.
struct TileIter {
    const uint32_t *bm;
    int nbw, wi, k0;
    uint32_t bits;
    __device__ TileIter(const uint32_t *bm_, int nbw_, int k0_) : bm(bm_), nbw(nbw_), wi(0), k0(k0_) {
        bits = nbw > 0 ? bm[0] : 0u;
    }
    __device__ int next() {
        while (bits == 0u) {
            if (++wi >= nbw) return -1;
            bits = bm[wi];
        }
        const int j = __ffs(int(bits)) - 1;
        bits &= bits - 1u;
        return k0 + 32 * wi + j;
    }
};

// One aligned 16-byte vector (words [c, c + 4)) of a mask row, zero outside
// [0, W); words at or past wlim read as zero.
__device__ __forceinline__ void mask_vec(const uint32_t *row, int64_t c, int64_t W, int64_t wlim, uint32_t (&x)[4]) {
    if (row != nullptr && c >= 0 && c + 4 <= W) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(row + c));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
        x[0] = x[1] = x[2] = x[3] = 0u;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (c + k >= wlim) x[k] = 0u;
}

template <int D, bool POS>
__global__ void __launch_bounds__(kThreads, Md<D>::CPS)
masked_dense_kernel(const MdParams p, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kvmap) {
    ptx::griddep_wait();               // the stream's previous kernel: complete and visible
    ptx::griddep_launch_dependents();
    using C = Md<D>;
    constexpr int BN = C::BN;
    constexpr int NW = C::NW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem + C::OFF_BITS);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::OFF_TSLOT);
    auto bar = [&](int i) { return ptx::smem_u32(bars + i); };

    // ---- the unit.  Groups launch last-first (the requests interleaved):
    // later queries usually see more keys, and the heaviest units starting
    // first leave the lightest for the last wave.
    const int unit = blockIdx.x;
    const int split = unit % p.ns;
    const int grp = unit / p.ns;
    const int b = grp % p.B;
    const int s0 = (p.groups - 1 - grp / p.B) * p.G;  // first query token of the group (window row)
    const int gv = min(p.G, p.S - s0);                // tokens of the group
    const int k0 = split * p.tps;                     // key tiles [k0, k1)
    const int k1 = min(k0 + p.tps, p.nt);
    const int nbw = k1 > k0 ? (k1 - k0 + 31) / 32 : 0;

    // key t of request b tests mask position t + ks; positions at or past
    // plim (the reserved word, the live end) admit nothing
    const uint32_t *mreq = p.mask + int64_t(b) * p.mask_rows * p.W;
    const int64_t ks = p.key_start_word ? int64_t(int32_t(__ldg(mreq + p.W - 1))) : 0;
    const int64_t wlim = p.W - p.key_start_word;
    int64_t plim = 32 * wlim;
    if (p.key_ends != nullptr) plim = min(plim, int64_t(__ldg(p.key_ends + b)));
    const int64_t t_lo = int64_t(k0) * BN;
    const int64_t t_hi = min(int64_t(k1) * BN, p.T);
    const int64_t p_lo = max(t_lo + ks, int64_t(0));
    const int64_t p_hi = min(t_hi + ks, plim);

    if (tid == 0) {
#pragma unroll 1
        for (int i = 0; i < C::NS; ++i) {
            ptx::mbar_init(bar(C::B_KV_FULL + i), 1);
            ptx::mbar_init(bar(C::B_KV_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar(C::B_S_FULL + i), 1);
            ptx::mbar_init(bar(C::B_S_EMPTY + i), 4);
            ptx::mbar_init(bar(C::B_P_FULL + i), 4);
            ptx::mbar_init(bar(C::B_PV_DONE + i), 1);
        }
        ptx::mbar_init(bar(C::B_Q), 1);
        ptx::mbar_init(bar(C::B_MMA_DONE), 1);
        ptx::fence_mbar_init();
    }
    if (warp == 5) {
        ptx::tmem_alloc(ptx::smem_u32(tslot), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    for (int i = tid; i < nbw; i += kThreads) bitmap[i] = 0u;
    __syncthreads();
    const int64_t qrow0 = (int64_t(b) * p.io_S + p.io_s0 + s0) * p.H;
    if (warp == 4 && lane == 0) {
        ptx::mbar_arrive_expect_tx(bar(C::B_Q), C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
            ptx::tma_load_2d(ptx::smem_u32(smem + C::OFF_Q + c * (kRows * 128)), &qmap, 64 * c, int32_t(qrow0),
                             bar(C::B_Q));
    }

    // ---- prologue: mark the key tiles some row of the group admits.  Item
    // (row, vector c) covers mask positions [128c, 128c + 128), clipped to
    // [p_lo, p_hi); tile = (position - ks) / BN.
    if (p_hi > p_lo && gv > 0) {
        const int64_t c_first = p_lo >> 7, c_last = (p_hi - 1) >> 7;
        const int nvec = int(c_last - c_first + 1);
        const int items = gv * nvec;
#pragma unroll 1
        for (int it = tid; it < items; it += kThreads) {
            const int rt = it / nvec;
            const int64_t c = c_first + (it - rt * nvec);
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(mreq + int64_t(s0 + rt) * p.W) + c);
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
            int first = -1, last = -1;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int64_t base = c * 128 + 32 * k;
                const int64_t lo = p_lo - base, hi = p_hi - base;   // keep bits j with lo <= j < hi
                uint32_t keep = 0xffffffffu;
                if (lo > 0) keep = lo >= 32 ? 0u : keep << uint32_t(lo);
                if (hi < 32) keep &= hi <= 0 ? 0u : (0xffffffffu >> uint32_t(32 - hi));
                w[k] &= keep;
                if (w[k] != 0u) {
                    if (first < 0) first = 32 * k + __ffs(int(w[k])) - 1;
                    last = 32 * k + 31 - __clz(int(w[k]));
                }
            }
            if (first >= 0) {
                const int64_t tf = (c * 128 + first - ks) / BN, tl = (c * 128 + last - ks) / BN;
                for (int64_t t = tf; t <= tl; ++t)
                    atomicOr(&bitmap[(t - k0) >> 5], 1u << uint32_t((t - k0) & 31));
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tbase = *tslot;
    int n_act = 0;
    for (int i = 0; i < nbw; ++i) n_act += __popc(bitmap[i]);
    if (warp >= 4) {
      if constexpr (C::CPS == 2) ptx::setmaxnreg_dec<kOtherRegs>();
      if (warp == 4) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            TileIter itr(bitmap, nbw, k0);
            int n = 0;
#pragma unroll 1
            for (int t = itr.next(); t >= 0; t = itr.next(), ++n) {
                const int st = n % C::NS;
                if (n >= C::NS && !wait_bar(bar(C::B_KV_EMPTY + st), ((n / C::NS) - 1) & 1, p.err)) break;
                ptx::mbar_arrive_expect_tx(bar(C::B_KV_FULL + st), C::STAGE);
                const int32_t y = int32_t(int64_t(b) * p.T + int64_t(t) * BN);
                const uint32_t dst = ptx::smem_u32(smem + C::OFF_KV + st * C::STAGE);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    ptx::tma_load_2d(dst + c * (BN * 128), &kvmap, 64 * c, y, bar(C::B_KV_FULL + st));
            }
            // every load issued has landed before the CTA may exit
            drain_wait(bar(C::B_Q), 0);
            for (int st = 0; st < C::NS && st < n; ++st) {
                const int last = st + ((n - 1 - st) / C::NS) * C::NS;   // the stage's last load
                drain_wait(bar(C::B_KV_FULL + st), (last / C::NS) & 1);
            }
        }
        __syncwarp();
      } else if (warp == 5) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(kRows, BN, false);
            constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(kRows, D, true);
            const uint32_t qa = ptx::smem_u32(smem + C::OFF_Q);
            auto kv_addr = [&](int n) { return ptx::smem_u32(smem + C::OFF_KV + (n % C::NS) * C::STAGE); };
            auto qk = [&](int n) -> bool {
                const int sb = n % C::NB;
                if (!wait_bar(bar(C::B_KV_FULL + n % C::NS), (n / C::NS) & 1, p.err)) return false;
                if (n >= C::NB && !wait_bar(bar(C::B_S_EMPTY + sb), ((n / C::NB) - 1) & 1, p.err)) return false;
                ptx::tc_fence_after();
                const uint32_t ka = kv_addr(n);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t ad = ptx::sdesc_sw128(qa + (k / 4) * (kRows * 128) + (k % 4) * 32, 16, 1024);
                    const uint64_t bd = ptx::sdesc_sw128(ka + (k / 4) * (BN * 128) + (k % 4) * 32, 16, 1024);
                    ptx::mma_ss(tbase + C::S_COL + sb * BN, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
                }
                ptx::mma_commit(bar(C::B_S_FULL + sb));
                return true;
            };
            auto pv = [&](int m) -> bool {
                const int sb = m % C::NB;
                if (!wait_bar(bar(C::B_P_FULL + sb), (m / C::NB) & 1, p.err)) return false;
                ptx::tc_fence_after();
                const uint32_t va = kv_addr(m);
#pragma unroll
                for (int t = 0; t < BN / 16; ++t) {
                    const uint64_t bd = ptx::sdesc_sw128(va + t * 2048, BN * 128, 1024);
                    ptx::mma_ts(tbase + C::O_COL, tbase + C::P_COL + sb * (BN / 2) + t * 8, bd, idesc_pv,
                                (m > 0 || t > 0) ? 1u : 0u);
                }
                ptx::mma_commit(bar(C::B_KV_EMPTY + m % C::NS));
                ptx::mma_commit(bar(C::B_PV_DONE + sb));
                return true;
            };
            bool ok = wait_bar(bar(C::B_Q), 0, p.err);
            ptx::tc_fence_after();
#pragma unroll 1
            for (int n = 0; ok && n < n_act; ++n) {
                ok = qk(n);
                if (ok && n >= 1) ok = pv(n - 1);
            }
            if (ok && n_act > 0) ok = pv(n_act - 1);
            ptx::mma_commit(bar(C::B_MMA_DONE));   // arrives once every MMA issued above has completed
        }
        __syncwarp();
      }
    } else {
        // ------------------------------------------------------------ softmax
        if constexpr (C::CPS == 2) ptx::setmaxnreg_inc<kSoftmaxRegs>();
        const int q4 = warp;
        const int r = q4 * 32 + lane;                  // this thread's row
        const int tok = r / p.H, h = r - tok * p.H;
        const bool row_ok = r < p.G * p.H && tok < gv;
        const uint32_t *mrow = row_ok ? mreq + int64_t(s0 + tok) * p.W : nullptr;
        const uint32_t lane_base = tbase + (uint32_t(q4 * 32) << 16);
        const float sc = p.scale_log2;

        // the row's mask bits for key tile t: bit c of word k admits key
        // t * BN + 32k + c (mask position p0 + 32k + c, p0 = t * BN + ks)
        // fast path (a tile whose positions start on a multiple of BN and lie
        // inside the row's admissible range and the T keys): one aligned
        // NW-word vector load, no shifts and no clipping
        const bool aligned_ks = (ks % BN) == 0;
        auto tile_bits = [&](int t, uint32_t (&w)[NW]) {
#pragma unroll
            for (int k = 0; k < NW; ++k) w[k] = 0u;
            if (t < 0 || mrow == nullptr) return;
            const int64_t p0 = int64_t(t) * BN + ks;
            if (aligned_ks && p0 >= 0 && p0 + BN <= plim && int64_t(t + 1) * BN <= p.T) {
                if constexpr (NW == 4) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(mrow + (p0 >> 5)));
                    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
                } else {
                    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(mrow + (p0 >> 5)));
                    w[0] = v.x; w[1] = v.y;
                }
                return;
            }
            const int64_t w0 = p0 >> 5;                 // floor
            const uint32_t sh = uint32_t(p0 & 31);
            const int64_t ca = w0 & ~int64_t(3);
            const int o = int(w0 - ca);
            uint32_t x[8];
            uint32_t xa[4], xb[4];
            mask_vec(mrow, ca, p.W, wlim, xa);
            if (o + NW + (sh != 0u ? 1 : 0) > 4) mask_vec(mrow, ca + 4, p.W, wlim, xb);
            else xb[0] = xb[1] = xb[2] = xb[3] = 0u;
#pragma unroll
            for (int k = 0; k < 4; ++k) { x[k] = xa[k]; x[4 + k] = xb[k]; }
            uint32_t y[NW + 1];
#pragma unroll
            for (int k = 0; k <= NW; ++k) y[k] = o == 0 ? x[k] : o == 1 ? x[k + 1] : o == 2 ? x[k + 2] : x[k + 3];
#pragma unroll
            for (int k = 0; k < NW; ++k) w[k] = __funnelshift_r(y[k], y[k + 1], sh);
            // keys past T and positions past plim admit nothing
            const int64_t cl = min(min(int64_t(BN), p.T - int64_t(t) * BN), plim - p0);
            if (cl < BN) {
#pragma unroll
                for (int k = 0; k < NW; ++k) {
                    const int64_t n = cl - 32 * k;      // bits of word k kept
                    w[k] &= n <= 0 ? 0u : n >= 32 ? 0xffffffffu : (0xffffffffu >> uint32_t(32 - n));
                }
            }
        };

        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        TileIter itr(bitmap, nbw, k0);
        int t_cur = itr.next();
        uint32_t wc[NW];
        tile_bits(t_cur, wc);
#pragma unroll 1
        for (int n = 0; t_cur >= 0; ++n) {
            const int t_nxt = itr.next();
            uint32_t wn[NW];
            tile_bits(t_nxt, wn);                       // prefetch the next tile's words
            const int sb = n % C::NB;
            if (!wait_all(bar(C::B_S_FULL + sb), (n / C::NB) & 1, p.err)) { ok = false; break; }
            ptx::tc_fence_after();
            float s[BN];
            {
                uint32_t raw[BN / 32][32];
#pragma unroll
                for (int k = 0; k < BN / 32; ++k) ptx::tmem_ld32(lane_base + C::S_COL + sb * BN + 32 * k, raw[k]);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < BN / 32; ++k)
#pragma unroll
                    for (int j = 0; j < 32; ++j) s[32 * k + j] = __uint_as_float(raw[k][j]);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(C::B_S_EMPTY + sb));

            // masked keys become -inf (in the scaled domain for a
            // non-positive scale); row maximum over 8 chains of 3-input maxima
#pragma unroll
            for (int k = 0; k < NW; ++k) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float v = POS ? s[32 * k + j] : s[32 * k + j] * sc;
                    s[32 * k + j] = ((wc[k] >> j) & 1u) ? v : -INFINITY;
                }
            }
            float mc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                constexpr int L = BN / 8;                   // values a chain
                float a = s[L * i];
#pragma unroll
                for (int e = 1; e + 1 < L; e += 2) a = ptx::max3(a, s[L * i + e], s[L * i + e + 1]);
                mc[i] = (L % 2 == 0) ? fmaxf(a, s[L * i + L - 1]) : a;
            }
            const float mx = ptx::max3(ptx::max3(mc[0], mc[1], mc[2]), ptx::max3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
            const float mt = POS ? mx * sc : mx;       // -inf when the row admits nothing here
            // lazy rescale: a new reference maximum only when it grows by more than 2^8
            float f = 1.f;
            if (mt > m_run + kRescaleLog2) {
                if (m_run != -INFINITY) f = ex2_approx(m_run - mt);
                m_run = mt;
                l_run *= f;
            }
            if (n > 0 && __any_sync(0xffffffffu, f != 1.f)) {
                // O holds P.V of the earlier tiles: wait for the last one, scale
                if (!wait_all(bar(C::B_PV_DONE + (n - 1) % C::NB), ((n - 1) / C::NB) & 1, p.err)) { ok = false; break; }
                ptx::tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o32[32];
                    ptx::tmem_ld32(lane_base + C::O_COL + 32 * c, o32);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o32[j] = __float_as_uint(__uint_as_float(o32[j]) * f);
                    ptx::tmem_st32(lane_base + C::O_COL + 32 * c, o32);
                }
                ptx::tmem_wait_st();
            }
            // P = 2^(x - m) (masked keys: 2^-inf = 0), bf16 pairs
            const float nm = m_run == -INFINITY ? 0.f : -m_run;
            const uint64_t sc2 = ptx::f2(sc, sc), nm2 = ptx::f2(nm, nm);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};   // packed partial sums
            // P buffer sb is free once the P.V of tile n - NB is done
            if (n >= C::NB && !wait_all(bar(C::B_PV_DONE + sb), ((n / C::NB) - 1) & 1, p.err)) { ok = false; break; }
            ptx::tc_fence_after();
            // 64 keys at a time, each half stored to TMEM as soon as it is packed
#pragma unroll
            for (int k = 0; k < BN / 64; ++k) {
                uint32_t q32[32];
#pragma unroll
                for (int c2 = 0; c2 < 32; ++c2) {
                    const int c = 32 * k + c2;
                    const uint64_t xy = ptx::f2(s[2 * c], s[2 * c + 1]);
                    float z0, z1;
                    ptx::f2_split(POS ? ptx::ffma2(xy, sc2, nm2) : ptx::fadd2(xy, nm2), z0, z1);
                    const float p0 = ex2_approx(z0), p1 = ex2_approx(z1);
                    acc[c & 3] = ptx::fadd2(acc[c & 3], ptx::f2(p0, p1));
                    q32[c2] = pack_bf16(p0, p1);
                }
                ptx::tmem_st32(lane_base + C::P_COL + sb * (BN / 2) + 32 * k, q32);
            }
            float l0, l1, l2, l3;
            ptx::f2_split(ptx::fadd2(acc[0], acc[1]), l0, l1);
            ptx::f2_split(ptx::fadd2(acc[2], acc[3]), l2, l3);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(C::B_P_FULL + sb));
            l_run += (l0 + l1) + (l2 + l3);
            t_cur = t_nxt;
#pragma unroll
            for (int k = 0; k < NW; ++k) wc[k] = wn[k];
        }

        // ------------------------------------------------------------ epilogue
        // one split: o = O * f, f = 2^(m-M) / (l 2^(m-M) + 2^(sink*log2e - M)),
        // M = max(m, sink*log2e) (the sink joins the denominator once, at the
        // end); splits: O / l and the log-sum-exp m + log2(l) per row.
        ok = wait_all(bar(C::B_MMA_DONE), 0, p.err) && ok;
        ptx::tc_fence_after();
        const bool have = n_act > 0 && ok;              // O in TMEM was written
        const int64_t tg = int64_t(b) * p.S + s0 + tok; // token of the call (window row)
        if (p.ns == 1) {
            const float sink2 = row_ok ? __ldg(p.sink + h) * kLog2e : 0.f;
            float f = 0.f;
            if (m_run != -INFINITY && sink2 != INFINITY) {
                const float M = fmaxf(m_run, sink2);
                const float e = ex2_approx(m_run - M);
                f = e / (l_run * e + ex2_approx(sink2 - M));
            }
            if (isnan(sink2) || isnan(m_run) || !ok) f = NAN;
            __nv_bfloat16 *dst = p.o + ((int64_t(b) * p.io_S + p.io_s0 + s0 + tok) * p.H + h) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o32[32];
                if (have) {
                    ptx::tmem_ld32(lane_base + C::O_COL + 32 * c, o32);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o32[j] = 0u;
                }
                if (row_ok) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(o32[8 * v + 0]) * f, __uint_as_float(o32[8 * v + 1]) * f);
                        w.y = pack_bf16(__uint_as_float(o32[8 * v + 2]) * f, __uint_as_float(o32[8 * v + 3]) * f);
                        w.z = pack_bf16(__uint_as_float(o32[8 * v + 4]) * f, __uint_as_float(o32[8 * v + 5]) * f);
                        w.w = pack_bf16(__uint_as_float(o32[8 * v + 6]) * f, __uint_as_float(o32[8 * v + 7]) * f);
                        *reinterpret_cast<uint4 *>(dst + 32 * c + 8 * v) = w;
                    }
                }
            }
        } else {
            const bool live = m_run != -INFINITY;
            float f = live ? 1.f / l_run : 0.f;
            if (!ok) f = NAN;
            const int64_t wrow = (tg * p.ns + split) * p.H + h;
            float *dst = p.ws_o + wrow * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o32[32];
                if (have) {
                    ptx::tmem_ld32(lane_base + C::O_COL + 32 * c, o32);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o32[j] = 0u;
                }
                if (row_ok) {
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        *reinterpret_cast<float4 *>(dst + 32 * c + 4 * v) =
                            make_float4(__uint_as_float(o32[4 * v]) * f, __uint_as_float(o32[4 * v + 1]) * f,
                                        __uint_as_float(o32[4 * v + 2]) * f, __uint_as_float(o32[4 * v + 3]) * f);
                }
            }
            if (row_ok) p.ws_lse[wrow] = !ok ? NAN : live ? m_run + __log2f(l_run) : -INFINITY;
        }
    }

    // ---------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        drain_wait(bar(C::B_MMA_DONE), 0);   // no MMA of this CTA is still running
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

constexpr int kMaxDev = 64;

template <int D>
cudaError_t prepare(int dev) {
    static std::once_flag once[kMaxDev];
    static cudaError_t err[kMaxDev];
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        err[dev] = cudaFuncSetAttribute(masked_dense_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        Md<D>::SMEM);
        if (err[dev] == cudaSuccess)
            err[dev] = cudaFuncSetAttribute(masked_dense_kernel<D, false>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, Md<D>::SMEM);
    });
    return err[dev];
}

// A bf16 [rows][D] tensor as a 2-D map with boxes of box_rows rows x 64
// columns (128 B), 128B-swizzled; rows past the end read as zeros.
cudaError_t encode_rows_map(CUtensorMap *m, const void *base, int64_t D, int64_t rows, int box_rows) {
    const auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
    if (enc == nullptr) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(D) * 2};
    cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_md(const AttnArgs &a, cudaStream_t stream) {
    using C = Md<D>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = prepare<D>(dev);
    if (e != cudaSuccess) return e;
    MdParams p{};
    e = device_error_word(&p.err);
    if (e != cudaSuccess) return e;
    const int64_t io_S = a.io_S > 0 ? a.io_S : a.S;
    p.sink = a.sink;
    p.mask = a.mask;
    p.key_ends = a.key_ends;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.ws_o = a.ws_o;
    p.ws_lse = a.ws_lse;
    p.mask_rows = a.mask_rows;
    p.W = a.mask_words;
    p.T = a.T;
    p.key_start_word = a.key_start_word;
    p.B = int(a.B);
    p.S = int(a.S);
    p.io_S = int(io_S);
    p.io_s0 = int(a.io_s0);
    p.H = int(a.H);
    p.G = int(kRows / a.H);
    p.groups = int((a.S + p.G - 1) / p.G);
    p.nt = int((a.T + C::BN - 1) / C::BN);
    p.ns = a.num_splits;
    p.tps = (p.nt + p.ns - 1) / p.ns;
    p.scale_log2 = a.scale * kLog2e;
    if (p.tps > kMaxTiles || p.ns < 1) return cudaErrorInvalidValue;
    CUtensorMap qmap, kvmap;
    e = encode_rows_map(&qmap, a.q, D, a.B * io_S * a.H, kRows);
    if (e != cudaSuccess) return e;
    e = encode_rows_map(&kvmap, a.kv, D, a.B * a.T, C::BN);
    if (e != cudaSuccess) return e;
    const int64_t ctas = a.B * int64_t(p.groups) * p.ns;
    if (a.scale > 0.f)
        e = launch_pdl(masked_dense_kernel<D, true>, dim3(unsigned(ctas)), dim3(kThreads), C::SMEM, stream, p, qmap, kvmap);
    else
        e = launch_pdl(masked_dense_kernel<D, false>, dim3(unsigned(ctas)), dim3(kThreads), C::SMEM, stream, p, qmap, kvmap);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool masked_dense_packed(int64_t D) { return D == 64 || D == 128 || D == 256; }

int masked_dense_splits(int64_t B, int64_t S, int64_t H, int64_t D, int64_t T, int num_splits, int num_sms) {
    if (!masked_dense_packed(D) || H < 1 || H > kRows || T < 1) return 0;
    const int64_t BN = D == 128 ? 128 : 64;
    const int64_t G = kRows / H;
    const int64_t units = B * ((S + G - 1) / G);
    const int64_t nt = (T + BN - 1) / BN;
    int64_t ns = num_splits;
    if (ns <= 0) {
        ns = 1;
        if (units > 0 && units < num_sms) ns = num_sms / units;
        const int64_t cap = nt / 4 > 1 ? nt / 4 : 1;   // at least 4 key tiles a split
        if (ns > cap) ns = cap;
    }
    if (ns > nt) ns = nt;
    const int64_t ns_min = (nt + kMaxTiles - 1) / kMaxTiles;
    if (ns < ns_min) ns = ns_min;
    if (ns < 1) ns = 1;
    return ns > 64 ? 0 : int(ns);
}

cudaError_t launch_masked_dense(const AttnArgs &a, cudaStream_t stream) {
    if (a.B * a.S == 0) return cudaSuccess;
    cudaError_t e;
    switch (a.D) {
        case 64: e = launch_md<64>(a, stream); break;
        case 128: e = launch_md<128>(a, stream); break;
        case 256: e = launch_md<256>(a, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    if (a.num_splits > 1) return launch_attn_combine(a, stream);
    return cudaSuccess;
}

}  // namespace sa
