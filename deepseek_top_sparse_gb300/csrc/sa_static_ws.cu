// sa_sparse_attn_fwd_static_ws: sparse_attn for callers that cannot allocate
// device memory.
//
// The split-KV path of sa_sparse_attn_fwd needs a float32 workspace for the
// per-split partial outputs, normally supplied by the caller.  Some callers
// have no way to provide one: a plain C host program linked against this
// library without any device allocator, a serving loop whose memory is
// planned once up front and that must not call cudaMalloc on the hot path
// (cudaMalloc can block on the device and fail under memory pressure), or a
// plugin running inside a host framework that owns every allocation.  For
// them this entry point uses a workspace that lives in the library itself: a
// file-scope device array of kStaticWsBytes bytes.  Nothing is allocated by
// the call; the array is part of the loaded module, so every GPU on which
// the library is used holds it until the process exits.
//
// Set-up: the first call on each device looks up the array's device address
// with cudaGetSymbolAddress (once per device, that device current).  Make the
// first call on a device before any stream capture begins.
//
// Sharing: all calls on a device share the one array and it keeps the last
// call's contents.  Nothing needs to start at zero: every partial row the
// combine reads is written by the same call first.  Calls that overlap on
// the GPU (different streams without ordering between them) race on the
// array and produce wrong results; serialise them on one stream or with
// events.
#include <mutex>

#include "sa_internal.h"

namespace {

// 32 MiB.  With the library's own split plan (num_splits = 0) and K <= 2048
// slots (one work unit per split) a split call never runs more units than
// the GPU has CTA slots, one per SM (half of them for D = 512), so on a
// 152-SM GB300 the partials take at most 152 x 128 x 256 x 4 bytes, about
// 20 MB, for H <= 128.  Larger K forces at least ceil(K / 2048) splits per
// token whatever the batch, and an explicit num_splits can ask for up to
// 64: such plans can exceed the array, and the call then returns
// SA_ERR_WORKSPACE.
constexpr size_t kStaticWsBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 64;
void *g_ws_ptr[kMaxDevices];
cudaError_t g_ws_err[kMaxDevices];
std::once_flag g_ws_once[kMaxDevices];

}  // namespace

extern "C" sa_status sa_sparse_attn_fwd_static_ws(const void *q, const void *kv, const float *attn_sink,
                                                 const int32_t *topk_idxs, float softmax_scale, void *o,
                                                 int64_t B, int64_t S, int64_t H, int64_t D, int64_t T,
                                                 int64_t K, int num_splits, sa_stream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SA_ERR_CUDA;
    std::call_once(g_ws_once[dev], [dev] {
        void *p = nullptr;
        g_ws_err[dev] = cudaGetSymbolAddress(&p, g_static_ws);
        g_ws_ptr[dev] = p;
    });
    if (g_ws_err[dev] != cudaSuccess || g_ws_ptr[dev] == nullptr) return SA_ERR_CUDA;
    // The regular entry point validates every argument first (so an invalid
    // argument is reported as such), then compares the planned workspace with
    // the array's size.
    return sa_sparse_attn_fwd_splits(q, kv, attn_sink, topk_idxs, softmax_scale, o, B, S, H, D, T, K,
                                     num_splits, g_ws_ptr[dev], kStaticWsBytes, stream);
}
