// moe_dispatch_noalloc: the dispatch sort (stable counting sort of routing
// slots by expert) without any device allocation.
//
// Some callers cannot allocate device memory when they need this step: an
// inference server whose memory pool owns the whole device, a plugin that is
// handed a fixed budget, or a latency-critical loop where cudaMalloc's
// implicit device synchronisation is not acceptable.  For them this entry
// point keeps its scratch (the per-block expert histograms and their scan) in
// a file-scope device array that is part of the loaded library, so the call
// itself allocates nothing; the caller passes only inputs and outputs.
//
// The array is process-wide: every GPU that loads the library holds its own
// copy until the process exits, all calls on one device share it, and it keeps
// the last call's contents.  Calls whose work overlaps on the GPU (different
// streams, or different host threads) race on it and must be serialised by
// the caller.  Every scratch entry a call reads is written earlier in the same
// call, so nothing has to be cleared between calls.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "moe.h"

namespace moe {
namespace {

constexpr int kTokensPerBlock = 32;
constexpr int kThreads = 256;
constexpr int kMaxDevices = 64;

// [blocks * E] histograms, then [E + 1] tile offsets, then [E + 1] active list
__device__ __align__(256) int32_t g_dispatch_scratch[MOE_DISPATCH_NOALLOC_SCRATCH_INTS];

// Device address of the array per device, with the unique id of the context it
// was looked up in: after a device reset the library's module is loaded again in
// a new context and the array may sit elsewhere, so a changed id means a new
// lookup.
std::mutex g_setup_mutex;
int32_t *g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// The current context's unique id (driver entry points fetched once), or 0.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

__global__ void __launch_bounds__(kThreads) static_hist_kernel(const int32_t *topk_idx, int T, int k, int E,
                                                                int32_t *blk_hist, int *bad) {
    __shared__ int hist[256];
    for (int e = threadIdx.x; e < E; e += kThreads) hist[e] = 0;
    __syncthreads();
    const int tok0 = blockIdx.x * kTokensPerBlock;
    const int n = max(0, min(kTokensPerBlock, T - tok0)) * k;
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const int e = topk_idx[(size_t)tok0 * k + i];
        if (e >= 0 && e < E)
            atomicAdd(&hist[e], 1);
        else
            *bad = 1;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) blk_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

__global__ void __launch_bounds__(kThreads) static_scatter_kernel(const int32_t *topk_idx, const int32_t *blk_base,
                                                                   int T, int k, int E, int32_t *sorted_tok,
                                                                   int32_t *slot_of) {
    __shared__ int e_s[kTokensPerBlock * 16];
    const int tok0 = blockIdx.x * kTokensPerBlock;
    const int n = max(0, min(kTokensPerBlock, T - tok0)) * k;
    const size_t ent0 = (size_t)tok0 * k;
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const int e = topk_idx[ent0 + i];
        e_s[i] = (e >= 0 && e < E) ? e : -1;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const int e = e_s[i];
        int slot = -1;
        if (e >= 0) {
            int rank = 0;  // earlier slots of the same expert in (token, slot) order
            for (int q = 0; q < i; ++q) rank += (e_s[q] == e);
            slot = blk_base[(size_t)blockIdx.x * E + e] + rank;
            sorted_tok[slot] = tok0 + i / k;
        }
        slot_of[ent0 + i] = slot;
    }
}

moe_status fail(moe_status st, const char *msg) {
    ::moe_set_last_error_internal(msg);
    return st;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_dispatch_noalloc(const int32_t *topk_idx, int T, int k, int E, int32_t *expert_offs,
                                           int32_t *sorted_token, int32_t *slot, int *bad_index,
                                           moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || k < 1 || k > 16 || E < 1 || E > 256)
        return fail(MOE_ERR_INVALID_ARG, "moe_dispatch_noalloc: need T >= 0, 1 <= k <= 16, 1 <= E <= 256");
    if (!expert_offs || !bad_index || (T > 0 && (!topk_idx || !sorted_token || !slot)))
        return fail(MOE_ERR_INVALID_ARG, "moe_dispatch_noalloc: NULL pointer");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T == 0) {  // no rows: every offset 0, no bad index
        if (cudaMemsetAsync(expert_offs, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess ||
            cudaMemsetAsync(bad_index, 0, sizeof(int), s) != cudaSuccess)
            return fail(MOE_ERR_CUDA, "moe_dispatch_noalloc: cudaMemsetAsync failed");
        return MOE_OK;
    }
    const long long nb = (T + kTokensPerBlock - 1) / kTokensPerBlock;
    if (nb * E + 2ll * (E + 1) > MOE_DISPATCH_NOALLOC_SCRATCH_INTS)
        return fail(MOE_ERR_UNSUPPORTED,
                    "moe_dispatch_noalloc: ceil(T/32)*E + 2*(E+1) exceeds the static scratch of "
                    "MOE_DISPATCH_NOALLOC_SCRATCH_INTS ints");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(MOE_ERR_CUDA, "moe_dispatch_noalloc: no usable current device");
    // make the device's primary context current on this thread (allocates nothing)
    if (cudaSetDevice(dev) != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_dispatch_noalloc: cudaSetDevice failed");
    int32_t *scratch = nullptr;
    {
        // first call on this device (or in a new context after a reset): the
        // device address of the array; host code only sees a host-side stand-in
        // for the symbol.  Without a context id the address is looked up each call.
        const unsigned long long ctx = current_context_id();
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (g_scratch_addr[dev] == nullptr || ctx == 0 || g_scratch_ctx[dev] != ctx) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
            if (e != cudaSuccess || p == nullptr)
                return fail(MOE_ERR_CUDA, "moe_dispatch_noalloc: cudaGetSymbolAddress failed");
            g_scratch_addr[dev] = static_cast<int32_t *>(p);
            g_scratch_ctx[dev] = ctx;
        }
        scratch = g_scratch_addr[dev];
    }
    int32_t *blk_hist = scratch;
    int32_t *tile_offs = scratch + nb * E;
    int32_t *active = tile_offs + (E + 1);
    e = cudaMemsetAsync(bad_index, 0, sizeof(int), s);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_dispatch_noalloc: cudaMemsetAsync failed");
    static_hist_kernel<<<(unsigned)nb, kThreads, 0, s>>>(topk_idx, T, k, E, blk_hist, bad_index);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_dispatch_noalloc: launch failed");
    ScanArgs sa{blk_hist, (int)nb, E, expert_offs, tile_offs, active};
    if ((e = launch_scan(sa, s)) != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_dispatch_noalloc: launch failed");
    static_scatter_kernel<<<(unsigned)nb, kThreads, 0, s>>>(topk_idx, blk_hist, T, k, E, sorted_token, slot);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_dispatch_noalloc: launch failed");
    return MOE_OK;
}
