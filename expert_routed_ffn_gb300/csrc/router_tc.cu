// Router logits on the tensor cores (K1, first half): 128 tokens per CTA.
//
// Logits l = X Wr^T are a [T, H] x [H, E] contraction: tcgen05.mma (M = 128
// tokens, N = E rounded up to 32, K = 16) with fp32 accumulation in TMEM, A =
// bf16 X and B = the fp32 router weights held as a three-way bf16 split
// Wr = hi + mid + lo (exact for normal fp32 values), whose three products are
// accumulated into the same accumulator.  Every product of two bf16 values is
// exact in fp32, so the logits carry fp32 accuracy.  When the router weights
// are exactly bf16 the split has one part.
//
// Epilogue: one thread per token moves its E fp32 logits from TMEM to global
// memory; the routing rule itself (scores, biased top-k, weights) runs in
// topk_kernel, one warp per token, so that it spreads over T/32 CTAs.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr int kMaxStages = 8;
constexpr int kABytes = 128 * 64 * 2;
constexpr int kMiscBytes = 1024;  // barriers and the TMEM slot
constexpr int kSmemMax = 232448;
constexpr uint64_t kDrainNs = 1000000000ull;

__global__ void __launch_bounds__(kThreads, 1) router_tc_kernel(const __grid_constant__ RouterTcArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    const uint32_t stage_bytes = kABytes + p.Np * 128;
    const uint32_t s0 = smem_u32(smem);
    uint8_t *misc = smem + S * stage_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(misc);  // full[8], empty[8], tfull, drain
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    const uint32_t tfull_bar = bar0 + 8u * (2 * kMaxStages);
    const uint32_t drain_bar = bar0 + 8u * (2 * kMaxStages + 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc + 8 * (2 * kMaxStages + 2));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    trace_mark(p.trace, 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(drain_bar, 1);
        fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.mapX);
        tma_prefetch_desc(&p.mapW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    trace_mark(p.trace, 1);
    pdl_trigger();
    const uint32_t tmem_base = *tmem_slot;
    // split-K: this CTA takes k-blocks [kb0, kb0 + nkb) and writes its partial logits
    const int kb0 = blockIdx.y * p.kb_per_split;
    const int nkb = min(p.H / 64 - kb0, p.kb_per_split);
    const int units = nkb * p.parts;  // (k-block, split part) pairs, each one stage
    const int row0 = blockIdx.x * 128;
    float *logits = p.logits + (size_t)blockIdx.y * p.T * p.Np;

    if (warp == 0) {
        if (lane == 0) {
            int u = 0;
            for (; u < units; ++u) {
                const int s = u % S;
                const uint32_t ph = (u / S) & 1u;
                if (!mbar_wait(empty_bar(s), ph ^ 1u, p.wait_ns, abort_flag)) break;
                const int kb = kb0 + u / p.parts, part = u % p.parts;
                mbar_arrive_expect_tx(full_bar(s), stage_bytes);
                tma_load_2d(s0 + s * stage_bytes, &p.mapX, full_bar(s), kb * 64, row0);
                tma_load_3d(s0 + s * stage_bytes + kABytes, &p.mapW, full_bar(s), kb * 64, 0, part);
            }
            if (u < units) {
                if (p.err) atomicOr(p.err, ERR_TIMEOUT);
                *abort_flag = 1;
                for (int i = 0; i < S && i < u; ++i) {
                    const int l = u - 1 - i;
                    mbar_wait(full_bar(l % S), (l / S) & 1u, kDrainNs, nullptr);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, p.Np);
            int u = 0;
            for (; u < units; ++u) {
                const int s = u % S;
                if (!mbar_wait(full_bar(s), (u / S) & 1u, p.wait_ns, abort_flag)) break;
                tc_fence_after();
                const uint64_t ad = smem_desc_k128(s0 + s * stage_bytes);
                const uint64_t bd = smem_desc_k128(s0 + s * stage_bytes + kABytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc_mma_bf16(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc, (u | kk) != 0);
                tc_commit(empty_bar(s));
            }
            if (u == units) {
                tc_commit(tfull_bar);
            } else {
                if (p.err) atomicOr(p.err, ERR_TIMEOUT);
                *abort_flag = 1;
                if (u > 0) {
                    tc_commit(drain_bar);
                    mbar_wait(drain_bar, 0, kDrainNs, nullptr);
                }
            }
        }
    } else {
        // epilogue: TMEM lane r = token row0 + r; 32 fp32 columns per load
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const int t = row0 + r;
        const bool ready = __all_sync(0xffffffffu, mbar_wait(tfull_bar, 0, p.wait_ns, abort_flag));
        if (!ready) {
            if (lane == 0) {
                if (p.err) atomicOr(p.err, ERR_TIMEOUT);
                *abort_flag = 1;
            }
        } else {
            tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < p.Np; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tb + c0, v);
                tmem_ld_wait();
                if (t < p.T) {
                    float4 *dst = reinterpret_cast<float4 *>(logits + (size_t)t * p.Np + c0);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                             __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    trace_exit(p.trace);
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// L2 prefetch of byte ranges (a hint; nothing is written).  Runs on a side
// stream next to the routing kernels: a CTA cannot retire before its bulk
// prefetches complete, so they must stay off the forward's dependency chain.
__global__ void __launch_bounds__(32) l2_prefetch_kernel(const PrefetchArgs p) {
    constexpr unsigned long long kChunk = 128 * 1024;
    const unsigned long long stride = (unsigned long long)gridDim.x * 32 * kChunk;
    for (int r = 0; r < 2; ++r) {
        const unsigned long long n = p.bytes[r];
        const char *base = static_cast<const char *>(p.ptr[r]);
        for (unsigned long long c = ((unsigned long long)blockIdx.x * 32 + threadIdx.x) * kChunk; c < n; c += stride) {
            const unsigned bytes = (unsigned)(n - c < kChunk ? n - c : kChunk);
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + c), "r"(bytes) : "memory");
        }
    }
}

// fp32 router weights -> three bf16 parts hi, mid, lo with hi + mid + lo == w
// (each part rounds the remainder left by the previous ones); flags bit 0: some
// weight needs mid, bit 1: some weight needs lo.
__global__ void split_router_kernel(const float *wr, size_t n, bf16 *parts, int *flags) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float w = wr[i];
        const bf16 hi = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(hi);
        const bf16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);
        const bf16 lo = __float2bfloat16_rn(r2);
        parts[i] = hi;
        parts[n + i] = mid;
        parts[2 * n + i] = lo;
        if (r1 != 0.f) atomicOr(flags, 1);
        if (r2 != 0.f) atomicOr(flags, 2);
    }
}

}  // namespace

RouterTcPlan plan_router_tc(int E, int parts) {
    RouterTcPlan pl;
    pl.Np = (E + 31) / 32 * 32;
    int cols = 32;
    while (cols < pl.Np) cols <<= 1;
    pl.tmem_cols = cols;
    const int stage = kABytes + pl.Np * 128;
    pl.stages = (kSmemMax - 1024 - kMiscBytes) / stage;
    if (pl.stages > kMaxStages) pl.stages = kMaxStages;
    pl.smem = pl.stages * stage + 1024 + kMiscBytes;
    pl.parts = parts;
    return pl;
}

cudaError_t launch_l2_prefetch(const PrefetchArgs &a, cudaStream_t s) {
    // runs beside the expert GEMM's CTAs: keep the SM's shared memory available to them
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(l2_prefetch_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    });
    l2_prefetch_kernel<<<64, 32, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_split_router(const float *wr, int E, int H, bf16 *parts, int *flags, cudaStream_t s) {
    const size_t n = (size_t)E * H;
    split_router_kernel<<<(unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0, s>>>(wr, n, parts, flags);
    return cudaGetLastError();
}

cudaError_t launch_router_tc(const RouterTcArgs &a, int smem, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    });
    const int nk = a.H / 64;
    const unsigned splits = (unsigned)((nk + a.kb_per_split - 1) / a.kb_per_split);
    return launch_pdl(router_tc_kernel, dim3((a.T + 127) / 128, splits), dim3(kThreads), (size_t)smem, s, a);
}

}  // namespace moe
