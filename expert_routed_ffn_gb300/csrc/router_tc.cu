// Router (K1) on the tensor cores, with the routing rule in the same launch.
//
// Logits l = X Wr^T are a [T, H] x [H, E] contraction: tcgen05.mma (M = 128
// tokens, N = E rounded up to 32, K = 16) with fp32 accumulation in TMEM, A =
// bf16 X and B = the fp32 router weights held as a three-way bf16 split
// Wr = hi + mid + lo (exact for normal fp32 values), whose three products are
// accumulated into the same accumulator.  Every product of two bf16 values is
// exact in fp32, so the logits carry fp32 accuracy.  When the router weights
// are exactly bf16 the split has one part.
//
// The H reduction is split over the S CTAs (1, 2, 4 or 8) of a thread-block
// cluster: CTA s of the cluster accumulates k-blocks [s*kb, (s+1)*kb) of the
// m-tile's 128 tokens.  Once every main loop is done (cluster barrier), each
// CTA stores the partial logits of token row r straight into the shared memory
// of the CTA that routes it (rank r / (128 / S)), and after a second cluster
// barrier each CTA adds the S partials of its 128 / S tokens from its own
// shared memory, in cluster rank order.  The routing rule (routing.cuh) runs
// on LPT lanes per token, lane `sub` holding experts 8*sub .. 8*sub + 7; each
// CTA writes the expert histogram of its tokens for the dispatch.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "routing.cuh"

namespace moe {
namespace {

constexpr int kThreads = 512;    // warp 0 TMA, warp 1 MMA, warps 2-5 TMEM epilogue; all route
constexpr int kMaxStages = 8;
constexpr int kABytes = 128 * 64 * 2;
constexpr int kMiscBytes = 1024;  // barriers and the TMEM slot
constexpr int kSmemMax = 232448;                   // per CTA, static + dynamic
constexpr int kDynSmemMax = kSmemMax - 256 * 4;    // less the static expert histogram
constexpr uint64_t kDrainNs = 1000000000ull;

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// address of the same shared-memory location in cluster CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32x4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// bulk copy of `bytes` from this CTA's shared memory to a cluster CTA's, completing
// on that CTA's mbarrier (both addresses mapped with map_to_rank)
__device__ __forceinline__ void bulk_to_cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "r"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int LPT>
__global__ void __launch_bounds__(kThreads, 1) router_tc_kernel(const __grid_constant__ RouterTcArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    __shared__ int hist[256];
    const int S = p.stages;
    const uint32_t b_bytes = (uint32_t)p.Np * 128;  // one weight part, Np rows x 64
    const uint32_t stage_bytes = kABytes + p.parts * b_bytes;
    const uint32_t s0 = smem_u32(smem);
    uint8_t *misc = smem + S * stage_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(misc);  // full[8], empty[8], tfull, drain, recv
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    const uint32_t tfull_bar = bar0 + 8u * (2 * kMaxStages);
    const uint32_t drain_bar = bar0 + 8u * (2 * kMaxStages + 1);
    const uint32_t recv_bar = bar0 + 8u * (2 * kMaxStages + 2);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc + 8 * (2 * kMaxStages + 3));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned long long *const stats = p.stats;
    trace_mark(p.trace, 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(drain_bar, 1);
        mbar_init(recv_bar, 1);
        fence_mbar_init();
        *abort_flag = 0;
    }
    for (int e = threadIdx.x; e < p.E; e += kThreads) hist[e] = 0;
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
    const uint64_t t_ready = stats ? global_timer_ns() : 0;
    const uint32_t tmem_base = *tmem_slot;
    // split-K: this CTA takes k-blocks [kb0, kb0 + nkb), each one stage with all weight parts
    const int nk = p.H / 64;
    const int kb0 = blockIdx.y * p.kb_per_split;
    const int nkb = max(0, min(nk - kb0, p.kb_per_split));
    const int row0 = blockIdx.x * 128;
    // receive buffer of the partial logits [128][Np + 4] fp32 (row sp * TT + i: token i of
    // this CTA's block from cluster rank sp), over the stage buffers once the main loops are done
    float *recv = reinterpret_cast<float *>(smem);
    const int ldp = p.Np + 4;

    if (warp == 0) {
        if (lane == 0) {
            int u = 0;
            for (; u < nkb; ++u) {
                const int s = u % S;
                const uint32_t ph = (u / S) & 1u;
                if (!mbar_wait(empty_bar(s), ph ^ 1u, p.wait_ns, abort_flag)) break;
                const int kb = kb0 + u;
                const uint32_t st = s0 + s * stage_bytes;
                mbar_arrive_expect_tx(full_bar(s), stage_bytes);
                tma_load_2d(st, &p.mapX, full_bar(s), kb * 64, row0);
                for (int q = 0; q < p.parts; ++q)
                    tma_load_3d(st + kABytes + q * b_bytes, &p.mapW, full_bar(s), kb * 64, 0, q);
            }
            if (u < nkb) {
                if (p.err) atomicOr(p.err, ERR_TIMEOUT);
                *abort_flag = 1;
                for (int i = 0; i < S && i < u; ++i) {
                    const int l = u - 1 - i;
                    mbar_wait(full_bar(l % S), (l / S) & 1u, kDrainNs, nullptr);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && nkb > 0) {
            const uint32_t idesc = idesc_bf16_f32(128, p.Np);
            int u = 0;
            for (; u < nkb; ++u) {
                const int s = u % S;
                if (!mbar_wait(full_bar(s), (u / S) & 1u, p.wait_ns, abort_flag)) break;
                tc_fence_after();
                const uint32_t st = s0 + s * stage_bytes;
                const uint64_t ad = smem_desc_k128(st);
                for (int q = 0; q < p.parts; ++q) {
                    const uint64_t bd = smem_desc_k128(st + kABytes + q * b_bytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc, (u | q | kk) != 0);
                }
                tc_commit(empty_bar(s));
            }
            if (u == nkb) {
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
    } else if (warp < 6 && nkb > 0) {
        // epilogue warps: wait until this CTA's accumulator is complete
        const bool ready = __all_sync(0xffffffffu, mbar_wait(tfull_bar, 0, p.wait_ns, abort_flag));
        if (!ready && lane == 0) {
            if (p.err) atomicOr(p.err, ERR_TIMEOUT);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    const uint64_t t_partials = stats ? global_timer_ns() : 0;
    // Exchange: TMEM lane r (token row0 + r) goes to the CTA that routes it, rank
    // r / TT, as row (my rank) * TT + r % TT of its receive buffer [S * TT][Np + 4].
    const int nsplit = p.splits, rank = (int)cluster_rank(), TT = 128 / nsplit;
    const uint32_t recv_addr = smem_u32(recv);
    const uint32_t row_bytes = (uint32_t)ldp * 4u;
    uint64_t t_cluster = 0;
    if (p.staged_push != 0 || nsplit == 1) {
        // Rows staged in this CTA's shared memory (stage buffers, after the receive
        // buffer), then one bulk copy per destination CTA completing on its receive
        // barrier: the cluster barrier only has to cover "every main loop is done".
        cluster_arrive();
        float *stage_rows = nsplit == 1 ? recv : recv + 128 * ldp;  // one CTA: rows stay in place
        if (threadIdx.x == 0 && nsplit > 1) mbar_arrive_expect_tx(recv_bar, 128u * row_bytes);
        if (warp >= 2 && warp < 6) {
            const int q = warp & 3;
            const int r = q * 32 + lane;
            float *dst = stage_rows + (size_t)r * ldp;
            if (nkb == 0 || *abort_flag != 0) {  // no k-blocks for this CTA (or a failed main loop): zeros
                for (int c = 0; c < p.Np; c += 4) *reinterpret_cast<float4 *>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                tc_fence_after();
                const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
                for (int c0 = 0; c0 < p.Np; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tb + c0, v);
                    tmem_ld_wait();
                    float4 *d4 = reinterpret_cast<float4 *>(dst + c0);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                            __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                }
            }
        }
        __syncthreads();
        cluster_wait();  // every CTA's stage buffers may now receive
        t_cluster = stats ? global_timer_ns() : 0;
        if (nsplit > 1) {
            // every CTA sends all its rows whatever happened before (zeros after a
            // failure), so each receive completes; the wait ignores the abort flag
            // and has its own bound, and nothing leaves while copies are in flight
            if (threadIdx.x == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // staged rows -> bulk-copy reads
                const uint32_t src0 = smem_u32(stage_rows), bytes = (uint32_t)TT * row_bytes;
                for (int d = 0; d < nsplit; ++d)
                    bulk_to_cluster(map_to_rank(recv_addr, (uint32_t)d) + (uint32_t)(rank * TT) * row_bytes,
                                    src0 + (uint32_t)(d * TT) * row_bytes, bytes, map_to_rank(recv_bar, (uint32_t)d));
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
            const bool got = __all_sync(0xffffffffu, mbar_wait(recv_bar, 0, kDrainNs, nullptr));
            if (!got && lane == 0 && p.err) atomicOr(p.err, ERR_TIMEOUT);
            if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        }
    } else {
        // no room for a staging copy: each epilogue thread stores its row into the
        // destination directly, and a second cluster barrier publishes the stores
        cluster_sync_all();  // every CTA's main loop is done: its stage buffers may receive
        t_cluster = stats ? global_timer_ns() : 0;
        if (warp >= 2 && warp < 6 && *abort_flag == 0) {
            const int q = warp & 3;
            const int r = q * 32 + lane;
            const uint32_t dst_row = map_to_rank(recv_addr, (uint32_t)(r / TT)) + (uint32_t)(rank * TT + r % TT) * row_bytes;
            if (nkb == 0) {
                for (int c = 0; c < p.Np; c += 4) st_cluster_f32x4(dst_row + 4u * c, make_float4(0.f, 0.f, 0.f, 0.f));
            } else {
                tc_fence_after();
                const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
                for (int c0 = 0; c0 < p.Np; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tb + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        st_cluster_f32x4(dst_row + 4u * (c0 + 4 * i),
                                         make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                     __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
                }
            }
        }
        cluster_sync_all();  // all partials of this CTA's tokens have arrived
    }
    const uint64_t t_pushed = stats ? global_timer_ns() : 0;
    uint64_t t_summed = t_pushed;

    // routing of tokens [rank * TT, (rank + 1) * TT) of the m-tile, LPT lanes per token
    constexpr int kGroups = kThreads / LPT;
    const int sub = threadIdx.x & (LPT - 1), grp = threadIdx.x / LPT;
    for (int base = 0; base < TT; base += kGroups) {
        const int tl = base + grp;
        const int t = row0 + rank * TT + tl;
        const bool valid = tl < TT && t < p.T;
        // a warp whose groups hold no token of this block skips the rule (warp-uniform)
        const int warp_t0 = row0 + rank * TT + base + warp * (32 / LPT);
        if (base + warp * (32 / LPT) >= TT || warp_t0 >= p.T) continue;
        float lg[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) lg[j] = 0.f;
        if (valid && 8 * sub < p.Np) {
            // the partials of the cluster's CTAs, added in rank order
            for (int sp = 0; sp < nsplit; ++sp) {
                const float4 *src = reinterpret_cast<const float4 *>(recv + (size_t)(sp * TT + tl) * ldp + 8 * sub);
                const float4 a = src[0], b = src[1];
                lg[0] += a.x; lg[1] += a.y; lg[2] += a.z; lg[3] += a.w;
                lg[4] += b.x; lg[5] += b.y; lg[6] += b.z; lg[7] += b.w;
            }
        }
        if (stats && threadIdx.x == 0 && base == 0) t_summed = global_timer_ns();  // thread 0's sums are in
        route_token_group<LPT, true>(lg, sub, valid, t, p.E, p.k, p.bias, p.score_func, p.route_norm,
                                     p.route_scale, p.topk_idx, p.topk_w, p.blk_hist ? hist : nullptr);
    }
    __syncthreads();
    const uint64_t t_routed = stats ? global_timer_ns() : 0;
    const int b = blockIdx.x * nsplit + rank;  // token block of TT tokens
    if (p.blk_hist != nullptr && b * TT < p.T)
        for (int e = threadIdx.x; e < p.E; e += kThreads)
            p.blk_hist[(size_t)b * p.hb + (size_t)e * p.he] = hist[e];
    __syncthreads();
    trace_exit(p.trace);
    if (stats && threadIdx.x == 0) {
        const uint64_t t_end = global_timer_ns();
        atomicAdd(stats + 0, (unsigned long long)(t_partials - t_ready));
        atomicAdd(stats + 1, (unsigned long long)(t_cluster - t_partials));
        atomicAdd(stats + 2, (unsigned long long)(t_pushed - t_cluster));
        atomicAdd(stats + 3, (unsigned long long)(t_routed - t_pushed));
        atomicAdd(stats + 4, (unsigned long long)(t_end - t_routed));
        atomicAdd(stats + 5, 1ull);
        atomicAdd(stats + 6, (unsigned long long)(t_summed - t_pushed));
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// L2 prefetch of byte ranges (a hint; nothing is written).  Runs on a side
// stream next to the routing kernels: a CTA cannot retire before its bulk
// prefetches complete, so they must stay off the forward's dependency chain.
// An SM's bulk-copy engine moves on the order of 100-200 GB/s, so the ranges are
// cut into one contiguous share per CTA over a grid of one CTA per SM, each
// share issued by the warp's lanes in 16-byte-aligned pieces.
__global__ void __launch_bounds__(32) l2_prefetch_kernel(const PrefetchArgs p) {
    const unsigned long long total = p.bytes[0] + p.bytes[1];
    const unsigned long long share = (total / gridDim.x + 32 * 16 - 1) / (32 * 16) * (32 * 16);
    const unsigned long long piece = share / 32;
    unsigned long long c = (unsigned long long)blockIdx.x * share + threadIdx.x * piece;
    unsigned long long left = piece;
    for (int r = 0; r < 2 && left > 0; ++r) {
        const unsigned long long n = p.bytes[r];
        if (c >= n) {
            c -= n;
            continue;
        }
        const unsigned long long len = n - c < left ? n - c : left;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const char *>(p.ptr[r]) + c),
                     "r"((unsigned)len)
                     : "memory");
        left -= len;
        c = 0;
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
    const int stage = kABytes + parts * pl.Np * 128;
    pl.stages = (kDynSmemMax - 1024 - kMiscBytes) / stage;
    if (pl.stages > kMaxStages) pl.stages = kMaxStages;
    // the partial logits [128][Np + 4] fp32 reuse the stage buffers
    const int part_bytes = 128 * (pl.Np + 4) * 4;
    if (pl.stages * stage < part_bytes) pl.stages = (part_bytes + stage - 1) / stage;
    pl.smem = pl.stages * stage + 1024 + kMiscBytes;
    pl.parts = parts;
    pl.staged_push = pl.stages * stage >= 2 * part_bytes ? 1 : 0;
    return pl;
}

cudaError_t launch_l2_prefetch(const PrefetchArgs &a, int grid, cudaStream_t s) {
    // runs beside the expert GEMM's CTAs: keep the SM's shared memory available to them
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(l2_prefetch_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    });
    if ((a.bytes[0] | a.bytes[1]) % 16 != 0 || grid < 1) return cudaErrorInvalidValue;
    // a piece must fit the instruction's 32-bit size
    if ((a.bytes[0] + a.bytes[1]) / (unsigned long long)grid / 32 >= (1ull << 31)) return cudaErrorInvalidValue;
    l2_prefetch_kernel<<<grid, 32, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_split_router(const float *wr, int E, int H, bf16 *parts, int *flags, cudaStream_t s) {
    const size_t n = (size_t)E * H;
    split_router_kernel<<<(unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0, s>>>(wr, n, parts, flags);
    return cudaGetLastError();
}

static int router_lpt(int E) {
    int l = 2;
    while (l * 8 < E) l <<= 1;
    return l;
}

cudaError_t launch_router_tc(const RouterTcArgs &a, int smem, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(router_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmemMax);
        cudaFuncSetAttribute(router_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmemMax);
        cudaFuncSetAttribute(router_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmemMax);
        cudaFuncSetAttribute(router_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmemMax);
        cudaFuncSetAttribute(router_tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmemMax);
    });
    if (smem > kDynSmemMax || a.splits < 1 || a.splits > kMaxRouterSplits || (a.splits & (a.splits - 1)) != 0)
        return cudaErrorInvalidValue;
    const dim3 grid((a.T + 127) / 128, a.splits), block(kThreads);
    switch (router_lpt(a.E)) {
    case 2: return launch_pdl_cluster(router_tc_kernel<2>, grid, block, (size_t)smem, s, dim3(1, a.splits, 1), a);
    case 4: return launch_pdl_cluster(router_tc_kernel<4>, grid, block, (size_t)smem, s, dim3(1, a.splits, 1), a);
    case 8: return launch_pdl_cluster(router_tc_kernel<8>, grid, block, (size_t)smem, s, dim3(1, a.splits, 1), a);
    case 16: return launch_pdl_cluster(router_tc_kernel<16>, grid, block, (size_t)smem, s, dim3(1, a.splits, 1), a);
    default: return launch_pdl_cluster(router_tc_kernel<32>, grid, block, (size_t)smem, s, dim3(1, a.splits, 1), a);
    }
}

}  // namespace moe
