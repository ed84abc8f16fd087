// Router (K1), dispatch sort (K2) and combine (K7) of the token-choice MoE block.
//
// Router: per token, fp32 logits l_e = x . Wr[e], scores s = sigmoid(l) (or
// softmax over e), the k largest s_e + b_e (b: expert_bias, for the choice
// only; equal values go to the lower expert index), weights gathered from the
// unbiased s, renormalised when route_norm is set, then times route_scale.
// (Arcee AFMoE issue, "Routing detail"; HF AFMoE docs, "expert routing".)
//
// Dispatch: a stable counting sort of the T*k routing slots by expert, so that
// each expert's rows are contiguous in (token, slot) order; deterministic, no
// global atomics.  The sorted rows of X are gathered into one bf16 buffer.
//
// Combine: Y[t] = sum_j w[t,j] * y_{idx[t,j]}(x_t) + y_shared(x_t), summed in
// fp32 in a fixed order (slots j = 0..k-1, then the shared expert) by reading
// the per-slot expert outputs back: no atomics.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "routing.cuh"

namespace moe {
namespace {

constexpr int kRouterThreads = 256;
constexpr int kHC = 64;        // H columns per shared-memory chunk
constexpr int kPad = kHC + 4;  // padded row length in floats

__device__ __forceinline__ void load8_as_f32(const void *X, int x_f32, size_t off, float (&v)[8]) {
    if (x_f32) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(X) + off));
        const float4 b =
            __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(X) + off + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const uint4 r = __ldg(reinterpret_cast<const uint4 *>(static_cast<const bf16 *>(X) + off));
        v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x); v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
        v[4] = bf16_lo(r.z); v[5] = bf16_hi(r.z); v[6] = bf16_lo(r.w); v[7] = bf16_hi(r.w);
    }
}

// One CTA = TT tokens.  Warp w owns tokens [w*TT/8, (w+1)*TT/8); lane l owns
// experts l, l+32, ... so each warp ends with its tokens' logits in registers.
template <int TT>
__global__ void __launch_bounds__(kRouterThreads) router_kernel(const RouterArgs a) {
    constexpr int TPW = TT / 8;  // tokens per warp
    extern __shared__ float sm[];
    float *xs = sm;                   // [TT][kPad]
    float *ws = sm + TT * kPad;       // [E][kPad]
    int *hist = reinterpret_cast<int *>(ws + a.E * kPad);  // [E]

    const int E = a.E, H = a.H, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * TT;
    trace_mark(a.trace, 0);
    pdl_wait();
    trace_mark(a.trace, 1);
    pdl_trigger();
    for (int e = tid; e < E; e += kRouterThreads) hist[e] = 0;

    float acc[TPW][8];
#pragma unroll
    for (int i = 0; i < TPW; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    for (int h0 = 0; h0 < H; h0 += kHC) {
        for (int f = tid; f < TT * (kHC / 8); f += kRouterThreads) {
            const int r = f / (kHC / 8), c = (f % (kHC / 8)) * 8, t = t0 + r;
            float v[8];
            if (t < a.T) {
                load8_as_f32(a.X, a.x_f32, (size_t)t * H + h0 + c, v);
                if (a.x_bf16 != nullptr) {
                    uint4 o;
                    o.x = pack_bf16x2(v[0], v[1]); o.y = pack_bf16x2(v[2], v[3]);
                    o.z = pack_bf16x2(v[4], v[5]); o.w = pack_bf16x2(v[6], v[7]);
                    *reinterpret_cast<uint4 *>(a.x_bf16 + (size_t)t * H + h0 + c) = o;
                }
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = 0.f;
            }
            float4 *dst = reinterpret_cast<float4 *>(xs + r * kPad + c);
            dst[0] = make_float4(v[0], v[1], v[2], v[3]);
            dst[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
        for (int f = tid; f < E * (kHC / 4); f += kRouterThreads) {
            const int e = f / (kHC / 4), c = (f % (kHC / 4)) * 4;
            *reinterpret_cast<float4 *>(ws + e * kPad + c) =
                __ldg(reinterpret_cast<const float4 *>(a.Wr + (size_t)e * H + h0 + c));
        }
        __syncthreads();
#pragma unroll 2
        for (int c = 0; c < kHC; c += 4) {
            float4 xv[TPW];
#pragma unroll
            for (int i = 0; i < TPW; ++i)
                xv[i] = *reinterpret_cast<const float4 *>(xs + (warp * TPW + i) * kPad + c);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = lane + 32 * j;
                if (e < E) {
                    const float4 wv = *reinterpret_cast<const float4 *>(ws + e * kPad + c);
#pragma unroll
                    for (int i = 0; i < TPW; ++i) {
                        acc[i][j] = fmaf(xv[i].x, wv.x, acc[i][j]);
                        acc[i][j] = fmaf(xv[i].y, wv.y, acc[i][j]);
                        acc[i][j] = fmaf(xv[i].z, wv.z, acc[i][j]);
                        acc[i][j] = fmaf(xv[i].w, wv.w, acc[i][j]);
                    }
                }
            }
        }
        __syncthreads();
    }

    // ---- scores, biased top-k, weights: one warp per token, registers only
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
        const int t = t0 + warp * TPW + i;
        if (t >= a.T) break;  // warp-uniform
        route_token_group<32>(acc[i], lane, true, t, a.E, a.k, a.bias, a.score_func, a.route_norm,
                              a.route_scale, a.topk_idx, a.topk_w, a.blk_hist ? hist : nullptr);
    }
    if (a.blk_hist != nullptr) {
        __syncthreads();
        for (int e = tid; e < E; e += kRouterThreads)
            a.blk_hist[(size_t)blockIdx.x * a.hb + (size_t)e * a.he] = hist[e];
    }
    __syncthreads();
    trace_exit(a.trace);
}

// Dispatch scan over block histograms, by one CTA of 1024 threads.  Per expert
// (one warp each): total over blocks; one warp scans the totals over experts
// (offs, tile_offs, active); then per expert the exclusive scan over blocks,
// offset by the expert's first row, replaces the block counts in place.
constexpr int kScanThreads = 1024;

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

__device__ void dispatch_scan_block(int32_t *blk_hist, int nb, int E, int hb, int he, int tile_m,
                                    int32_t *offs, int32_t *tile_offs, int32_t *active) {
    __shared__ int cnt[256];
    __shared__ int base[256];
    if (hb == 0 && he == 0) {
        hb = E;
        he = 1;
    }
    if (tile_m <= 0) tile_m = kGemmBM;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int kWarps = blockDim.x / 32;
    for (int e = warp; e < E; e += kWarps) {
        int s = 0;
        for (int b = lane; b < nb; b += 32) s += __ldcg(blk_hist + (size_t)b * hb + (size_t)e * he);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) cnt[e] = s;
    }
    __syncthreads();
    if (warp == 0) {
        int run = 0, trun = 0, nact = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int c = e < E ? cnt[e] : 0;
            const int tl = (c + tile_m - 1) / tile_m;
            const int inc = warp_incl_scan(c, lane), tinc = warp_incl_scan(tl, lane);
            const unsigned act = __ballot_sync(0xffffffffu, c > 0);
            if (e < E) {
                base[e] = run + inc - c;
                offs[e] = run + inc - c;
                tile_offs[e] = trun + tinc - tl;
                if (c > 0) active[nact + __popc(act & ((1u << lane) - 1u))] = e;
            }
            run += __shfl_sync(0xffffffffu, inc, 31);
            trun += __shfl_sync(0xffffffffu, tinc, 31);
            nact += __popc(act);
        }
        if (lane == 0) {
            offs[E] = run;
            tile_offs[E] = trun;
            active[E] = nact;
        }
    }
    __syncthreads();
    for (int e = warp; e < E; e += kWarps) {
        int carry = base[e];
        for (int b0 = 0; b0 < nb; b0 += 32) {
            const int b = b0 + lane;
            const int v = b < nb ? __ldcg(blk_hist + (size_t)b * hb + (size_t)e * he) : 0;
            const int inc = warp_incl_scan(v, lane);
            if (b < nb) blk_hist[(size_t)b * hb + (size_t)e * he] = carry + inc - v;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
    }
}

size_t router_smem(int TT, int E) { return (size_t)(TT + E) * kPad * 4 + (size_t)E * 4; }

// ------------------------------------------------------------------- scan

__global__ void __launch_bounds__(kScanThreads) scan_kernel(const ScanArgs a) {
    pdl_wait();
    pdl_trigger();
    dispatch_scan_block(a.blk_hist, a.nb, a.E, a.hb, a.he, a.tile_m, a.offs, a.tile_offs, a.active);
}

// ---------------------------------------------------------------- scatter

constexpr int kScatterThreads = 256;
constexpr int kMaxTT = 128;

// grid (token blocks, gather_split).  Every CTA first derives, from the block
// histograms, the expert offsets (offs[e] = rows of experts < e) and its own
// block's first row per expert (offs[e] + rows of expert e in earlier blocks):
// independent loads and shared-memory sums, no serial pass; CTA (0, 0) also
// writes offs, tile_offs (ceil(count / tile_m) prefix) and the active-expert
// list.  Then, per expert, the bitmask of the block's tokens that chose it
// gives the rank of slot (t, j) among its expert's rows in the block (a
// token's k experts are distinct; a repeat is reported and dropped).  CTA
// y = 0 writes the index arrays; the CTAs of a block share the copy of X rows.
__global__ void __launch_bounds__(kScatterThreads) scatter_kernel(const ScatterArgs a) {
    __shared__ uint32_t masks[256][kMaxTT / 32];
    __shared__ int e_s[kMaxTT * 16];
    __shared__ int slot_s[kMaxTT * 16];
    __shared__ int cnt[256], pre[256], base[256];
    const int TT = a.tokens_per_block, k = a.k, E = a.E, H = a.H;
    const int hb = (a.hb | a.he) ? a.hb : E, he = (a.hb | a.he) ? a.he : 1;
    const int words = (TT + 31) / 32;
    const int tok0 = blockIdx.x * TT;
    const int nbk = gridDim.x, b = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int e = threadIdx.x; e < E; e += kScatterThreads) cnt[e] = pre[e] = 0;
    for (int i = threadIdx.x; i < E * words; i += kScatterThreads) masks[i / words][i % words] = 0;
    trace_mark(a.trace, 0);
    pdl_wait();
    trace_mark(a.trace, 1);
    if (a.tok_done != nullptr && blockIdx.y == 0)  // this block's per-token counters of the combine
        for (int i = threadIdx.x; i < TT && tok0 + i < a.T; i += kScatterThreads) a.tok_done[tok0 + i] = 0;
    // the expert GEMM is launched only when every CTA has reached the end of its
    // gather (launch_dependents below): launched earlier, its one-per-SM CTAs
    // would take the shared memory that this grid's later waves need
    __syncthreads();
    {
        // cnt[e] = rows of expert e, pre[e] = its rows in the blocks before this one:
        // G threads per expert (a power of two dividing 32) sum strided blocks, eight
        // loads in flight each, then a shuffle reduction.  No shared-memory atomics
        // (with a few experts and many blocks they serialise on one address).
        int G = 1;
        while (G * 2 * E <= kScatterThreads && G < 32) G *= 2;
        const int e = threadIdx.x / G, g = threadIdx.x % G;
        int c = 0, pr = 0;
        if (e < E) {
            constexpr int kU = 8;
            for (int b0 = g; b0 < nbk; b0 += kU * G) {
                int v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int bb = b0 + u * G;
                    v[u] = bb < nbk ? __ldg(a.blk_hist + (size_t)bb * hb + (size_t)e * he) : 0;
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    c += v[u];
                    if (b0 + u * G < b) pr += v[u];
                }
            }
        }
        for (int o = G / 2; o > 0; o >>= 1) {
            c += __shfl_xor_sync(0xffffffffu, c, o);
            pr += __shfl_xor_sync(0xffffffffu, pr, o);
        }
        if (e < E && g == 0) {
            cnt[e] = c;
            pre[e] = pr;
        }
    }
    __syncthreads();
    if (warp == 0) {
        const int tile_m = a.tile_m > 0 ? a.tile_m : kGemmBM;
        const bool writer = blockIdx.x == 0 && blockIdx.y == 0;
        int run = 0, trun = 0, nact = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int c = e < E ? cnt[e] : 0;
            const int tl = (c + tile_m - 1) / tile_m;
            const int inc = warp_incl_scan(c, lane), tinc = warp_incl_scan(tl, lane);
            const unsigned act = __ballot_sync(0xffffffffu, c > 0);
            if (e < E) {
                base[e] = run + inc - c + pre[e];
                if (writer) {
                    a.offs[e] = run + inc - c;
                    a.tile_offs[e] = trun + tinc - tl;
                    if (c > 0) a.active[nact + __popc(act & ((1u << lane) - 1u))] = e;
                }
            }
            run += __shfl_sync(0xffffffffu, inc, 31);
            trun += __shfl_sync(0xffffffffu, tinc, 31);
            nact += __popc(act);
        }
        if (writer && lane == 0) {
            a.offs[E] = run;
            a.tile_offs[E] = trun;
            a.active[E] = nact;
        }
        if (writer && a.tile_counters != nullptr && lane < 2) a.tile_counters[lane] = 0;
        if (writer && a.ready != nullptr) {
            for (int i = lane; i < trun * a.ready_per_tile; i += 32) a.ready[i] = 0;
            for (int i = lane; i < a.ready_shared_count; i += 32) a.ready[a.ready_shared_base + i] = 0;
        }
    }
    const int n = max(0, min(TT, a.T - tok0)) * k;
    const size_t ent0 = (size_t)tok0 * k;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kScatterThreads) {
        int e = a.topk_idx[ent0 + i];
        if (e < 0 || e >= E) {
            if (blockIdx.y == 0) atomicOr(a.err, ERR_BOUNDS);
            e = -1;
        } else {
            const int tl = i / k;
            const uint32_t bit = 1u << (tl & 31);
            if (atomicOr(&masks[e][tl >> 5], bit) & bit) {
                if (blockIdx.y == 0) atomicOr(a.err, ERR_BOUNDS);
                e = -1;
            }
        }
        e_s[i] = e;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kScatterThreads) {
        const int e = e_s[i];
        int slot = -1;
        if (e >= 0) {
            const int tl = i / k;
            int rank = __popc(masks[e][tl >> 5] & ((1u << (tl & 31)) - 1u));
            for (int w = 0; w < (tl >> 5); ++w) rank += __popc(masks[e][w]);
            slot = base[e] + rank;
            if (blockIdx.y == 0) a.sorted_tok[slot] = tok0 + tl;
        }
        if (blockIdx.y == 0) a.slot_of[ent0 + i] = slot;
        slot_s[i] = slot;
    }
    __syncthreads();
    // row copy in units of (row, batch of 32 * kG 16-byte chunks), dealt round-robin to
    // the block's warps so that every warp copies the same number of bytes (a warp per
    // row left some warps a third more rows when a row is several batches long); each
    // lane has up to kG chunks in flight, all loads of a batch before its stores
    constexpr int kG = 8;
    const int nw = kScatterThreads / 32, chunks = H / 8;
    const int batches = (chunks + 32 * kG - 1) / (32 * kG);
    for (int w = blockIdx.y * nw + warp; w < n * batches; w += gridDim.y * nw) {
        const int i = w / batches;
        const int slot = slot_s[i];
        if (slot < 0) continue;
        const size_t src = (size_t)(tok0 + i / k) * H, dst = (size_t)slot * H;
        {
            const int c0 = lane + (w % batches) * 32 * kG;
            uint4 o[kG];
#pragma unroll
            for (int u = 0; u < kG; ++u) {
                const int c = c0 + 32 * u;
                if (c >= chunks) break;
                if (a.x_f32) {
                    float v[8];
                    load8_as_f32(a.X, 1, src + 8 * c, v);
                    o[u].x = pack_bf16x2(v[0], v[1]); o[u].y = pack_bf16x2(v[2], v[3]);
                    o[u].z = pack_bf16x2(v[4], v[5]); o[u].w = pack_bf16x2(v[6], v[7]);
                } else {
                    o[u] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const bf16 *>(a.X) + src + 8 * c));
                }
            }
#pragma unroll
            for (int u = 0; u < kG; ++u) {
                const int c = c0 + 32 * u;
                if (c >= chunks) break;
                *reinterpret_cast<uint4 *>(a.x_sorted + dst + 8 * c) = o[u];
            }
        }
    }
    pdl_trigger();
    __syncthreads();
    trace_exit(a.trace);
}

// ---------------------------------------------------------------- combine

// One CTA per token row, one thread per 8 columns: blockDim = 32 * ceil(H / 256)
// (H <= 8192).  Loads go out in batches of four slot rows per thread.
constexpr int kRowMaxThreads = 1024;
constexpr int kSlotBatch = 2;  // fp32 rows: two slots (64 bytes per thread) in flight keep the 1024-thread CTA unspilled

// 8 fp32 values at p (32-byte aligned)
__device__ __forceinline__ void ld8(const float *p, float4 (&r)[2]) {
    r[0] = __ldg(reinterpret_cast<const float4 *>(p));
    r[1] = __ldg(reinterpret_cast<const float4 *>(p) + 1);
}

__device__ __forceinline__ void fma8(float w, const float4 (&r)[2], float (&acc)[8]) {
    acc[0] = fmaf(w, r[0].x, acc[0]); acc[1] = fmaf(w, r[0].y, acc[1]);
    acc[2] = fmaf(w, r[0].z, acc[2]); acc[3] = fmaf(w, r[0].w, acc[3]);
    acc[4] = fmaf(w, r[1].x, acc[4]); acc[5] = fmaf(w, r[1].y, acc[5]);
    acc[6] = fmaf(w, r[1].z, acc[6]); acc[7] = fmaf(w, r[1].w, acc[7]);
}

__device__ __forceinline__ void add8(const float4 (&r)[2], float (&acc)[8]) {
    acc[0] += r[0].x; acc[1] += r[0].y; acc[2] += r[0].z; acc[3] += r[0].w;
    acc[4] += r[1].x; acc[5] += r[1].y; acc[6] += r[1].z; acc[7] += r[1].w;
}

// Sum of the token's fp32 slot outputs (weights w) plus the shared outputs, in
// fp32, in a fixed order (slots 0..k-1, then the shared expert's parts 0..P-1)
// for the 8 columns at c.
__device__ __forceinline__ void combine_columns(const CombineArgs &a, int t, int c, const int *s_slot,
                                                const float *s_w, float (&acc)[8]) {
    const int H = a.H;
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    for (int j0 = 0; j0 < a.k; j0 += kSlotBatch) {
        float4 r[kSlotBatch][2];
#pragma unroll
        for (int u = 0; u < kSlotBatch; ++u) {
            const int slot = j0 + u < a.k ? s_slot[j0 + u] : -1;
            if (slot >= 0)
                ld8(a.yslot + (size_t)slot * H + c, r[u]);
            else
                r[u][0] = r[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kSlotBatch; ++u)
            if (j0 + u < a.k && s_slot[j0 + u] >= 0) fma8(s_w[j0 + u], r[u], acc);
    }
    if (a.ys != nullptr) {
        for (int p0 = 0; p0 < a.ys_parts; p0 += kSlotBatch) {
            float4 r[kSlotBatch][2];
#pragma unroll
            for (int u = 0; u < kSlotBatch; ++u)
                if (p0 + u < a.ys_parts) ld8(a.ys + (p0 + u) * a.ys_part_stride + (size_t)t * H + c, r[u]);
#pragma unroll
            for (int u = 0; u < kSlotBatch; ++u)
                if (p0 + u < a.ys_parts) add8(r[u], acc);
        }
    }
}

__device__ __forceinline__ void store8(void *Y, int y_f32, size_t off, const float (&v)[8]) {
    if (y_f32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(Y) + off);
        dst[0] = make_float4(v[0], v[1], v[2], v[3]);
        dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
        uint4 o;
        o.x = pack_bf16x2(v[0], v[1]); o.y = pack_bf16x2(v[2], v[3]);
        o.z = pack_bf16x2(v[4], v[5]); o.w = pack_bf16x2(v[6], v[7]);
        *reinterpret_cast<uint4 *>(static_cast<bf16 *>(Y) + off) = o;
    }
}

// The 8 gains at column c: g = w (norm 1) or 1 + w (norm 2)
__device__ __forceinline__ void gain8(const float *w, int norm, int c, float (&g)[8]) {
    const float4 lo = __ldg(reinterpret_cast<const float4 *>(w + c));
    const float4 hi = __ldg(reinterpret_cast<const float4 *>(w + c + 4));
    g[0] = lo.x; g[1] = lo.y; g[2] = lo.z; g[3] = lo.w; g[4] = hi.x; g[5] = hi.y; g[6] = hi.z; g[7] = hi.w;
    if (norm == 2) {
#pragma unroll
        for (int q = 0; q < 8; ++q) g[q] += 1.0f;
    }
}

// Sum over the CTA in a fixed order (lanes by butterfly, then warps in index
// order); every thread gets the total.
__device__ __forceinline__ float row_sum(float v, float *s_red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
    __syncthreads();
    float tot = 0.f;
    const int nw = blockDim.x >> 5;
    for (int w = 0; w < nw; ++w) tot += s_red[w];
    return tot;
}

// NORM: out = residual + y * g / sqrt(mean(y^2) + eps) on the fp32 row y.
template <bool NORM>
__global__ void __launch_bounds__(kRowMaxThreads) combine_kernel(const CombineArgs a) {
    __shared__ int s_slot[2][16];
    __shared__ float s_w[2][16];
    __shared__ float s_red[kRowMaxThreads / 32];
    const int k = a.k, H = a.H, c = threadIdx.x * 8;
    const bool on = c < H;
    trace_mark(a.trace, 0);
    // The tokens' slots and weights come from the router and the dispatch, which
    // completed before the expert GEMM (this grid's predecessor) passed its own
    // wait and let this grid launch: the first token's are read ahead of the wait,
    // from L2, and each next token's while the current one is summed.
    int t = blockIdx.x;
    if (threadIdx.x < k && t < a.T) {
        s_slot[0][threadIdx.x] = __ldcg(a.slot_of + (size_t)t * k + threadIdx.x);
        s_w[0][threadIdx.x] = __ldcg(a.topk_w + (size_t)t * k + threadIdx.x);
    }
    float g[8];
    if (NORM && on) gain8(a.post_w, a.norm, c, g);  // weights: not written by any kernel
    pdl_wait();
    trace_mark(a.trace, 1);
    pdl_trigger();
    __syncthreads();
    for (int b = 0; t < a.T; t += gridDim.x, b ^= 1) {
        const int tn = t + gridDim.x;
        if (threadIdx.x < k && tn < a.T) {
            s_slot[b ^ 1][threadIdx.x] = __ldcg(a.slot_of + (size_t)tn * k + threadIdx.x);
            s_w[b ^ 1][threadIdx.x] = __ldcg(a.topk_w + (size_t)tn * k + threadIdx.x);
        }
        float acc[8];
        if (on) combine_columns(a, t, c, s_slot[b], s_w[b], acc);
        if (!NORM) {
            if (on) store8(a.Y, a.y_f32, (size_t)t * H + c, acc);
        } else {
            float x[8], ss = 0.f;
            if (on) {
                load8_as_f32(a.residual, a.y_f32, (size_t)t * H + c, x);
#pragma unroll
                for (int q = 0; q < 8; ++q) ss = fmaf(acc[q], acc[q], ss);
            }
            const float inv = 1.0f / sqrtf(row_sum(ss, s_red) / (float)H + a.eps);
            if (on) {
#pragma unroll
                for (int q = 0; q < 8; ++q) x[q] += acc[q] * inv * g[q];
                store8(a.Y, a.y_f32, (size_t)t * H + c, x);
            }
        }
        __syncthreads();  // the next token's slots are in; this token's buffer may be refilled
    }
    trace_exit(a.trace);
}

// Without the post-norm every output element depends on its own column only.
// The work is T * H / 4 units (token, 4-column group), consecutive units on
// consecutive groups of a row; each CTA takes one contiguous range of units (a
// multiple of its thread count) and walks it kFlatTok tokens at a time: it stages
// those tokens' slot ids and weights in shared memory (one coalesced round trip),
// then each thread takes units of the range, so a warp reads 512 contiguous bytes
// of each term.  A unit's terms are its k slot rows (weights w) and then its P
// shared parts (weight 1: fmaf(1, x, acc) rounds exactly as acc + x), in that
// fixed order, in batches of kFlatBatch whose loads are all issued before any is
// added: one round trip per unit and batch, up to kFlatBatch 16-byte loads in
// flight per thread.
constexpr int kFlatThreads = 256;
constexpr int kFlatBatch = 8;
constexpr int kFlatTok = 64;

// Overlapped with the expert GEMM (a.tok_done): each 64-token chunk first waits until
// its tokens' rows are stored (loads then bypass L1), and the wait on the GEMM grid
// comes at the end.
__device__ __forceinline__ bool wait_tokens(const CombineArgs &a, int ts, int nt, const int *s_slot, int parts) {
    bool good = true;
    if (threadIdx.x < 32)
        for (int i = threadIdx.x; i < nt; i += 32) {
            int valid = parts;
            for (int j = 0; j < a.k; ++j) valid += s_slot[i * a.k + j] >= 0;
            good = good && wait_at_least(a.tok_done + ts + i, a.tok_unit * valid, a.wait_ns);
        }
    if (!good && a.err != nullptr) atomicOr(a.err, ERR_TIMEOUT);
    return good;
}

__global__ void __launch_bounds__(kFlatThreads, 3) combine_flat_kernel(const CombineArgs a) {
    __shared__ int s_slot[kFlatTok * 16];
    __shared__ float s_w[kFlatTok * 16];
    const bool ovl = a.tok_done != nullptr;
    trace_mark(a.trace, 0);
    if (!ovl) {
        pdl_wait();
        trace_mark(a.trace, 1);
    }
    pdl_trigger();
    const int k = a.k, H = a.H, groups = H / 4;
    const int parts = a.ys != nullptr ? a.ys_parts : 0, terms = k + parts;
    const long long units = (long long)a.T * groups;
    long long per = (units + gridDim.x - 1) / gridDim.x;
    per = (per + kFlatThreads - 1) / kFlatThreads * kFlatThreads;
    const long long u_begin = blockIdx.x * per, u_end = min(units, u_begin + per);
    if (u_begin >= u_end) {
        if (ovl) pdl_wait();
        trace_exit(a.trace);
        return;
    }
    const int t_last = (int)((u_end - 1) / groups);
    for (int ts = (int)(u_begin / groups); ts <= t_last; ts += kFlatTok) {
        const int nt = min(kFlatTok, t_last + 1 - ts);
        __syncthreads();  // the previous tokens' ids are no longer read
        for (int i = threadIdx.x; i < nt * k; i += kFlatThreads) {
            s_slot[i] = __ldg(a.slot_of + (size_t)ts * k + i);
            s_w[i] = __ldg(a.topk_w + (size_t)ts * k + i);
        }
        __syncthreads();
        if (ovl) {
            wait_tokens(a, ts, nt, s_slot, parts);
            __syncthreads();
        }
        const long long lo = max(u_begin, (long long)ts * groups);
        const long long hi = min(u_end, (long long)(ts + nt) * groups);
        for (long long u = lo + threadIdx.x; u < hi; u += kFlatThreads) {
            const int t = (int)(u / groups);
            const int tl = t - ts;
            const int c = (int)(u - (long long)t * groups) * 4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j0 = 0; j0 < terms; j0 += kFlatBatch) {
                float4 r[kFlatBatch];
                float w[kFlatBatch];
                bool on[kFlatBatch];
#pragma unroll
                for (int v = 0; v < kFlatBatch; ++v) {
                    const int j = j0 + v;
                    const float *src = nullptr;
                    w[v] = 1.f;
                    if (j < k) {
                        const int slot = s_slot[tl * k + j];
                        if (slot >= 0) {
                            src = a.yslot + (size_t)slot * H + c;
                            w[v] = s_w[tl * k + j];
                        }
                    } else if (j < terms) {
                        src = a.ys + (size_t)(j - k) * a.ys_part_stride + (size_t)t * H + c;
                    }
                    on[v] = src != nullptr;
                    if (on[v])
                        r[v] = ovl ? __ldcg(reinterpret_cast<const float4 *>(src))
                                   : __ldg(reinterpret_cast<const float4 *>(src));
                }
#pragma unroll
                for (int v = 0; v < kFlatBatch; ++v) {
                    if (on[v]) {
                        acc.x = fmaf(w[v], r[v].x, acc.x);
                        acc.y = fmaf(w[v], r[v].y, acc.y);
                        acc.z = fmaf(w[v], r[v].z, acc.z);
                        acc.w = fmaf(w[v], r[v].w, acc.w);
                    }
                }
            }
            const size_t off = (size_t)t * H + c;
            if (a.y_f32) {
                *reinterpret_cast<float4 *>(static_cast<float *>(a.Y) + off) = acc;
            } else {
                uint2 o;
                o.x = pack_bf16x2(acc.x, acc.y);
                o.y = pack_bf16x2(acc.z, acc.w);
                *reinterpret_cast<uint2 *>(static_cast<bf16 *>(a.Y) + off) = o;
            }
        }
    }
    if (ovl) {  // the grid ends after the expert GEMM's
        pdl_wait();
        trace_mark(a.trace, 1);
    }
    trace_exit(a.trace);
}

// Without the post-norm, with bulk copies: the work is T * H / kBulkCols units
// (token, chunk of kBulkCols columns); each CTA takes a contiguous range of units and
// stages the ids and weights of their tokens in shared memory.  Warp w takes units w,
// w + kBulkWarps, ... of the range: lane 0 copies a unit's terms (its k slot rows,
// then the P shared parts, kBulkCols fp32 each) with cp.async.bulk into one of the
// warp's two stages, completing on the stage's mbarrier, so that the next unit's
// copies are in flight while the warp adds the current one.  The sum is the flat
// kernel's: fmaf in the fixed term order from zero, weight 1 for the shared parts.
//
// Used when a unit has at most kBulkMaxTerms terms, where the flat kernel has few
// loads in flight per thread.  Measured on GB300: MiniMax-M3 block (4 slots + 1
// shared part, H = 6144) 53 against 61.5 us; with 7 terms (AFMoE prefill) 61 against
// 56 us and with 9 (Nano decode) 10.2 against 8.2 us, so those stay on the flat
// kernel; 512- or 1024-column units (4 or 2 warps) are slower still.
constexpr int kBulkCols = 256;
constexpr int kBulkWarps = 8;
constexpr int kBulkVec = kBulkCols / 128;  // float4 per lane and term
constexpr int kBulkTok = 64;
constexpr int kBulkMaxTerms = 5;
constexpr uint64_t kBulkDrainNs = 1000000000ull;

__global__ void __launch_bounds__(kBulkWarps * 32) combine_bulk_kernel(const CombineArgs a) {
    extern __shared__ __align__(128) uint8_t bulk_smem[];
    __shared__ __align__(8) uint64_t bars[kBulkWarps][2];
    __shared__ int s_slot[kBulkTok * 16];
    __shared__ float s_w[kBulkTok * 16];
    trace_mark(a.trace, 0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = a.k, H = a.H, chunks = H / kBulkCols;
    const int parts = a.ys != nullptr ? a.ys_parts : 0, terms = k + parts;
    constexpr uint32_t kTermBytes = kBulkCols * 4;
    const uint32_t stage_bytes = (uint32_t)terms * kTermBytes;
    const uint32_t stage0 = smem_u32(bulk_smem) + (uint32_t)(2 * warp) * stage_bytes;
    const float *stage_f = reinterpret_cast<const float *>(bulk_smem) + (size_t)(2 * warp) * terms * kBulkCols;
    const uint32_t bar0 = smem_u32(&bars[warp][0]);
    if (lane == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar0 + 8, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const bool ovl = a.tok_done != nullptr;
    if (!ovl) {
        pdl_wait();
        trace_mark(a.trace, 1);
    }
    pdl_trigger();
    const long long units = (long long)a.T * chunks;
    const long long per = (units + gridDim.x - 1) / gridDim.x;
    const long long u_begin = blockIdx.x * per, u_end = min(units, u_begin + per);
    uint32_t issued = 0, done = 0;  // this warp's units copied / added (stage = count & 1)
    bool ok = true;
    for (long long ub = u_begin; ub < u_end && ok;) {
        // a pass: the units of at most kBulkTok tokens
        const int ts = (int)(ub / chunks);
        const int nt = (int)min((long long)kBulkTok, (u_end - 1) / chunks + 1 - ts);
        const long long ue = min(u_end, (long long)(ts + nt) * chunks);
        for (int i = threadIdx.x; i < nt * k; i += kBulkWarps * 32) {
            s_slot[i] = __ldg(a.slot_of + (size_t)ts * k + i);
            s_w[i] = __ldg(a.topk_w + (size_t)ts * k + i);
        }
        __syncthreads();
        if (ovl) {
            wait_tokens(a, ts, nt, s_slot, parts);
            __syncthreads();
        }
        auto issue = [&](long long u) {
            const uint32_t st = issued & 1u;
            if (lane == 0) {
                const int t = (int)(u / chunks), tl = t - ts, c0 = (int)(u - (long long)t * chunks) * kBulkCols;
                const uint32_t bar = bar0 + 8u * st, dst = stage0 + st * stage_bytes;
                int valid = parts;
                for (int j = 0; j < k; ++j) valid += s_slot[tl * k + j] >= 0;
                // the stage was last read by this warp's lanes (generic proxy) before __syncwarp;
                // with the overlap, the rows were stored by the GEMM's generic stores
                asm volatile("fence.proxy.async;" ::: "memory");
                mbar_arrive_expect_tx(bar, (uint32_t)valid * kTermBytes);
                for (int j = 0; j < k; ++j) {
                    const int slot = s_slot[tl * k + j];
                    if (slot >= 0) bulk_g2s(dst + j * kTermBytes, a.yslot + (size_t)slot * H + c0, kTermBytes, bar);
                }
                for (int q = 0; q < parts; ++q)
                    bulk_g2s(dst + (k + q) * kTermBytes, a.ys + q * a.ys_part_stride + (size_t)t * H + c0, kTermBytes,
                             bar);
            }
            ++issued;
        };
        long long un = ub + warp;
        if (un < ue) issue(un);
        for (long long u = un; u < ue; u += kBulkWarps) {
            if (u + kBulkWarps < ue) issue(u + kBulkWarps);  // the other stage: read two units ago
            const uint32_t st = done & 1u, ph = (done >> 1) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8u * st, ph, a.wait_ns, nullptr))) {
                if (lane == 0 && a.err != nullptr) atomicOr(a.err, ERR_TIMEOUT);
                ok = false;
                break;
            }
            const int t = (int)(u / chunks), tl = t - ts, c0 = (int)(u - (long long)t * chunks) * kBulkCols;
            const float *sf = stage_f + (size_t)st * terms * kBulkCols;
            float4 acc[kBulkVec];
#pragma unroll
            for (int h = 0; h < kBulkVec; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < terms; ++j) {
                float w = 1.f;
                if (j < k) {
                    if (s_slot[tl * k + j] < 0) continue;
                    w = s_w[tl * k + j];
                }
#pragma unroll
                for (int h = 0; h < kBulkVec; ++h) {
                    const float4 x = *reinterpret_cast<const float4 *>(sf + j * kBulkCols + 128 * h + 4 * lane);
                    acc[h].x = fmaf(w, x.x, acc[h].x);
                    acc[h].y = fmaf(w, x.y, acc[h].y);
                    acc[h].z = fmaf(w, x.z, acc[h].z);
                    acc[h].w = fmaf(w, x.w, acc[h].w);
                }
            }
            __syncwarp();  // every lane has read the stage before lane 0 refills it
            ++done;
#pragma unroll
            for (int h = 0; h < kBulkVec; ++h) {
                const size_t off = (size_t)t * H + c0 + 128 * h + 4 * lane;
                if (a.y_f32) {
                    *reinterpret_cast<float4 *>(static_cast<float *>(a.Y) + off) = acc[h];
                } else {
                    uint2 o;
                    o.x = pack_bf16x2(acc[h].x, acc[h].y);
                    o.y = pack_bf16x2(acc[h].z, acc[h].w);
                    *reinterpret_cast<uint2 *>(static_cast<bf16 *>(a.Y) + off) = o;
                }
            }
        }
        ub = ue;
        // every warp is done with this pass's ids (and agrees whether to go on)
        ok = __syncthreads_and(ok) != 0;
    }
    if (!ok) {
        // copies still in flight land before the CTA's shared memory is released
        for (; done < issued; ++done)
            mbar_wait(bar0 + 8u * (done & 1u), (done >> 1) & 1u, kBulkDrainNs, nullptr);
    }
    __syncthreads();
    if (ovl) {  // the grid ends after the expert GEMM's
        pdl_wait();
        trace_mark(a.trace, 1);
    }
    trace_exit(a.trace);
}

// ------------------------------------------------------------- pre-MLP norm

__global__ void __launch_bounds__(kRowMaxThreads) rmsnorm_kernel(const NormArgs a) {
    __shared__ float s_red[kRowMaxThreads / 32];
    const int t = blockIdx.x, H = a.H, c = threadIdx.x * 8;
    const bool on = c < H;
    trace_mark(a.trace, 0);
    float g[8];
    if (on) gain8(a.w, a.norm, c, g);
    pdl_wait();
    trace_mark(a.trace, 1);
    pdl_trigger();
    if (t == 0) {
        for (int i = threadIdx.x; i < a.zero_a_n; i += blockDim.x) a.zero_a[i] = 0;
        for (int i = threadIdx.x; i < a.zero_b_n; i += blockDim.x) a.zero_b[i] = 0;
    }
    const size_t off = (size_t)t * H + c;
    float v[8], ss = 0.f;
    if (on) {
        load8_as_f32(a.X, a.x_f32, off, v);
#pragma unroll
        for (int q = 0; q < 8; ++q) ss = fmaf(v[q], v[q], ss);
    }
    const float inv = 1.0f / sqrtf(row_sum(ss, s_red) / (float)H + a.eps);
    if (on) {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = v[q] * inv * g[q];
        store8(a.out, a.x_f32, off, v);
    }
    __syncthreads();
    trace_exit(a.trace);
}

}  // namespace

// The routing kernels overlap the expert GEMM's CTAs (programmatic dependent
// launch): ask for the largest shared-memory carveout so that an SM running
// them can still take a GEMM CTA.
template <typename K>
static void max_smem_carveout(K kernel) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

int router_tokens_per_block(int T, int num_sms) { return (T + 31) / 32 >= num_sms ? 32 : 16; }

cudaError_t launch_router(const RouterArgs &a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] {
        const int max_smem = (int)router_smem(32, 256);
        cudaFuncSetAttribute(router_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        cudaFuncSetAttribute(router_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        max_smem_carveout(router_kernel<16>);
        max_smem_carveout(router_kernel<32>);
    });
    const int TT = a.tokens_per_block;
    const int nb = (a.T + TT - 1) / TT;
    const size_t smem = router_smem(TT, a.E);
    if (TT == 32) return launch_pdl(router_kernel<32>, dim3(nb), dim3(kRouterThreads), smem, s, a);
    return launch_pdl(router_kernel<16>, dim3(nb), dim3(kRouterThreads), smem, s, a);
}

cudaError_t launch_scan(const ScanArgs &a, cudaStream_t s) {
    return launch_pdl(scan_kernel, dim3(1), dim3(kScanThreads), 0, s, a);
}

int scatter_ctas_per_sm() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scatter_kernel, kScatterThreads, 0) != cudaSuccess ||
            n < 1) {
            cudaGetLastError();
            n = 1;
        }
    });
    return n;
}

cudaError_t launch_scatter(const ScatterArgs &a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] { max_smem_carveout(scatter_kernel); });
    const int nb = (a.T + a.tokens_per_block - 1) / a.tokens_per_block;
    return launch_pdl(scatter_kernel, dim3(nb, a.gather_split > 0 ? a.gather_split : 1), dim3(kScatterThreads),
                      0, s, a);
}

// threads of a row kernel: one per 8 columns, whole warps
static int row_threads(int H) { return ((H / 8 + 31) / 32) * 32; }

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] {
        max_smem_carveout(combine_kernel<true>);
        max_smem_carveout(combine_flat_kernel);
    });
    if (a.H % 8 != 0 || row_threads(a.H) > kRowMaxThreads || a.k > 16 || (a.ys != nullptr && a.ys_parts < 1))
        return cudaErrorInvalidValue;
    // four CTAs per SM, each looping over tokens (measured on GB300: 2 us faster than one
    // CTA per token at AFMoE prefill sizes, equal at decode sizes)
    constexpr int kCombineCtasPerSm = 4;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidValue;
    if (a.norm != 0) {
        if (a.residual == nullptr || a.post_w == nullptr) return cudaErrorInvalidValue;
        const int grid = a.T < sms * kCombineCtasPerSm ? a.T : sms * kCombineCtasPerSm;
        return launch_pdl(combine_kernel<true>, dim3(grid), dim3(row_threads(a.H)), 0, s, a);
    }
    // bulk copies when a unit's terms fit two stages per warp
    const int terms = a.k + (a.ys != nullptr ? a.ys_parts : 0);
    if (a.H % kBulkCols == 0 && terms >= 1 && terms <= kBulkMaxTerms &&
        kBulkWarps * 2 * terms * kBulkCols * 4 <= 200 * 1024) {
        const int smem = kBulkWarps * 2 * terms * kBulkCols * 4;
        static int bulk_per_sm[kBulkMaxTerms + 1] = {};
        static std::once_flag bulk_once;
        std::call_once(bulk_once, [] {
            cudaFuncSetAttribute(combine_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
            for (int tm = 1; tm <= kBulkMaxTerms; ++tm) {
                const int sb = kBulkWarps * 2 * tm * kBulkCols * 4;
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bulk_per_sm[tm], combine_bulk_kernel,
                                                                  kBulkWarps * 32, sb) != cudaSuccess ||
                    bulk_per_sm[tm] < 1)
                    bulk_per_sm[tm] = 1;
            }
        });
        const long long units = (long long)a.T * (a.H / kBulkCols);
        const long long need = (units + kBulkWarps - 1) / kBulkWarps;
        const long long cap = (long long)sms * bulk_per_sm[terms];
        const int grid = (int)(need < cap ? need : cap);
        return launch_pdl(combine_bulk_kernel, dim3(grid), dim3(kBulkWarps * 32), (size_t)smem, s, a);
    }
    // the flat kernel: as many CTAs as are resident at once on every SM, capped by the chunks
    static int flat_per_sm = 0;
    static std::once_flag occ;
    std::call_once(occ, [] {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&flat_per_sm, combine_flat_kernel, kFlatThreads, 0) !=
                cudaSuccess || flat_per_sm < 1)
            flat_per_sm = 1;
    });
    // CTAs: as many as are resident at once, at most one per kFlatThreads units
    const long long units = (long long)a.T * (a.H / 4);
    const long long need = (units + kFlatThreads - 1) / kFlatThreads;
    const int grid = (int)(need < (long long)sms * flat_per_sm ? need : (long long)sms * flat_per_sm);
    return launch_pdl(combine_flat_kernel, dim3(grid), dim3(kFlatThreads), 0, s, a);
}

cudaError_t launch_rmsnorm(const NormArgs &a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] { max_smem_carveout(rmsnorm_kernel); });
    if (a.H % 8 != 0 || row_threads(a.H) > kRowMaxThreads) return cudaErrorInvalidValue;
    return launch_pdl(rmsnorm_kernel, dim3(a.T), dim3(row_threads(a.H)), 0, s, a);
}

}  // namespace moe
