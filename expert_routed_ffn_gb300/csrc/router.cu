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
    // the expert GEMM is launched only when every CTA has reached the end of its
    // gather (launch_dependents below): launched earlier, its one-per-SM CTAs
    // would take the shared memory that this grid's later waves need
    __syncthreads();
    {
        // eight independent loads in flight per thread, then the shared sums
        constexpr int kU = 8;
        const int tot = E * nbk;
        for (int i0 = threadIdx.x; i0 < tot; i0 += kU * kScatterThreads) {
            int v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = i0 + u * kScatterThreads;
                const int e = i / nbk, bb = i - e * nbk;
                v[u] = i < tot ? __ldg(a.blk_hist + (size_t)bb * hb + (size_t)e * he) : 0;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = i0 + u * kScatterThreads;
                if (v[u]) {
                    const int e = i / nbk, bb = i - e * nbk;
                    atomicAdd(&cnt[e], v[u]);
                    if (bb < b) atomicAdd(&pre[e], v[u]);
                }
            }
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
    // row copy: a warp per row, each lane up to kG 16-byte chunks in flight
    // (all loads of a batch before its stores)
    constexpr int kG = 8;
    const int nw = kScatterThreads / 32, chunks = H / 8;
    for (int i = blockIdx.y * nw + warp; i < n; i += gridDim.y * nw) {
        const int slot = slot_s[i];
        if (slot < 0) continue;
        const size_t src = (size_t)(tok0 + i / k) * H, dst = (size_t)slot * H;
        for (int c0 = lane; c0 < chunks; c0 += 32 * kG) {
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

constexpr int kCombineThreads = 128;
constexpr int kCombineMaxChunks = 8;  // H <= 8 * 128 * 8 = 8192

// Sum of the token's slot outputs (weights w) plus the shared outputs, in fp32,
// in a fixed order (slots 0..k-1, then the shared expert's parts) for the 8
// columns at c.
__device__ __forceinline__ void combine_columns(const CombineArgs &a, int t, int c, const int *s_slot,
                                                const float *s_w, float (&acc)[8]) {
    const int H = a.H;
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    for (int j = 0; j < a.k; ++j) {
        const int slot = s_slot[j];
        if (slot < 0) continue;
        const float w = s_w[j];
        const uint4 r = __ldg(reinterpret_cast<const uint4 *>(a.yslot + (size_t)slot * H + c));
        acc[0] = fmaf(w, bf16_lo(r.x), acc[0]); acc[1] = fmaf(w, bf16_hi(r.x), acc[1]);
        acc[2] = fmaf(w, bf16_lo(r.y), acc[2]); acc[3] = fmaf(w, bf16_hi(r.y), acc[3]);
        acc[4] = fmaf(w, bf16_lo(r.z), acc[4]); acc[5] = fmaf(w, bf16_hi(r.z), acc[5]);
        acc[6] = fmaf(w, bf16_lo(r.w), acc[6]); acc[7] = fmaf(w, bf16_hi(r.w), acc[7]);
    }
    const __nv_bfloat16 *sh[2] = {a.ys, a.ys2};
#pragma unroll
    for (int p = 0; p < 2; ++p) {  // the shared expert (and its second K half)
        if (sh[p] == nullptr) continue;
        const uint4 r = __ldg(reinterpret_cast<const uint4 *>(sh[p] + (size_t)t * H + c));
        acc[0] += bf16_lo(r.x); acc[1] += bf16_hi(r.x); acc[2] += bf16_lo(r.y);
        acc[3] += bf16_hi(r.y); acc[4] += bf16_lo(r.z); acc[5] += bf16_hi(r.z);
        acc[6] += bf16_lo(r.w); acc[7] += bf16_hi(r.w);
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

// One CTA per token.  NORM: the token's whole output row stays in registers
// (8 columns per thread per chunk), its sum of squares is reduced over the CTA
// (lanes, then warps, in a fixed order), and out = residual + y * g * inv.
template <bool NORM>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
    __shared__ int s_slot[16];
    __shared__ float s_w[16];
    __shared__ float s_red[kCombineThreads / 32];
    const int t = blockIdx.x, k = a.k, H = a.H;
    trace_mark(a.trace, 0);
    // The token's slots and weights come from the router and the dispatch, which
    // completed before the expert GEMM (this grid's predecessor) passed its own
    // wait and let this grid launch: they are read ahead of the wait, from L2.
    if (threadIdx.x < k) {
        s_slot[threadIdx.x] = __ldcg(a.slot_of + (size_t)t * k + threadIdx.x);
        s_w[threadIdx.x] = __ldcg(a.topk_w + (size_t)t * k + threadIdx.x);
    }
    pdl_wait();
    trace_mark(a.trace, 1);
    pdl_trigger();
    __syncthreads();
    if (!NORM) {
        for (int c = threadIdx.x * 8; c < H; c += kCombineThreads * 8) {
            float acc[8];
            combine_columns(a, t, c, s_slot, s_w, acc);
            store8(a.Y, a.y_f32, (size_t)t * H + c, acc);
        }
    } else {
        float acc[kCombineMaxChunks][8];
        float ss = 0.f;
#pragma unroll
        for (int ci = 0; ci < kCombineMaxChunks; ++ci) {
            const int c = (threadIdx.x + ci * kCombineThreads) * 8;
            if (c < H) {
                combine_columns(a, t, c, s_slot, s_w, acc[ci]);
#pragma unroll
                for (int q = 0; q < 8; ++q) ss = fmaf(acc[ci][q], acc[ci][q], ss);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kCombineThreads / 32; ++w) tot += s_red[w];
        const float inv = 1.0f / sqrtf(tot / (float)H + a.eps);
#pragma unroll
        for (int ci = 0; ci < kCombineMaxChunks; ++ci) {
            const int c = (threadIdx.x + ci * kCombineThreads) * 8;
            if (c < H) {
                float x[8], o[8];
                load8_as_f32(a.residual, a.y_f32, (size_t)t * H + c, x);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float g = a.norm == 2 ? 1.0f + __ldg(a.post_w + c + q) : __ldg(a.post_w + c + q);
                    o[q] = x[q] + acc[ci][q] * inv * g;
                }
                store8(a.Y, a.y_f32, (size_t)t * H + c, o);
            }
        }
    }
    __syncthreads();
    trace_exit(a.trace);
}

// ------------------------------------------------------------- pre-MLP norm

constexpr int kNormThreads = 256;  // 8 warps, one row each

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const NormArgs a) {
    const int lane = threadIdx.x & 31, t = blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5);
    trace_mark(a.trace, 0);
    pdl_wait();
    trace_mark(a.trace, 1);
    pdl_trigger();
    if (t < a.T) {
        const int H = a.H;
        const size_t row = (size_t)t * H;
        float ss = 0.f;
        for (int c = lane * 8; c < H; c += 256) {
            float v[8];
            load8_as_f32(a.X, a.x_f32, row + c, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) ss = fmaf(v[q], v[q], ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = 1.0f / sqrtf(ss / (float)H + a.eps);
        for (int c = lane * 8; c < H; c += 256) {
            float v[8];
            load8_as_f32(a.X, a.x_f32, row + c, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float g = a.norm == 2 ? 1.0f + __ldg(a.w + c + q) : __ldg(a.w + c + q);
                v[q] = v[q] * inv * g;
            }
            store8(a.out, a.x_f32, row + c, v);
        }
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

cudaError_t launch_scatter(const ScatterArgs &a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] { max_smem_carveout(scatter_kernel); });
    const int nb = (a.T + a.tokens_per_block - 1) / a.tokens_per_block;
    return launch_pdl(scatter_kernel, dim3(nb, a.gather_split > 0 ? a.gather_split : 1), dim3(kScatterThreads),
                      0, s, a);
}

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] {
        max_smem_carveout(combine_kernel<false>);
        max_smem_carveout(combine_kernel<true>);
    });
    if (a.norm != 0) {
        if (a.H > kCombineMaxChunks * kCombineThreads * 8 || a.residual == nullptr || a.post_w == nullptr)
            return cudaErrorInvalidValue;
        return launch_pdl(combine_kernel<true>, dim3(a.T), dim3(kCombineThreads), 0, s, a);
    }
    return launch_pdl(combine_kernel<false>, dim3(a.T), dim3(kCombineThreads), 0, s, a);
}

cudaError_t launch_rmsnorm(const NormArgs &a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] { max_smem_carveout(rmsnorm_kernel); });
    const int rows = kNormThreads / 32;
    return launch_pdl(rmsnorm_kernel, dim3((a.T + rows - 1) / rows), dim3(kNormThreads), 0, s, a);
}

}  // namespace moe
