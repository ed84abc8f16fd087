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

__device__ __forceinline__ bool better(float c, int e, float bc, int be) {
    return c > bc || (c == bc && e < be);
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
        float s[8], c[8];
        if (a.score_func == 1) {
            float m = -INFINITY;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (lane + 32 * j < E) m = fmaxf(m, acc[i][j]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float z = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                s[j] = (lane + 32 * j < E) ? expf(acc[i][j] - m) : 0.f;
                z += s[j];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
#pragma unroll
            for (int j = 0; j < 8; ++j) s[j] = s[j] / z;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) s[j] = 1.0f / (1.0f + expf(-acc[i][j]));
        }
        uint32_t open = 0;  // bit j: expert lane+32j is a candidate
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane + 32 * j;
            if (e < E) {
                const float cj = s[j] + (a.bias ? __ldg(a.bias + e) : 0.f);
                c[j] = (cj != cj) ? -INFINITY : cj;  // NaN never wins
                open |= 1u << j;
            } else {
                c[j] = -INFINITY;
            }
        }
        float wsum = 0.f, my_s = 0.f;
        int my_e = 0;
        for (int r = 0; r < a.k; ++r) {
            float bc = -INFINITY;
            int be = 0x7fffffff;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if ((open >> j & 1u) && better(c[j], lane + 32 * j, bc, be)) {
                    bc = c[j];
                    be = lane + 32 * j;
                }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float oc = __shfl_xor_sync(0xffffffffu, bc, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (better(oc, oe, bc, be)) {
                    bc = oc;
                    be = oe;
                }
            }
            const int owner = be & 31, jj = be >> 5;
            float sv = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j == jj) sv = s[j];
            if (lane == owner) open &= ~(1u << jj);
            sv = __shfl_sync(0xffffffffu, sv, owner);
            wsum += sv;
            if (lane == r) {
                my_e = be;
                my_s = sv;
            }
        }
        if (lane < a.k) {
            float w = my_s;
            if (a.route_norm) w = w / wsum;
            w = w * a.route_scale;
            a.topk_idx[(size_t)t * a.k + lane] = my_e;
            a.topk_w[(size_t)t * a.k + lane] = w;
            if (a.blk_hist != nullptr) atomicAdd(&hist[my_e], 1);
        }
    }
    if (a.blk_hist != nullptr) {
        __syncthreads();
        for (int e = tid; e < E; e += kRouterThreads)
            a.blk_hist[(size_t)blockIdx.x * E + e] = hist[e];
    }
}

size_t router_smem(int TT, int E) { return (size_t)(TT + E) * kPad * 4 + (size_t)E * 4; }

// ------------------------------------------------------------------- scan

constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) scan_kernel(const ScanArgs a) {
    __shared__ int cnt[256];
    __shared__ int base[257];
    const int E = a.E, nb = a.nb;
    for (int e = threadIdx.x; e < E; e += kScanThreads) {
        int run = 0;
        for (int b = 0; b < nb; ++b) {  // exclusive scan over blocks, per expert
            const int v = a.blk_hist[(size_t)b * E + e];
            a.blk_hist[(size_t)b * E + e] = run;
            run += v;
        }
        cnt[e] = run;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int o = 0, to = 0, n = 0;
        for (int e = 0; e < E; ++e) {
            base[e] = o;
            a.offs[e] = o;
            a.tile_offs[e] = to;
            o += cnt[e];
            to += (cnt[e] + kGemmBM - 1) / kGemmBM;
            if (cnt[e] > 0) a.active[n++] = e;
        }
        a.offs[E] = o;
        a.tile_offs[E] = to;
        a.active[E] = n;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nb * E; i += kScanThreads) a.blk_hist[i] += base[i % E];
}

// ---------------------------------------------------------------- scatter

constexpr int kScatterThreads = 256;

__global__ void __launch_bounds__(kScatterThreads) scatter_kernel(const ScatterArgs a) {
    __shared__ int e_s[32 * 16];
    __shared__ int slot_s[32 * 16];
    const int TT = a.tokens_per_block, k = a.k, E = a.E, H = a.H;
    const int tok0 = blockIdx.x * TT;
    const int n = max(0, min(TT, a.T - tok0)) * k;
    const size_t ent0 = (size_t)tok0 * k;
    for (int i = threadIdx.x; i < n; i += kScatterThreads) {
        int e = a.topk_idx[ent0 + i];
        if (e < 0 || e >= E) {
            atomicOr(a.err, ERR_BOUNDS);
            e = -1;
        }
        e_s[i] = e;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kScatterThreads) {
        const int e = e_s[i];
        int slot = -1;
        if (e >= 0) {
            int rank = 0;  // entries of the same expert earlier in (token, slot) order
            for (int q = 0; q < i; ++q) rank += (e_s[q] == e);
            slot = a.blk_base[(size_t)blockIdx.x * E + e] + rank;
            a.sorted_tok[slot] = tok0 + i / k;
        }
        a.slot_of[ent0 + i] = slot;
        slot_s[i] = slot;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < n; i += kScatterThreads / 32) {
        const int slot = slot_s[i];
        if (slot < 0) continue;
        const size_t src = (size_t)(tok0 + i / k) * H, dst = (size_t)slot * H;
        for (int c = lane * 8; c < H; c += 256) {
            uint4 o;
            if (a.x_f32) {
                float v[8];
                load8_as_f32(a.X, 1, src + c, v);
                o.x = pack_bf16x2(v[0], v[1]); o.y = pack_bf16x2(v[2], v[3]);
                o.z = pack_bf16x2(v[4], v[5]); o.w = pack_bf16x2(v[6], v[7]);
            } else {
                o = __ldg(reinterpret_cast<const uint4 *>(static_cast<const bf16 *>(a.X) + src + c));
            }
            *reinterpret_cast<uint4 *>(a.x_sorted + dst + c) = o;
        }
    }
}

// ---------------------------------------------------------------- combine

constexpr int kCombineThreads = 128;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
    const int t = blockIdx.x, k = a.k, H = a.H;
    for (int c = threadIdx.x * 8; c < H; c += kCombineThreads * 8) {
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.f;
        for (int j = 0; j < k; ++j) {
            const int slot = __ldg(a.slot_of + (size_t)t * k + j);
            if (slot < 0) continue;
            const float w = __ldg(a.topk_w + (size_t)t * k + j);
            const uint4 r = __ldg(reinterpret_cast<const uint4 *>(a.yslot + (size_t)slot * H + c));
            acc[0] = fmaf(w, bf16_lo(r.x), acc[0]); acc[1] = fmaf(w, bf16_hi(r.x), acc[1]);
            acc[2] = fmaf(w, bf16_lo(r.y), acc[2]); acc[3] = fmaf(w, bf16_hi(r.y), acc[3]);
            acc[4] = fmaf(w, bf16_lo(r.z), acc[4]); acc[5] = fmaf(w, bf16_hi(r.z), acc[5]);
            acc[6] = fmaf(w, bf16_lo(r.w), acc[6]); acc[7] = fmaf(w, bf16_hi(r.w), acc[7]);
        }
        if (a.ys != nullptr) {
            const uint4 r = __ldg(reinterpret_cast<const uint4 *>(a.ys + (size_t)t * H + c));
            acc[0] += bf16_lo(r.x); acc[1] += bf16_hi(r.x); acc[2] += bf16_lo(r.y);
            acc[3] += bf16_hi(r.y); acc[4] += bf16_lo(r.z); acc[5] += bf16_hi(r.z);
            acc[6] += bf16_lo(r.w); acc[7] += bf16_hi(r.w);
        }
        if (a.y_f32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.Y) + (size_t)t * H + c);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        } else {
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]); o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]); o.w = pack_bf16x2(acc[6], acc[7]);
            *reinterpret_cast<uint4 *>(static_cast<bf16 *>(a.Y) + (size_t)t * H + c) = o;
        }
    }
}

}  // namespace

int router_tokens_per_block(int T, int num_sms) { return (T + 31) / 32 >= num_sms ? 32 : 16; }

cudaError_t launch_router(const RouterArgs &a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] {
        const int max_smem = (int)router_smem(32, 256);
        cudaFuncSetAttribute(router_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        cudaFuncSetAttribute(router_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    });
    const int TT = a.tokens_per_block;
    const int nb = (a.T + TT - 1) / TT;
    const size_t smem = router_smem(TT, a.E);
    if (TT == 32)
        router_kernel<32><<<nb, kRouterThreads, smem, s>>>(a);
    else
        router_kernel<16><<<nb, kRouterThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_scan(const ScanArgs &a, cudaStream_t s) {
    scan_kernel<<<1, kScanThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_scatter(const ScatterArgs &a, cudaStream_t s) {
    const int nb = (a.T + a.tokens_per_block - 1) / a.tokens_per_block;
    scatter_kernel<<<nb, kScatterThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s) {
    combine_kernel<<<a.T, kCombineThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
