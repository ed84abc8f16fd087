// Weight-streaming decode kernels (K6) for few tokens per expert.
//
// With a handful of tokens per expert the block is bound by reading the
// touched experts' weights once from HBM.  A persistent grid takes blocks of
// output rows of the active experts (and of the shared expert) round-robin;
// for each it stages that expert's token rows in shared memory and streams the
// weight rows with 128-bit loads that bypass L1, one warp reducing one output
// row with shuffles.  Only experts that received tokens are visited (the
// dispatch sort lists them).
//
// Gate/up: h[r, i] = act(Wg[e][i,:] . x_r, Wu[e][i,:] . x_r)   (bf16 out)
// Down:    y[r, j] = Wd[e][j,:] . h_r                           (fp32 out)
// (stacked [out, in] expert weights: Arcee AFMoE issue, "Checkpoint weight layout")
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerCta = kWarps;  // one output row per warp
constexpr int kMT = 8;               // token rows staged per pass
constexpr int kMaxK = 8192;          // longest staged row (H, I or S)
constexpr int kUnroll = 8;           // 16-byte loads per lane in flight (x2 for gate and up)
constexpr int kCtasPerSm = 4;        // persistent grid (residency permitting: kMT x K x 2 staged bytes each)

__device__ __forceinline__ uint4 ld_stream(const bf16 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float dot8(const uint4 w, const uint4 x) {
    float s = bf16_lo(w.x) * bf16_lo(x.x);
    s = fmaf(bf16_hi(w.x), bf16_hi(x.x), s);
    s = fmaf(bf16_lo(w.y), bf16_lo(x.y), s);
    s = fmaf(bf16_hi(w.y), bf16_hi(x.y), s);
    s = fmaf(bf16_lo(w.z), bf16_lo(x.z), s);
    s = fmaf(bf16_hi(w.z), bf16_hi(x.z), s);
    s = fmaf(bf16_lo(w.w), bf16_lo(x.w), s);
    s = fmaf(bf16_hi(w.w), bf16_hi(x.w), s);
    return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Work items: blocks of kRowsPerCta output rows of the active routed experts (in the
// dispatch's order), then of the shared expert.  A persistent grid takes them
// round-robin, so no CTA is launched for an expert without tokens.
__device__ __forceinline__ bool work_item(const DecodeGroups &g, int item, int nb_routed, int nb_shared, int &expert,
                                          int &rb, int &row0, int &m) {
    const int n_routed = g.active[g.E] * nb_routed;
    if (item < n_routed) {
        expert = g.active[item / nb_routed];
        rb = item % nb_routed;
        row0 = g.offs[expert];
        m = g.offs[expert + 1] - row0;
        return true;
    }
    item -= n_routed;
    if (!g.shared || item >= nb_shared) return false;
    expert = -1;
    rb = item;
    row0 = 0;
    m = g.T;
    return true;
}

__device__ __forceinline__ void stage_rows(bf16 *xs, const bf16 *src, int rows, int K) {
    const int per_row = K / 8;
    for (int f = threadIdx.x; f < rows * per_row; f += kThreads) {
        const int r = f / per_row, c = (f % per_row) * 8;
        *reinterpret_cast<uint4 *>(xs + (size_t)r * K + c) =
            __ldg(reinterpret_cast<const uint4 *>(src + (size_t)r * K + c));
    }
}

// One output row per warp: lane-strided 16-byte weight loads (the weights are read
// once; the token rows come from shared memory).
__global__ void __launch_bounds__(kThreads) decode_glu_kernel(const DecodeGluArgs a) {
    extern __shared__ __align__(16) unsigned char dsm[];
    bf16 *xs = reinterpret_cast<bf16 *>(dsm);  // [kMT][H]
    pdl_wait();
    pdl_trigger();
    const int H = a.H;
    const int nb_routed = (a.I + kRowsPerCta - 1) / kRowsPerCta, nb_shared = (a.S + kRowsPerCta - 1) / kRowsPerCta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int expert, rb, row0, m;
    for (int item = blockIdx.x; work_item(a.g, item, nb_routed, nb_shared, expert, rb, row0, m); item += gridDim.x) {
        const bool shared = expert < 0;
        const int W = shared ? a.S : a.I;
        const bf16 *src = shared ? a.x_shared : a.x_routed + (size_t)row0 * H;
        const bf16 *Wg = shared ? a.sh_gate : a.gate + (size_t)expert * a.I * H;
        const bf16 *Wu = shared ? a.sh_up : a.up + (size_t)expert * a.I * H;
        bf16 *out = shared ? a.h_shared : a.h_routed + (size_t)row0 * a.I;
        const int i = rb * kRowsPerCta + warp;  // this warp's output row
        for (int tc = 0; tc < m; tc += kMT) {
            const int mt = min(kMT, m - tc);
            __syncthreads();
            stage_rows(xs, src + (size_t)tc * H, mt, H);
            __syncthreads();
            if (i >= W) continue;
            float ag[kMT], au[kMT];
#pragma unroll
            for (int t = 0; t < kMT; ++t) ag[t] = au[t] = 0.f;
            const bf16 *wg = Wg + (size_t)i * H, *wu = Wu + (size_t)i * H;
#pragma unroll kUnroll
            for (int h = lane * 8; h < H; h += 256) {
                const uint4 vg = ld_stream(wg + h), vu = ld_stream(wu + h);
#pragma unroll
                for (int t = 0; t < kMT; ++t) {
                    if (t < mt) {
                        const uint4 xv = *reinterpret_cast<const uint4 *>(xs + (size_t)t * H + h);
                        ag[t] += dot8(vg, xv);
                        au[t] += dot8(vu, xv);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kMT; ++t) {
                if (t < mt) {
                    const float g = warp_sum(ag[t]), u = warp_sum(au[t]);
                    if (lane == t)
                        out[(size_t)(tc + t) * W + i] =
                            __float2bfloat16_rn(glu_act(g, u, a.act, a.alpha, a.limit, a.beta));
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads) decode_down_kernel(const DecodeDownArgs a) {
    extern __shared__ __align__(16) unsigned char dsm[];
    bf16 *hs = reinterpret_cast<bf16 *>(dsm);  // [kMT][K]
    pdl_wait();
    pdl_trigger();
    const int H = a.H;
    const int nb = (H + kRowsPerCta - 1) / kRowsPerCta;  // row blocks of every group
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int expert, rb, row0, m;
    for (int item = blockIdx.x; work_item(a.g, item, nb, nb, expert, rb, row0, m); item += gridDim.x) {
        const bool shared = expert < 0;
        const int K = shared ? a.S : a.I;
        const bf16 *src = shared ? a.h_shared : a.h_routed + (size_t)row0 * a.I;
        const bf16 *Wd = shared ? a.sh_down : a.down + (size_t)expert * H * a.I;
        float *out = shared ? a.y_shared : a.y_routed + (size_t)row0 * H;
        const int j = rb * kRowsPerCta + warp;
        for (int tc = 0; tc < m; tc += kMT) {
            const int mt = min(kMT, m - tc);
            __syncthreads();
            stage_rows(hs, src + (size_t)tc * K, mt, K);
            __syncthreads();
            if (j >= H) continue;
            float acc[kMT];
#pragma unroll
            for (int t = 0; t < kMT; ++t) acc[t] = 0.f;
            const bf16 *wd = Wd + (size_t)j * K;
#pragma unroll kUnroll
            for (int c = lane * 8; c < K; c += 256) {
                const uint4 vw = ld_stream(wd + c);
#pragma unroll
                for (int t = 0; t < kMT; ++t)
                    if (t < mt) acc[t] += dot8(vw, *reinterpret_cast<const uint4 *>(hs + (size_t)t * K + c));
            }
#pragma unroll
            for (int t = 0; t < kMT; ++t) {
                if (t < mt) {
                    const float y = warp_sum(acc[t]);
                    if (lane == t) out[(size_t)(tc + t) * H + j] = y;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_decode_glu(const DecodeGluArgs &a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(decode_glu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMT * kMaxK * 2);
    });
    if (a.H > kMaxK || a.H % 8 != 0 || a.num_sms < 1) return cudaErrorInvalidValue;
    return launch_pdl(decode_glu_kernel, dim3(a.num_sms * kCtasPerSm), dim3(kThreads), (size_t)kMT * a.H * 2, s, a);
}

cudaError_t launch_decode_down(const DecodeDownArgs &a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(decode_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMT * kMaxK * 2);
    });
    const int K = a.g.shared ? max(a.I, a.S) : a.I;
    if (K > kMaxK || a.I % 8 != 0 || a.S % 8 != 0 || a.num_sms < 1) return cudaErrorInvalidValue;
    return launch_pdl(decode_down_kernel, dim3(a.num_sms * kCtasPerSm), dim3(kThreads), (size_t)kMT * K * 2, s, a);
}

}  // namespace moe
