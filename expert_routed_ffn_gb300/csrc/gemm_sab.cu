// Expert GEMMs for few tokens per expert, on the tensor cores with the
// operands swapped (K3/K4/K5, decode-sized T).
//
// With m tokens per expert and m much smaller than 128, the weight rows are
// the natural M = 128 operand of tcgen05.mma and the tokens a small N (32 or
// 64): a pipeline stage is 16 KB of weights plus N x 128 B of token rows, so
// about ten stages of mostly weight bytes are in flight per SM, and a tile is
// small enough that the tiles of all touched experts spread evenly over the
// SMs.
//
//   gate/up (glu = 1): D[128, N] = [Wg[g][i0:i0+64]; Wu[g][i0:i0+64]] . A[r0:r0+N]^T
//       TMEM lanes 0-63 hold gate, 64-127 up for the same 64 outputs i; the
//       epilogue warps of lanes 64-127 hand their values to those of lanes
//       0-63 through shared memory, which apply the activation and store
//       h[r][i0 + lane] (bf16)
//   down    (glu = 0): D[128, N] = Wd[g][j0:j0+128] . h[r0:r0+N]^T
//       lane l stores y[r][j0 + l] (fp32)
// (stacked [out, in] expert weights: Arcee AFMoE issue, "Checkpoint weight
// layout"; activation: HF AFMoE docs hidden_act silu, MiniMax-M3 issue
// clamp-SwiGLU.)  Segments, persistent scheduling and bounded waits follow
// gemm_tc.cu.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr int kABytes = 128 * 64 * 2;  // 16 KB of weight rows per stage
constexpr int kMaxStages = 12;
constexpr int kSmemMax = 232448 - 4096;  // dynamic budget; the rest holds the static offset tables
constexpr uint64_t kDrainNs = 1000000000ull;

struct Tile {
    int seg, group, wt, nt, row0, m_valid;
};

// offs / toffs: shared-memory copies of segment 0's dispatch offsets (only
// segment 0 may be grouped)
template <int N>
__device__ __forceinline__ int seg_tiles(const SabSegment &s, const int *toffs) {
    if (s.dense) return ((s.m_dense + N - 1) / N) * s.w_tiles;
    return toffs[s.num_groups] * s.w_tiles;
}

// token tiles (nt) of one weight tile (wt) are adjacent, so concurrent CTAs
// share the weight tile in L2 when an expert has more than N tokens
template <int N>
__device__ __forceinline__ Tile decode_tile(const SabArgs &p, int tile, int tiles0, const int *offs,
                                            const int *toffs) {
    Tile t;
    t.seg = 0;
    if (tile >= tiles0) {
        t.seg = 1;
        tile -= tiles0;
    }
    const SabSegment &s = p.seg[t.seg];
    if (s.dense) {
        const int nts = (s.m_dense + N - 1) / N;
        t.group = 0;
        t.wt = tile / nts;
        t.nt = tile % nts;
        t.row0 = t.nt * N;
        t.m_valid = min(N, s.m_dense - t.row0);
    } else {
        int lo = 0, hi = s.num_groups - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (toffs[mid] * s.w_tiles <= tile)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int nts = toffs[lo + 1] - toffs[lo];
        const int local = tile - toffs[lo] * s.w_tiles;
        t.group = lo;
        t.wt = local / nts;
        t.nt = local % nts;
        t.row0 = offs[lo] + t.nt * N;
        t.m_valid = min(N, offs[lo + 1] - t.row0);
    }
    return t;
}

__device__ __forceinline__ void raise_abort(int *err, volatile int *abort_flag) {
    if (err != nullptr) atomicOr(err, ERR_TIMEOUT);
    *abort_flag = 1;
}

// Named barrier 1 of the four epilogue warps (128 threads).
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// AND of v over the four epilogue warps (barrier 1): every epilogue thread gets
// the same answer, so they stop or go on together.
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v)
        : "memory");
    return out != 0;
}

template <bool GLU, int N>
__global__ void __launch_bounds__(kThreads, 1) gemm_sab_kernel(const __grid_constant__ SabArgs p) {
    constexpr int kBBytes = N * 128;
    constexpr int kStage = kABytes + kBBytes;
    constexpr uint32_t kTmemCols = (2 * N < 32) ? 32 : 2 * N;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    const uint32_t s0 = smem_u32(smem);
    float *xch = reinterpret_cast<float *>(smem + S * kStage);        // [2][64][N + 1]
    uint8_t *misc = smem + S * kStage + (GLU ? 2 * 64 * (N + 1) * 4 : 0);
    uint64_t *bars = reinterpret_cast<uint64_t *>(misc);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    auto tfull_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kMaxStages + a); };
    auto tempty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kMaxStages + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kMaxStages + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kMaxStages + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (uint32_t a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 128);
        }
        mbar_init(drain_bar, 1);
        fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.Wa0);
        if (GLU) tma_prefetch_desc(&p.Wb0);
        tma_prefetch_desc(&p.X0);
        if (p.num_segs > 1) {
            tma_prefetch_desc(&p.Wa1);
            if (GLU) tma_prefetch_desc(&p.Wb1);
            tma_prefetch_desc(&p.X1);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    pdl_trigger();
    // every role decodes every tile: keep the dispatch offsets on chip
    __shared__ int s_offs[257], s_toffs[257];
    if (!p.seg[0].dense)
        for (int i = threadIdx.x; i <= p.seg[0].num_groups; i += blockDim.x) {
            s_offs[i] = p.seg[0].offs[i];
            s_toffs[i] = p.seg[0].tile_offs[i];
        }
    __syncthreads();
    const uint32_t tmem_base = *tmem_slot;
    const int tiles0 = seg_tiles<N>(p.seg[0], s_toffs);
    const int total = tiles0 + (p.num_segs > 1 ? seg_tiles<N>(p.seg[1], s_toffs) : 0);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t L = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const Tile t = decode_tile<N>(p, tile, tiles0, s_offs, s_toffs);
                const SabSegment &sg = p.seg[t.seg];
                const CUtensorMap *mWa = t.seg ? &p.Wa1 : &p.Wa0;
                const CUtensorMap *mWb = t.seg ? &p.Wb1 : &p.Wb0;
                const CUtensorMap *mX = t.seg ? &p.X1 : &p.X0;
                const int g = sg.group_base + t.group;
                for (int kb = 0; kb < sg.k_blocks; ++kb) {
                    const int s = L % S;
                    const uint32_t ph = (L / S) & 1u;
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, p.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = s0 + s * kStage;
                    mbar_arrive_expect_tx(full_bar(s), kStage);
                    if (GLU) {
                        tma_load_3d(st, mWa, full_bar(s), kb * 64, t.wt * 64, g);
                        tma_load_3d(st + kABytes / 2, mWb, full_bar(s), kb * 64, t.wt * 64, g);
                    } else {
                        tma_load_3d(st, mWa, full_bar(s), kb * 64, t.wt * 128, g);
                    }
                    tma_load_2d(st + kABytes, mX, full_bar(s), kb * 64, t.row0);
                    ++L;
                }
            }
            if (!ok) {
                raise_abort(p.err, abort_flag);
                for (uint32_t i = 0; i < (uint32_t)S && i < L; ++i) {
                    const uint32_t l = L - 1 - i;
                    mbar_wait(full_bar(l % S), (l / S) & 1u, kDrainNs, nullptr);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, N);
            uint32_t L = 0, n_acc = 0;
            bool ok = true, issued = false;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const Tile t = decode_tile<N>(p, tile, tiles0, s_offs, s_toffs);
                const SabSegment &sg = p.seg[t.seg];
                const uint32_t a = n_acc & 1u, aph = (n_acc >> 1) & 1u;
                if (!mbar_wait(tempty_bar(a), aph ^ 1u, p.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + a * N;
                for (int kb = 0; kb < sg.k_blocks; ++kb) {
                    const int s = L % S;
                    if (!mbar_wait(full_bar(s), (L / S) & 1u, p.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_k128(s0 + s * kStage);
                    const uint64_t bd = smem_desc_k128(s0 + s * kStage + kABytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) tc_mma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    issued = true;
                    tc_commit(empty_bar(s));
                    ++L;
                }
                if (!ok) break;
                tc_commit(tfull_bar(a));
                ++n_acc;
            }
            if (!ok) {
                raise_abort(p.err, abort_flag);
                if (issued) {
                    tc_commit(drain_bar);
                    mbar_wait(drain_bar, 0, kDrainNs, nullptr);
                }
            }
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int r = q * 32 + lane;  // TMEM lane = weight row of the tile
        uint32_t n_acc = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Tile t = decode_tile<N>(p, tile, tiles0, s_offs, s_toffs);
            const SabSegment &sg = p.seg[t.seg];
            const uint32_t a = n_acc & 1u, aph = (n_acc >> 1) & 1u;
            const bool ready = __all_sync(0xffffffffu, mbar_wait(tfull_bar(a), aph, p.wait_ns, abort_flag));
            // the four epilogue warps leave together (they share named barriers)
            if (!epi_all(ready)) {
                if (lane == 0) raise_abort(p.err, abort_flag);
                break;
            }
            tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + a * N;
            if (GLU) {
                float *x = xch + a * 64 * (N + 1);
                if (q >= 2) {  // up rows: hand over
#pragma unroll
                    for (int c0 = 0; c0 < N; c0 += 32) {
                        uint32_t v[32];
                        tmem_ld32(tb + c0, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[(r - 64) * (N + 1) + c0 + i] = __uint_as_float(v[i]);
                    }
                }
                epi_bar();
                if (q < 2) {  // gate rows: activation and store
                    const int col = t.wt * 64 + r;
                    const bool col_ok = col < sg.n_out;
#pragma unroll
                    for (int c0 = 0; c0 < N; c0 += 32) {
                        uint32_t v[32];
                        tmem_ld32(tb + c0, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int c = c0 + i;
                            if (col_ok && c < t.m_valid) {
                                const float h = glu_act(__uint_as_float(v[i]), x[r * (N + 1) + c], p.act,
                                                        p.alpha, p.limit, p.beta);
                                static_cast<bf16 *>(sg.out)[(size_t)(t.row0 + c) * sg.ldo + col] = __float2bfloat16_rn(h);
                            }
                        }
                    }
                }
            } else {
                const int col = t.wt * 128 + r;
                const bool col_ok = col < sg.n_out;
#pragma unroll
                for (int c0 = 0; c0 < N; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tb + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int c = c0 + i;
                        if (col_ok && c < t.m_valid)
                            static_cast<float *>(sg.out)[(size_t)(t.row0 + c) * sg.ldo + col] = __uint_as_float(v[i]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(tempty_bar(a));
            ++n_acc;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <bool GLU, int N>
int sab_smem(int stages) {
    return stages * (kABytes + N * 128) + (GLU ? 2 * 64 * (N + 1) * 4 : 0) + 1024 /*align*/ + 256 /*barriers*/;
}

template <bool GLU, int N>
int sab_stages() {
    int s = (kSmemMax - sab_smem<GLU, N>(0)) / (kABytes + N * 128);
    return s > kMaxStages ? kMaxStages : s;
}

template <bool GLU, int N>
cudaError_t launch_one(SabArgs a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(gemm_sab_kernel<GLU, N>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    });
    a.stages = sab_stages<GLU, N>();
    return launch_pdl(gemm_sab_kernel<GLU, N>, dim3(a.num_ctas), dim3(kThreads),
                      (size_t)sab_smem<GLU, N>(a.stages), s, a);
}

}  // namespace

cudaError_t launch_gemm_sab(const SabArgs &a, int n_tokens, cudaStream_t s) {
    if (a.glu) return n_tokens == 32 ? launch_one<true, 32>(a, s) : launch_one<true, 64>(a, s);
    return n_tokens == 32 ? launch_one<false, 32>(a, s) : launch_one<false, 64>(a, s);
}

}  // namespace moe
