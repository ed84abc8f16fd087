// Expert GEMMs on block-scaled (MX) weights for few tokens per expert, with the
// operands swapped and the weights decoded straight into tensor memory.
//
// The weights are OCP microscaling codes (E4M3 or E2M1) with one E8M0 scale per
// 32 consecutive input values of a row (the 4-bit and MXFP8 checkpoints of the
// Arcee AFMoE issue, "Checkpoint confirmed"); the activations stay bf16.  With m
// tokens per expert and m much smaller than 128, the weight rows are the MMA's
// M = 128 operand and the tokens a small N (32 or 64):
//
//   gate/up (glu = 1): D[128, N] = [Wg[g][i0:i0+64]; Wu[g][i0:i0+64]] . A[r0:r0+N]^T
//       TMEM lanes 0-63 gate, 64-127 up for the same 64 outputs i; the epilogue
//       warps of lanes 64-127 hand their values to those of lanes 0-63 through
//       shared memory, which apply the activation and store h[r][i0 + lane]
//   down    (glu = 0): D[128, N] = Wd[g][j0:j0+128] . h[r0:r0+N]^T
//
// tcgen05.mma takes its A operand from tensor memory here: thread r of the four
// converter warps owns TMEM lane r = weight row r of the tile, decodes the row's
// 64 codes of a k-block (and its two scales) in registers and writes the 32
// packed bf16 pairs with one tcgen05.st.  Shared memory then carries only the
// weight codes (1 or 1/2 byte per weight, via TMA) and the token rows, so the
// weight stream is not throttled by a shared-memory round trip of the decoded
// tile.  Decoding is exact (every decoded weight is a bf16 number unless the
// scale pushes it out of bf16's range, where it rounds to nearest), so the MMA
// multiplies the same bf16 values as the bf16 path would on decoded weights.
//
// Measured on GB300 (Nano decode, role timers): the kernel is bound by issuing its
// MMAs.  A 128 x 32 x 16 tcgen05.mma costs about 280 cycles to issue whatever its N,
// and with the weights as M one instruction covers 128 x 16 weights, half of what the
// grouped kernel's 128 x 256 x 16 (weights as N) covers; converter count, TMEM depth,
// code width (MXFP8 or MXFP4) and the number of copies per k-block leave the time
// unchanged.  It stays selectable (MOE_OPT_PATH 3) and exact; the auto path takes the
// grouped kernel.
//
// One CTA per SM, static round-robin over tiles (segment, group, weight tile,
// token tile), 14 warps:
//   warp 0     TMA: per tile the scales of its 128 weight rows (all of K, into one of
//              two tile buffers); per k-block stage the N token rows (bf16, 128-byte
//              swizzle) and the tile's codes (128 rows x 64 values)
//   warp 1     tcgen05.mma issue (kind::f16, A from TMEM, B from shared memory)
//   warps 2-5  epilogue (TMEM accumulators -> activation -> bf16 stores)
//   warps 6-   converters (one weight row per thread), kConvSets sets of four
// Every wait is bounded: on timeout the kernel records ERR_TIMEOUT, stops every
// role, drains its copies and MMAs and returns.
#include <cuda_fp16.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// converter warps: kConvSets sets of four (one per TMEM lane quadrant); set c decodes
// the k-blocks L with L % kConvSets == c, so one set's decode overlaps the other's
// tensor-memory stores and barrier hand-over
constexpr int kConvSets = 2;
constexpr int kConvWarps = 4;  // converter warps arriving per k-block (one set)
constexpr int kThreads = 32 * (6 + 4 * kConvSets);
// TMEM A buffers, one k-block (32 columns) each: the k-blocks a decoded A may run ahead
// of the MMA (each buffer's round trip is decode, tensor-memory store, MMA, commit)
constexpr int kAStages = 8;
constexpr int kMaxStages = 12;
constexpr int kSmemMax = 232448 - 4096;  // dynamic budget; the rest holds the static offset tables
constexpr uint64_t kDrainNs = 1000000000ull;

template <int WF>
struct MxtCfg {
    static constexpr int kRawRow = WF == kWeightsMxfp8 ? 64 : 32;  // code bytes of one row's k-block
    static constexpr int kCodes = 128 * kRawRow;
};

template <int WF, int N>
__host__ __device__ constexpr int mxt_stage_bytes() {
    return (N * 128 + MxtCfg<WF>::kCodes + 1023) / 1024 * 1024;
}

struct Tile {
    int seg, group, wt, nt, row0, m_valid;
};

template <int N>
__device__ __forceinline__ int seg_tiles(const SabSegment &s, const int *toffs) {
    if (s.dense) return ((s.m_dense + N - 1) / N) * s.w_tiles;
    return toffs[s.num_groups] * s.w_tiles;
}

// token tiles (nt) of one weight tile (wt) are adjacent
template <int N>
__device__ __forceinline__ Tile decode_tile(const MxtArgs &p, int tile, int tiles0, const int *offs,
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

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
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

// ------------------------------------------------------------ decoding
// f16x2 of two MX codes (hardware unpack) -> the bits of bf16x2 of value * 2^-112:
// every E4M3 / E2M1 value is a normal f16 (or zero) whose low 7 mantissa bits are
// zero, so dropping 3 bits keeps sign, exponent field and mantissa; one bf16x2
// multiply by 2^(scale - 15) then applies the E8M0 scale 2^(scale - 127).
__device__ __forceinline__ uint32_t f16x2_as_bf16x2_scaled(uint32_t h) {
    return ((h & 0x7fff7fffu) >> 3) | (h & 0x80008000u);
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t pair16) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)pair16));
    return h;
}
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte) {
    uint32_t h;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(byte));
    return h;
}
// 2^(code - 127) for an E8M0 code (255: NaN; 0: 2^-127, an fp32 subnormal)
__device__ __forceinline__ float e8m0_f32(uint32_t code) {
    if (code == 0u) return __uint_as_float(0x00400000u);
    if (code == 255u) return __uint_as_float(0x7fc00000u);
    return __uint_as_float(code << 23);
}
// one word: the f16x2 pair h scaled by an E8M0 code; fast: the code's multiplier is a
// normal bf16 (code + 112 <= 254), so one bf16x2 multiply is exact where representable
template <bool FAST>
__device__ __forceinline__ uint32_t scaled_pair(uint32_t h, uint32_t code) {
    if (FAST) return bf16x2_mul(f16x2_as_bf16x2_scaled(h), ((code + 112u) << 7) * 0x00010001u);
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    const float s = e8m0_f32(code);
    return pack_bf16x2(f.x * s, f.y * s);
}

template <int WF, bool FAST>
__device__ __forceinline__ void decode_row_as(const uint8_t *codes, uint32_t s0, uint32_t s1, uint32_t (&w)[32]) {
    if (WF == kWeightsMxfp8) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // 16 codes: values 16q .. 16q + 15
            const uint4 v = *reinterpret_cast<const uint4 *>(codes + 16 * q);
            const uint32_t s = q < 2 ? s0 : s1;
            const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w[8 * q + 2 * i] = scaled_pair<FAST>(e4m3x2_f16x2(x[i]), s);
                w[8 * q + 2 * i + 1] = scaled_pair<FAST>(e4m3x2_f16x2(x[i] >> 16), s);
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < 2; ++q) {  // 16 bytes: values 32q .. 32q + 31, two per byte
            const uint4 v = *reinterpret_cast<const uint4 *>(codes + 16 * q);
            const uint32_t s = q == 0 ? s0 : s1;
            const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    w[16 * q + 4 * i + b] = scaled_pair<FAST>(e2m1x2_f16x2((x[i] >> (8 * b)) & 0xffu), s);
        }
    }
}

// Row r's k-block: 64 values -> 32 words (word i = values 2i, 2i+1, the lower K in
// the low half), values 0-31 scaled by code s0, 32-63 by s1.
template <int WF>
__device__ __forceinline__ void decode_row(const uint8_t *codes, uint32_t s0, uint32_t s1, uint32_t (&w)[32]) {
    if (s0 + 112u <= 254u && s1 + 112u <= 254u)
        decode_row_as<WF, true>(codes, s0, s1, w);
    else
        decode_row_as<WF, false>(codes, s0, s1, w);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
        " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
        " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, fp32 accumulation; issued by one thread.
__device__ __forceinline__ void tc_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

template <bool GLU, int WF, int N>
__global__ void __launch_bounds__(kThreads, 1) gemm_mxt_kernel(const __grid_constant__ MxtArgs p) {
    using M = MxtCfg<WF>;
    constexpr int kStage = mxt_stage_bytes<WF, N>();
    constexpr int kTok = N * 128;                    // token rows of one k-block
    constexpr uint32_t kTxBytes = kTok + M::kCodes;
    constexpr uint32_t kAcol = 2 * N;                // first TMEM column of the A buffers
    constexpr uint32_t kTmemCols = 2 * N + kAStages * 32 <= 256 ? 256 : 512;
    static_assert(2 * N + kAStages * 32 <= 512, "accumulators and A buffers fit tensor memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    const uint32_t s0 = smem_u32(smem);
    // per-tile scale buffers [2]: gate/up [gate | up][K/32][64 rows], down [K/32][128 rows]
    const int sbuf = 128 * p.sblk;
    uint8_t *sbufs = smem + S * kStage;
    float *xch = reinterpret_cast<float *>(sbufs + 2 * sbuf);  // [2][64][N + 1] (gate/up)
    uint8_t *misc = sbufs + 2 * sbuf + (GLU ? 2 * 64 * (N + 1) * 4 : 0);
    uint64_t *bars = reinterpret_cast<uint64_t *>(misc);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    auto afull_bar = [&](int s) { return bar0 + 8u * (2 * kMaxStages + s); };
    auto aempty_bar = [&](int s) { return bar0 + 8u * (2 * kMaxStages + kAStages + s); };
    auto tfull_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kMaxStages + 2 * kAStages + a); };
    auto tempty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kMaxStages + 2 * kAStages + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kMaxStages + 2 * kAStages + 4);
    auto sfull_bar = [&](uint32_t b) { return bar0 + 8u * (2 * kMaxStages + 2 * kAStages + 5 + b); };
    auto sempty_bar = [&](uint32_t b) { return bar0 + 8u * (2 * kMaxStages + 2 * kAStages + 7 + b); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kMaxStages + 2 * kAStages + 9);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1 + kConvWarps);  // the MMA's commit and each converter warp
        }
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(afull_bar(s), kConvWarps);
            mbar_init(aempty_bar(s), 1);
        }
        for (uint32_t a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 128);
        }
        mbar_init(drain_bar, 1);
        for (uint32_t b = 0; b < 2; ++b) {
            mbar_init(sfull_bar(b), 1);
            mbar_init(sempty_bar(b), 4 * kConvSets);  // every converter warp, at the end of each tile
        }
        fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.Wa0);
        tma_prefetch_desc(&p.Sa0);
        if (GLU) {
            tma_prefetch_desc(&p.Wb0);
            tma_prefetch_desc(&p.Sb0);
        }
        tma_prefetch_desc(&p.X0);
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
            uint32_t L = 0, n_tile = 0;
            uint64_t w_empty = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const Tile t = decode_tile<N>(p, tile, tiles0, s_offs, s_toffs);
                const SabSegment &sg = p.seg[t.seg];
                const CUtensorMap *mWa = t.seg ? &p.Wa1 : &p.Wa0, *mWb = t.seg ? &p.Wb1 : &p.Wb0;
                const CUtensorMap *mSa = t.seg ? &p.Sa1 : &p.Sa0, *mSb = t.seg ? &p.Sb1 : &p.Sb0;
                const CUtensorMap *mX = t.seg ? &p.X1 : &p.X0;
                const int g = sg.group_base + t.group;
                const int rows0 = GLU ? t.wt * 64 : t.wt * 128;
                // the tile's scales: every 32-value block of its rows, one copy per half
                const uint32_t tb = n_tile & 1u;
                if (!mbar_wait(sempty_bar(tb), ((n_tile >> 1) & 1u) ^ 1u, p.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                const int nblk = 2 * sg.k_blocks;
                const uint32_t sd = smem_u32(sbufs + tb * sbuf);
                mbar_arrive_expect_tx(sfull_bar(tb), 128u * nblk);
                tma_load_3d(sd, mSa, sfull_bar(tb), rows0, 0, g);
                if (GLU) tma_load_3d(sd + 64 * nblk, mSb, sfull_bar(tb), rows0, 0, g);
                ++n_tile;
                for (int kb = 0; kb < sg.k_blocks; ++kb) {
                    const int s = L % S;
                    const uint64_t t0 = p.stats ? global_timer_ns() : 0;
                    if (!mbar_wait(empty_bar(s), ((L / S) & 1u) ^ 1u, p.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (p.stats) w_empty += global_timer_ns() - t0;
                    const uint32_t st = s0 + s * kStage, codes = st + kTok;
                    const int xb = WF == kWeightsMxfp8 ? kb * 64 : kb * 32;  // byte of the k-block in a code row
                    mbar_arrive_expect_tx(full_bar(s), kTxBytes);
                    tma_load_2d(st, mX, full_bar(s), kb * 64, t.row0);
                    tma_load_3d(codes, mWa, full_bar(s), xb, rows0, g);
                    if (GLU) tma_load_3d(codes + 64 * M::kRawRow, mWb, full_bar(s), xb, rows0, g);
                    ++L;
                }
            }
            if (!ok) {
                raise_abort(p.err, abort_flag);
                for (uint32_t i = 0; i < (uint32_t)S && i < L; ++i) {
                    const uint32_t l = L - 1 - i;
                    mbar_wait(full_bar(l % S), (l / S) & 1u, kDrainNs, nullptr);
                }
                for (uint32_t i = 0; i < 2u && i < n_tile; ++i) {  // scale copies in flight
                    const uint32_t n = n_tile - 1 - i;
                    mbar_wait(sfull_bar(n & 1u), (n >> 1) & 1u, kDrainNs, nullptr);
                }
            }
            if (p.stats) atomicAdd(p.stats + 0, (unsigned long long)w_empty);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, N);
            uint32_t L = 0, n_acc = 0;
            uint64_t w_ops = 0, w_acc = 0;
            bool ok = true, issued = false;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const Tile t = decode_tile<N>(p, tile, tiles0, s_offs, s_toffs);
                const SabSegment &sg = p.seg[t.seg];
                const uint32_t a = n_acc & 1u, aph = (n_acc >> 1) & 1u;
                const uint64_t t0 = p.stats ? global_timer_ns() : 0;
                if (!mbar_wait(tempty_bar(a), aph ^ 1u, p.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                if (p.stats) w_acc += global_timer_ns() - t0;
                tc_fence_after();
                const uint32_t d = tmem_base + a * N;
                for (int kb = 0; kb < sg.k_blocks; ++kb) {
                    const int s = L % S, sa = L % kAStages;
                    const uint64_t t1 = p.stats ? global_timer_ns() : 0;
                    if (!mbar_wait(full_bar(s), (L / S) & 1u, p.wait_ns, abort_flag) ||
                        !mbar_wait(afull_bar(sa), (L / kAStages) & 1u, p.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (p.stats) w_ops += global_timer_ns() - t1;
                    tc_fence_after();
                    const uint64_t bd = smem_desc_k128(s0 + s * kStage);
                    const uint32_t at = tmem_base + kAcol + sa * 32;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) tc_mma_bf16_ta(d, at + 8 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    issued = true;
                    tc_commit(aempty_bar(sa));
                    tc_commit(empty_bar(s));
                    ++L;
                }
                if (!ok) break;
                tc_commit(tfull_bar(a));
                ++n_acc;
            }
            if (p.stats) {
                atomicAdd(p.stats + 3, (unsigned long long)w_ops);
                atomicAdd(p.stats + 4, (unsigned long long)w_acc);
                atomicAdd(p.stats + 7, (unsigned long long)n_acc);
            }
            if (!ok) {
                raise_abort(p.err, abort_flag);
                if (issued) {
                    tc_commit(drain_bar);
                    mbar_wait(drain_bar, 0, kDrainNs, nullptr);
                }
            }
        }
    } else if (warp >= 6) {
        // -------------------------------------------------------- converters
        const int q = warp & 3, r = q * 32 + lane;  // TMEM lane = weight row of the tile
        const int set = (warp - 6) >> 2;
        uint32_t L = 0, n_tile = 0;
        uint64_t w_full = 0, w_aempty = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++n_tile) {
            const Tile t = decode_tile<N>(p, tile, tiles0, s_offs, s_toffs);
            const int kbs = p.seg[t.seg].k_blocks;
            const uint32_t tb = n_tile & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(sfull_bar(tb), (n_tile >> 1) & 1u, p.wait_ns, abort_flag))) {
                if (lane == 0) raise_abort(p.err, abort_flag);
                break;
            }
            // this row's scales in the tile buffer: block b at sc[b * sstep]
            const int nblk = 2 * kbs;
            const uint8_t *sc = sbufs + tb * sbuf + (GLU ? (r >> 6) * 64 * nblk + (r & 63) : r);
            const int sstep = GLU ? 64 : 128;
            for (int kb = 0; kb < kbs; ++kb, ++L) {
                if ((int)(L % kConvSets) != set) continue;
                const int s = L % S, sa = L % kAStages;
                const uint64_t t0 = p.stats ? global_timer_ns() : 0;
                bool got = __all_sync(0xffffffffu, mbar_wait(full_bar(s), (L / S) & 1u, p.wait_ns, abort_flag));
                const uint64_t t1 = p.stats ? global_timer_ns() : 0;
                got = got && __all_sync(0xffffffffu, mbar_wait(aempty_bar(sa), ((L / kAStages) & 1u) ^ 1u,
                                                               p.wait_ns, abort_flag));
                if (p.stats) {
                    w_full += t1 - t0;
                    w_aempty += global_timer_ns() - t1;
                }
                if (!got) {
                    if (lane == 0) raise_abort(p.err, abort_flag);
                    ok = false;
                    break;
                }
                const uint8_t *codes = smem + s * kStage + kTok;
                uint32_t w[32];
                decode_row<WF>(codes + r * M::kRawRow, sc[2 * kb * sstep], sc[(2 * kb + 1) * sstep], w);
                tc_fence_after();
                tmem_st32(tmem_base + ((uint32_t)(q * 32) << 16) + kAcol + sa * 32, w);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(afull_bar(sa));
                    mbar_arrive(empty_bar(s));
                }
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(sempty_bar(tb));  // this warp has read the tile's scales
        }
        if (p.stats && lane == 0) {
            atomicAdd(p.stats + 1, (unsigned long long)w_full);
            atomicAdd(p.stats + 2, (unsigned long long)w_aempty);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int r = q * 32 + lane;  // TMEM lane = weight row of the tile
        uint32_t n_acc = 0;
        uint64_t w_tfull = 0, w_work = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Tile t = decode_tile<N>(p, tile, tiles0, s_offs, s_toffs);
            const SabSegment &sg = p.seg[t.seg];
            const uint32_t a = n_acc & 1u, aph = (n_acc >> 1) & 1u;
            const uint64_t t0 = p.stats ? global_timer_ns() : 0;
            const bool ready = __all_sync(0xffffffffu, mbar_wait(tfull_bar(a), aph, p.wait_ns, abort_flag));
            const uint64_t t1 = p.stats ? global_timer_ns() : 0;
            w_tfull += t1 - t0;
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
                                const float h = glu_act(__uint_as_float(v[i]), x[r * (N + 1) + c], p.act, p.alpha,
                                                        p.limit, p.beta);
                                static_cast<bf16 *>(sg.out)[(size_t)(t.row0 + c) * sg.ldo + col] = __float2bfloat16_rn(h);
                            }
                        }
                    }
                }
                epi_bar();  // the exchange buffer of this accumulator is read before its next use
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
            if (p.stats) w_work += global_timer_ns() - t1;
            ++n_acc;
        }
        if (p.stats && q == 0 && lane == 0) {
            atomicAdd(p.stats + 5, (unsigned long long)w_tfull);
            atomicAdd(p.stats + 6, (unsigned long long)w_work);
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

template <bool GLU, int WF, int N>
int mxt_smem(int stages) {
    return stages * mxt_stage_bytes<WF, N>() + (GLU ? 2 * 64 * (N + 1) * 4 : 0) + 1024 /*align*/ + 512 /*barriers*/;
}

template <bool GLU, int WF, int N>
int mxt_stages(int sblk) {
    int s = (kSmemMax - mxt_smem<GLU, WF, N>(0) - 2 * 128 * sblk) / mxt_stage_bytes<WF, N>();
    return s > kMaxStages ? kMaxStages : s;
}

template <bool GLU, int WF, int N>
cudaError_t launch_one(MxtArgs a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(gemm_mxt_kernel<GLU, WF, N>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    });
    if (a.sblk < 2 || a.sblk > 256) return cudaErrorInvalidValue;
    a.stages = mxt_stages<GLU, WF, N>(a.sblk);
    if (a.stages < 2) return cudaErrorInvalidValue;
    return launch_pdl(gemm_mxt_kernel<GLU, WF, N>, dim3(a.num_ctas), dim3(kThreads),
                      (size_t)(mxt_smem<GLU, WF, N>(a.stages) + 2 * 128 * a.sblk), s, a);
}

template <int WF>
cudaError_t launch_wf(const MxtArgs &a, int n_tokens, cudaStream_t s) {
    if (a.glu) return n_tokens == 32 ? launch_one<true, WF, 32>(a, s) : launch_one<true, WF, 64>(a, s);
    return n_tokens == 32 ? launch_one<false, WF, 32>(a, s) : launch_one<false, WF, 64>(a, s);
}

}  // namespace

cudaError_t launch_gemm_mxt(const MxtArgs &a, int n_tokens, cudaStream_t s) {
    if (n_tokens != 32 && n_tokens != 64) return cudaErrorInvalidValue;
    if (a.wfmt == kWeightsMxfp8) return launch_wf<kWeightsMxfp8>(a, n_tokens, s);
    if (a.wfmt == kWeightsMxfp4) return launch_wf<kWeightsMxfp4>(a, n_tokens, s);
    return cudaErrorInvalidValue;
}

}  // namespace moe
