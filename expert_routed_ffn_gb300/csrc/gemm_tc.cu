// Grouped GEMMs of the expert MLPs on the 5th-generation tensor cores (K3, K4, K5).
//
//   gate/up (glu = 1):  H_out[r, i] = act( A[r,:] . Wg[g][i,:],  A[r,:] . Wu[g][i,:] )
//   down    (glu = 0):  Y_out[r, j] = A[r,:] . Wd[g][j,:]
//
// One launch covers up to four segments: the routed experts (rows grouped by
// expert through the dispatch offsets, weight slice = expert id) and the
// shared expert (all T token rows, one weight slice), for the gate/up
// projection, the down projection, or both.  Weights are the pre-stacked
// [groups, out, in] tensors (Arcee AFMoE issue, "Checkpoint weight layout";
// the packed shared expert of the MiniMax-M3 issue is slice E).  When both
// projections share a launch, a down tile first waits until every gate/up
// tile of its 128 rows has been stored (a per-m-tile counter), so the down
// tiles of early experts overlap the gate/up tail and the second launch's ramp
// disappears.  Gate/up tiles never wait, tiles are claimed in increasing
// order, and each CTA's roles take its tiles in claim order with all CTAs
// resident (one per SM): a down tile only waits for tiles claimed before it,
// which do not wait, so the waits end.
//
// CTA pairs (256-row m-tiles): an expert's m-tile of at most 128 rows (its last, or
// its only one) runs with the operands swapped, the pair's 256 weight rows as M and
// the tile's rows, rounded up to 32, as N: each CTA loads half of those token rows
// and 128 weight rows (a gate/up tile: 64 gate and 64 up rows of the same 64
// features), and the MMA skips most of the padding rows that a 256-row token tile
// would carry.  Each output is the same K-ordered sum of the same products, so the
// results are bit-identical to the unswapped tile (tested).  Measured on GB300:
// AFMoE prefill 552 against 571 us, Zipf T = 4096 575 against 595 us; a bound of 64
// or 96 rows instead of 128 is slower.
//
// Persistent kernel, one CTA per SM, 6 warps:
//   warp 0     TMA producer: A tile 128 x 64 and B tile 256 x 64 (gate/up: 128
//              gate rows + 128 up rows) per stage, 128-byte swizzle, 4 stages
//   warp 1     allocates 512 TMEM columns; lane 0 issues tcgen05.mma
//              (M 128, N 256, K 16, bf16 in, fp32 accumulate) into one of two
//              TMEM accumulators, so the epilogue of one tile overlaps the
//              main loop of the next
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//              32*(w%4)..+31 = tile rows), activation, bf16 rows (gate/up) or fp32
//              rows (down projections); 128-row and CTA-pair tiles stage each
//              32-row slice in shared memory and write it with one TMA store
//              (measured on GB300: AFMoE prefill 549 -> 525 us against a 16-byte
//              store per lane and row), thin tiles store from registers
// Tiles are (segment, group, m-tile, n-tile) in a fixed order; the producer
// claims them from a launch-wide ticket (the CTA that is free first takes the
// next tile) and passes each id to the MMA and epilogue warps through a ring
// in shared memory.  Inside a group the m-tiles of one n-tile are adjacent so
// concurrent CTAs share the weight tile in L2.  Every wait is bounded: on timeout the kernel records
// ERR_TIMEOUT, stops all roles, drains its in-flight copies and MMAs, frees
// TMEM and returns.
#include <cuda_fp16.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kABytes = kGemmBM * kGemmBK * 2;  // 16 KB
// Epilogue warps: kEpiParts per TMEM lane quadrant, each a 1/kEpiParts slice of the
// tile's columns (measured: 4 warps are as fast as 8 at decode sizes and 1% faster
// at prefill, with the fast activation below)
constexpr int kEpiParts = 1;
constexpr int kEpiWarps = 4 * kEpiParts;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;     // warp 0 TMA, warp 1 MMA, then the epilogue warps
constexpr uint32_t kTmemCols = 512;             // two 128 x 256 fp32 accumulators
constexpr uint64_t kDrainNs = 1000000000ull;    // bound of the drain after an abort
constexpr uint64_t kPairDrainNs = 1000000ull;   // CTA pair: grace for the copies in flight after an abort
constexpr int kRing = 8;                        // tile ids in flight from the producer to the other roles
// CTA pairs: the last waves of tiles are claimed, not assigned.  Measured on GB300 (step
// us, static order / 1 / 2 / 4 claimed waves): AFMoE prefill 547 / 542.5 / 542.9 / 545.3,
// Zipf T = 4096 571 / 564.7 / 566.2 / 563.8, T = 16384 1820 / 1792 / 1788 / 1791; a fully
// claimed order keeps fewer weight tiles shared in L2 (578 us on AFMoE prefill).
constexpr int kTailWaves = 2;

// Per-variant layout.  One CTA: stage = one k-block of 64, A 128 x 64 + B
// 256 x 64 (48 KB), 4 stages.  CTA pair: each CTA stages its own 128 A rows and
// half of B (128 rows), two k-blocks per stage loaded as one box each (A and B
// 32 KB: larger copies keep a CTA's TMA stream near the MMA's rate), 3 stages;
// a tile is 256 rows (128 per CTA).  A stage holds kKB consecutive 16 KB
// (A) and kBBytes / kKB (B) k-block tiles.
// THIN (one CTA, decode sizes): tiles of kThinRows = 32 rows (the dispatch counts
// 32-row m-tiles), A rows in boxes of 32 rows (4 KB), so six stages of 36 KB keep
// 192 KB of weights in flight instead of 128 KB; the MMA still reads 128 rows of A,
// the rows past the box being whatever shared memory follows (their outputs are
// never stored).
constexpr int kThinRows = 32;
template <bool PAIR, bool THIN = false>
struct GemmCfg {
    static constexpr int kKB = PAIR ? 2 : 1;     // k-blocks per stage
    static constexpr int kStages = PAIR ? 3 : (THIN ? 6 : 4);
    static constexpr int kBBytes = (PAIR ? kGemmBN / 2 : kGemmBN) * kGemmBK * 2 * kKB;
    static constexpr int kAStage = (THIN ? kThinRows * kGemmBK * 2 : kABytes) * kKB;
    static constexpr int kStageBytes = kAStage + kBBytes;
    // CTA pairs: the gate values' hand-over buffer of swapped gate/up tiles, 2 x 32 x 32 fp32
    static constexpr int kXBufBytes = PAIR ? 8192 : 0;
    // the epilogue's store staging: one [32 rows][128 bytes] slice per TMEM lane quadrant,
    // 1024-byte aligned.  Thin tiles store from registers: their one quadrant of rows is
    // mostly partial, and staging it measured slower (Nano decode 68.6 -> 74.4 us)
    static constexpr int kEpiOff = (kStages * kStageBytes + 512 + kXBufBytes + 1023) / 1024 * 1024;
    static constexpr int kEpiBufBytes = THIN ? 0 : 4 * 4096;
    static constexpr int kSmemBytes = kEpiOff + kEpiBufBytes + 1024 /*align*/;
    static constexpr int kBM = PAIR ? 2 * kGemmBM : (THIN ? kThinRows : kGemmBM);  // rows per tile
};

struct Tile {
    int seg, group, mt, nt, ks, row0, m_valid, ready;  // ks: K range; row0, m_valid: this CTA's rows;
                                                       // ready: its m-tile's counter
    int swp;  // swapped operands (CTA pairs): row0, m_valid = the whole m-tile's rows
};

// Swapped-operand tiles of a CTA pair: the MMA's N (token columns, a multiple of 32,
// half of them in each CTA's shared memory) and the rows of the token box each CTA loads.
__device__ __forceinline__ int swap_n(int rows) { return (rows + 31) / 32 * 32; }
__device__ __forceinline__ int swap_box(int rows) { return swap_n(rows) / 2 <= 32 ? 32 : 64; }

// offs / toffs: shared-memory copies of the grouped segments' dispatch offsets
// (toffs counts tiles of BM rows)
template <int BM>
__device__ __forceinline__ int seg_tiles(const GemmSegment &s, const int *toffs) {
    if (s.dense) return ((s.m_dense + BM - 1) / BM) * s.n_tiles * max(s.k_splits, 1);
    return toffs[s.num_groups] * s.n_tiles;
}

// The launch's segments, copied from the kernel parameters into shared memory when
// a kernel of this file starts (load_segments): every role reads them per tile, and a
// parameter read that misses the constant cache costs about a microsecond under load.
__shared__ GemmSegment s_seg[kGemmMaxSegments];
__device__ __forceinline__ void load_segments(const GemmArgs &p) {
    static_assert(sizeof(GemmSegment) % 4 == 0, "segments copied as words");
    constexpr int kWords = (int)(sizeof(GemmSegment) * kGemmMaxSegments / 4);
    const int *src = reinterpret_cast<const int *>(p.seg);
    int *dst = reinterpret_cast<int *>(s_seg);
    for (int i = threadIdx.x; i < kWords; i += blockDim.x) dst[i] = src[i];
}

// Tile -> segment, group, m-tile, n-tile.  With CTA pairs (BM = 256) the CTA of
// cluster rank `half` takes rows [128 * half, 128 * half + 128) of the tile, and
// the per-128-row counters are numbered 2 * m-tile + half.
template <int BM>
__device__ __forceinline__ Tile decode_tile(const GemmArgs &p, int tile, const int *seg_end, const int *offs,
                                            const int *toffs, int half) {
    Tile t;
    t.seg = 0;
    t.swp = 0;
    while (t.seg + 1 < p.num_segs && tile >= seg_end[t.seg]) ++t.seg;
    if (t.seg > 0) tile -= seg_end[t.seg - 1];
    const GemmSegment &s = s_seg[t.seg];
    constexpr int kRows = BM < kGemmBM ? BM : kGemmBM;  // rows of a tile per CTA
    constexpr int kSub = BM / kRows;                    // CTA parts of a tile (2 with CTA pairs)
    if (s.dense) {
        const int mtiles = (s.m_dense + BM - 1) / BM;
        t.group = 0;
        t.ks = tile / (mtiles * s.n_tiles);
        tile -= t.ks * mtiles * s.n_tiles;
        t.nt = tile / mtiles;
        t.mt = tile % mtiles;
        t.row0 = t.mt * BM + half * kRows;
        t.m_valid = min(kRows, s.m_dense - t.row0);
        t.ready = s.ready_base + kSub * t.mt + half;
    } else {
        // largest group whose first tile is <= tile (empty groups own no tiles)
        int lo = 0, hi = s.num_groups - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (toffs[mid] * s.n_tiles <= tile)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int mt_g = toffs[lo + 1] - toffs[lo];
        const int local = tile - toffs[lo] * s.n_tiles;
        t.group = lo;
        t.ks = 0;
        t.nt = local / mt_g;
        t.mt = local % mt_g;
        const int start = offs[lo];
        const int rows = min(BM, offs[lo + 1] - (start + t.mt * BM));  // of the m-tile
        if (kSub == 2 && p.swap_rem && rows <= kSwapMaxRows) {
            // weights as M, the m-tile's rows as N: both CTAs' outputs cover all its rows
            t.swp = 1;
            t.row0 = start + t.mt * BM;
            t.m_valid = rows;
        } else {
            t.row0 = start + t.mt * BM + half * kRows;
            t.m_valid = min(kRows, offs[lo + 1] - t.row0);  // <= 0: the odd CTA of a pair past the group's rows
        }
        t.ready = s.ready_base + kSub * (toffs[lo] + t.mt) + half;
    }
    return t;
}

__device__ __forceinline__ void raise_abort(int *err, volatile int *abort_flag) {
    if (err != nullptr) atomicOr(err, ERR_TIMEOUT);
    *abort_flag = 1;
}
// CTA pair: also stop the other CTA's roles
__device__ __forceinline__ void raise_abort_pair(int *err, volatile int *abort_flag) {
    raise_abort(err, abort_flag);
    const uint32_t peer = mapa_shared(smem_u32(const_cast<int *>(abort_flag)), cluster_ctarank() ^ 1u);
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer), "r"(1u) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait (bounded, like mbar_wait) until *p >= target.
__device__ __forceinline__ bool wait_counter(const int *p, int target, uint64_t limit_ns, volatile int *abort) {
    if (ld_acquire(p) >= target) return true;
    if (limit_ns == 0) return false;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        __nanosleep(64);
        if (ld_acquire(p) >= target) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// Named barrier 1 of the four epilogue warps; and the AND of v over them.
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v), "n"(kEpiThreads)
        : "memory");
    return out != 0;
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async;" ::: "memory"); }
// the same ordering for this thread's shared-memory stores only (operands the MMA reads)
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}


// Barrier addresses and shared state the epilogue warps use (every kernel lays
// out ring_full[kRing], ring_empty[kRing], tfull[2], tempty[2] contiguously).
struct EpiCtx {
    uint32_t ring_full0, ring_empty0, tfull0, tempty0;
    volatile int *ring;
    volatile int *abort_flag;
    uint32_t tmem_base;
    int total;
    const int *s_seg_end, *s_offs, *s_toffs;
    int half;
    float *xbuf;  // CTA pairs: [2][32][32] hand-over of swapped gate/up tiles
    // store staging, [ebuf_quads][32 rows][128 bytes] (quadrant q uses slice q % ebuf_quads);
    // 0: none, every row stored from registers
    uint32_t ebuf;
    int ebuf_quads;
};

// One warp's staged store of a [32 rows][128 bytes] slice: lane i has written row i into
// its 128-byte-swizzled staging buffer `sb` (16-byte unit j at j ^ (i % 8)).  All 32 rows
// valid: one TMA store of the box at (x, y) by lane 0.  Fewer (`rows`): 16-byte stores
// of the valid rows, eight lanes per row, row i at `dst + i * ld_bytes` (coalesced).
__device__ __forceinline__ void epi_flush(const CUtensorMap *map, uint32_t sb, int rows, int x, int y, char *dst,
                                          size_t ld_bytes, int lane) {
    if (rows == 32) {
        fence_proxy_async_smem();  // the rows' generic writes -> the TMA's reads
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(map, sb, x, y);
            bulk_commit();
        }
    } else {
        __syncwarp();
        const int u = lane & 7;
        for (int i = lane >> 3; i < rows; i += 4) {
            uint4 v;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(sb + (uint32_t)i * 128u + ((uint32_t)(u ^ (i & 7)) << 4)));
            *reinterpret_cast<uint4 *>(dst + (size_t)i * ld_bytes + 16 * u) = v;
        }
        __syncwarp();  // the buffer is read before the next slice overwrites it
    }
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Epilogue role (kEpiWarps warps, named barrier 1): for each tile id from the
// ring, wait for its accumulator, apply the activation and store bf16 rows
// (gate/up) or store the fp32 rows (down projections), release the accumulator, and publish the m-tile's completion.  HALVES = 2:
// 256-row tiles in one CTA, one accumulator of 2 x 256 columns (half h's rows in
// columns 256 h ..), no second buffer.
template <bool PAIR, int kBM, int HALVES = 1>
__device__ __forceinline__ void epilogue_role(const GemmArgs &p, const EpiCtx &c, int warp, int lane) {
    auto ring_full = [&](int i) { return c.ring_full0 + 8u * i; };
    auto ring_empty = [&](int i) { return c.ring_empty0 + 8u * i; };
    auto tfull_bar = [&](uint32_t a) { return c.tfull0 + 8u * a; };
    auto tempty_bar = [&](uint32_t a) { return c.tempty0 + 8u * a; };
    volatile int *ring = c.ring;
    volatile int *abort_flag = c.abort_flag;
    const uint32_t tmem_base = c.tmem_base;
    const int total = c.total, half = c.half;
    const int *s_seg_end = c.s_seg_end, *s_offs = c.s_offs, *s_toffs = c.s_toffs;
    unsigned long long *const stats = p.stats;
    const int act = p.act;  // loop-invariant: read the parameters once
    const float alpha = p.alpha, limit = p.limit, beta = p.beta;
    auto abort_all = [&]() {
        if (PAIR)
            raise_abort_pair(p.err, abort_flag);
        else
            raise_abort(p.err, abort_flag);
    };
    const int q = warp & 3;               // TMEM lane quadrant this warp may read
    const int part = (warp - 2) / 4;      // which slice of the tile's columns
    const bool lead_thread = q == 0 && part == 0 && lane == 0;
    const int r = q * 32 + lane;
    uint32_t n_acc = 0;
    uint64_t w_tfull = 0, w_work = 0;
    for (int n = 0;; ++n) {
        const int slot = n % kRing;
        const uint64_t t0 = stats ? global_timer_ns() : 0;
        const bool have = __all_sync(0xffffffffu, mbar_wait(ring_full(slot), (n / kRing) & 1u, p.wait_ns, abort_flag));
        const int tile = have ? ring[slot] : total;
        // all four epilogue warps agree to go on or stop (they share barrier 1), and
        // have read the id before it is released; the tcgen05.ld below is .sync.aligned
        if (!epi_all(have)) {
            if (lane == 0) abort_all();
            break;
        }
        if (lead_thread) mbar_arrive(ring_empty(slot));
        if (tile >= total) break;
        const Tile tile0 = decode_tile<kBM>(p, tile, s_seg_end, s_offs, s_toffs, HALVES == 2 ? 0 : half);
        const GemmSegment &sg = s_seg[tile0.seg];
        const uint32_t a = HALVES == 2 ? 0u : n_acc & 1u, aph = HALVES == 2 ? n_acc & 1u : (n_acc >> 1) & 1u;
        const bool ready = __all_sync(0xffffffffu, PAIR ? mbar_wait_cluster(tfull_bar(a), aph, p.wait_ns, abort_flag)
                                                        : mbar_wait(tfull_bar(a), aph, p.wait_ns, abort_flag));
        const uint64_t t1 = stats ? global_timer_ns() : 0;
        w_tfull += t1 - t0;
        if (!epi_all(ready)) {
            if (lane == 0) abort_all();
            break;
        }
        tc_fence_after();
        if (PAIR && tile0.swp) {
            // Swapped operands: TMEM lane r = weight row r of this CTA's half, column j =
            // token row0 + j.  Gate/up: lanes 0-63 gate and 64-127 up of the features
            // nt * 128 + 64 * half + (r % 64).  Down: lane r = output column
            // nt * 256 + 128 * half + r.
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + a * kGemmBN;
            const int R = tile0.m_valid, nch = swap_n(R) / 32;
            if (sg.glu) {
                // warps q and q + 2 hold the gate and up values of the same 32 features; per
                // chunk of 32 tokens the gate warp activates tokens 0-15 and the up warp 16-31,
                // each handing the other the half it needs
                const bool gate_w = q < 2;
                const int f = tile0.nt * 128 + 64 * half + 32 * (q & 1) + lane;
                float *xg = c.xbuf + (q & 1) * 1024, *xu = xg + 512;  // [16][32] each
#pragma unroll 1
                for (int ch = 0; ch < nch; ++ch) {
                    uint32_t v[32];
                    tmem_ld32(tb + 32 * ch, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (gate_w)
                            xg[j * 32 + lane] = __uint_as_float(v[16 + j]);
                        else
                            xu[j * 32 + lane] = __uint_as_float(v[j]);
                    }
                    epi_bar();
                    const int t0 = 32 * ch + (gate_w ? 0 : 16);
                    if (f < sg.n_out) {
                        bf16 *o = static_cast<bf16 *>(sg.out) + (size_t)(tile0.row0 + t0) * sg.ldo + f;
                        const int nj = min(16, R - t0);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (j < nj)
                                o[(size_t)j * sg.ldo] = __float2bfloat16_rn(
                                    gate_w ? glu_act(__uint_as_float(v[j]), xu[j * 32 + lane], act, alpha, limit, beta)
                                           : glu_act(xg[j * 32 + lane], __uint_as_float(v[16 + j]), act, alpha, limit, beta));
                    }
                    epi_bar();
                }
            } else {
                const int col = tile0.nt * kGemmBN + 128 * half + 32 * q + lane;
#pragma unroll 1
                for (int ch = 0; ch < nch; ++ch) {
                    uint32_t v[32];
                    tmem_ld32(tb + 32 * ch, v);
                    tmem_ld_wait();
                    if (col < sg.n_out) {
                        float *o = static_cast<float *>(sg.out) + (size_t)(tile0.row0 + 32 * ch) * sg.ldo + col;
                        const int nj = min(32, R - 32 * ch);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nj) o[(size_t)j * sg.ldo] = __uint_as_float(v[j]);
                    }
                }
                if (sg.tok_done != nullptr) {  // this CTA's half of every row is stored
                    __threadfence();
                    epi_bar();
                    for (int j = q * 32 + lane; j < R; j += kEpiThreads)
                        atomicAdd(sg.tok_done + sg.row_tok[tile0.row0 + j], 1);
                }
            }
        } else
#pragma unroll 1
        for (int hh = 0; hh < HALVES; ++hh) {
        const Tile t = hh == 0 ? tile0 : decode_tile<kBM>(p, tile, s_seg_end, s_offs, s_toffs, hh);
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (a + hh) * kGemmBN;
        const bool row_ok = r < t.m_valid;
        const size_t orow = t.ks * sg.split_stride + (size_t)(t.row0 + (row_ok ? r : 0)) * sg.ldo;
        if (c.ebuf != 0 && sg.map_out != 0) {
            // Staged: each 32-column (fp32) or 64-column (bf16) slice of this warp's 32 rows
            // goes through shared memory and leaves as one TMA store (or coalesced stores
            // when the quadrant holds fewer valid rows), instead of one row per lane
            const int rows = min(32, t.m_valid - q * 32);
            if (rows > 0) {  // warp-uniform
                const uint32_t sb = c.ebuf + (uint32_t)(q % c.ebuf_quads) * 4096u;
                const uint32_t srow = sb + (uint32_t)lane * 128u;
                const int sw = lane & 7;
                const CUtensorMap *map = &p.maps[sg.map_out];
                const int y = (t.ks != 0 ? t.ks * (int)(sg.split_stride / sg.ldo) : 0) + t.row0 + q * 32;
                const size_t esz = sg.glu ? 2 : 4;
                char *const obase = static_cast<char *>(sg.out) + (t.ks * sg.split_stride + (size_t)(t.row0 + q * 32) * sg.ldo) * esz;
                const size_t ld_bytes = (size_t)sg.ldo * esz;
                if (sg.glu) {
                    static_assert(128 / kEpiParts % 64 == 0, "bf16 slices of 64 columns");
#pragma unroll 1
                    for (int c0 = part * (128 / kEpiParts); c0 < (part + 1) * (128 / kEpiParts); c0 += 64) {
                        const int col = t.nt * 128 + c0;
                        if (col >= sg.n_out) break;
                        if (lane == 0) bulk_wait_read_all();  // the previous slice's store has read the buffer
                        __syncwarp();
#pragma unroll 1
                        for (int h2 = 0; h2 < 2; ++h2) {
                            uint32_t g[32], u[32];
                            tmem_ld32(tb + c0 + 32 * h2, g);
                            tmem_ld32(tb + 128 + c0 + 32 * h2, u);
                            tmem_ld_wait();
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pk[i] = pack_bf16x2(
                                    glu_act(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i]), act, alpha, limit, beta),
                                    glu_act(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1]), act, alpha, limit, beta));
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                st_shared_v4(srow + ((uint32_t)((4 * h2 + v) ^ sw) << 4), pk[4 * v], pk[4 * v + 1],
                                             pk[4 * v + 2], pk[4 * v + 3]);
                        }
                        epi_flush(map, sb, rows, col, y, obase + (size_t)col * 2, ld_bytes, lane);
                    }
                } else {
                    constexpr int kSpan = kGemmBN / kEpiParts;
#pragma unroll 1
                    for (int c0 = part * kSpan; c0 < (part + 1) * kSpan; c0 += 32) {
                        const int col = t.nt * kGemmBN + c0;
                        if (col >= sg.n_out) break;
                        uint32_t v32[32];
                        tmem_ld32(tb + c0, v32);
                        tmem_ld_wait();
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            st_shared_v4(srow + ((uint32_t)(v ^ sw) << 4), v32[4 * v], v32[4 * v + 1], v32[4 * v + 2],
                                         v32[4 * v + 3]);
                        epi_flush(map, sb, rows, col, y, obase + (size_t)col * 4, ld_bytes, lane);
                    }
                }
                if (sg.tok_done != nullptr) {  // the rows are stored: this tile's columns of each token
                    if (lane == 0) {
                        bulk_wait_all();
                        fence_proxy_async();
                    }
                    __syncwarp();
                    if (row_ok) {
                        const int row = t.row0 + r;
                        __threadfence();
                        atomicAdd(sg.tok_done + (sg.row_tok != nullptr ? sg.row_tok[row] : row), 2);
                    }
                }
            }
        } else if (sg.glu) {
            constexpr int kSpan = 128 / kEpiParts;  // output columns per slice
#pragma unroll 1
            for (int c0 = part * kSpan; c0 < (part + 1) * kSpan; c0 += 32) {
                uint32_t g[32], u[32];
                tmem_ld32(tb + c0, g);
                tmem_ld32(tb + 128 + c0, u);
                tmem_ld_wait();
                const int col = t.nt * 128 + c0;
                if (row_ok && col < sg.n_out) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16x2(
                            glu_act(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i]), act, alpha, limit, beta),
                            glu_act(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1]),
                                    act, alpha, limit, beta));
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<bf16 *>(sg.out) + orow + col);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
        } else {
            constexpr int kSpan = kGemmBN / kEpiParts;
#pragma unroll 1
            for (int c0 = part * kSpan; c0 < (part + 1) * kSpan; c0 += 32) {
                uint32_t v32[32];
                tmem_ld32(tb + c0, v32);
                tmem_ld_wait();
                const int col = t.nt * kGemmBN + c0;
                if (row_ok && col < sg.n_out) {  // fp32 rows: the combine rounds once
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<float *>(sg.out) + orow + col);
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        dst[v] = make_uint4(v32[4 * v], v32[4 * v + 1], v32[4 * v + 2], v32[4 * v + 3]);
                }
            }
            if (sg.tok_done != nullptr && row_ok) {  // this row's columns of the tile are stored
                const int row = t.row0 + r;
                __threadfence();
                atomicAdd(sg.tok_done + (sg.row_tok != nullptr ? sg.row_tok[row] : row), 2);
            }
        }
        }  // halves
        tc_fence_before();
        if (PAIR)  // rank 0's barrier counts both CTAs' epilogue threads
            mbar_arrive_cluster(mapa_shared(tempty_bar(a), 0));
        else
            mbar_arrive(tempty_bar(a));
        if (sg.signal != nullptr) {
            // publish the stored rows: this warp's TMA stores complete, proxy fence for the
            // consumer's TMA reads, device-scope fence, all four warps done, then one
            // release increment
            if (c.ebuf != 0 && lane == 0) bulk_wait_all();
            fence_proxy_async();
            __threadfence();
            epi_bar();
            if (lead_thread)
                for (int hh = 0; hh < HALVES; ++hh) atomicAdd(sg.signal + tile0.ready + hh, 1);
        }
        if (stats) w_work += global_timer_ns() - t1;
        ++n_acc;
    }
    if (c.ebuf != 0 && lane == 0) bulk_wait_all();  // no store may still read the buffer when the CTA exits
    if (stats && lead_thread) {
        atomicAdd(stats + 4, (unsigned long long)w_tfull);
        atomicAdd(stats + 5, (unsigned long long)w_work);
    }
}

template <bool PAIR, bool THIN = false>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmArgs p) {
    using C = GemmCfg<PAIR, THIN>;
    constexpr int kStages = C::kStages, kBBytes = C::kBBytes, kStageBytes = C::kStageBytes, kBM = C::kBM;
    constexpr int kKB = C::kKB, kAStage = C::kAStage;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + kStages * kAStage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    const uint32_t bar0 = smem_u32(bars);
    // barriers: full[kStages], empty[kStages], tfull[2], tempty[2], drain, ring_full[kRing], ring_empty[kRing]
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto tfull_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kStages + a); };
    auto tempty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kStages + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
    auto ring_full = [&](int i) { return bar0 + 8u * (2 * kStages + 5 + i); };
    auto ring_empty = [&](int i) { return bar0 + 8u * (2 * kStages + 5 + kRing + i); };
    // CTA pairs, tiles claimed at the tail: rank 0 hands each claimed id to rank 1 through
    // a two-slot mailbox in rank 1's shared memory (claim_full in rank 1, claim_empty in rank 0)
    auto claim_full = [&](uint32_t i) { return bar0 + 8u * (2 * kStages + 5 + 2 * kRing + i); };
    auto claim_empty = [&](uint32_t i) { return bar0 + 8u * (2 * kStages + 5 + 2 * kRing + 2 + i); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kStages + 5 + 2 * kRing + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *ring = reinterpret_cast<volatile int *>(tmem_slot + 2);  // [kRing] tile ids
    volatile int *mailbox = ring + kRing;                                   // [2] claimed tile ids
    static_assert(8 * (2 * kStages + 5 + 2 * kRing + 4) + 8 + 4 * kRing + 8 <= 512, "barrier block");
    float *xbuf = reinterpret_cast<float *>(smem + kStages * kStageBytes + 512);  // C::kXBufBytes

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTA pair: rank 0 issues the MMAs; the full and accumulator-empty barriers
    // that count both CTAs are rank 0's
    const int half = PAIR ? (int)cluster_ctarank() : 0;
    const bool leader = half == 0;
    auto abort_all = [&]() {
        if (PAIR)
            raise_abort_pair(p.err, abort_flag);
        else
            raise_abort(p.err, abort_flag);
    };
    trace_mark(p.trace, 0);
    load_segments(p);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (uint32_t a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), PAIR ? 2 * kEpiThreads : kEpiThreads);  // the epilogue threads (of both CTAs)
        }
        mbar_init(drain_bar, 1);
        for (int i = 0; i < kRing; ++i) {
            mbar_init(ring_full(i), 1);
            mbar_init(ring_empty(i), 2);  // the MMA thread and the epilogue have read the id
        }
        for (uint32_t i = 0; i < 2; ++i) {
            mbar_init(claim_full(i), 1);   // rank 0's hand-over (rank 1's barrier)
            mbar_init(claim_empty(i), 1);  // rank 1 has read the id (rank 0's barrier)
        }
        fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0 && lane == 0)
        for (int m = 0; m < kGemmMaxMaps; ++m) tma_prefetch_desc(&p.maps[m]);
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // both CTAs' barriers exist before any copy or arrival crosses over
    tc_fence_after();
    // the prologue above overlaps the previous kernel; the dispatch results
    // (offsets, tile counts) and the A rows are read only after this point
    pdl_wait();
    trace_mark(p.trace, 1);
    pdl_trigger();
    unsigned long long *const stats = p.stats;
    const uint64_t t_ready = stats ? global_timer_ns() : 0;
    // every role decodes every tile: keep the dispatch offsets on chip
    __shared__ int s_offs[257], s_toffs[257];
    __shared__ int s_seg_end[kGemmMaxSegments];
    int grouped = -1;
    for (int s = 0; s < p.num_segs; ++s)
        if (!s_seg[s].dense) grouped = s;
    if (grouped >= 0)
        for (int i = threadIdx.x; i <= s_seg[grouped].num_groups; i += blockDim.x) {
            s_offs[i] = s_seg[grouped].offs[i];
            s_toffs[i] = s_seg[grouped].tile_offs[i];
        }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int s = 0; s < p.num_segs; ++s) {
            run += seg_tiles<kBM>(s_seg[s], s_toffs);
            s_seg_end[s] = run;
        }
    }
    __syncthreads();
    const uint32_t tmem_base = *tmem_slot;
    const int total = s_seg_end[p.num_segs - 1];

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t L = 0;  // loads issued so far; stage = L % kStages
            bool ok = true;
            uint64_t w_empty = 0, w_dep = 0;
            // tiles: claimed in order from the launch-wide ticket, or round-robin.  The
            // next tile is claimed three k-blocks before the current one's loads end,
            // so the atomic's latency hides behind them while the claim stays late.
            const bool dyn = !PAIR && p.tile_counter != nullptr;
            const int stride = PAIR ? (int)gridDim.x / 2 : (int)gridDim.x;
            // CTA pairs: tiles in static round-robin order up to n_static (neighbouring pairs on
            // neighbouring tiles of one weight tile, which then stays in L2), the last kTailWaves
            // waves claimed from the ticket by whichever pair is free first
            const int n_static = PAIR && p.tile_counter != nullptr ? max(0, total - kTailWaves * stride) : total;
            uint32_t n_claim = 0;
            auto claim_pair = [&](int &out) -> bool {
                const uint32_t c = n_claim++, slot = c & 1u, ph = (c >> 1) & 1u;
                if (leader) {
                    if (!mbar_wait(claim_empty(slot), ph ^ 1u, p.wait_ns, abort_flag)) return false;
                    out = n_static + atomicAdd(p.tile_counter, 1);
                    st_cluster_s32(mapa_shared(smem_u32(const_cast<int *>(mailbox + slot)), 1), out);
                    mbar_arrive_cluster(mapa_shared(claim_full(slot), 1));
                } else {
                    if (!mbar_wait_cluster(claim_full(slot), ph, p.wait_ns, abort_flag)) return false;
                    out = mailbox[slot];
                    mbar_arrive_cluster(mapa_shared(claim_empty(slot), 0));
                }
                return true;
            };
            // the tile after `cur`: the static one, or a claimed one past the static part
            auto next_tile = [&](int cur, int &out) -> bool {
                if (!PAIR) {
                    out = dyn ? atomicAdd(p.tile_counter, 1) : cur + stride;
                    return true;
                }
                if (cur + stride < n_static) {
                    out = cur + stride;
                    return true;
                }
                return claim_pair(out);
            };
            int next = 0;
            if (!next_tile((PAIR ? (int)blockIdx.x / 2 : (int)blockIdx.x) - stride, next)) ok = false;
            for (int n = 0; ok; ++n) {
                const int tile = next < total ? next : total;  // total: the end marker
                const int slot = n % kRing;
                if (!mbar_wait(ring_empty(slot), ((n / kRing) & 1u) ^ 1u, p.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                ring[slot] = tile;
                mbar_arrive(ring_full(slot));
                if (tile >= total) break;
                const Tile t = decode_tile<kBM>(p, tile, s_seg_end, s_offs, s_toffs, half);
                const GemmSegment &sg = s_seg[t.seg];
                const int g = sg.group_base + t.group;
                const int claim_at = sg.k_blocks > 3 * kKB ? sg.k_blocks - 3 * kKB : 0;
                if (sg.wait != nullptr) {  // A rows written earlier in this launch
                    const uint64_t t0 = stats ? global_timer_ns() : 0;
                    // a swapped tile reads rows of both 128-row halves of its m-tile
                    if (!wait_counter(sg.wait + t.ready - (t.swp ? half : 0), sg.wait_count, p.wait_ns, abort_flag) ||
                        (t.swp && !wait_counter(sg.wait + t.ready - half + 1, sg.wait_count, p.wait_ns, abort_flag))) {
                        ok = false;
                        break;
                    }
                    if (stats) w_dep += global_timer_ns() - t0;
                    fence_proxy_async();  // order the A rows' generic-proxy stores before our TMA reads
                }
                const CUtensorMap *mA = &p.maps[sg.map_a];
                const CUtensorMap *mB = &p.maps[sg.map_b0];
                const CUtensorMap *mB2 = &p.maps[sg.map_b1];
                for (int kb = 0; kb < sg.k_blocks; kb += kKB) {
                    const int s = L % kStages;
                    const uint32_t ph = (L / kStages) & 1u;
                    if ((kb == claim_at || (kKB > 1 && kb + 1 == claim_at)) && !next_tile(tile, next)) {
                        ok = false;
                        break;
                    }
                    const uint64_t t0 = stats ? global_timer_ns() : 0;
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, p.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (stats) w_empty += global_timer_ns() - t0;
                    if (PAIR && t.swp) {
                        // swapped: this CTA's token rows (half of the MMA's N) in a 32- or 64-row
                        // box, and 128 weight rows: the down tile's half, or 64 gate and 64 up
                        // rows of the same features (one box per k-block and projection)
                        const uint32_t fb = mapa_shared(full_bar(s), 0);
                        const int box = swap_box(t.m_valid), nh = swap_n(t.m_valid) / 2;
                        if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * (kBBytes + box * kGemmBK * 2 * kKB));
                        const int kc = sg.k_base + t.ks * sg.k_blocks + kb;
                        tma_load_3d_pair(sA + s * kAStage, &p.maps[sg.map_aw[box == 64]], fb, 0, t.row0 + half * nh, kc);
                        if (sg.glu) {
                            const int f0 = t.nt * 128 + 64 * half;
#pragma unroll
                            for (int j = 0; j < kKB; ++j) {
                                const uint32_t dst = sB + s * kBBytes + j * (kBBytes / kKB);
                                tma_load_3d_pair(dst, &p.maps[sg.map_bw0], fb, (kc + j) * kGemmBK, f0, g);
                                tma_load_3d_pair(dst + kBBytes / kKB / 2, &p.maps[sg.map_bw1], fb, (kc + j) * kGemmBK, f0, g);
                            }
                        } else {
                            tma_load_4d_pair(sB + s * kBBytes, mB, fb, 0, t.nt * kGemmBN + half * 128, kc, g);
                        }
                    } else if (PAIR) {
                        // both CTAs' copies complete on rank 0's full barrier; rank 0 expects their bytes.
                        // Maps view K as (64, K / 64) so that one box brings k-blocks kb, kb + 1
                        // (past the last k-block: zero fill, no MMA)
                        const uint32_t fb = mapa_shared(full_bar(s), 0);
                        if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * kStageBytes);
                        const int kc = sg.k_base + t.ks * sg.k_blocks + kb;
                        tma_load_3d_pair(sA + s * kAStage, mA, fb, 0, t.row0, kc);
                        if (sg.glu)  // gate rows in rank 0, up rows in rank 1: accumulator columns 0-127 / 128-255
                            tma_load_4d_pair(sB + s * kBBytes, leader ? mB : mB2, fb, 0, t.nt * 128, kc, g);
                        else
                            tma_load_4d_pair(sB + s * kBBytes, mB, fb, 0, t.nt * kGemmBN + half * 128, kc, g);
                    } else {
                        const int kx = (sg.k_base + t.ks * sg.k_blocks + kb) * kGemmBK;
                        mbar_arrive_expect_tx(full_bar(s), kStageBytes);
                        tma_load_2d(sA + s * kAStage, mA, full_bar(s), kx, t.row0);
                        if (sg.glu) {
                            tma_load_3d(sB + s * kBBytes, mB, full_bar(s), kx, t.nt * 128, g);
                            tma_load_3d(sB + s * kBBytes + kBBytes / 2, mB2, full_bar(s), kx, t.nt * 128, g);
                        } else {
                            tma_load_3d(sB + s * kBBytes, mB, full_bar(s), kx, t.nt * kGemmBN, g);
                        }
                    }
                    ++L;
                }
                if (!ok) break;
            }
            if (stats) {
                atomicAdd(stats + 0, (unsigned long long)w_empty);
                atomicAdd(stats + 1, (unsigned long long)w_dep);
            }
            if (!ok) {
                abort_all();
                if (PAIR) {
                    // a stage's copies complete on rank 0's barrier together with the other
                    // CTA's, which may never be issued after an abort: wait a fixed time instead
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < kPairDrainNs) __nanosleep(1000);
                } else {
                    // wait for the copies still in flight (the last load of each stage)
                    for (uint32_t i = 0; i < (uint32_t)kStages && i < L; ++i) {
                        const uint32_t l = L - 1 - i;
                        mbar_wait(full_bar(l % kStages), (l / kStages) & 1u, kDrainNs, nullptr);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue
        if (PAIR && !leader && lane == 0) {
            // rank 1 issues nothing; it only releases its ring slots
            for (int n = 0;; ++n) {
                const int slot = n % kRing;
                if (!mbar_wait(ring_full(slot), (n / kRing) & 1u, p.wait_ns, abort_flag)) break;
                const int tile = ring[slot];
                mbar_arrive(ring_empty(slot));
                if (tile >= total) break;
            }
        } else if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(PAIR ? 2 * kGemmBM : kGemmBM, kGemmBN);
            uint32_t L = 0, n_acc = 0;
            bool ok = true, issued = false;
            uint64_t w_full = 0, w_acc = 0;
            for (int n = 0; ok; ++n) {
                const int slot = n % kRing;
                if (!mbar_wait(ring_full(slot), (n / kRing) & 1u, p.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                const int tile = ring[slot];
                mbar_arrive(ring_empty(slot));
                if (tile >= total) break;
                const Tile t = decode_tile<kBM>(p, tile, s_seg_end, s_offs, s_toffs, half);
                const GemmSegment &sg = s_seg[t.seg];
                const uint32_t a = n_acc & 1u, aph = (n_acc >> 1) & 1u;
                const uint64_t t0 = stats ? global_timer_ns() : 0;
                if (!(PAIR ? mbar_wait_cluster(tempty_bar(a), aph ^ 1u, p.wait_ns, abort_flag)
                           : mbar_wait(tempty_bar(a), aph ^ 1u, p.wait_ns, abort_flag))) {
                    ok = false;
                    break;
                }
                if (stats) w_acc += global_timer_ns() - t0;
                tc_fence_after();
                const uint32_t d = tmem_base + a * kGemmBN;
                // swapped: A = the weight rows (B's stage), B = the token rows, N = swap_n(rows)
                const bool swp = PAIR && t.swp;
                const uint32_t id = swp ? idesc_bf16_f32(2 * kGemmBM, swap_n(t.m_valid)) : idesc;
                const uint32_t tok_kb = swp ? (uint32_t)swap_box(t.m_valid) * kGemmBK * 2 : (uint32_t)kABytes;
                for (int kb = 0; kb < sg.k_blocks; kb += kKB) {
                    const int s = L % kStages;
                    const uint32_t ph = (L / kStages) & 1u;
                    const uint64_t t1 = stats ? global_timer_ns() : 0;
                    if (!mbar_wait(full_bar(s), ph, p.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (stats) w_full += global_timer_ns() - t1;
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < kKB; ++j) {
                        if (kKB > 1 && kb + j >= sg.k_blocks) break;
                        const uint64_t td = smem_desc_k128(sA + s * kAStage + j * tok_kb);
                        const uint64_t wd = smem_desc_k128(sB + s * kBBytes + j * (kBBytes / kKB));
                        const uint64_t ad = swp ? wd : td, bd = swp ? td : wd;
#pragma unroll
                        for (int kk = 0; kk < kGemmBK / 16; ++kk) {  // +32 bytes per K step of 16
                            if (PAIR)
                                tc_mma_bf16_pair(d, ad + 2 * kk, bd + 2 * kk, id, (kb | j | kk) != 0);
                            else
                                tc_mma_bf16(d, ad + 2 * kk, bd + 2 * kk, id, (kb | j | kk) != 0);
                        }
                    }
                    issued = true;
                    // frees the stage (in both CTAs of a pair) once these MMAs have read it
                    if (PAIR)
                        tc_commit_pair(empty_bar(s), 3);
                    else
                        tc_commit(empty_bar(s));
                    ++L;
                }
                if (!ok) break;
                if (PAIR)  // accumulator complete, in both CTAs' TMEM
                    tc_commit_pair(tfull_bar(a), 3);
                else
                    tc_commit(tfull_bar(a));
                ++n_acc;
            }
            if (stats) {
                atomicAdd(stats + 2, (unsigned long long)w_full);
                atomicAdd(stats + 3, (unsigned long long)w_acc);
                atomicAdd(stats + 7, (unsigned long long)n_acc);
            }
            if (!ok) {
                abort_all();
                if (issued) {
                    if (PAIR)
                        tc_commit_pair(drain_bar, 1);
                    else
                        tc_commit(drain_bar);
                    mbar_wait(drain_bar, 0, kDrainNs, nullptr);
                }
            }
        }
    } else {
        // ----------------------------------------------------------- epilogue
        EpiCtx c{ring_full(0), ring_empty(0), tfull_bar(0), tempty_bar(0), ring, abort_flag, tmem_base, total,
                 s_seg_end, s_offs, s_toffs, half, xbuf, THIN ? 0u : smem_u32(smem + C::kEpiOff),
                 C::kEpiBufBytes / 4096 > 0 ? C::kEpiBufBytes / 4096 : 1};
        epilogue_role<PAIR, kBM>(p, c, warp, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // neither CTA leaves while the other may still reach its memory
    trace_exit(p.trace);
    if (stats && threadIdx.x == 0) atomicAdd(stats + 6, (unsigned long long)(global_timer_ns() - t_ready));
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------------
// Expert GEMM on block-scaled (OCP microscaling) weights.
//
// The weights are stored as MX element codes with one E8M0 scale per 32
// consecutive K values of a row (the checkpoint formats the Arcee AFMoE issue
// lists: "Checkpoint confirmed", 4-bit and MXFP8 variants).  A weight is
// code_value * 2^(scale - 127).  The activations stay bf16, so the block still
// multiplies bf16 tokens by the exact decoded weights: every decoded value is a
// bf16 number (3 or 1 mantissa bits times a power of two), the MMA is the same
// bf16 tcgen05 MMA as above, and only the weight bytes streamed from HBM shrink
// (1 byte per weight for E4M3, half a byte for E2M1, plus 1/32 byte of scale).
//
// One CTA per SM, 15 warps (7 + kConvWarps = 8 converters):
//   warp 0     TMA producer of the weight codes and scales (the HBM stream): a
//              raw ring of kRawStages k-blocks, 256 rows x 64 codes + 2 x 256 scales
//   warp 1     tcgen05.mma issue (as above): A from the A ring, B from the B ring
//   warps 2-5  epilogue (as above)
//   warp 6     TMA producer of the A rows (bf16, 128-byte swizzle) into the A ring
//   warps 7-14 converters: decode a raw k-block into the B ring's bf16 tile, written
//              in the 128-byte-swizzled K-major layout the MMA descriptor reads
// Three rings: raw (kRawStages, freed by the converters), A (kAStages, freed by the
// MMA) and converted B (kBStages, freed by the MMA), so the weight stream and the
// A rows each run several k-blocks ahead of the MMA while B is being converted.
// Every k-block moves about 130 KB through shared memory (codes in and out, the
// bf16 B tile in and out, the A tile in and out), which bounds this design at
// roughly one k-block per 1000 cycles.
//
// 256-row tiles (M256, where the host picks the CTA-pair tile size): one CTA loads both
// 128-row halves of the A rows and issues two M = 128 MMAs on every decoded weight
// tile into one accumulator of 2 x 256 TMEM columns, so each decoded weight serves
// twice the rows; the epilogue then runs between tiles (one accumulator).  Measured:
// AFMoE MXFP8 prefill expert GEMM 555 against 758 us with 128-row tiles; a CTA-pair
// version (each CTA decoding half of the weight tile, rank 1 relaying its k-blocks to
// rank 0's cta_group::2 MMAs) took 1028 us.  Bit-identical to the bf16 CTA-pair path.
template <int WF, bool M256 = false, int CW = 8>
struct MxCfg {
    // B rows converted per k-block (the tile's 256 columns)
    static constexpr int kBRows = kGemmBN;
    static constexpr int kRawRow = WF == kWeightsMxfp8 ? kGemmBK : kGemmBK / 2;  // bytes of a row's k-block
    static constexpr int kRawCodes = kBRows * kRawRow;                          // 16 KB / 8 KB
    // scales [row half][32-value block][128 rows]: every copy lands 128-byte aligned, as a
    // tensor copy's shared-memory destination must
    static constexpr int kScaleStride = 128;
    static constexpr int kScaleBytes = (kBRows / 128) * 2 * kScaleStride;
    static constexpr int kRawStage = kRawCodes + kScaleBytes;
    // ring depths measured on GB300 (Nano decode and AFMoE prefill, MXFP8 and MXFP4):
    // three converted B stages beat two by 2-4%; deeper A or raw rings change nothing.
    // 256-row tiles (M256): an A stage holds both 128-row halves (32 KB), two of them.
    static constexpr int kRawStages = M256 ? (WF == kWeightsMxfp8 ? 3 : 4) : (WF == kWeightsMxfp8 ? 4 : 6);
    static constexpr int kAStages = M256 ? 2 : 3;
    static constexpr int kBStages = 3;
    static constexpr int kAStageBytes = (M256 ? 2 : 1) * kABytes;
    static constexpr int kBBytes = kBRows * kGemmBK * 2;  // converted B tile, 32 KB
    static constexpr int kBarBytes = 1024;
    static constexpr int kSmemBytes =
        kBStages * kBBytes + kAStages * kAStageBytes + kRawStages * kRawStage + 1024 /*align*/ + kBarBytes;
    // converter warps: 8, or 16 where the weight stream of 128-row tiles outruns eight
    // (GemmArgs::mx_conv16)
    static constexpr int kConvWarps = CW;
    static constexpr int kThreads = 32 * (7 + kConvWarps);  // warps 0-6 as listed, then the converters
    static_assert(kRawStage % 128 == 0, "raw stages stay 128-byte aligned");
};

// 2^(code - 127) for an E8M0 scale code (255 is NaN; 0 is 2^-127, an fp32 subnormal).
__device__ __forceinline__ float e8m0_to_f32(uint32_t code) {
    if (code == 0u) return __uint_as_float(0x00400000u);
    if (code == 255u) return __uint_as_float(0x7fc00000u);
    return __uint_as_float(code << 23);
}

// Two E4M3 codes (low byte = lower K index) -> bf16x2 of code * scale.  The
// hardware conversion to f16 is exact (every E4M3 value is a normal f16 or
// zero); the product by a power of two is exact in fp32 and in bf16 unless it
// leaves bf16's range, where it rounds to nearest.
__device__ __forceinline__ uint32_t e4m3x2_scaled(uint32_t pair16, float scale) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)pair16));
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    return pack_bf16x2(f.x * scale, f.y * scale);
}

// Two E2M1 codes in one byte (low nibble = lower K index) -> bf16x2 of code * scale.
__device__ __forceinline__ uint32_t e2m1x2_scaled(uint32_t byte, float scale) {
    uint32_t h;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(byte));
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    return pack_bf16x2(f.x * scale, f.y * scale);
}

// Decoders that keep the conversion pipe nearly idle.  A bf16x2 word whose bit
// patterns are built from the codes represents code * 2^-b exactly (zero, the
// codes' subnormals and their normals all map onto the same form of bf16), and
// one bf16x2 multiply by 2^(scale - 127 + b) applies the E8M0 scale: exact when
// the product is a bf16 number, rounded to nearest otherwise.  The multiplier
// must itself be a normal bf16: scale + b <= 254, checked per block.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// 2^(code + bias - 127) in both halves of a bf16x2 (its exponent field is code + bias)
__device__ __forceinline__ uint32_t pow2_bf16x2(uint32_t code, int bias) {
    return ((code + bias) << 7) * 0x00010001u;
}
// f16x2 of two MX codes (hardware unpack) -> the same bits as bf16x2 of value * 2^-112:
// every E4M3 / E2M1 value is a normal f16 (or zero) with its low 7 mantissa bits zero,
// so dropping 3 bits keeps sign, exponent field and mantissa.
__device__ __forceinline__ uint32_t f16x2_as_bf16x2_scaled(uint32_t h) {
    return ((h & 0x7fff7fffu) >> 3) | (h & 0x80008000u);
}
// Four E4M3 codes (byte i = K index i) -> bf16x2 (codes 0, 1) and (2, 3) of value * 2^-120:
// the code's 7 magnitude bits become bf16 bits 4..10 (exponent field = the code's
// exponent field, mantissa = its 3 bits), its sign bit 15.
__device__ __forceinline__ void e4m3x4_as_bf16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t m = w & 0x7f7f7f7fu, sg = w & 0x80808080u;
    lo = __byte_perm(m, 0u, 0x4140) * 16u + __byte_perm(sg, 0u, 0x1404);
    hi = __byte_perm(m, 0u, 0x4342) * 16u + __byte_perm(sg, 0u, 0x3424);
}

// Decoder: 0 = fp32 products (conversion pipe), 1 = f16 unpack + bit reinterpretation +
// one bf16x2 multiply, 2 = (E4M3) integer bit spreading + one bf16x2 multiply.  Measured
// on GB300 (Nano decode): all three run at the same speed; the converters are bound by
// shared-memory traffic, not by their arithmetic.
#ifndef MOE_MX_CVT
#define MOE_MX_CVT 1
#endif

// Converter warp cw (of kConvWarps): rows [cw * kRows / kConvWarps, + kRows / kConvWarps)
// of one raw k-block (kRows = 256, or 128 in a CTA pair) -> bf16 B
// tile.  Row r's 16-byte chunk j (K values 8j..8j+7) goes to r * 128 + ((j ^ (r % 8))
// * 16): the 128-byte swizzle of a 1024-byte-aligned tile.  Lanes read consecutive
// 16-byte pieces of the raw rows and store chunks of 8 distinct swizzle positions
// per quarter-warp, so neither side has bank conflicts.  The scale codes of the
// warp's rows are read first: when all of them allow the bf16 multiplier (the usual
// case) the loop has no per-row branch and its code loads are issued together
// (measured: 0.35 against 0.58 us per k-block for eight warps with the branch).
template <int WF, int kRows, int CW>
__device__ __forceinline__ void mx_convert(const uint8_t *raw, const uint8_t *sc, uint8_t *out, int cw, int lane) {
    using M = MxCfg<WF, false, CW>;
    constexpr int kRowsPerWarp = kRows / M::kConvWarps;
    static_assert(kRowsPerWarp % 16 == 0, "converter rows");
    constexpr int kRowsPerIt = WF == kWeightsMxfp8 ? 8 : 16;  // rows a warp covers per iteration
    constexpr int kIt = kRowsPerWarp / kRowsPerIt;
    constexpr int kB = (WF == kWeightsMxfp8 && MOE_MX_CVT == 2) ? 120 : 112;  // the decoders' 2^-b
    // fp8: lane -> row + lane / 4, 16 codes (K 16c .. 16c + 15, c = lane % 4);
    // fp4: lane -> row + lane / 2, 32 codes (K 32c .. 32c + 31, c = lane % 2)
    const int c = WF == kWeightsMxfp8 ? (lane & 3) : (lane & 1);
    const int r_lane = WF == kWeightsMxfp8 ? (lane >> 2) : (lane >> 1);
    const int sblk = WF == kWeightsMxfp8 ? (c >> 1) : c;  // 32-value scale block of the lane's codes
    uint32_t code[kIt];
    bool fast = MOE_MX_CVT != 0;
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
        const int row = cw * kRowsPerWarp + it * kRowsPerIt + r_lane;
        code[it] = sc[((row >> 7) * 2 + sblk) * M::kScaleStride + (row & 127)];
        fast = fast && code[it] + kB <= 254u;
    }
    if (__all_sync(0xffffffffu, fast)) {
        constexpr int U = kIt < 4 ? kIt : 4;
#pragma unroll
        for (int i0 = 0; i0 < kIt; i0 += U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int row = cw * kRowsPerWarp + (i0 + u) * kRowsPerIt + r_lane;
                v[u] = *reinterpret_cast<const uint4 *>(raw + row * M::kRawRow + c * 16);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int row = cw * kRowsPerWarp + (i0 + u) * kRowsPerIt + r_lane;
                const uint32_t s2 = pow2_bf16x2(code[i0 + u], kB);
                uint8_t *rp = out + row * 128;
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                if (WF == kWeightsMxfp8) {
                    uint32_t r[8];
                    if (MOE_MX_CVT == 2) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) e4m3x4_as_bf16x2(w[i], r[2 * i], r[2 * i + 1]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t h0, h1;
                            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h0) : "h"((unsigned short)w[i]));
                            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h1) : "h"((unsigned short)(w[i] >> 16)));
                            r[2 * i] = f16x2_as_bf16x2_scaled(h0);
                            r[2 * i + 1] = f16x2_as_bf16x2_scaled(h1);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) r[i] = bf16x2_mul(r[i], s2);
                    *reinterpret_cast<uint4 *>(rp + (((2 * c) ^ (row & 7)) << 4)) = make_uint4(r[0], r[1], r[2], r[3]);
                    *reinterpret_cast<uint4 *>(rp + (((2 * c + 1) ^ (row & 7)) << 4)) =
                        make_uint4(r[4], r[5], r[6], r[7]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {  // chunk 4c + q: K 32c + 8q .. + 7 = the four bytes of w[q]
                        uint32_t r[4];
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            uint32_t h;
                            asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
                                : "=r"(h) : "r"(w[q] >> (8 * b)));
                            r[b] = bf16x2_mul(f16x2_as_bf16x2_scaled(h), s2);
                        }
                        *reinterpret_cast<uint4 *>(rp + (((4 * c + q) ^ (row & 7)) << 4)) =
                            make_uint4(r[0], r[1], r[2], r[3]);
                    }
                }
            }
        }
        return;
    }
    // some scale of the warp's rows leaves the bf16 multiplier's range (or the fp32
    // decoder is selected): fp32 products, rounded once to bf16
#pragma unroll 1
    for (int it = 0; it < kIt; ++it) {
        const int row = cw * kRowsPerWarp + it * kRowsPerIt + r_lane;
        const uint4 v = *reinterpret_cast<const uint4 *>(raw + row * M::kRawRow + c * 16);
        const float f = e8m0_to_f32(sc[((row >> 7) * 2 + sblk) * M::kScaleStride + (row & 127)]);
        uint8_t *rp = out + row * 128;
        if (WF == kWeightsMxfp8) {
            const uint4 o0 = make_uint4(e4m3x2_scaled(v.x, f), e4m3x2_scaled(v.x >> 16, f), e4m3x2_scaled(v.y, f),
                                        e4m3x2_scaled(v.y >> 16, f));
            const uint4 o1 = make_uint4(e4m3x2_scaled(v.z, f), e4m3x2_scaled(v.z >> 16, f), e4m3x2_scaled(v.w, f),
                                        e4m3x2_scaled(v.w >> 16, f));
            *reinterpret_cast<uint4 *>(rp + (((2 * c) ^ (row & 7)) << 4)) = o0;
            *reinterpret_cast<uint4 *>(rp + (((2 * c + 1) ^ (row & 7)) << 4)) = o1;
        } else {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 o = make_uint4(e2m1x2_scaled(w[q] & 0xffu, f), e2m1x2_scaled((w[q] >> 8) & 0xffu, f),
                                           e2m1x2_scaled((w[q] >> 16) & 0xffu, f), e2m1x2_scaled(w[q] >> 24, f));
                *reinterpret_cast<uint4 *>(rp + (((4 * c + q) ^ (row & 7)) << 4)) = o;
            }
        }
    }
}

template <int WF, bool M256, int CW = 8>
__global__ void __launch_bounds__(MxCfg<WF, M256, CW>::kThreads, 1) gemm_mx_kernel(const __grid_constant__ GemmArgs p) {
    using M = MxCfg<WF, M256, CW>;
    constexpr int R = M::kRawStages, RA = M::kAStages, P = M::kBStages, NCW = M::kConvWarps;
    constexpr int kBM = M256 ? 2 * kGemmBM : kGemmBM;  // rows per tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    // converted B stages (32 KB), A stages (16 KB, or 32 KB for 256-row tiles; both
    // 1024-byte aligned), raw stages, barriers
    auto opB = [&](int s) { return smem + s * M::kBBytes; };
    auto opA = [&](int s) { return smem + P * M::kBBytes + s * M::kAStageBytes; };
    uint8_t *const raw0 = smem + P * M::kBBytes + RA * M::kAStageBytes;
    auto rawS = [&](int s) { return raw0 + s * M::kRawStage; };
    uint64_t *bars = reinterpret_cast<uint64_t *>(raw0 + R * M::kRawStage);
    const uint32_t bar0 = smem_u32(bars);
    // barriers: ring_full[kRing], ring_empty[kRing], tfull[2], tempty[2] (the epilogue's
    // contiguous block), then raw_full[R], raw_empty[R], a_full[RA], a_empty[RA], op_full[P],
    // op_empty[P] (op: the converted B ring), drain
    auto ring_full = [&](int i) { return bar0 + 8u * i; };
    auto ring_empty = [&](int i) { return bar0 + 8u * (kRing + i); };
    auto tfull_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kRing + a); };
    auto tempty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kRing + 2 + a); };
    constexpr int kB0 = 2 * kRing + 4;
    auto raw_full = [&](int s) { return bar0 + 8u * (kB0 + s); };
    auto raw_empty = [&](int s) { return bar0 + 8u * (kB0 + R + s); };
    auto a_full = [&](int s) { return bar0 + 8u * (kB0 + 2 * R + s); };
    auto a_empty = [&](int s) { return bar0 + 8u * (kB0 + 2 * R + RA + s); };
    auto op_full = [&](int s) { return bar0 + 8u * (kB0 + 2 * R + 2 * RA + s); };
    auto op_empty = [&](int s) { return bar0 + 8u * (kB0 + 2 * R + 2 * RA + P + s); };
    const uint32_t drain_bar = bar0 + 8u * (kB0 + 2 * R + 2 * RA + 2 * P);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kB0 + 2 * R + 2 * RA + 2 * P + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *ring = reinterpret_cast<volatile int *>(tmem_slot + 2);  // [kRing] tile ids
    static_assert(8 * (kB0 + 2 * R + 2 * RA + 2 * P + 1) + 8 + 4 * kRing <= M::kBarBytes, "barrier block");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 256-row tiles: both 128-row halves in this CTA, one accumulator of 2 x 256 columns
    // (no second buffer: the epilogue of a tile precedes the next tile's MMAs)
    const int half = 0;
    auto abort_all = [&]() { raise_abort(p.err, abort_flag); };
    trace_mark(p.trace, 0);
    load_segments(p);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(ring_full(i), 1);
            mbar_init(ring_empty(i), 3 + NCW);  // MMA, epilogue, A producer, each converter warp
        }
        for (uint32_t a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), kEpiThreads);
        }
        for (int s = 0; s < R; ++s) {
            mbar_init(raw_full(s), 1);
            mbar_init(raw_empty(s), NCW);
        }
        for (int s = 0; s < RA; ++s) {
            mbar_init(a_full(s), 1);   // the A copy
            mbar_init(a_empty(s), 1);  // the MMA's commit
        }
        for (int s = 0; s < P; ++s) {
            mbar_init(op_full(s), NCW);  // each converter warp
            mbar_init(op_empty(s), 1);   // the MMA's commit
        }
        mbar_init(drain_bar, 1);
        fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0 && lane == 0)
        for (int m = 0; m < kGemmMaxMaps; ++m) tma_prefetch_desc(&p.maps[m]);
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    trace_mark(p.trace, 1);
    pdl_trigger();
    unsigned long long *const stats = p.stats;
    const uint64_t t_ready = stats ? global_timer_ns() : 0;
    __shared__ int s_offs[257], s_toffs[257];
    __shared__ int s_seg_end[kGemmMaxSegments];
    int grouped = -1;
    for (int s = 0; s < p.num_segs; ++s)
        if (!s_seg[s].dense) grouped = s;
    if (grouped >= 0)
        for (int i = threadIdx.x; i <= s_seg[grouped].num_groups; i += blockDim.x) {
            s_offs[i] = s_seg[grouped].offs[i];
            s_toffs[i] = s_seg[grouped].tile_offs[i];
        }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int s = 0; s < p.num_segs; ++s) {
            run += seg_tiles<kBM>(s_seg[s], s_toffs);
            s_seg_end[s] = run;
        }
    }
    __syncthreads();
    const uint32_t tmem_base = *tmem_slot;
    const int total = s_seg_end[p.num_segs - 1];

    if (warp == 0) {
        // ------------------------------------------- weight codes and scales
        if (lane == 0) {
            uint32_t L = 0;
            bool ok = true;
            uint64_t w_empty = 0;
            // tiles: from the launch-wide ticket, or round-robin
            const bool dyn = p.tile_counter != nullptr;
            const int stride = (int)gridDim.x;
            int next = dyn ? atomicAdd(p.tile_counter, 1) : (int)blockIdx.x;
            for (int n = 0;; ++n) {
                const int tile = next < total ? next : total;
                const int slot = n % kRing;
                if (!mbar_wait(ring_empty(slot), ((n / kRing) & 1u) ^ 1u, p.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                ring[slot] = tile;
                mbar_arrive(ring_full(slot));
                if (tile >= total) break;
                const Tile t = decode_tile<kBM>(p, tile, s_seg_end, s_offs, s_toffs, half);
                const GemmSegment &sg = s_seg[t.seg];
                const int g = sg.group_base + t.group;
                const int claim_at = sg.k_blocks > 3 ? sg.k_blocks - 3 : 0;
                // rows of the B tile's two 128-row halves: gate and up rows of n-tile nt,
                // or the 256 rows of a down tile
                const int r0 = sg.glu ? t.nt * 128 : t.nt * kGemmBN, r1 = sg.glu ? r0 : r0 + 128;
                const CUtensorMap *mC0 = &p.maps[sg.map_b0], *mC1 = &p.maps[sg.glu ? sg.map_b1 : sg.map_b0];
                const CUtensorMap *mS0 = &p.maps[sg.map_s0], *mS1 = &p.maps[sg.glu ? sg.map_s1 : sg.map_s0];
                for (int kb = 0; kb < sg.k_blocks; ++kb) {
                    const int s = L % R;
                    const uint32_t ph = (L / R) & 1u;
                    if (kb == claim_at) next = dyn ? atomicAdd(p.tile_counter, 1) : tile + stride;
                    const uint64_t t0 = stats ? global_timer_ns() : 0;
                    if (!mbar_wait(raw_empty(s), ph ^ 1u, p.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (stats) w_empty += global_timer_ns() - t0;
                    const int kx = (sg.k_base + t.ks * sg.k_blocks + kb) * kGemmBK;  // first K value
                    const int xb = WF == kWeightsMxfp8 ? kx : kx / 2;                // its byte in a code row
                    const uint32_t dst = smem_u32(rawS(s));
                    mbar_arrive_expect_tx(raw_full(s), M::kRawStage);
                    tma_load_3d(dst, mC0, raw_full(s), xb, r0, g);
                    tma_load_3d(dst + M::kRawCodes, mS0, raw_full(s), r0, kx / 32, g);
                    tma_load_3d(dst + 128 * M::kRawRow, mC1, raw_full(s), xb, r1, g);
                    tma_load_3d(dst + M::kRawCodes + 2 * M::kScaleStride, mS1, raw_full(s), r1, kx / 32, g);
                    ++L;
                }
                if (!ok) break;
            }
            if (stats) atomicAdd(stats + 0, (unsigned long long)w_empty);
            if (!ok) {
                abort_all();
                for (uint32_t i = 0; i < (uint32_t)R && i < L; ++i) {  // copies still in flight
                    const uint32_t l = L - 1 - i;
                    mbar_wait(raw_full(l % R), (l / R) & 1u, kDrainNs, nullptr);
                }
            }
        }
    } else if (warp == 6) {
        // ------------------------------------------------------------ A rows
        if (lane == 0) {
            uint32_t L = 0;
            bool ok = true;
            uint64_t w_dep = 0;
            for (int n = 0;; ++n) {
                const int slot = n % kRing;
                if (!mbar_wait(ring_full(slot), (n / kRing) & 1u, p.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                const int tile = ring[slot];
                mbar_arrive(ring_empty(slot));
                if (tile >= total) break;
                const Tile t = decode_tile<kBM>(p, tile, s_seg_end, s_offs, s_toffs, half);
                const GemmSegment &sg = s_seg[t.seg];
                if (sg.wait != nullptr) {  // A rows written earlier in this launch (both halves)
                    const uint64_t t0 = stats ? global_timer_ns() : 0;
                    if (!wait_counter(sg.wait + t.ready, sg.wait_count, p.wait_ns, abort_flag) ||
                        (M256 && !wait_counter(sg.wait + t.ready + 1, sg.wait_count, p.wait_ns, abort_flag))) {
                        ok = false;
                        break;
                    }
                    if (stats) w_dep += global_timer_ns() - t0;
                    fence_proxy_async();
                }
                const CUtensorMap *mA = &p.maps[sg.map_a];
                for (int kb = 0; kb < sg.k_blocks; ++kb) {
                    const int s = L % RA;
                    const uint32_t ph = (L / RA) & 1u;
                    if (!mbar_wait(a_empty(s), ph ^ 1u, p.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int kx = (sg.k_base + t.ks * sg.k_blocks + kb) * kGemmBK;
                    mbar_arrive_expect_tx(a_full(s), M::kAStageBytes);
                    tma_load_2d(smem_u32(opA(s)), mA, a_full(s), kx, t.row0);
                    if (M256) tma_load_2d(smem_u32(opA(s)) + kABytes, mA, a_full(s), kx, t.row0 + 128);
                    ++L;
                }
                if (!ok) break;
            }
            if (stats) atomicAdd(stats + 1, (unsigned long long)w_dep);
            if (!ok) {
                abort_all();
                for (uint32_t i = 0; i < (uint32_t)RA && i < L; ++i) {  // copies still in flight
                    const uint32_t l = L - 1 - i;
                    mbar_wait(a_full(l % RA), (l / RA) & 1u, kDrainNs, nullptr);
                }
            }
        }
    } else if (warp >= 7) {
        // -------------------------------------------------------- converters
        const int cw = warp - 7;
        uint32_t L = 0;
        bool ok = true;
        for (int n = 0; ok; ++n) {
            const int slot = n % kRing;
            const bool have = __all_sync(0xffffffffu, mbar_wait(ring_full(slot), (n / kRing) & 1u, p.wait_ns, abort_flag));
            if (!have) {
                if (lane == 0) abort_all();
                break;
            }
            const int tile = ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(ring_empty(slot));
            if (tile >= total) break;
            const Tile t = decode_tile<kBM>(p, tile, s_seg_end, s_offs, s_toffs, half);
            const int kbs = s_seg[t.seg].k_blocks;
            for (int kb = 0; kb < kbs; ++kb) {
                const int rs = L % R, os = L % P;
                const bool got = __all_sync(0xffffffffu, mbar_wait(raw_full(rs), (L / R) & 1u, p.wait_ns, abort_flag) &&
                                                             mbar_wait(op_empty(os), ((L / P) & 1u) ^ 1u, p.wait_ns, abort_flag));
                if (!got) {
                    if (lane == 0) abort_all();
                    ok = false;
                    break;
                }
                mx_convert<WF, M::kBRows, CW>(rawS(rs), rawS(rs) + M::kRawCodes, opB(os), cw, lane);
                fence_proxy_async_smem();  // the generic-proxy stores, before the MMA (async proxy) reads them
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(raw_empty(rs));
                    mbar_arrive(op_full(os));
                }
                ++L;
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kGemmBM, kGemmBN);
            uint32_t L = 0, n_acc = 0;
            bool ok = true, issued = false;
            uint64_t w_full = 0, w_acc = 0;
            for (int n = 0; ok; ++n) {
                const int slot = n % kRing;
                if (!mbar_wait(ring_full(slot), (n / kRing) & 1u, p.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                const int tile = ring[slot];
                mbar_arrive(ring_empty(slot));
                if (tile >= total) break;
                const Tile t = decode_tile<kBM>(p, tile, s_seg_end, s_offs, s_toffs, half);
                const GemmSegment &sg = s_seg[t.seg];
                // two accumulators in turn, or (256-row tiles) one of 2 x 256 columns
                const uint32_t a = M256 ? 0u : n_acc & 1u, aph = M256 ? n_acc & 1u : (n_acc >> 1) & 1u;
                const uint64_t t0 = stats ? global_timer_ns() : 0;
                if (!mbar_wait(tempty_bar(a), aph ^ 1u, p.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                if (stats) w_acc += global_timer_ns() - t0;
                tc_fence_after();
                const uint32_t d = tmem_base + a * kGemmBN;
                for (int kb = 0; kb < sg.k_blocks; ++kb) {
                    const int sa = L % RA, sb = L % P;
                    const uint64_t t1 = stats ? global_timer_ns() : 0;
                    if (!mbar_wait(a_full(sa), (L / RA) & 1u, p.wait_ns, abort_flag) ||
                        !mbar_wait(op_full(sb), (L / P) & 1u, p.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (stats) w_full += global_timer_ns() - t1;
                    tc_fence_after();
                    const uint64_t bd = smem_desc_k128(smem_u32(opB(sb)));
                    // each 128-row half of the tile's A rows against the same decoded B tile
#pragma unroll
                    for (int hh = 0; hh < (M256 ? 2 : 1); ++hh) {
                        const uint64_t ad = smem_desc_k128(smem_u32(opA(sa)) + hh * kABytes);
#pragma unroll
                        for (int kk = 0; kk < kGemmBK / 16; ++kk)
                            tc_mma_bf16(d + hh * kGemmBN, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    }
                    issued = true;
                    tc_commit(a_empty(sa));
                    tc_commit(op_empty(sb));
                    ++L;
                }
                if (!ok) break;
                tc_commit(tfull_bar(a));
                ++n_acc;
            }
            if (stats) {
                atomicAdd(stats + 2, (unsigned long long)w_full);
                atomicAdd(stats + 3, (unsigned long long)w_acc);
                atomicAdd(stats + 7, (unsigned long long)n_acc);
            }
            if (!ok) {
                abort_all();
                if (issued) {
                    tc_commit(drain_bar);
                    mbar_wait(drain_bar, 0, kDrainNs, nullptr);
                }
            }
        }
    } else {
        // ----------------------------------------------------------- epilogue
        EpiCtx c{ring_full(0), ring_empty(0), tfull_bar(0), tempty_bar(0), ring, abort_flag, tmem_base, total,
                 s_seg_end, s_offs, s_toffs, half, nullptr, 0u, 1};
        epilogue_role<false, kBM, M256 ? 2 : 1>(p, c, warp, lane);
    }

    tc_fence_before();
    __syncthreads();
    trace_exit(p.trace);
    if (stats && threadIdx.x == 0) atomicAdd(stats + 6, (unsigned long long)(global_timer_ns() - t_ready));
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

size_t gemm_tc_smem_bytes() { return GemmCfg<false>::kSmemBytes; }

CUresult encode_map_a(CUtensorMap *m, const void *ptr, int rows, int K) {
    return encode_map_a_box(m, ptr, rows, K, kGemmBM);
}

CUresult encode_map_a_box(CUtensorMap *m, const void *ptr, int rows, int K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kGemmBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_map_out(CUtensorMap *m, const void *ptr, int rows, int cols, int f32) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t es = f32 ? 4 : 2;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * es};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / es), 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_map_b(CUtensorMap *m, const void *ptr, int groups, int rows, int K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)groups};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)rows * K * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kGemmBK, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// The same tensors viewed with K split as (64, K / 64), box of two 64-column
// chunks: one copy brings two consecutive k-blocks, each a 128-byte-swizzled
// [rows][64] tile, one after the other in shared memory (CTA-pair GEMM).
CUresult encode_map_a_kb2(CUtensorMap *m, const void *ptr, int rows, int K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[3] = {(cuuint64_t)kGemmBK, (cuuint64_t)rows, (cuuint64_t)(K / kGemmBK)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)kGemmBK * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kGemmBK, (cuuint32_t)box_rows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_map_b_kb2(CUtensorMap *m, const void *ptr, int groups, int rows, int K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[4] = {(cuuint64_t)kGemmBK, (cuuint64_t)rows, (cuuint64_t)(K / kGemmBK), (cuuint64_t)groups};
    const cuuint64_t strides[3] = {(cuuint64_t)K * 2, (cuuint64_t)kGemmBK * 2, (cuuint64_t)rows * K * 2};
    const cuuint32_t box[4] = {(cuuint32_t)kGemmBK, (cuuint32_t)box_rows, 2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_map_mx_codes(CUtensorMap *m, const void *ptr, int groups, int rows, int K, int wfmt, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
    const int row_bytes = wfmt == kWeightsMxfp8 ? K : K / 2;
    const cuuint64_t dims[3] = {(cuuint64_t)row_bytes, (cuuint64_t)rows, (cuuint64_t)groups};
    const cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows * row_bytes};
    const cuuint32_t box[3] = {(cuuint32_t)(wfmt == kWeightsMxfp8 ? kGemmBK : kGemmBK / 2), (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_map_mx_scales(CUtensorMap *m, const void *ptr, int groups, int rows, int K, int box_rows,
                              int box_blocks) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[3] = {(cuuint64_t)rows, (cuuint64_t)(K / 32), (cuuint64_t)groups};
    const cuuint64_t strides[2] = {(cuuint64_t)rows, (cuuint64_t)rows * (K / 32)};
    const cuuint32_t box[3] = {(cuuint32_t)box_rows, (cuuint32_t)box_blocks, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

cudaError_t launch_gemm_tc(const GemmArgs &a, cudaStream_t s) {
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(gemm_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GemmCfg<false>::kSmemBytes);
        cudaFuncSetAttribute(gemm_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GemmCfg<true>::kSmemBytes);
        cudaFuncSetAttribute(gemm_tc_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GemmCfg<false, true>::kSmemBytes);
        cudaFuncSetAttribute(gemm_mx_kernel<kWeightsMxfp8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             MxCfg<kWeightsMxfp8>::kSmemBytes);
        cudaFuncSetAttribute(gemm_mx_kernel<kWeightsMxfp4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             MxCfg<kWeightsMxfp4>::kSmemBytes);
        cudaFuncSetAttribute(gemm_mx_kernel<kWeightsMxfp8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             MxCfg<kWeightsMxfp8, true>::kSmemBytes);
        cudaFuncSetAttribute(gemm_mx_kernel<kWeightsMxfp4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             MxCfg<kWeightsMxfp4, true>::kSmemBytes);
        cudaFuncSetAttribute(gemm_mx_kernel<kWeightsMxfp8, false, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             MxCfg<kWeightsMxfp8, false, 16>::kSmemBytes);
        cudaFuncSetAttribute(gemm_mx_kernel<kWeightsMxfp4, false, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             MxCfg<kWeightsMxfp4, false, 16>::kSmemBytes);
    });
    if (a.wfmt == kWeightsMxfp8 || a.wfmt == kWeightsMxfp4) {
        const bool f8 = a.wfmt == kWeightsMxfp8;
        if (a.pair) {  // 256-row tiles (the dispatch counted them), one CTA each
            if (f8)
                return launch_pdl(gemm_mx_kernel<kWeightsMxfp8, true>, dim3(a.num_ctas),
                                  dim3(MxCfg<kWeightsMxfp8>::kThreads), (size_t)MxCfg<kWeightsMxfp8, true>::kSmemBytes,
                                  s, a);
            return launch_pdl(gemm_mx_kernel<kWeightsMxfp4, true>, dim3(a.num_ctas), dim3(MxCfg<kWeightsMxfp4>::kThreads),
                              (size_t)MxCfg<kWeightsMxfp4, true>::kSmemBytes, s, a);
        }
        if (a.mx_conv16) {
            if (f8)
                return launch_pdl(gemm_mx_kernel<kWeightsMxfp8, false, 16>, dim3(a.num_ctas),
                                  dim3(MxCfg<kWeightsMxfp8, false, 16>::kThreads),
                                  (size_t)MxCfg<kWeightsMxfp8, false, 16>::kSmemBytes, s, a);
            return launch_pdl(gemm_mx_kernel<kWeightsMxfp4, false, 16>, dim3(a.num_ctas),
                              dim3(MxCfg<kWeightsMxfp4, false, 16>::kThreads),
                              (size_t)MxCfg<kWeightsMxfp4, false, 16>::kSmemBytes, s, a);
        }
        if (f8)
            return launch_pdl(gemm_mx_kernel<kWeightsMxfp8, false>, dim3(a.num_ctas),
                              dim3(MxCfg<kWeightsMxfp8>::kThreads), (size_t)MxCfg<kWeightsMxfp8>::kSmemBytes, s, a);
        return launch_pdl(gemm_mx_kernel<kWeightsMxfp4, false>, dim3(a.num_ctas), dim3(MxCfg<kWeightsMxfp4>::kThreads),
                          (size_t)MxCfg<kWeightsMxfp4>::kSmemBytes, s, a);
    }
    if (a.wfmt != kWeightsBf16) return cudaErrorInvalidValue;
    if (a.pair) {
        if (a.num_ctas < 2 || (a.num_ctas & 1)) return cudaErrorInvalidValue;
        return launch_pdl_cluster(gemm_tc_kernel<true>, dim3(a.num_ctas), dim3(kThreads),
                                  (size_t)GemmCfg<true>::kSmemBytes, s, dim3(2, 1, 1), a);
    }
    if (a.thin)
        return launch_pdl(gemm_tc_kernel<false, true>, dim3(a.num_ctas), dim3(kThreads),
                          (size_t)GemmCfg<false, true>::kSmemBytes, s, a);
    return launch_pdl(gemm_tc_kernel<false>, dim3(a.num_ctas), dim3(kThreads), (size_t)GemmCfg<false>::kSmemBytes,
                      s, a);
}

}  // namespace moe
