// Host-side launchers of the MoE kernels (internal to libmoe.so).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace moe {

// Launch `kernel` with programmatic dependent launch allowed (the kernel calls
// pdl_wait() before touching memory that earlier kernels on the stream use),
// in thread-block clusters of `cluster` CTAs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                      dim3 cluster, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster.x;
    attr[1].val.clusterDim.y = cluster.y;
    attr[1].val.clusterDim.z = cluster.z;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same without clusters.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

using bf16 = __nv_bfloat16;

// Bits of the device error word.
enum : int { ERR_TIMEOUT = 1, ERR_BOUNDS = 2 };

// ---------------------------------------------------------------- router (K1)
// Per token: fp32 logits against the fp32 router weights, sigmoid (or softmax)
// scores, top-k of score + bias (ties to the lower expert index), weights
// gathered from the unbiased scores, optional renormalisation, route_scale.
// Each CTA also writes the expert histogram of its tokens to blk_hist.
struct RouterArgs {
    const void *X;         // [T, H], bf16 or fp32
    int x_f32;             // 1 when X is fp32
    int T, H, E, k;
    const float *Wr;       // [E, H]
    const float *bias;     // [E] or nullptr
    int score_func;        // 0 sigmoid, 1 softmax
    int route_norm;
    float route_scale;
    int32_t *topk_idx;     // [T, k]
    float *topk_w;         // [T, k]
    int32_t *blk_hist;     // block histograms or nullptr; count (b, e) at b*hb + e*he
    int hb, he;
    __nv_bfloat16 *x_bf16; // [T, H] bf16 copy of fp32 X, or nullptr
    int tokens_per_block;  // 16 or 32
    unsigned long long *trace;  // 5 slots, or nullptr
};
int router_tokens_per_block(int T, int num_sms);
cudaError_t launch_router(const RouterArgs &a, cudaStream_t s);

// Tensor-core router with the routing rule (router_tc.cu): grid (ceil(T/128),
// splits) in clusters of (1, splits); the splits CTAs of an m-tile share its
// H reduction and each routes 128 / splits of its tokens.  The fp32 router
// weights are held as `parts` bf16 slices [parts, E, H] whose sum is exact
// (see launch_split_router).
constexpr int kMaxRouterSplits = 8;
struct RouterTcArgs {
    CUtensorMap mapX;      // X [T, H] bf16, box 128 x 64
    CUtensorMap mapW;      // router weight parts [parts, E, H] bf16, box Np x 64
    int T, H, E, Np, parts, stages, tmem_cols;
    int kb_per_split;      // 64-wide k-blocks per CTA of a cluster
    int splits;            // cluster size: 1, 2, 4 or 8
    int staged_push;       // 1: the stage buffers hold two [128][Np + 4] fp32 arrays (plan)
    int k;
    const float *bias;     // [E] or nullptr
    int score_func, route_norm;
    float route_scale;
    int32_t *topk_idx;     // [T, k]
    float *topk_w;         // [T, k]
    int32_t *blk_hist;     // histogram of each (128 / splits)-token block, or nullptr
    int hb, he;            // its strides, as in ScanArgs
    int *err;
    unsigned long long wait_ns;
    unsigned long long *trace;
    // nullptr, or kRouterStats ns sums over CTAs: main loop, first cluster
    // barrier, pushing the partials with the second barrier, adding them and
    // routing, histogram; then the number of CTAs; then the part of "adding them
    // and routing" spent adding the partials
    unsigned long long *stats;
};
constexpr int kRouterStats = 8;
struct RouterTcPlan {
    int Np, tmem_cols, stages, smem, parts, staged_push;
};
RouterTcPlan plan_router_tc(int E, int parts);
cudaError_t launch_router_tc(const RouterTcArgs &a, int smem, cudaStream_t s);
// L2 prefetch of bytes[i] bytes from ptr[i] (16-byte multiples), a hint only.
struct PrefetchArgs {
    const void *ptr[2];
    unsigned long long bytes[2];
};
cudaError_t launch_l2_prefetch(const PrefetchArgs &a, int grid, cudaStream_t s);
// Split fp32 weights w into bf16 hi + mid + lo == w; *flags |= 1 when some w
// needs mid, |= 2 when some w needs lo.
cudaError_t launch_split_router(const float *wr, int E, int H, bf16 *parts, int *flags, cudaStream_t s);

// ------------------------------------------------------- dispatch sort (K2)
// offs[e] = first sorted row of expert e (exclusive scan of the counts),
// tile_offs[e] = exclusive scan of ceil(count_e / 128), active[0..n) = experts
// with rows, active[E] = n.  blk_hist becomes the first row of each
// (block, expert) pair.  Rows are ordered by (expert, token, slot): stable.
struct ScanArgs {
    int32_t *blk_hist;  // in: counts, out: base rows; (b, e) at b*hb + e*he
    int nb, E;
    int32_t *offs;      // [E + 1]
    int32_t *tile_offs; // [E + 1]
    int32_t *active;    // [E + 1]
    int hb, he;         // 0, 0: row-major [nb, E]
    int tile_m;         // m-tile counted by tile_offs; 0: kGemmBM
};
cudaError_t launch_scan(const ScanArgs &a, cudaStream_t s);

struct ScatterArgs {
    const int32_t *topk_idx;  // [T, k]; the k experts of a token are distinct
    const int32_t *blk_hist;  // expert counts of each token block; (b, e) at b*hb + e*he
    int hb, he;
    int32_t *offs, *tile_offs, *active;  // written by CTA (0, 0): as in ScanArgs
    int tile_m;                          // 0: kGemmBM
    // CTA (0, 0) zeroes the fused expert GEMM's counters: ready[0, routed m-tiles)
    // and ready[ready_shared_base, + ready_shared_count)
    int *ready;
    int ready_per_tile;    // counters per routed tile of tile_m rows (2 with CTA pairs)
    int ready_shared_base, ready_shared_count;
    int *tile_counters;    // [2] tile tickets of the expert GEMM launches, zeroed by CTA (0, 0), or nullptr
    unsigned long long *trace;
    int T, k, E, H;
    int tokens_per_block;     // <= 128: the router's blocking
    int gather_split;         // CTAs per token block sharing the row gather
    const void *X;            // [T, H]
    int x_f32;
    int32_t *sorted_tok;      // [T*k]
    int32_t *slot_of;         // [T*k]
    __nv_bfloat16 *x_sorted;  // [T*k, H]
    int *err;
    int *tok_done;            // [T] per-token output counters, zeroed here (CTAs y = 0), or nullptr
};
cudaError_t launch_scatter(const ScatterArgs &a, cudaStream_t s);
// CTAs of the dispatch kernel resident at once on one SM (occupancy query, cached)
int scatter_ctas_per_sm();

// --------------------------------------------------------------- combine (K7)
// Y[t] = sum_j w[t,j] * Yslot[slot_of[t,j]] + Ys[t]  (fp32 sum, fixed order).
// The slot and shared outputs are fp32: the one rounding to the output dtype is
// the combine's.
struct CombineArgs {
    const float *yslot;          // [T*k, H]
    const float *ys;             // shared output part 0 [T, H], or nullptr
    int ys_parts;                // parts of a K-split shared down projection (>= 1), summed in order
    size_t ys_part_stride;       // elements from one part to the next
    const float *topk_w;         // [T, k]
    const int32_t *slot_of;      // [T, k]
    int T, k, H;
    void *Y;                     // [T, H]
    int y_f32;
    unsigned long long *trace;
    // post_mlp norm and residual (norm != 0): Y = residual + y * g / sqrt(mean(y^2) + eps),
    // g = post_w (norm 1) or 1 + post_w (norm 2); residual in Y's dtype
    int norm;
    float eps;
    const float *post_w;
    const void *residual;
    int *err;                    // ERR_TIMEOUT when a bounded wait gives up (or nullptr)
    unsigned long long wait_ns;  // bound of each wait
    // Overlap with the expert GEMM (no post-norm): instead of waiting for the GEMM to
    // finish, a token is combined once tok_done[t] reaches tok_unit * (its valid slots +
    // ys_parts) (the down tiles' epilogues count its stored rows); nullptr: wait first
    const int *tok_done;
    int tok_unit;
};
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s);

// pre_mlp norm of each token row: out = x * g / sqrt(mean(x^2) + eps), g = w (norm 1)
// or 1 + w (norm 2), in the dtype of X (x_f32), one CTA per row.  After its
// dependency wait the first CTA also zeroes zero_a[0, zero_a_n) and
// zero_b[0, zero_b_n) (counters of the kernels that follow), or nothing.
struct NormArgs {
    const void *X;
    int x_f32;
    int T, H;
    const float *w;
    int norm;
    float eps;
    void *out;
    unsigned long long *trace;
    int *zero_a;
    int zero_a_n;
    int *zero_b;
    int zero_b_n;
};
cudaError_t launch_rmsnorm(const NormArgs &a, cudaStream_t s);

// ------------------------------------------- tcgen05 grouped GEMMs (K3/K4/K5)
constexpr int kGemmBM = 128;   // rows (tokens) per tile: the MMA's M
constexpr int kGemmBK = 64;    // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kGemmBN = 256;   // MMA N; gate/up tiles hold 128 gate + 128 up columns

constexpr int kGemmMaxSegments = 5;
constexpr int kGemmMaxMaps = 20;

// Storage of the expert weights (the B operand): bf16, or OCP microscaling
// (MX) codes with one E8M0 scale per 32 consecutive K values.
enum WeightFormat { kWeightsBf16 = 0, kWeightsMxfp8 = 1, kWeightsMxfp4 = 2 };
struct GemmSegment {
    int dense;             // 1: one group of m_dense rows from row 0; 0: groups by offs
    int num_groups;
    int group_base;        // weight-map coordinate of group 0
    int m_dense;
    const int32_t *offs;   // [num_groups + 1] (grouped; every grouped segment of a launch shares them)
    const int32_t *tile_offs;
    int n_tiles;           // output tiles per group along N
    int k_blocks;          // K / 64 (of this segment)
    int k_base;            // first 64-wide k-block of A's columns and B's columns
    int n_out;             // valid output columns
    void *out;             // [rows, ldo]: bf16 activations (glu), fp32 projection outputs (otherwise)
    int ldo;
    int glu;               // 1: gate/up pair (maps b0, b1) with the activation; 0: one projection (map b0)
    int map_a, map_b0, map_b1;  // indices into GemmArgs::maps
    // Dependencies inside one launch, per m-tile index (tile_offs[g] + mt, or mt when dense, plus
    // ready_base): `signal` gets +1 after a tile's outputs are stored; before loading a tile's A
    // rows the producer waits until wait[index] >= wait_count.
    int *signal;
    const int *wait;
    int wait_count;
    int ready_base;
    // dense segments: K split into k_splits consecutive ranges of k_blocks each (0 or 1:
    // no split); range j starts at k-block k_base + j * k_blocks and stores its partial
    // product at out + j * split_stride
    int k_splits;
    size_t split_stride;
    // MX weights: maps of the E8M0 scales of b0 and b1 ([groups, K / 32, rows] uint8)
    int map_s0, map_s1;
    // CTA pairs, grouped segments: an m-tile of at most kSwapMaxRows rows runs with the
    // operands swapped (the weight rows as M = 256, the tokens as N); its token rows come
    // from map_aw[0] (boxes of 32 rows, two k-blocks) or map_aw[1] (64 rows), and a
    // gate/up tile's weights from map_bw0 / map_bw1 (boxes of 64 rows, one k-block)
    int map_aw[2];
    int map_bw0, map_bw1;
    // down projections feeding a combine that overlaps the launch: after a tile's rows are
    // stored, tok_done[token] += 2 for each of its rows (swapped pair tiles: += 1 from each
    // CTA, which stores half of every row's columns); token = row_tok[row], or the row
    // itself when row_tok is nullptr (dense segments)
    int *tok_done;
    const int32_t *row_tok;
    // tiles with the tokens as M: the output's store map (encode_map_out: boxes of 32 rows of
    // 128 bytes), through which the epilogue writes each 32-row slice whose rows are all
    // valid; 0: none (map 0 is always an A operand), every row stored from registers
    int map_out;
};
constexpr int kSwapMaxRows = 128;

struct GemmArgs {
    CUtensorMap maps[kGemmMaxMaps];
    GemmSegment seg[kGemmMaxSegments];
    int num_segs;          // tiles of segment s precede those of segment s + 1
    int act;
    float alpha, limit, beta;
    int *err;
    unsigned long long wait_ns;
    int num_ctas;
    int pair;              // 1: CTA pairs (cta_group::2, 256-row tiles; num_ctas even,
                           //    tile_offs counting 256-row tiles; all maps from encode_map_*_kb2)
    int *tile_counter;     // zeroed ticket: tiles claimed in order (one CTA per tile: every tile; CTA
                           // pairs: the last waves, after a static round-robin part); nullptr: round-robin
    unsigned long long *trace;
    // nullptr, or kGemmStats ns sums over CTAs: producer waiting for a free
    // stage, producer waiting for gate/up rows, MMA waiting for data, MMA
    // waiting for an accumulator, epilogue waiting for an accumulator,
    // epilogue working, CTA time past the dependency wait, tiles
    unsigned long long *stats;
    int wfmt;              // WeightFormat of every segment's B maps; MX only without CTA pairs
    int thin;              // one CTA per tile, bf16, every m-tile <= 32 rows: A maps with boxes of 32
                           // rows, six stages (gemm_tc.cu, kThinRows)
    int swap_rem;          // CTA pairs: grouped m-tiles of <= kSwapMaxRows rows with swapped operands
    int mx_conv16;         // MX weights, 128-row tiles: 16 converter warps instead of 8
};
constexpr int kGemmStats = 8;
cudaError_t launch_gemm_tc(const GemmArgs &a, cudaStream_t s);
size_t gemm_tc_smem_bytes();

// Swapped-operand expert GEMMs for few tokens per expert (gemm_sab.cu): weight
// rows are the MMA's M = 128, n_tokens (32 or 64) token rows its N.
struct SabSegment {
    int dense, num_groups, group_base, m_dense;
    const int32_t *offs;       // [num_groups + 1] (grouped)
    const int32_t *tile_offs;  // [num_groups + 1] prefix of ceil(m_g / n_tokens)
    int w_tiles;               // weight tiles per group (64 gate/up outputs, or 128 down outputs)
    int k_blocks;              // K / 64
    int n_out;                 // valid output columns
    void *out;                 // [rows, ldo]: bf16 activations (gate/up), fp32 outputs (down)
    int ldo;
};
struct SabArgs {
    // segment 0: weights Wa0 (+Wb0 = up for gate/up), tokens X0; segment 1 likewise
    CUtensorMap Wa0, Wb0, X0, Wa1, Wb1, X1;
    SabSegment seg[2];
    int num_segs, glu, act;
    float alpha, limit, beta;
    int *err;
    unsigned long long wait_ns;
    int num_ctas, stages;
};
cudaError_t launch_gemm_sab(const SabArgs &a, int n_tokens, cudaStream_t s);

// Swapped-operand expert GEMMs on MX weights (gemm_mxt.cu): the weight rows are
// the MMA's A operand (M = 128), decoded from their codes and scales by one thread
// per row straight into tensor memory; n_tokens (32 or 64) token rows from shared
// memory are its N.  Segments as in SabArgs; per segment, W?a / W?b map the codes of
// gate (or down) and up with boxes of 64 rows (gate/up) or 128 rows (down), S?a / S?b
// their scales with boxes of those rows x all K / 32 blocks of the segment (one copy
// per tile), and X? the token rows (box n_tokens x 64).  sblk: the largest K / 32 of
// the segments (sizes the per-tile scale buffers).
struct MxtArgs {
    CUtensorMap Wa0, Wb0, Sa0, Sb0, X0;
    CUtensorMap Wa1, Wb1, Sa1, Sb1, X1;
    SabSegment seg[2];
    int num_segs, glu, act;
    float alpha, limit, beta;
    int *err;
    unsigned long long wait_ns;
    int num_ctas, stages, wfmt, sblk;
    // nullptr, or kGemmStats ns sums over CTAs: producer waiting for a free stage,
    // converters waiting for codes, converters waiting for a free TMEM buffer, MMA
    // waiting for operands, MMA waiting for an accumulator, epilogue waiting for an
    // accumulator, epilogue working; then the tiles
    unsigned long long *stats;
};
cudaError_t launch_gemm_mxt(const MxtArgs &a, int n_tokens, cudaStream_t s);

// Tensor maps (TMA descriptors) for the GEMMs.  A: [rows, K] bf16, box 128 x 64.
// B: [groups, rows, K] bf16, box box_rows x 64.  Both with 128-byte swizzle.
CUresult encode_map_a(CUtensorMap *m, const void *ptr, int rows, int K);
// K viewed as (64, K / 64), box 64 x box_rows x 2 chunks (CTA-pair expert GEMM)
CUresult encode_map_a_kb2(CUtensorMap *m, const void *ptr, int rows, int K, int box_rows = 128);
CUresult encode_map_b_kb2(CUtensorMap *m, const void *ptr, int groups, int rows, int K, int box_rows);
CUresult encode_map_a_box(CUtensorMap *m, const void *ptr, int rows, int K, int box_rows);
// [rows, cols] bf16 (f32 = 0) or fp32 (f32 = 1) output: boxes of 32 rows x 128 bytes,
// 128-byte swizzle (the GEMM epilogue's TMA stores)
CUresult encode_map_out(CUtensorMap *m, const void *ptr, int rows, int cols, int f32);
CUresult encode_map_b(CUtensorMap *m, const void *ptr, int groups, int rows, int K, int box_rows);
// MX weights: element codes [groups, rows, K] (E4M3, one byte each) or [groups,
// rows, K / 2] (E2M1, two per byte, element 2j in the low nibble), box of one
// 64-element k-block x 128 rows; E8M0 scales [groups, K / 32, rows], box 128
// rows x 2 (the k-block's two scale blocks).  No swizzle.
CUresult encode_map_mx_codes(CUtensorMap *m, const void *ptr, int groups, int rows, int K, int wfmt,
                             int box_rows = 128);
CUresult encode_map_mx_scales(CUtensorMap *m, const void *ptr, int groups, int rows, int K, int box_rows = 128,
                              int box_blocks = 2);

// ------------------------------------------------- decode streamers (K6)
// CUDA-core kernels for few tokens per expert: each CTA streams a block of
// weight rows of one expert once (128-bit loads) and applies it to that
// expert's tokens, staged in shared memory.
struct DecodeGroups {
    const int32_t *offs;     // [E + 1] routed rows per expert
    const int32_t *active;   // [E + 1] active experts, count at active[E]
    int E;
    int shared;              // 1: one more group, the shared expert, over rows [0, T)
    int T;
};
struct DecodeGluArgs {
    DecodeGroups g;
    const __nv_bfloat16 *x_routed;  // [T*k, H] expert-sorted rows
    const __nv_bfloat16 *x_shared;  // [T, H]
    const __nv_bfloat16 *gate, *up; // [E', I, H]
    const __nv_bfloat16 *sh_gate, *sh_up;  // [S, H]
    int H, I, S;
    __nv_bfloat16 *h_routed;        // [T*k, I]
    __nv_bfloat16 *h_shared;        // [T, S]
    int act;
    float alpha, limit, beta;
    int num_sms;                    // persistent grid: kDecodeCtasPerSm CTAs per SM
};
cudaError_t launch_decode_glu(const DecodeGluArgs &a, cudaStream_t s);

struct DecodeDownArgs {
    DecodeGroups g;
    const __nv_bfloat16 *h_routed;  // [T*k, I]
    const __nv_bfloat16 *h_shared;  // [T, S]
    const __nv_bfloat16 *down;      // [E', H, I]
    const __nv_bfloat16 *sh_down;   // [H, S]
    int H, I, S;
    float *y_routed;                // [T*k, H]
    float *y_shared;                // [T, H]
    int num_sms;
};
cudaError_t launch_decode_down(const DecodeDownArgs &a, cudaStream_t s);

}  // namespace moe

// Sets the calling thread's moe_last_error() message (defined with the C ABI).
__attribute__((visibility("hidden"))) void moe_set_last_error_internal(const char *msg);
