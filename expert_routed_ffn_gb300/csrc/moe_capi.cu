// Host runtime and C ABI of libmoe.so (declared in include/moe.h).
//
// A handle owns one device allocation (the workspace, sized by max_tokens),
// the TMA descriptors of the borrowed weight tensors and of its workspace
// buffers, and a device error word.  moe_forward enqueues, on the caller's
// stream:
//   router (K1) -> dispatch scan + stable scatter/gather (K2) ->
//   gate/up + activation (K3/K5) -> down (K4/K5) -> combine (K7)
// where the two expert stages are either the tcgen05 grouped GEMMs (routed and
// shared expert tiles in one persistent launch each) or, for few tokens, the
// weight-streaming decode kernels (K6).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <string>

#include "kernels.h"
#include "moe.h"

using moe::bf16;

namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

moe_status cuda_fail(cudaError_t e, const char *what) {
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int kPathAuto = 0, kPathDecode = 1, kPathGrouped = 2, kPathSwapped = 3;
// Auto path: the tcgen05 grouped GEMMs (path 2) at every size, for bf16 and MX
// weights.  Measured on GB300: the CUDA-core decode kernels (path 1) are slower
// from T = 1 up (Zipf T = 1: 82 against 60 us per step; T = 8: 277 against 120);
// the swapped-operand GEMMs (path 3) tie path 2 at decode sizes (Nano: 40.3 + 25.0
// against 42.8 + 22.7 us) and lose 1.7x on the MiniMax-M3 block, where the shared
// expert's 2048 tokens re-read every weight tile per token tile; with MX weights
// path 3 is slower at every size (Nano MXFP8: 47 + 29 against 51 us: each of its
// 128 x 32 x 16 MMAs costs about 280 cycles to issue and it needs twice as many
// per weight as the grouped kernel's 128 x 256 x 16).  Paths 1 and 3 stay
// selectable with MOE_OPT_PATH as diagnostic alternatives.
// L2 share for the weight prefetch issued while routing, in tenths of the
// device's L2 (GB300: 126.5 MB reported).  Measured on GB300 (Nano decode, two
// runs of 50 steps each): 88 MB (0.7) 62.4 / 62.9 us per step, 72 MB 63.3 / 63.3,
// 104 MB 63.5 / 63.6.  The prefetch never exceeds the experts' gate/up weights.
// rows of an m-tile at decode sizes (gemm_tc.cu kThinRows)
constexpr int kThinRows = 32;
// 32-row m-tiles pay while the experts average at most 16 routed rows: above that, many
// experts need two or more of them and their weight tiles are streamed once per m-tile.
// Measured on GB300 (step us, 32-row tiles up to 32 / up to 16 rows per expert on
// average): MiniMax-M3 block T = 768 2138 / 1885, T = 1024 2410 / 1951; Nano decode
// T = 384 76.7 / 73.3, T = 512 87.1 / 80.1; AFMoE Zipf T = 256 217 / 206, T = 341
// 233 / 211; equal at 16 rows (Nano decode T = 256: 68.4 / 68.9).
constexpr int kThinAvgRows = 16;
#ifndef MOE_PREFETCH_L2_TENTHS
#define MOE_PREFETCH_L2_TENTHS 7
#endif
// CTAs issuing the prefetch (0: one per SM).  Measured on GB300 (Nano decode):
// from 18 CTAs the prefetch lands while the router runs without slowing it; from
// one CTA per SM it takes memory bandwidth from the latency-bound router and the
// step gets no faster.
#ifndef MOE_PREFETCH_GRID
#define MOE_PREFETCH_GRID 18
#endif

}  // namespace

void moe_set_last_error_internal(const char *msg) { g_last_error = msg; }

struct moe_handle {
    moe_config cfg;
    moe_weights w;
    int device = 0, num_sms = 0;
    unsigned long long l2_bytes = 0;  // the device's L2 size (sizes the weight prefetch)
    int H = 0, E = 0, Ep = 0, k = 0, I = 0, S = 0;  // S: shared width actually used (I when packed)
    bool has_shared = false, x_f32 = false;
    bool dense = false;        // num_experts == 0: a dense MLP layer (the shared segments only)
    int norm = 0;              // moe_norm of the sandwich norms
    float eps = 0.f;
    void *x_norm = nullptr;    // pre_mlp norm output [max_tokens, H] in the activation dtype
    const bf16 *sh_gate = nullptr, *sh_up = nullptr, *sh_down = nullptr;  // shared tensors (or slice E)
    int path_opt = kPathAuto;
    bool thin_now = false;  // this forward: 32-row m-tiles, the GEMM's 32-row A boxes (gemm_tc.cu THIN)
    unsigned long long wait_ns = 500000000ull;

    // workspace
    void *ws = nullptr;
    size_t ws_bytes = 0;
    int32_t *topk_idx = nullptr, *blk_hist = nullptr, *offs = nullptr, *tile_offs = nullptr,
            *active = nullptr, *sorted_tok = nullptr, *slot_of = nullptr;
    float *topk_w = nullptr;
    bf16 *x_sorted = nullptr, *x_bf16 = nullptr, *hbuf = nullptr, *hs = nullptr;
    // per-slot, shared and K-split partial outputs of the down projections: fp32, so
    // that the combine rounds to the output dtype once
    float *yslot = nullptr, *ys = nullptr, *ys_split = nullptr;
    void *x_stage = nullptr, *y_stage = nullptr;
    int *err = nullptr;
    bf16 *wr_parts = nullptr;  // router weights as exact bf16 splits [3, E, H]
    int *ready = nullptr;      // per-m-tile gate/up completion counters of the fused expert GEMM
    int *tile_counters = nullptr;  // [2] tile tickets of the expert GEMM launches
    int *tok_done = nullptr;   // [max_tokens] rows stored per token, for the overlapped combine
    bool combine_overlap = true;  // the combine waits per token instead of for the whole GEMM
    bool staged_stores = true;    // the expert GEMM's epilogue stores through shared memory
    bool ovl_now = false;      // this forward: combine overlapped with the grouped GEMM
    int ready_shared_base = 0; // first counter of the shared expert's m-tiles
    bool fuse_experts = true;  // gate/up and down in one persistent launch
    int pair_opt = 2;          // CTA-pair expert GEMM: 0 never, 1 always, 2 at tensor-bound sizes
    bool pair_swap = true;     // CTA pairs: m-tiles of <= 128 rows with swapped operands
    bool pair_now = false;     // the current forward's choice
    int shared_parts = 1;      // K ranges of the shared (dense) down projection this forward
    bool prefetch_opt = true;  // L2 prefetch of expert weights during routing
    cudaStream_t side = nullptr;               // the prefetch runs here, beside the routing kernels
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    int hist_stride = 0;       // block histograms are [E, hist_stride]
    unsigned long long *trace = nullptr;  // [kMaxStages][kTraceSlots] device trace (MOE_OPT_TRACE)
    bool trace_on = false;
    unsigned long long *gemm_stats = nullptr;  // [moe::kGemmStats] (MOE_OPT_TRACE)
    unsigned long long *router_stats = nullptr;  // [moe::kRouterStats] (MOE_OPT_TRACE)
    int *wr_flags = nullptr;
    moe::RouterTcPlan rplan{};

    // TMA descriptors fixed at create
    CUtensorMap m_xsorted, m_hbuf, m_hs, m_xbf16, m_gate, m_up, m_down, m_shg, m_shu, m_shd, m_wr;
    // the grouped GEMM's output store maps: routed and shared activations, routed slot rows,
    // shared output and its K-split partials
    CUtensorMap m_out_hbuf, m_out_hs, m_out_yslot, m_out_ys, m_out_ysp;
    // swapped-operand GEMMs: weight boxes of 64 (gate/up) and 128 (down) rows,
    // token boxes of 32 ([0]) or 64 ([1]) rows
    CUtensorMap m_gate64, m_up64, m_down128, m_shg64, m_shu64, m_shd128;
    CUtensorMap m_xs_n[2], m_hb_n[2], m_hs_n[2], m_xbf_n[2], m_x_n[2];
    const void *m_x_n_ptr[2] = {nullptr, nullptr};
    int m_x_n_rows[2] = {0, 0};
    // CTA-pair expert GEMM: the same tensors with K viewed as (64, K / 64), two
    // k-blocks per box (A: 128 rows; weights: 128 rows)
    CUtensorMap m_xs2, m_hb2, m_hs2, m_xbf2, m_gate2, m_up2, m_down2, m_shg2, m_shu2, m_shd2, m_x2;
    // and the token rows of its swapped-operand tiles: two k-blocks, 32 ([0]) or 64 ([1]) rows
    CUtensorMap m_xs2_n[2], m_hb2_n[2];
    // MX weights: m_gate ... m_shd map the element codes; these map their E8M0 scales
    int wfmt = 0;  // moe_weight_format
    CUtensorMap m_gate_s, m_up_s, m_down_s, m_shg_s, m_shu_s, m_shd_s;
    // and with boxes of a whole tile's scales (the swapped MX kernel: 64 rows x H/32 for
    // gate/up, 128 rows x K/32 for down; its gate/up codes go in m_gate64 ...)
    CUtensorMap m_gate_st, m_up_st, m_down_st, m_shg_st, m_shu_st, m_shd_st;
    const void *m_x2_ptr = nullptr;
    int m_x2_rows = 0;
    // descriptor of the caller's X for the shared-expert GEMM (cached by pointer and T)
    CUtensorMap m_x;
    const void *m_x_ptr = nullptr;
    int m_x_rows = 0;

    int last_path = 0, last_launches = 0, last_T = 0;

    // optional per-kernel timing of moe_forward
    static constexpr int kMaxStages = 8;
    bool stage_events = false;
    // moe_forward_host replayed from a CUDA graph: the copy in, the forward and the copy
    // out, captured on the second call with the same buffers, T and options
    bool graph_opt = true;
    unsigned opt_gen = 0;  // bumped by every option change
    cudaGraphExec_t graph_exec = nullptr;
    const void *g_x = nullptr;
    void *g_y = nullptr;
    int g_T = -1;
    unsigned g_gen = 0;
    int g_seen = 0;        // consecutive eager calls with this key
    cudaStream_t hstream = nullptr;  // the graph runs here when the caller passes the legacy stream
    cudaEvent_t ev_host = nullptr;
    cudaEvent_t ev[kMaxStages + 1] = {};
    int ev_recorded = 0;
    const char *stage_name[kMaxStages] = {};
};

namespace {

moe_status validate_config(const moe_config *c, int *S_eff) {
    if (c->hidden_size < 64 || c->hidden_size % 64 != 0 || c->hidden_size > 8192)
        return fail(MOE_ERR_UNSUPPORTED, "hidden_size %d: need a multiple of 64 in [64, 8192]",
                    c->hidden_size);
    if (c->mlp_norm != MOE_NORM_NONE && c->mlp_norm != MOE_NORM_RMS && c->mlp_norm != MOE_NORM_GEMMA)
        return fail(MOE_ERR_INVALID_ARG, "mlp_norm %d", c->mlp_norm);
    if (c->mlp_norm != MOE_NORM_NONE && !(std::isfinite(c->rms_norm_eps) && c->rms_norm_eps >= 0.f))
        return fail(MOE_ERR_INVALID_ARG, "rms_norm_eps must be finite and >= 0");
    if (c->num_shared_experts < 0 || c->shared_intermediate_size < 0)
        return fail(MOE_ERR_INVALID_ARG, "negative shared expert count or width");
    if (c->weight_format != MOE_WEIGHTS_BF16 && c->weight_format != MOE_WEIGHTS_MXFP8 &&
        c->weight_format != MOE_WEIGHTS_MXFP4)
        return fail(MOE_ERR_INVALID_ARG, "weight_format %d", c->weight_format);
    if (c->num_experts == 0) {
        // a dense MLP layer: no router, the shared tensors are its gate/up/down
        if (c->num_experts_per_tok != 0 || c->shared_packed)
            return fail(MOE_ERR_INVALID_ARG, "a dense layer (num_experts 0) has num_experts_per_tok 0, no packing");
        const int S = c->shared_intermediate_size;
        if (S < 64 || S % 64 != 0 || S > 16384)
            return fail(MOE_ERR_UNSUPPORTED, "dense width %d: need a multiple of 64 in [64, 16384]", S);
        if (c->hidden_act != MOE_ACT_SILU && c->hidden_act != MOE_ACT_SWIGLU_OAI)
            return fail(MOE_ERR_INVALID_ARG, "hidden_act %d", c->hidden_act);
        if (c->act_dtype == MOE_DTYPE_F32)  // the dense layers run bf16 activations
            return fail(MOE_ERR_UNSUPPORTED, "a dense layer takes bf16 activations");
        if (c->act_dtype != MOE_DTYPE_BF16)
            return fail(MOE_ERR_INVALID_ARG, "act_dtype %d", c->act_dtype);
        if (c->max_tokens < 1 || c->max_tokens > (1 << 24))
            return fail(MOE_ERR_INVALID_ARG, "max_tokens %d: need 1..2^24", c->max_tokens);
        *S_eff = S;
        return MOE_OK;
    }
    if (c->num_experts < 1 || c->num_experts > 256)
        return fail(MOE_ERR_UNSUPPORTED, "num_experts %d: need 0 (dense) or 1..256", c->num_experts);
    if (c->num_experts_per_tok < 1 || c->num_experts_per_tok > c->num_experts ||
        c->num_experts_per_tok > 16)
        return fail(MOE_ERR_INVALID_ARG, "num_experts_per_tok %d: need 1..min(num_experts, 16)",
                    c->num_experts_per_tok);
    if (c->moe_intermediate_size < 64 || c->moe_intermediate_size % 64 != 0 ||
        c->moe_intermediate_size > 8192)
        return fail(MOE_ERR_UNSUPPORTED, "moe_intermediate_size %d: need a multiple of 64 in [64, 8192]",
                    c->moe_intermediate_size);
    int S = 0;
    if (c->shared_packed) {
        if (c->shared_intermediate_size != 0 && c->shared_intermediate_size != c->moe_intermediate_size)
            return fail(MOE_ERR_INVALID_ARG,
                        "a packed shared expert has the routed width (%d), got shared_intermediate_size %d",
                        c->moe_intermediate_size, c->shared_intermediate_size);
        S = c->moe_intermediate_size;
    } else {
        S = c->shared_intermediate_size ? c->shared_intermediate_size
                                        : c->num_shared_experts * c->moe_intermediate_size;
        if (S % 64 != 0 || S > 8192)
            return fail(MOE_ERR_UNSUPPORTED, "shared width %d: need a multiple of 64, at most 8192", S);
    }
    if (c->score_func != MOE_SCORE_SIGMOID && c->score_func != MOE_SCORE_SOFTMAX)
        return fail(MOE_ERR_INVALID_ARG, "score_func %d", c->score_func);
    if (c->hidden_act != MOE_ACT_SILU && c->hidden_act != MOE_ACT_SWIGLU_OAI)
        return fail(MOE_ERR_INVALID_ARG, "hidden_act %d", c->hidden_act);
    if (c->act_dtype != MOE_DTYPE_BF16 && c->act_dtype != MOE_DTYPE_F32)
        return fail(MOE_ERR_INVALID_ARG, "act_dtype %d", c->act_dtype);
    if (!std::isfinite(c->route_scale))
        return fail(MOE_ERR_INVALID_ARG, "route_scale is not finite");
    if (c->max_tokens < 1 || (long long)c->max_tokens * c->num_experts_per_tok > (1ll << 24))
        return fail(MOE_ERR_INVALID_ARG, "max_tokens %d: need 1..2^24/k", c->max_tokens);
    *S_eff = S;
    return MOE_OK;
}

// elements of the K-split partial-output buffer: parts * T * H <= SMs * 128 * 256
// whenever a split is taken (parts * output tiles <= CTAs or CTA pairs)
size_t split_elems(const moe_handle *h) { return (size_t)h->num_sms * moe::kGemmBM * moe::kGemmBN; }

// K ranges of the shared (dense) down projection on the grouped path.  Its tiles
// are few at small T and each streams a whole K = S of weights: a MoE layer
// splits K in two when the tiles fill at most a quarter of the SMs (one CTA per
// tile); a dense layer, whose down projection is the whole second half of its
// work, takes the largest power of two (<= 16) that keeps parts x tiles within
// the CTAs (CTA pairs) and at least 4 k-blocks (an even number with CTA pairs)
// per part.
int shared_parts(const moe_handle *h, int T) {
    const int bm = h->pair_now ? 2 * moe::kGemmBM : moe::kGemmBM;
    const long long tiles = (long long)((T + bm - 1) / bm) * ((h->H + moe::kGemmBN - 1) / moe::kGemmBN);
    const int kb = h->S / 64;
    int parts = 1;
    if (!h->dense) {
        if (!h->pair_now && kb % 2 == 0 && tiles * 4 <= h->num_sms) parts = 2;
    } else {
        const int units = h->pair_now ? h->num_sms / 2 : h->num_sms;
        for (int p = 16; p >= 2; p >>= 1) {
            const int per = kb / p;
            if (kb % p == 0 && per >= 4 && (!h->pair_now || per % 2 == 0) && tiles * p <= units) {
                parts = p;
                break;
            }
        }
    }
    while (parts > 1 && (size_t)parts * T * h->H > split_elems(h)) parts >>= 1;
    return parts;
}

struct Carver {
    size_t off = 0;
    template <class T>
    T *take(void *base, size_t count) {
        off = round_up(off, 256);
        T *p = base ? reinterpret_cast<T *>(static_cast<char *>(base) + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

void carve(moe_handle *h, void *base) {
    const size_t MT = h->cfg.max_tokens, k = h->k, H = h->H, E = h->E;
    const size_t nb = (MT + 7) / 8;  // token blocks of at least 8
    const size_t elt = h->x_f32 ? 4 : 2;
    Carver c;
    h->err = c.take<int>(base, 64);
    h->topk_idx = c.take<int32_t>(base, MT * k);
    h->topk_w = c.take<float>(base, MT * k);
    h->hist_stride = (int)nb;
    h->blk_hist = c.take<int32_t>(base, nb * E);
    h->offs = c.take<int32_t>(base, E + 1);
    h->tile_offs = c.take<int32_t>(base, E + 1);
    h->active = c.take<int32_t>(base, E + 1);
    h->sorted_tok = c.take<int32_t>(base, MT * k);
    h->slot_of = c.take<int32_t>(base, MT * k);
    h->x_sorted = c.take<bf16>(base, MT * k * H);
    h->x_bf16 = h->x_f32 ? c.take<bf16>(base, MT * H) : nullptr;
    h->hbuf = c.take<bf16>(base, MT * k * h->I);
    h->hs = h->has_shared ? c.take<bf16>(base, MT * h->S) : nullptr;
    h->yslot = c.take<float>(base, MT * k * H);
    h->ys = h->has_shared ? c.take<float>(base, MT * H) : nullptr;
    // partial products of a K-split shared down projection: the split is taken only
    // while parts x output tiles fit the SMs, so parts * T * H <= SMs * 128 * 256
    h->ys_split = h->has_shared ? c.take<float>(base, split_elems(h)) : nullptr;
    h->x_stage = c.take<char>(base, MT * H * elt);
    h->x_norm = h->norm ? c.take<char>(base, MT * H * elt) : nullptr;
    h->y_stage = c.take<char>(base, MT * H * elt);
    h->wr_parts = c.take<bf16>(base, 3 * E * H);
    h->trace = c.take<unsigned long long>(base, MOE_TRACE_FIELDS * moe_handle::kMaxStages);
    h->gemm_stats = c.take<unsigned long long>(base, moe::kGemmStats);
    h->router_stats = c.take<unsigned long long>(base, moe::kRouterStats);
    // routed m-tiles number at most T*k/32 + E (32-row m-tiles at decode sizes; with
    // CTA pairs 2 counters per 256-row tile: at most T*k/128 + 2E + 2); the shared
    // expert's follow (at most ceil(T/32) + 2)
    h->ready_shared_base = (int)(MT * k / kThinRows + 2 * E + 2);
    const size_t shared_counters = std::max((MT + kThinRows - 1) / kThinRows, 2 * ((MT + 255) / 256)) + 2;
    h->ready = c.take<int>(base, (size_t)h->ready_shared_base + shared_counters);
    h->wr_flags = c.take<int>(base, 64);
    h->tile_counters = c.take<int>(base, 64);
    h->tok_done = c.take<int>(base, (size_t)MT);
    h->ws_bytes = round_up(c.off, 256);
}

moe_status build_maps(moe_handle *h) {
    const int MT = h->cfg.max_tokens, k = h->k, H = h->H, I = h->I, S = h->S, Ep = h->Ep;
    CUresult r = CUDA_SUCCESS;
#define MAP(call)                                                                        \
    do {                                                                                 \
        r = (call);                                                                      \
        if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", #call, (int)r); \
    } while (0)
    if (!h->dense) {
    MAP(moe::encode_map_out(&h->m_out_hbuf, h->hbuf, MT * k, I, 0));
    MAP(moe::encode_map_out(&h->m_out_yslot, h->yslot, MT * k, H, 1));
    MAP(moe::encode_map_a(&h->m_xsorted, h->x_sorted, MT * k, H));
    MAP(moe::encode_map_a(&h->m_hbuf, h->hbuf, MT * k, I));
    MAP(moe::encode_map_a_kb2(&h->m_xs2, h->x_sorted, MT * k, H));
    MAP(moe::encode_map_a_kb2(&h->m_hb2, h->hbuf, MT * k, I));
    for (int v = 0; v < 2; ++v) {
        MAP(moe::encode_map_a_kb2(&h->m_xs2_n[v], h->x_sorted, MT * k, H, v ? 64 : 32));
        MAP(moe::encode_map_a_kb2(&h->m_hb2_n[v], h->hbuf, MT * k, I, v ? 64 : 32));
    }
    MAP(moe::encode_map_b(&h->m_wr, h->wr_parts, h->rplan.parts, h->E, H, h->rplan.Np));
    if (h->wfmt != MOE_WEIGHTS_BF16) {
        MAP(moe::encode_map_mx_codes(&h->m_gate, h->w.gate, Ep, I, H, h->wfmt));
        MAP(moe::encode_map_mx_codes(&h->m_up, h->w.up, Ep, I, H, h->wfmt));
        MAP(moe::encode_map_mx_codes(&h->m_down, h->w.down, Ep, H, I, h->wfmt));
        MAP(moe::encode_map_mx_scales(&h->m_gate_s, h->w.gate_scale, Ep, I, H));
        MAP(moe::encode_map_mx_scales(&h->m_up_s, h->w.up_scale, Ep, I, H));
        MAP(moe::encode_map_mx_scales(&h->m_down_s, h->w.down_scale, Ep, H, I));
        MAP(moe::encode_map_mx_codes(&h->m_gate64, h->w.gate, Ep, I, H, h->wfmt, 64));
        MAP(moe::encode_map_mx_codes(&h->m_up64, h->w.up, Ep, I, H, h->wfmt, 64));
        MAP(moe::encode_map_mx_scales(&h->m_gate_st, h->w.gate_scale, Ep, I, H, 64, H / 32));
        MAP(moe::encode_map_mx_scales(&h->m_up_st, h->w.up_scale, Ep, I, H, 64, H / 32));
        MAP(moe::encode_map_mx_scales(&h->m_down_st, h->w.down_scale, Ep, H, I, 128, I / 32));
    } else {
    MAP(moe::encode_map_b_kb2(&h->m_gate2, h->w.gate, Ep, I, H, 128));
    MAP(moe::encode_map_b_kb2(&h->m_up2, h->w.up, Ep, I, H, 128));
    MAP(moe::encode_map_b_kb2(&h->m_down2, h->w.down, Ep, H, I, 128));
    MAP(moe::encode_map_b(&h->m_gate, h->w.gate, Ep, I, H, 128));
    MAP(moe::encode_map_b(&h->m_up, h->w.up, Ep, I, H, 128));
    MAP(moe::encode_map_b(&h->m_down, h->w.down, Ep, H, I, moe::kGemmBN));
    MAP(moe::encode_map_b(&h->m_gate64, h->w.gate, Ep, I, H, 64));
    MAP(moe::encode_map_b(&h->m_up64, h->w.up, Ep, I, H, 64));
    MAP(moe::encode_map_b(&h->m_down128, h->w.down, Ep, H, I, 128));
    }
    }
    for (int v = 0; v < 2; ++v) {
        const int n = v ? 64 : 32;
        if (!h->dense) {
            MAP(moe::encode_map_a_box(&h->m_xs_n[v], h->x_sorted, MT * k, H, n));
            MAP(moe::encode_map_a_box(&h->m_hb_n[v], h->hbuf, MT * k, I, n));
        }
        if (h->has_shared) MAP(moe::encode_map_a_box(&h->m_hs_n[v], h->hs, MT, S, n));
        if (h->has_shared && h->x_f32) MAP(moe::encode_map_a_box(&h->m_xbf_n[v], h->x_bf16, MT, H, n));
    }
    if (h->has_shared) {
        MAP(moe::encode_map_out(&h->m_out_hs, h->hs, MT, S, 0));
        MAP(moe::encode_map_out(&h->m_out_ys, h->ys, MT, H, 1));
        MAP(moe::encode_map_out(&h->m_out_ysp, h->ys_split, (int)(split_elems(h) / H), H, 1));
        MAP(moe::encode_map_a(&h->m_hs, h->hs, MT, S));
        if (h->x_f32) MAP(moe::encode_map_a(&h->m_xbf16, h->x_bf16, MT, H));
        MAP(moe::encode_map_a_kb2(&h->m_hs2, h->hs, MT, S));
        if (h->x_f32) MAP(moe::encode_map_a_kb2(&h->m_xbf2, h->x_bf16, MT, H));
        if (h->cfg.shared_packed) {
            h->m_shg = h->m_gate;
            h->m_shu = h->m_up;
            h->m_shd = h->m_down;
            h->m_shg_s = h->m_gate_s;
            h->m_shu_s = h->m_up_s;
            h->m_shd_s = h->m_down_s;
            h->m_shg_st = h->m_gate_st;
            h->m_shu_st = h->m_up_st;
            h->m_shd_st = h->m_down_st;
            h->m_shg64 = h->m_gate64;
            h->m_shu64 = h->m_up64;
            h->m_shd128 = h->m_down128;
            h->m_shg2 = h->m_gate2;
            h->m_shu2 = h->m_up2;
            h->m_shd2 = h->m_down2;
        } else if (h->wfmt != MOE_WEIGHTS_BF16) {
            MAP(moe::encode_map_mx_codes(&h->m_shg, h->w.sh_gate, 1, S, H, h->wfmt));
            MAP(moe::encode_map_mx_codes(&h->m_shu, h->w.sh_up, 1, S, H, h->wfmt));
            MAP(moe::encode_map_mx_codes(&h->m_shd, h->w.sh_down, 1, H, S, h->wfmt));
            MAP(moe::encode_map_mx_scales(&h->m_shg_s, h->w.sh_gate_scale, 1, S, H));
            MAP(moe::encode_map_mx_scales(&h->m_shu_s, h->w.sh_up_scale, 1, S, H));
            MAP(moe::encode_map_mx_scales(&h->m_shd_s, h->w.sh_down_scale, 1, H, S));
            MAP(moe::encode_map_mx_codes(&h->m_shg64, h->w.sh_gate, 1, S, H, h->wfmt, 64));
            MAP(moe::encode_map_mx_codes(&h->m_shu64, h->w.sh_up, 1, S, H, h->wfmt, 64));
            MAP(moe::encode_map_mx_scales(&h->m_shg_st, h->w.sh_gate_scale, 1, S, H, 64, H / 32));
            MAP(moe::encode_map_mx_scales(&h->m_shu_st, h->w.sh_up_scale, 1, S, H, 64, H / 32));
            MAP(moe::encode_map_mx_scales(&h->m_shd_st, h->w.sh_down_scale, 1, H, S, 128, S / 32));
        } else {
            MAP(moe::encode_map_b(&h->m_shg, h->w.sh_gate, 1, S, H, 128));
            MAP(moe::encode_map_b(&h->m_shu, h->w.sh_up, 1, S, H, 128));
            MAP(moe::encode_map_b(&h->m_shd, h->w.sh_down, 1, H, S, moe::kGemmBN));
            MAP(moe::encode_map_b(&h->m_shg64, h->w.sh_gate, 1, S, H, 64));
            MAP(moe::encode_map_b(&h->m_shu64, h->w.sh_up, 1, S, H, 64));
            MAP(moe::encode_map_b(&h->m_shd128, h->w.sh_down, 1, H, S, 128));
            MAP(moe::encode_map_b_kb2(&h->m_shg2, h->w.sh_gate, 1, S, H, 128));
            MAP(moe::encode_map_b_kb2(&h->m_shu2, h->w.sh_up, 1, S, H, 128));
            MAP(moe::encode_map_b_kb2(&h->m_shd2, h->w.sh_down, 1, H, S, 128));
        }
    }
#undef MAP
    return MOE_OK;
}

moe_status check_launch(cudaError_t e, const char *what) {
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, what);
}

// Event after kernel number n (n = 0: before the first kernel).
void mark(moe_handle *h, int n, cudaStream_t s) {
    if (!h->stage_events || n > moe_handle::kMaxStages) return;
    cudaEventRecord(h->ev[n], s);
    h->ev_recorded = n + 1;
}

// Count a launch (named by `what`, e.g. "router_logits") and mark its end.
moe_status launched(moe_handle *h, cudaError_t e, const char *what, int *n, cudaStream_t s) {
    if (e != cudaSuccess) return cuda_fail(e, what);
    if (*n < moe_handle::kMaxStages) h->stage_name[*n] = what;
    ++*n;
    mark(h, *n, s);
    return MOE_OK;
}

// Trace slots of the kernel about to be launched as number n, or nullptr.
unsigned long long *trace_slot(const moe_handle *h, int n) {
    return h->trace_on && n < moe_handle::kMaxStages ? h->trace + MOE_TRACE_FIELDS * n : nullptr;
}

// TMA descriptor of the caller's bf16 X (router and shared-expert A operand),
// re-encoded only when the pointer or T changes.
moe_status x_map(moe_handle *h, const void *X, int T) {
    if (h->m_x_ptr == X && h->m_x_rows == T) return MOE_OK;
    CUresult r = moe::encode_map_a(&h->m_x, X, T, h->H);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled(X) failed: %d", (int)r);
    h->m_x_ptr = X;
    h->m_x_rows = T;
    return MOE_OK;
}

// TMA descriptor of the caller's bf16 X with a box of 32 (v = 0) or 64 (v = 1)
// rows, cached by pointer and T.
moe_status x_map_box(moe_handle *h, const void *X, int T, int v, const CUtensorMap **out) {
    if (h->m_x_n_ptr[v] != X || h->m_x_n_rows[v] != T) {
        CUresult r = moe::encode_map_a_box(&h->m_x_n[v], X, T, h->H, v ? 64 : 32);
        if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled(X) failed: %d", (int)r);
        h->m_x_n_ptr[v] = X;
        h->m_x_n_rows[v] = T;
    }
    *out = &h->m_x_n[v];
    return MOE_OK;
}

// Cluster size of the tensor-core router: the largest power of two that keeps
// about one CTA per SM and at least one k-block per CTA, up to 8 for at most 8
// m-tiles (the clusters then fit on the GPU at once) and 4 beyond.
int router_splits(const moe_handle *h, int T) {
    const int nk = h->H / 64, mtiles = (T + 127) / 128;
    const int cap = mtiles <= 8 ? moe::kMaxRouterSplits : 4;
    int want = h->num_sms / mtiles, sp = 1;
    while (sp * 2 <= want && sp * 2 <= cap && sp * 2 <= nk) sp *= 2;
    return sp;
}

// Router for bf16 X: logits on the tensor cores and the routing rule, one
// launch (clusters of router_splits CTAs per m-tile).  Token blocks of the
// histograms hold 128 / router_splits tokens.
moe_status run_router_tc(moe_handle *h, const void *X, int T, int32_t *topk_idx, float *topk_w,
                         int32_t *blk_hist, cudaStream_t s, int *n) {
    moe_status st = x_map(h, X, T);
    if (st != MOE_OK) return st;
    moe::RouterTcArgs ra{};
    ra.mapX = h->m_x;
    ra.mapW = h->m_wr;
    ra.T = T;
    ra.H = h->H;
    ra.E = h->E;
    ra.Np = h->rplan.Np;
    ra.parts = h->rplan.parts;
    ra.stages = h->rplan.stages;
    ra.tmem_cols = h->rplan.tmem_cols;
    ra.splits = router_splits(h, T);
    ra.staged_push = h->rplan.staged_push;
    ra.kb_per_split = (h->H / 64 + ra.splits - 1) / ra.splits;
    ra.k = h->k;
    ra.bias = h->w.expert_bias;
    ra.score_func = h->cfg.score_func;
    ra.route_norm = h->cfg.route_norm;
    ra.route_scale = h->cfg.route_scale;
    ra.topk_idx = topk_idx;
    ra.topk_w = topk_w;
    ra.blk_hist = blk_hist;
    ra.hb = 1;  // expert-major histograms: each expert's blocks are contiguous
    ra.he = h->hist_stride;
    ra.err = h->err;
    ra.wait_ns = h->wait_ns;
    ra.trace = trace_slot(h, *n);
    ra.stats = h->trace_on ? h->router_stats : nullptr;
    return launched(h, moe::launch_router_tc(ra, h->rplan.smem, s), "router", n, s);
}

// Router + dispatch, shared by all paths (tile_m: rows per tile counted by
// tile_offs).  Returns launches through *n.
moe_status run_front(moe_handle *h, const void *X, int T, cudaStream_t s, int *n, int tile_m) {
    // bf16 X: tensor-core router; fp32 X: CUDA-core router
    const int TT = h->x_f32 ? moe::router_tokens_per_block(T, h->num_sms) : 128 / router_splits(h, T);
    const int nb = (T + TT - 1) / TT;
    if (!h->x_f32) {
        moe_status st = run_router_tc(h, X, T, h->topk_idx, h->topk_w, h->blk_hist, s, n);
        if (st != MOE_OK) return st;
    } else {
    moe::RouterArgs ra{};
    ra.X = X;
    ra.x_f32 = h->x_f32;
    ra.T = T;
    ra.H = h->H;
    ra.E = h->E;
    ra.k = h->k;
    ra.Wr = h->w.router_w;
    ra.bias = h->w.expert_bias;
    ra.score_func = h->cfg.score_func;
    ra.route_norm = h->cfg.route_norm;
    ra.route_scale = h->cfg.route_scale;
    ra.topk_idx = h->topk_idx;
    ra.topk_w = h->topk_w;
    ra.blk_hist = h->blk_hist;
    ra.x_bf16 = h->x_f32 && h->has_shared ? h->x_bf16 : nullptr;
    ra.hb = 1;
    ra.he = h->hist_stride;
    ra.tokens_per_block = TT;
    ra.trace = trace_slot(h, *n);
    moe_status st = launched(h, moe::launch_router(ra, s), "router", n, s);
    if (st != MOE_OK) return st;
    }

    moe_status st = MOE_OK;

    moe::ScatterArgs xa{};
    xa.topk_idx = h->topk_idx;
    xa.blk_hist = h->blk_hist;
    xa.hb = 1;
    xa.he = h->hist_stride;
    xa.offs = h->offs;
    xa.tile_offs = h->tile_offs;
    xa.active = h->active;
    xa.tile_m = tile_m;
    xa.ready = h->ready;
    xa.ready_shared_base = h->ready_shared_base;
    xa.ready_per_tile = h->pair_now ? 2 : 1;
    xa.ready_shared_count = h->pair_now ? 2 * ((T + 255) / 256) : (h->thin_now ? (T + kThinRows - 1) / kThinRows
                                                                               : (T + 127) / 128);
    xa.tile_counters = h->tile_counters;
    xa.T = T;
    xa.k = h->k;
    xa.E = h->E;
    xa.H = h->H;
    xa.tokens_per_block = TT;
    {
        // spread the row gather over about two CTAs per SM, at least 8 rows per CTA and no
        // more CTAs than are resident at once; then take a split whose busiest SM copies at
        // least 10% fewer rows (ceil(nb * g / SMs) / g blocks' worth), if every SM still
        // gets a CTA (measured: MiniMax-M3 dispatch 36.3 -> 31.2 us with 7 instead of 5)
        const int per_block_rows = TT * h->k;
        const int gmax = std::max(1, std::min((per_block_rows + 7) / 8, moe::scatter_ctas_per_sm() * h->num_sms / nb));
        const int g = std::min(std::max(1, (2 * h->num_sms + nb - 1) / nb), gmax);
        auto busiest = [&](int x) { return (double)((nb * x + h->num_sms - 1) / h->num_sms) / x; };
        int best = g;
        for (int x = 1; x <= gmax; ++x)
            if (nb * x >= h->num_sms && busiest(x) < 0.9 * busiest(best)) best = x;
        xa.gather_split = best;
    }
    xa.X = X;
    xa.x_f32 = h->x_f32;
    xa.sorted_tok = h->sorted_tok;
    xa.slot_of = h->slot_of;
    xa.x_sorted = h->x_sorted;
    xa.err = h->err;
    xa.tok_done = h->tok_done;
    xa.trace = trace_slot(h, *n);
    st = launched(h, moe::launch_scatter(xa, s), "dispatch_scatter", n, s);
    if (st != MOE_OK) return st;
    return MOE_OK;
}

// tcgen05 grouped GEMMs (tokens as M): routed and shared segments of the
// gate/up and down projections, in one persistent launch (the down tiles wait
// per m-tile for their gate/up rows) or in two launches.
moe_status run_grouped(moe_handle *h, const void *X, int T, cudaStream_t s, int *n) {
    const int H = h->H, I = h->I, S = h->S, E = h->E;
    enum { kXs = 0, kX = 1, kHb = 2, kHs = 3, kG = 4, kU = 5, kSG = 6, kSU = 7, kD = 8, kSD = 9,
           kGs = 10, kUs = 11, kSGs = 12, kSUs = 13, kDs = 14, kSDs = 15 };
    // bf16 CTA pairs (no scale maps): the swapped tiles' token and 64-row weight maps
    enum { kXw32 = 10, kXw64 = 11, kHw32 = 12, kHw64 = 13, kGw = 14, kUw = 15 };
    // the epilogue's output store maps
    enum { kOutH = 16, kOutHs = 17, kOutY = 18, kOutYs = 19 };
    const bool mx = h->wfmt != MOE_WEIGHTS_BF16;
    moe::GemmArgs g{};
    g.err = h->err;
    g.wait_ns = h->wait_ns;
    g.act = h->cfg.hidden_act;
    g.alpha = h->cfg.act_alpha;
    g.limit = h->cfg.act_limit;
    g.beta = h->cfg.act_beta;
    // CTA pairs: an even grid, static tile order, down weights in 128-row boxes
    // (each CTA of a pair loads half of a 256-row tile); the bf16 kernel's pair stages
    // hold two k-blocks (maps with two-k-block boxes), the MX kernel's one
    const bool pair = h->pair_now;
    const bool kb2 = pair && !mx;
    g.pair = pair ? 1 : 0;
    g.num_ctas = pair ? h->num_sms / 2 * 2 : h->num_sms;
    // unused slots hold a valid descriptor (a dense layer has only the shared ones)
    for (auto &m : g.maps) m = h->dense ? h->m_hs : h->m_xsorted;
    if (!h->dense) {
        g.maps[kXs] = kb2 ? h->m_xs2 : h->m_xsorted;
        g.maps[kHb] = kb2 ? h->m_hb2 : h->m_hbuf;
        g.maps[kG] = kb2 ? h->m_gate2 : h->m_gate;
        g.maps[kU] = kb2 ? h->m_up2 : h->m_up;
        g.maps[kD] = kb2 ? h->m_down2 : h->m_down;
        if (mx) {
            g.maps[kGs] = h->m_gate_s;
            g.maps[kUs] = h->m_up_s;
            g.maps[kDs] = h->m_down_s;
        }
    }
    // expert tiles of at most 128 rows on CTA pairs: weights as M, tokens as N
    const bool swap = pair && !mx && !h->dense && h->pair_swap;
    g.swap_rem = swap ? 1 : 0;
    if (swap) {
        g.maps[kXw32] = h->m_xs2_n[0];
        g.maps[kXw64] = h->m_xs2_n[1];
        g.maps[kHw32] = h->m_hb2_n[0];
        g.maps[kHw64] = h->m_hb2_n[1];
        g.maps[kGw] = h->m_gate64;
        g.maps[kUw] = h->m_up64;
    }
    if (h->has_shared) {
        if (h->x_f32) {
            g.maps[kX] = kb2 ? h->m_xbf2 : h->m_xbf16;
        } else if (kb2) {
            if (h->m_x2_ptr != X || h->m_x2_rows != T) {
                CUresult r = moe::encode_map_a_kb2(&h->m_x2, X, T, H);
                if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled(X) failed: %d", (int)r);
                h->m_x2_ptr = X;
                h->m_x2_rows = T;
            }
            g.maps[kX] = h->m_x2;
        } else {
            moe_status st = x_map(h, X, T);
            if (st != MOE_OK) return st;
            g.maps[kX] = h->m_x;
        }
        g.maps[kHs] = kb2 ? h->m_hs2 : h->m_hs;
        g.maps[kSG] = kb2 ? h->m_shg2 : h->m_shg;
        g.maps[kSU] = kb2 ? h->m_shu2 : h->m_shu;
        g.maps[kSD] = kb2 ? h->m_shd2 : h->m_shd;
        if (mx) {
            g.maps[kSGs] = h->m_shg_s;
            g.maps[kSUs] = h->m_shu_s;
            g.maps[kSDs] = h->m_shd_s;
        }
    }
    g.wfmt = h->wfmt;
    // MX weights on 128-row tiles with at least 32 routed rows per expert on average: the
    // weight stream outruns eight converter warps (measured on GB300: MiniMax-M3 MXFP8
    // 2797 -> 2636 us with sixteen; at Nano decode sizes, 16 rows per expert, sixteen
    // are slower: 76.2 -> 77.2 us)
    g.mx_conv16 = mx && !pair && E > 0 && (long long)T * h->k >= 32ll * E ? 1 : 0;
    // decode sizes: 32-row m-tiles (the dispatch counted them), A rows in 32-row
    // boxes, so the ring holds more weights
    const bool thin = h->thin_now;
    g.thin = thin ? 1 : 0;
    if (thin) {
        if (!h->dense) {
            g.maps[kXs] = h->m_xs_n[0];
            g.maps[kHb] = h->m_hb_n[0];
        }
        if (h->has_shared) {
            if (h->x_f32) {
                g.maps[kX] = h->m_xbf_n[0];
            } else {
                const CUtensorMap *mx32 = nullptr;
                moe_status st = x_map_box(h, X, T, 0, &mx32);
                if (st != MOE_OK) return st;
                g.maps[kX] = *mx32;
            }
            g.maps[kHs] = h->m_hs_n[0];
        }
    }
    const int sh_base = h->cfg.shared_packed ? E : 0;
    const int nt_gu = (I + 127) / 128, nt_sgu = (S + 127) / 128, nt_d = (H + moe::kGemmBN - 1) / moe::kGemmBN;
    const bool fused = h->fuse_experts;
    int *sig = fused ? h->ready : nullptr;
    moe::GemmSegment gu{0, E, 0, 0, h->offs, h->tile_offs, nt_gu, H / 64, 0, I, h->hbuf, I,
                              1, kXs, kG, kU, sig, nullptr, 0, 0, 0, 0, kGs, kUs,
                              {swap ? kXw32 : 0, swap ? kXw64 : 0}, swap ? kGw : 0, swap ? kUw : 0};
    moe::GemmSegment sgu{1, 1, sh_base, T, nullptr, nullptr, nt_sgu, H / 64, 0, S, h->hs, S,
                               1, kX, kSG, kSU, sig, nullptr, 0, h->ready_shared_base, 0, 0, kSGs, kSUs};
    int *const tok_done = h->ovl_now ? h->tok_done : nullptr;  // the combine waits per token
    moe::GemmSegment dn{0, E, 0, 0, h->offs, h->tile_offs, nt_d, I / 64, 0, H, h->yslot, H,
                              0, kHb, kD, kD, nullptr, fused ? h->ready : nullptr, nt_gu, 0, 0, 0, kDs, kDs,
                              {swap ? kHw32 : 0, swap ? kHw64 : 0}, 0, 0, tok_done, h->sorted_tok};
    // At small T the shared down projection (K = S) is the longest tile chain: its K
    // runs as `parts` ranges into as many partial outputs, which the combine adds in
    // fixed order (for two concatenated shared experts of width I and two parts,
    // the parts are exactly the two experts).
    const int parts = h->shared_parts;
    moe::GemmSegment sdn{1, 1, sh_base, T, nullptr, nullptr, nt_d, S / 64 / parts, 0, H,
                         parts > 1 ? h->ys_split : h->ys, H, 0, kHs, kSD, kSD, nullptr,
                         fused ? h->ready : nullptr, nt_sgu, h->ready_shared_base, parts, (size_t)T * H,
                         kSDs, kSDs, {0, 0}, 0, 0, tok_done, nullptr};
    // output store maps (the epilogue of tiles with the tokens as M); the K-split partials
    // are rows ks * T + token of one [parts * T, H] map
    if (h->staged_stores) {
        g.maps[kOutH] = h->dense ? g.maps[kOutH] : h->m_out_hbuf;
        g.maps[kOutY] = h->dense ? g.maps[kOutY] : h->m_out_yslot;
        if (h->has_shared) {
            g.maps[kOutHs] = h->m_out_hs;
            g.maps[kOutYs] = parts > 1 ? h->m_out_ysp : h->m_out_ys;
        }
        gu.map_out = kOutH;
        dn.map_out = kOutY;
        sgu.map_out = kOutHs;
        sdn.map_out = kOutYs;
    }
    if (fused) {
        int ns = 0;
        if (!h->dense) g.seg[ns++] = gu;
        if (h->has_shared) g.seg[ns++] = sgu;
        if (!h->dense) g.seg[ns++] = dn;
        if (h->has_shared) g.seg[ns++] = sdn;
        g.num_segs = ns;
        // CTA pairs claim only their last waves of tiles; MX 256-row tiles keep the static order
        g.tile_counter = pair && mx ? nullptr : h->tile_counters;
        g.trace = trace_slot(h, *n);
        g.stats = h->trace_on ? h->gemm_stats : nullptr;
        return launched(h, moe::launch_gemm_tc(g, s), "experts_gemm", n, s);
    }
    g.num_segs = 0;
    if (!h->dense) g.seg[g.num_segs++] = gu;
    if (h->has_shared) g.seg[g.num_segs++] = sgu;
    g.tile_counter = pair && mx ? nullptr : h->tile_counters;
    g.trace = trace_slot(h, *n);
    moe_status st = launched(h, moe::launch_gemm_tc(g, s), "gate_up_gemm", n, s);
    if (st != MOE_OK) return st;
    g.num_segs = 0;
    if (!h->dense) g.seg[g.num_segs++] = dn;
    if (h->has_shared) g.seg[g.num_segs++] = sdn;
    g.tile_counter = pair && mx ? nullptr : h->tile_counters + 1;
    g.trace = trace_slot(h, *n);
    return launched(h, moe::launch_gemm_tc(g, s), "down_gemm", n, s);
}

// Swapped-operand expert GEMMs on MX weights (gemm_mxt.cu): gate/up, then down,
// routed and shared segments in each launch, n_tok token rows per tile.
moe_status run_mx_swapped(moe_handle *h, const void *X, int T, cudaStream_t s, int *n, int n_tok) {
    const int H = h->H, I = h->I, S = h->S, E = h->E, v = n_tok == 32 ? 0 : 1;
    moe::MxtArgs g{};
    g.err = h->err;
    g.wait_ns = h->wait_ns;
    g.act = h->cfg.hidden_act;
    g.alpha = h->cfg.act_alpha;
    g.limit = h->cfg.act_limit;
    g.beta = h->cfg.act_beta;
    g.num_ctas = h->num_sms;
    g.wfmt = h->wfmt;
    const int sh_base = h->cfg.shared_packed ? E : 0;
    // unused map slots hold a valid descriptor
    g.Wa0 = g.Wb0 = g.Wa1 = g.Wb1 = g.Sa0 = g.Sb0 = g.Sa1 = g.Sb1 = h->m_down;
    g.X0 = g.X1 = h->m_xs_n[v];

    g.glu = 1;
    g.Wa0 = h->m_gate64;
    g.Wb0 = h->m_up64;
    g.Sa0 = h->m_gate_st;
    g.Sb0 = h->m_up_st;
    g.sblk = H / 32;
    g.X0 = h->m_xs_n[v];
    g.seg[0] = moe::SabSegment{0, E, 0, 0, h->offs, h->tile_offs, (I + 63) / 64, H / 64, I, h->hbuf, I};
    g.num_segs = 1;
    if (h->has_shared) {
        if (h->x_f32) {
            g.X1 = h->m_xbf_n[v];
        } else {
            const CUtensorMap *mx = nullptr;
            moe_status st = x_map_box(h, X, T, v, &mx);
            if (st != MOE_OK) return st;
            g.X1 = *mx;
        }
        g.Wa1 = h->m_shg64;
        g.Wb1 = h->m_shu64;
        g.Sa1 = h->m_shg_st;
        g.Sb1 = h->m_shu_st;
        g.seg[1] = moe::SabSegment{1, 1, sh_base, T, nullptr, nullptr, (S + 63) / 64, H / 64, S, h->hs, S};
        g.num_segs = 2;
    }
    g.stats = h->trace_on ? h->gemm_stats : nullptr;
    moe_status st = launched(h, moe::launch_gemm_mxt(g, n_tok, s), "gate_up_gemm_swapped", n, s);
    if (st != MOE_OK) return st;

    g.glu = 0;
    g.stats = nullptr;  // the statistics describe the gate/up launch
    g.Wa0 = g.Wb0 = h->m_down;
    g.Sa0 = g.Sb0 = h->m_down_st;
    g.sblk = I / 32;
    g.X0 = h->m_hb_n[v];
    g.seg[0] = moe::SabSegment{0, E, 0, 0, h->offs, h->tile_offs, (H + 127) / 128, I / 64, H, h->yslot, H};
    g.num_segs = 1;
    if (h->has_shared) {
        g.Wa1 = g.Wb1 = h->m_shd;
        g.Sa1 = g.Sb1 = h->m_shd_st;
        g.sblk = I > S ? I / 32 : S / 32;
        g.X1 = h->m_hs_n[v];
        g.seg[1] = moe::SabSegment{1, 1, sh_base, T, nullptr, nullptr, (H + 127) / 128, S / 64, H, h->ys, H};
        g.num_segs = 2;
    }
    return launched(h, moe::launch_gemm_mxt(g, n_tok, s), "down_gemm_swapped", n, s);
}

moe_status run_decode(moe_handle *h, const void *X, int T, cudaStream_t s, int *n) {
    moe::DecodeGroups grp{h->offs, h->active, h->E, h->has_shared ? 1 : 0, T};
    moe::DecodeGluArgs ga{};
    ga.g = grp;
    ga.x_routed = h->x_sorted;
    ga.x_shared = h->x_f32 ? h->x_bf16 : static_cast<const bf16 *>(X);
    ga.gate = static_cast<const bf16 *>(h->w.gate);
    ga.up = static_cast<const bf16 *>(h->w.up);
    ga.sh_gate = h->sh_gate;
    ga.sh_up = h->sh_up;
    ga.H = h->H;
    ga.I = h->I;
    ga.S = h->S;
    ga.h_routed = h->hbuf;
    ga.h_shared = h->hs;
    ga.act = h->cfg.hidden_act;
    ga.alpha = h->cfg.act_alpha;
    ga.limit = h->cfg.act_limit;
    ga.beta = h->cfg.act_beta;
    ga.num_sms = h->num_sms;
    moe_status st = launched(h, moe::launch_decode_glu(ga, s), "decode_gate_up", n, s);
    if (st != MOE_OK) return st;
    moe::DecodeDownArgs da{};
    da.g = grp;
    da.h_routed = h->hbuf;
    da.h_shared = h->hs;
    da.down = static_cast<const bf16 *>(h->w.down);
    da.sh_down = h->sh_down;
    da.H = h->H;
    da.I = h->I;
    da.S = h->S;
    da.y_routed = h->yslot;
    da.y_shared = h->ys;
    da.num_sms = h->num_sms;
    st = launched(h, moe::launch_decode_down(da, s), "decode_down", n, s);
    if (st != MOE_OK) return st;
    return MOE_OK;
}

// Swapped-operand expert GEMMs (weights as M, n_tok tokens as N), routed and
// shared tiles in one launch per projection.
moe_status run_swapped(moe_handle *h, const void *X, int T, cudaStream_t s, int *n, int n_tok) {
    const int H = h->H, I = h->I, S = h->S, E = h->E, v = n_tok == 32 ? 0 : 1;
    moe::SabArgs g{};
    g.err = h->err;
    g.wait_ns = h->wait_ns;
    g.act = h->cfg.hidden_act;
    g.alpha = h->cfg.act_alpha;
    g.limit = h->cfg.act_limit;
    g.beta = h->cfg.act_beta;
    g.num_ctas = h->num_sms;
    const int sh_base = h->cfg.shared_packed ? E : 0;

    g.glu = 1;
    g.Wa0 = h->m_gate64;
    g.Wb0 = h->m_up64;
    g.X0 = h->m_xs_n[v];
    g.seg[0] = moe::SabSegment{0, E, 0, 0, h->offs, h->tile_offs, (I + 63) / 64, H / 64, I, h->hbuf, I};
    g.num_segs = 1;
    if (h->has_shared) {
        if (h->x_f32) {
            g.X1 = h->m_xbf_n[v];
        } else {
            const CUtensorMap *mx = nullptr;
            moe_status st = x_map_box(h, X, T, v, &mx);
            if (st != MOE_OK) return st;
            g.X1 = *mx;
        }
        g.Wa1 = h->m_shg64;
        g.Wb1 = h->m_shu64;
        g.seg[1] = moe::SabSegment{1, 1, sh_base, T, nullptr, nullptr, (S + 63) / 64, H / 64, S, h->hs, S};
        g.num_segs = 2;
    }
    moe_status st = launched(h, moe::launch_gemm_sab(g, n_tok, s), "gate_up_gemm_swapped", n, s);
    if (st != MOE_OK) return st;

    g.glu = 0;
    g.Wa0 = h->m_down128;
    g.X0 = h->m_hb_n[v];
    g.seg[0] = moe::SabSegment{0, E, 0, 0, h->offs, h->tile_offs, (H + 127) / 128, I / 64, H, h->yslot, H};
    g.num_segs = 1;
    if (h->has_shared) {
        g.Wa1 = h->m_shd128;
        g.X1 = h->m_hs_n[v];
        g.seg[1] = moe::SabSegment{1, 1, sh_base, T, nullptr, nullptr, (H + 127) / 128, S / 64, H, h->ys, H};
        g.num_segs = 2;
    }
    return launched(h, moe::launch_gemm_sab(g, n_tok, s), "down_gemm_swapped", n, s);
}

moe_status forward_device(moe_handle *h, const void *X, int T, void *Y, cudaStream_t s) {
    int n = 0;
    const long long slots = (long long)T * h->k;
    int path = h->path_opt == kPathAuto ? kPathGrouped : h->path_opt;
    if (h->dense) path = kPathGrouped;  // a dense layer: the grouped GEMM's shared segments
    const int n_tok = slots <= 24ll * h->E ? 32 : 64;  // token tile of the swapped GEMMs
    h->ev_recorded = 0;
    // Decode-sized batches touch nearly every expert (about two or more tokens
    // per expert expected): while the routing kernels run, a side stream warms
    // L2 with the first experts' gate and up slices, the fused GEMM's first tiles.
    // Not when the dispatch's copy of the token rows alone would sweep L2 (more
    // than a quarter of it): measured on GB300, the prefetch then costs 0.2-0.7%
    // (AFMoE prefill, MiniMax-M3, Zipf T = 4096) instead of saving 2-6% (Nano
    // decode, Zipf T = 64 and 512).
    const bool prefetch = h->prefetch_opt && !h->dense && path == kPathGrouped && h->fuse_experts &&
                          slots >= 2ll * h->E && (unsigned long long)slots * h->H * 2 <= h->l2_bytes / 4 &&
                          h->side != nullptr;
    if (prefetch) {
        // bytes of one expert's gate (or up) slice: bf16, or MX codes (1 or 1/2 byte per weight)
        const unsigned long long slice = (unsigned long long)h->I * h->H *
                                         (h->wfmt == MOE_WEIGHTS_BF16 ? 4 : h->wfmt == MOE_WEIGHTS_MXFP8 ? 2 : 1) / 2;
        const unsigned long long budget = h->l2_bytes * MOE_PREFETCH_L2_TENTHS / 10;
        const unsigned long long each = budget / 2 / slice * slice, all = slice * h->E;
        moe::PrefetchArgs pa{{h->w.gate, h->w.up}, {each < all ? each : all, each < all ? each : all}};
        cudaError_t e = cudaEventRecord(h->ev_fork, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->ev_fork, 0);
        if (e == cudaSuccess) e = moe::launch_l2_prefetch(pa, MOE_PREFETCH_GRID > 0 ? MOE_PREFETCH_GRID : h->num_sms, h->side);
        if (e == cudaSuccess) e = cudaEventRecord(h->ev_join, h->side);
        if (e != cudaSuccess) return cuda_fail(e, "weight prefetch");
    }
    if (h->trace_on) {  // every slot starts at ~0 and only shrinks (atomicMin)
        cudaError_t e =
            cudaMemsetAsync(h->trace, 0xff, MOE_TRACE_FIELDS * moe_handle::kMaxStages * sizeof(unsigned long long), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(h->gemm_stats, 0, moe::kGemmStats * sizeof(unsigned long long), s);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(h->router_stats, 0, moe::kRouterStats * sizeof(unsigned long long), s);
        if (e != cudaSuccess) return cuda_fail(e, "trace reset");
    }
    // CTA pairs once the weight tiles are reused by enough rows on average: 160 with bf16
    // weights (measured on GB300, step us without / with pairs: AFMoE-shaped T = 1536
    // (144 rows) 308 / 303, T = 2048 (192) 363 / 355, Zipf T = 2048 375 / 348, Zipf
    // T = 1024 255 / 269; the HBM-bound MiniMax-M3 shape at 128 rows 2977 / 3007), 256
    // with MX weights (256-row tiles in one CTA each, two MMAs on every decoded weight
    // tile); a dense layer: T >= 256.  Not for narrow experts (I < 512): their down
    // tiles have a short K and the tile epilogues dominate (Nano-shaped, I = 256, T =
    // 4096: 216 / 245, T = 2048: 136 / 167).
    const long long pair_rows = h->wfmt == MOE_WEIGHTS_BF16 ? 160 : 256;
    h->pair_now = path == kPathGrouped && h->num_sms >= 2 &&
                  (h->pair_opt == 1 ||
                   (h->pair_opt == 2 && (h->dense ? T >= 256 : (h->I >= 512 && slots >= pair_rows * h->E))));
    // 32-row m-tiles at decode sizes: at most 16 routed rows per expert on average
    // (T * k <= 16 E) or at most 32 tokens (then no m-tile has more than 32 rows)
    h->thin_now = path == kPathGrouped && !h->pair_now && h->wfmt == MOE_WEIGHTS_BF16 &&
                  (T <= kThinRows || (h->E > 0 && slots <= (long long)kThinAvgRows * h->E));
    h->shared_parts = path == kPathGrouped && h->has_shared ? shared_parts(h, T) : 1;
    // the combine (no post-norm) overlaps the grouped expert GEMM: it waits per token for
    // the down tiles' counts instead of for the whole launch
    h->ovl_now = path == kPathGrouped && !h->dense && h->norm == 0 && h->combine_overlap;
    mark(h, 0, s);
    moe_status st = MOE_OK;
    const void *Xm = X;  // the MLP's input: X, or pre_mlp_norm(X)
    // a dense layer has no router and no dispatch: its GEMM's counters (zeroed by
    // the dispatch in a MoE layer) are zeroed by the pre-norm kernel, or here
    int *const zero_a = h->dense ? h->ready + h->ready_shared_base : nullptr;
    const int zero_a_n = h->dense ? std::max((T + kThinRows - 1) / kThinRows, 2 * ((T + 255) / 256)) + 2 : 0;
    int *const zero_b = h->dense ? h->tile_counters : nullptr;
    const int zero_b_n = h->dense ? 2 : 0;
    if (h->norm) {
        moe::NormArgs na{X, h->x_f32 ? 1 : 0, T, h->H, h->w.pre_norm_w, h->norm, h->eps, h->x_norm,
                         trace_slot(h, n), zero_a, zero_a_n, zero_b, zero_b_n};
        st = launched(h, moe::launch_rmsnorm(na, s), "pre_norm", &n, s);
        Xm = h->x_norm;
    } else if (h->dense) {
        cudaError_t e = cudaMemsetAsync(zero_a, 0, sizeof(int) * (size_t)zero_a_n, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(zero_b, 0, sizeof(int) * (size_t)zero_b_n, s);
        if (e != cudaSuccess) st = cuda_fail(e, "counter reset");
    }
    if (st == MOE_OK && !h->dense)
        st = run_front(h, Xm, T, s, &n,
                       path == kPathSwapped ? n_tok
                                            : (h->pair_now ? 2 * moe::kGemmBM : (h->thin_now ? kThinRows : moe::kGemmBM)));
    if (st == MOE_OK) {
        if (path == kPathDecode)
            st = run_decode(h, Xm, T, s, &n);
        else if (path == kPathSwapped)
            st = h->wfmt != MOE_WEIGHTS_BF16 ? run_mx_swapped(h, Xm, T, s, &n, n_tok) : run_swapped(h, Xm, T, s, &n, n_tok);
        else
            st = run_grouped(h, Xm, T, s, &n);
    }
    if (st == MOE_OK) {
        const bool split = h->shared_parts > 1;
        moe::CombineArgs ca{h->yslot, h->has_shared ? (split ? h->ys_split : h->ys) : nullptr, h->shared_parts,
                            (size_t)T * h->H, h->topk_w, h->slot_of,
                            T, h->k, h->H, Y, h->x_f32 ? 1 : 0, trace_slot(h, n),
                            h->norm, h->eps, h->w.post_norm_w, X, h->err, h->wait_ns,
                            h->ovl_now ? h->tok_done : nullptr, 2 * ((h->H + moe::kGemmBN - 1) / moe::kGemmBN)};
        st = launched(h, moe::launch_combine(ca, s), "combine", &n, s);
    }
    if (prefetch) {  // the caller's stream ends ordered after the side stream
        cudaError_t e = cudaStreamWaitEvent(s, h->ev_join, 0);
        if (e != cudaSuccess && st == MOE_OK) st = cuda_fail(e, "join of the prefetch stream");
    }
    h->last_path = path;
    h->last_launches = n;
    h->last_T = T;
    return st;
}

}  // namespace

extern "C" {

moe_status moe_create(const moe_config *config, const moe_weights *weights, moe_handle **out) {
    if (out == nullptr) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (config == nullptr || weights == nullptr) return fail(MOE_ERR_INVALID_ARG, "config or weights is NULL");
    int S = 0;
    moe_status st = validate_config(config, &S);
    if (st != MOE_OK) return st;
    const moe_weights &w = *weights;
    const bool dense = config->num_experts == 0;
    if (!dense && (!w.router_w || !w.gate || !w.up || !w.down))
        return fail(MOE_ERR_INVALID_ARG, "router_w, gate, up and down are required");
    if (config->mlp_norm != MOE_NORM_NONE && (!w.pre_norm_w || !w.post_norm_w))
        return fail(MOE_ERR_INVALID_ARG, "mlp_norm needs pre_norm_w and post_norm_w");
    const void *ptrs[] = {w.router_w, w.expert_bias, w.gate, w.up, w.down, w.sh_gate, w.sh_up, w.sh_down,
                          w.pre_norm_w, w.post_norm_w};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "weight pointer %p is not 16-byte aligned", p);
    const bool has_shared = S > 0;
    if (has_shared && !config->shared_packed && (!w.sh_gate || !w.sh_up || !w.sh_down))
        return fail(MOE_ERR_INVALID_ARG, "shared width %d needs sh_gate, sh_up and sh_down", S);
    const bool mx = config->weight_format != MOE_WEIGHTS_BF16;
    if (mx) {
        if (!dense && (!w.gate_scale || !w.up_scale || !w.down_scale))
            return fail(MOE_ERR_INVALID_ARG, "MX weights need gate_scale, up_scale and down_scale");
        if (has_shared && !config->shared_packed && (!w.sh_gate_scale || !w.sh_up_scale || !w.sh_down_scale))
            return fail(MOE_ERR_INVALID_ARG, "MX shared weights need sh_gate_scale, sh_up_scale and sh_down_scale");
        const void *sp[] = {w.gate_scale, w.up_scale, w.down_scale, w.sh_gate_scale, w.sh_up_scale, w.sh_down_scale};
        for (const void *p : sp)
            if (p && !aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "scale pointer %p is not 16-byte aligned", p);
    }

    moe_handle *h = new moe_handle();
    h->cfg = *config;
    h->w = w;
    h->H = config->hidden_size;
    h->E = config->num_experts;
    h->Ep = config->num_experts + (config->shared_packed ? 1 : 0);
    h->k = config->num_experts_per_tok;
    h->I = config->moe_intermediate_size;
    h->S = S;
    h->has_shared = has_shared;
    h->x_f32 = config->act_dtype == MOE_DTYPE_F32;
    h->dense = dense;
    h->norm = config->mlp_norm;
    h->eps = config->rms_norm_eps;
    h->wfmt = config->weight_format;
    if (config->shared_packed) {
        const size_t slice = (size_t)h->E * h->I * h->H;
        h->sh_gate = static_cast<const bf16 *>(w.gate) + slice;
        h->sh_up = static_cast<const bf16 *>(w.up) + slice;
        h->sh_down = static_cast<const bf16 *>(w.down) + slice;
    } else {
        h->sh_gate = static_cast<const bf16 *>(w.sh_gate);
        h->sh_up = static_cast<const bf16 *>(w.sh_up);
        h->sh_down = static_cast<const bf16 *>(w.sh_down);
    }
    cudaError_t e = cudaGetDevice(&h->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
    int l2 = 0;
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, h->device);
    h->l2_bytes = (unsigned long long)(l2 > 0 ? l2 : 0);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e, "device query");
    }
    carve(h, nullptr);
    e = cudaMalloc(&h->ws, h->ws_bytes);
    if (e != cudaSuccess) {
        const size_t h_bytes = h->ws_bytes;
        cudaGetLastError();
        delete h;
        return fail(MOE_ERR_OOM, "workspace of %zu bytes: %s", h_bytes, cudaGetErrorString(e));
    }
    carve(h, h->ws);
    e = cudaMemset(h->err, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(h->wr_flags, 0, sizeof(int));
    int flags = 0;
    if (!dense) {
        if (e == cudaSuccess) e = moe::launch_split_router(w.router_w, h->E, h->H, h->wr_parts, h->wr_flags, 0);
        if (e == cudaSuccess) e = cudaMemcpy(&flags, h->wr_flags, sizeof(int), cudaMemcpyDeviceToHost);
    }
    if (e != cudaSuccess) {
        cudaFree(h->ws);
        delete h;
        return cuda_fail(e, "router weight split");
    }
    if (!dense) h->rplan = moe::plan_router_tc(h->E, (flags & 2) ? 3 : (flags & 1) ? 2 : 1);
    if (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        h->side = nullptr;  // no prefetch without its stream
    }
    if (cudaStreamCreateWithFlags(&h->hstream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_host, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        h->hstream = nullptr;  // graphs then only on a caller's non-legacy stream
    }
    st = build_maps(h);
    if (st != MOE_OK) {
        cudaFree(h->ws);
        delete h;
        return st;
    }
    *out = h;
    return MOE_OK;
}

moe_status moe_route(moe_handle *h, const void *X, int T, int32_t *topk_idx, float *topk_w,
                     moe_stream_t stream) {
    if (h == nullptr) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0 || T > h->cfg.max_tokens)
        return fail(MOE_ERR_INVALID_ARG, "T = %d outside [0, max_tokens = %d]", T, h->cfg.max_tokens);
    h->last_launches = 0;
    if (T == 0) return MOE_OK;
    if (!X || !topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "X, topk_idx and topk_w are required");
    if (!aligned16(X)) return fail(MOE_ERR_INVALID_ARG, "X is not 16-byte aligned");
    if (h->dense) return fail(MOE_ERR_UNSUPPORTED, "a dense layer (num_experts 0) has no router");
    int n = 0;
    if (h->norm) {  // the router sees pre_mlp_norm(X)
        moe::NormArgs na{X, h->x_f32 ? 1 : 0, T, h->H, h->w.pre_norm_w, h->norm, h->eps, h->x_norm, nullptr};
        moe_status st = launched(h, moe::launch_rmsnorm(na, reinterpret_cast<cudaStream_t>(stream)), "pre_norm", &n,
                                 reinterpret_cast<cudaStream_t>(stream));
        if (st != MOE_OK) return st;
        X = h->x_norm;
    }
    if (!h->x_f32) {
        moe_status st =
            run_router_tc(h, X, T, topk_idx, topk_w, nullptr, reinterpret_cast<cudaStream_t>(stream), &n);
        h->last_launches = n;
        return st;
    }
    moe::RouterArgs ra{};
    ra.X = X;
    ra.x_f32 = h->x_f32;
    ra.T = T;
    ra.H = h->H;
    ra.E = h->E;
    ra.k = h->k;
    ra.Wr = h->w.router_w;
    ra.bias = h->w.expert_bias;
    ra.score_func = h->cfg.score_func;
    ra.route_norm = h->cfg.route_norm;
    ra.route_scale = h->cfg.route_scale;
    ra.topk_idx = topk_idx;
    ra.topk_w = topk_w;
    ra.blk_hist = nullptr;
    ra.x_bf16 = nullptr;
    ra.tokens_per_block = moe::router_tokens_per_block(T, h->num_sms);
    moe_status st = launched(h, moe::launch_router(ra, reinterpret_cast<cudaStream_t>(stream)), "router", &n,
                             reinterpret_cast<cudaStream_t>(stream));
    h->last_launches = n;
    return st;
}

moe_status moe_forward(moe_handle *h, const void *X, int T, void *Y, moe_stream_t stream) {
    if (h == nullptr) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0 || T > h->cfg.max_tokens)
        return fail(MOE_ERR_INVALID_ARG, "T = %d outside [0, max_tokens = %d]", T, h->cfg.max_tokens);
    h->last_launches = 0;
    if (T == 0) return MOE_OK;
    if (!X || !Y) return fail(MOE_ERR_INVALID_ARG, "X and Y are required");
    if (!aligned16(X) || !aligned16(Y)) return fail(MOE_ERR_INVALID_ARG, "X and Y must be 16-byte aligned");
    const size_t bytes = (size_t)T * h->H * (h->x_f32 ? 4 : 2);
    const char *xb = static_cast<const char *>(X), *yb = static_cast<const char *>(Y);
    if (xb < yb + bytes && yb < xb + bytes) return fail(MOE_ERR_INVALID_ARG, "X and Y overlap");
    return forward_device(h, X, T, Y, reinterpret_cast<cudaStream_t>(stream));
}

namespace {

// The host-buffer forward's stream work: copy X in, the block, copy Y out.
// Copy of n 16-byte words from the caller's page-locked host buffer: the GPU reads it
// itself over the host link.  Measured on GB300 around a 60 us step with 512 KB each
// way: 7 us per step for two such copies, against 15 us through the copy engines.
__global__ void __launch_bounds__(256) copy_words_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                         size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

// Device address of a page-locked host buffer, or nullptr (pageable memory, or the
// query failed: the copy engines then move the bytes)
void *mapped_host(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// xm, ym: mapped_host(X_host), mapped_host(Y_host)
moe_status forward_host_ops(moe_handle *h, const void *X_host, const void *xm, int T, void *Y_host, void *ym,
                            cudaStream_t s) {
    const size_t bytes = (size_t)T * h->H * (h->x_f32 ? 4 : 2);
    const size_t words = bytes / 16;
    const bool direct = xm != nullptr && ym != nullptr && bytes % 16 == 0 &&
                        ((reinterpret_cast<uintptr_t>(xm) | reinterpret_cast<uintptr_t>(ym)) & 15) == 0;
    const int grid = (int)std::min<size_t>((size_t)2 * h->num_sms, (words + 255) / 256);
    cudaError_t e = cudaSuccess;
    if (direct) {
        copy_words_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4 *>(xm), static_cast<uint4 *>(h->x_stage), words);
        e = cudaGetLastError();
    } else {
        e = cudaMemcpyAsync(h->x_stage, X_host, bytes, cudaMemcpyHostToDevice, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy of X");
    // page-locked Y: the block's last kernel (the combine) stores its rows there itself
    moe_status st = forward_device(h, h->x_stage, T, direct ? ym : h->y_stage, s);
    if (st != MOE_OK || direct) return st;
    e = cudaMemcpyAsync(Y_host, h->y_stage, bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy of Y");
    return MOE_OK;
}

// Capture forward_host_ops into h->graph_exec; false (and no graph) if anything fails.
// Only called with page-locked host buffers: a capture whose copy touched pageable
// memory crashed the host process on GB300 (pinned X, pageable Y).
bool capture_forward_host(moe_handle *h, const void *X_host, const void *xm, int T, void *Y_host, void *ym,
                          cudaStream_t s) {
    if (h->graph_exec) {
        cudaGraphExecDestroy(h->graph_exec);
        h->graph_exec = nullptr;
    }
    cudaGraph_t graph = nullptr;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    const moe_status st = forward_host_ops(h, X_host, xm, T, Y_host, ym, s);
    const cudaError_t e = cudaStreamEndCapture(s, &graph);
    bool ok = st == MOE_OK && e == cudaSuccess && graph != nullptr;
    if (ok) ok = cudaGraphInstantiate(&h->graph_exec, graph, 0) == cudaSuccess;
    if (graph) cudaGraphDestroy(graph);
    if (!ok) {
        h->graph_exec = nullptr;
        cudaGetLastError();
    }
    return ok;
}

}  // namespace

moe_status moe_forward_host(moe_handle *h, const void *X_host, int T, void *Y_host, moe_stream_t stream) {
    if (h == nullptr) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0 || T > h->cfg.max_tokens)
        return fail(MOE_ERR_INVALID_ARG, "T = %d outside [0, max_tokens = %d]", T, h->cfg.max_tokens);
    h->last_launches = 0;
    if (T == 0) return MOE_OK;
    if (!X_host || !Y_host) return fail(MOE_ERR_INVALID_ARG, "X_host and Y_host are required");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // graphs only without per-kernel events or traces (those read host-side state per call);
    // the legacy stream cannot be captured: the call (synchronous anyway) then runs on the
    // handle's own stream, after the work already queued on the caller's
    const bool graphable = h->graph_opt && !h->stage_events && !h->trace_on && (s != nullptr || h->hstream != nullptr);
    if (graphable && s == nullptr) {
        cudaError_t e = cudaEventRecord(h->ev_host, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->hstream, h->ev_host, 0);
        if (e != cudaSuccess) return cuda_fail(e, "ordering after the caller's stream");
        s = h->hstream;
    }
    const bool same = h->g_x == X_host && h->g_y == Y_host && h->g_T == T && h->g_gen == h->opt_gen;
    if (graphable && same && h->graph_exec != nullptr) {
        cudaError_t e = cudaGraphLaunch(h->graph_exec, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "graph launch of the host-buffer forward");
        return MOE_OK;
    }
    if (!same && h->graph_exec != nullptr) {  // captured for other buffers, T or options
        cudaGraphExecDestroy(h->graph_exec);
        h->graph_exec = nullptr;
    }
    h->g_seen = same ? h->g_seen + 1 : 1;
    h->g_x = X_host;
    h->g_y = Y_host;
    h->g_T = T;
    h->g_gen = h->opt_gen;
    void *xm = mapped_host(X_host), *ym = mapped_host(Y_host);
    if (graphable && h->g_seen >= 2 && xm != nullptr && ym != nullptr &&
        capture_forward_host(h, X_host, xm, T, Y_host, ym, s)) {
        // the launches recorded in the graph keep the counts and names of the eager forward
        cudaError_t e = cudaGraphLaunch(h->graph_exec, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "graph launch of the host-buffer forward");
        return MOE_OK;
    }
    moe_status st = forward_host_ops(h, X_host, xm, T, Y_host, ym, s);
    if (st != MOE_OK) return st;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
    return MOE_OK;
}

moe_status moe_sync_status(moe_handle *h) {
    if (h == nullptr) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "synchronise");
    int word = 0;
    e = cudaMemcpy(&word, h->err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(h->err, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "read of the device error word");
    if (word & moe::ERR_TIMEOUT)
        return fail(MOE_ERR_TIMEOUT, "a device wait ran out of its bound (error word 0x%x)", word);
    if (word & moe::ERR_BOUNDS)
        return fail(MOE_ERR_DEVICE_CHECK, "a device bounds check failed (error word 0x%x)", word);
    return MOE_OK;
}

void moe_destroy(moe_handle *h) {
    if (h == nullptr) return;
    cudaDeviceSynchronize();
    if (h->graph_exec) cudaGraphExecDestroy(h->graph_exec);
    if (h->hstream) cudaStreamDestroy(h->hstream);
    if (h->ev_host) cudaEventDestroy(h->ev_host);
    for (auto &e : h->ev)
        if (e != nullptr) cudaEventDestroy(e);
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    if (h->side) cudaStreamDestroy(h->side);
    cudaFree(h->ws);
    delete h;
}

const char *moe_last_error(void) { return g_last_error.c_str(); }

moe_status moe_set_option(moe_handle *h, int option, long long value) {
    if (h == nullptr) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
    ++h->opt_gen;  // a captured forward no longer matches the options
    switch (option) {
    case MOE_OPT_GRAPH:
        if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "graph %lld", value);
        h->graph_opt = value != 0;
        return MOE_OK;
    case MOE_OPT_PATH:
        if (value < kPathAuto || value > kPathSwapped) return fail(MOE_ERR_INVALID_ARG, "path %lld", value);
        if (h->wfmt != MOE_WEIGHTS_BF16 && value == kPathDecode)
            return fail(MOE_ERR_UNSUPPORTED, "MX weights run on the tensor-core paths only (2 grouped, 3 swapped)");
        h->path_opt = (int)value;
        return MOE_OK;
    case MOE_OPT_WAIT_LIMIT_NS:
        if (value < 0) return fail(MOE_ERR_INVALID_ARG, "wait limit %lld", value);
        h->wait_ns = (unsigned long long)value;
        return MOE_OK;
    case MOE_OPT_PREFETCH:
        if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "prefetch %lld", value);
        h->prefetch_opt = value != 0;
        return MOE_OK;
    case MOE_OPT_FUSE_EXPERTS:
        if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "fuse experts %lld", value);
        h->fuse_experts = value != 0;
        return MOE_OK;
    case MOE_OPT_GEMM_PAIR:
        if (value < 0 || value > 2) return fail(MOE_ERR_INVALID_ARG, "gemm pair %lld", value);
        h->pair_opt = (int)value;
        return MOE_OK;
    case MOE_OPT_COMBINE_OVERLAP:
        if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "combine overlap %lld", value);
        h->combine_overlap = value != 0;
        return MOE_OK;
    case MOE_OPT_STAGED_STORES:
        if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "staged stores %lld", value);
        h->staged_stores = value != 0;
        return MOE_OK;
    case MOE_OPT_PAIR_SWAP:
        if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "pair swap %lld", value);
        h->pair_swap = value != 0;
        return MOE_OK;
    case MOE_OPT_TRACE:
        if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "trace %lld", value);
        h->trace_on = value != 0;
        return MOE_OK;
    case MOE_OPT_STAGE_EVENTS:
        if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "stage events %lld", value);
        if (value && h->ev[0] == nullptr) {
            for (auto &e : h->ev) {
                cudaError_t r = cudaEventCreate(&e);
                if (r != cudaSuccess) return cuda_fail(r, "cudaEventCreate");
            }
        }
        h->stage_events = value != 0;
        h->ev_recorded = 0;
        return MOE_OK;
    default:
        return fail(MOE_ERR_INVALID_ARG, "unknown option %d", option);
    }
}

moe_status moe_get_stats(const moe_handle *h, moe_stats *out) {
    if (h == nullptr || out == nullptr) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    out->path = h->last_path;
    out->kernel_launches = h->last_launches;
    out->workspace_bytes = (long long)h->ws_bytes;
    return MOE_OK;
}

moe_status moe_get_stage_times(moe_handle *h, float *ms, int max, int *n) {
    if (h == nullptr || ms == nullptr || n == nullptr) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    if (!h->stage_events || h->ev_recorded < 2)
        return fail(MOE_ERR_INVALID_ARG, "no timed forward (enable MOE_OPT_STAGE_EVENTS first)");
    cudaError_t e = cudaEventSynchronize(h->ev[h->ev_recorded - 1]);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    int count = 0;
    for (int i = 0; i + 1 < h->ev_recorded && count < max; ++i) {
        e = cudaEventElapsedTime(&ms[count], h->ev[i], h->ev[i + 1]);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
        ++count;
    }
    *n = count;
    return MOE_OK;
}

moe_status moe_get_trace(moe_handle *h, double *t_us, int max, int *n) {
    if (h == nullptr || t_us == nullptr || n == nullptr) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    if (!h->trace_on || h->last_launches < 1)
        return fail(MOE_ERR_INVALID_ARG, "no traced forward (enable MOE_OPT_TRACE first)");
    cudaError_t e = cudaSetDevice(h->device);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    unsigned long long raw[MOE_TRACE_FIELDS * moe_handle::kMaxStages];
    if (e == cudaSuccess) e = cudaMemcpy(raw, h->trace, sizeof(raw), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "trace read");
    const int kernels = h->last_launches < moe_handle::kMaxStages ? h->last_launches : moe_handle::kMaxStages;
    const unsigned long long none = ~0ull;
    unsigned long long t0 = none;
    for (int i = 0; i < kernels; ++i)
        if (raw[MOE_TRACE_FIELDS * i] < t0) t0 = raw[MOE_TRACE_FIELDS * i];
    int count = 0;
    for (int i = 0; i < kernels && count < max; ++i, ++count) {
        const unsigned long long *r = raw + MOE_TRACE_FIELDS * i;
        // slots 2 and 4 hold the complement of a maximum
        const unsigned long long v[MOE_TRACE_FIELDS] = {r[0], r[1], ~r[2], r[3], ~r[4]};
        const bool ok = r[0] != none && r[1] != none && r[2] != none && r[3] != none && r[4] != none;
        for (int f = 0; f < MOE_TRACE_FIELDS; ++f)
            t_us[MOE_TRACE_FIELDS * i + f] = ok ? (double)(v[f] - t0) * 1e-3 : -1.0;
    }
    *n = count;
    return MOE_OK;
}

const char *moe_get_stage_name(const moe_handle *h, int i) {
    if (h == nullptr || i < 0 || i >= h->last_launches || i >= moe_handle::kMaxStages) return nullptr;
    return h->stage_name[i];
}

moe_status moe_inspect(const moe_handle *h, int buffer, void *dst, size_t bytes, moe_stream_t stream) {
    if (h == nullptr || dst == nullptr) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    const size_t MT = h->cfg.max_tokens, k = h->k;
    const void *src = nullptr;
    size_t cap = 0;
    switch (buffer) {
    case MOE_BUF_TOPK_IDX: src = h->topk_idx; cap = MT * k * 4; break;
    case MOE_BUF_TOPK_W: src = h->topk_w; cap = MT * k * 4; break;
    case MOE_BUF_EXPERT_OFFS: src = h->offs; cap = (h->E + 1) * 4; break;
    case MOE_BUF_SORTED_TOKEN: src = h->sorted_tok; cap = MT * k * 4; break;
    case MOE_BUF_SLOT: src = h->slot_of; cap = MT * k * 4; break;
    case MOE_BUF_HIDDEN: src = h->hbuf; cap = MT * k * h->I * 2; break;
    case MOE_BUF_GEMM_STATS: src = h->gemm_stats; cap = moe::kGemmStats * 8; break;
    case MOE_BUF_ROUTER_STATS: src = h->router_stats; cap = moe::kRouterStats * 8; break;
    case MOE_BUF_NORMED_X: src = h->x_norm; cap = MT * h->H * (h->x_f32 ? 4 : 2); break;
    case MOE_BUF_SHARED_HIDDEN: src = h->hs; cap = MT * h->S * 2; break;
    default: return fail(MOE_ERR_INVALID_ARG, "unknown buffer %d", buffer);
    }
    if (src == nullptr) return fail(MOE_ERR_UNSUPPORTED, "buffer %d does not exist in this layer", buffer);
    if (bytes > cap) return fail(MOE_ERR_INVALID_ARG, "%zu bytes requested, buffer holds %zu", bytes, cap);
    cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice,
                                    reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "inspect copy");
}

}  // extern "C"
