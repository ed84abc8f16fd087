/*
 * moe.h - C ABI of libmoe.so: the token-choice mixture-of-experts feed-forward
 * block of AFMoE (Arcee Trinity) and of MiniMax-M3, on one GB300 (sm_103a).
 *
 * What the block computes, per token x = X[t,:] (H values):
 *   logits   l_e = x . Wr[e,:]                  in fp32, e in [0, E)
 *   scores   s_e = sigmoid(l_e)  (or softmax over e)
 *   select   the k experts with the largest s_e + b_e (b = expert_bias, used for
 *            the choice only; ties go to the lower expert index), in
 *            descending biased score
 *   weights  w_j = s_{idx_j}; if route_norm: w_j /= sum_j w_j; w_j *= route_scale
 *   experts  y_e = Wd[e] . act(Wg[e] . x, Wu[e] . x)
 *   shared   y_s = the same MLP over the shared tensors (or the packed slice E),
 *            weight 1.0, never selected, never normalised, never scaled
 *   output   Y[t,:] = sum_j w_j y_{idx_j} + y_s
 * Sources: Arcee AFMoE issue (mlxcel #845), "Routing detail" (sigmoid scores,
 * selection-only expert_bias, route_norm then route_scale) and "Checkpoint
 * weight layout" (pre-stacked experts.{gate,up,down}_proj, router.gate,
 * expert_bias, shared_experts); HF Transformers AFMoE docs, AfmoeConfig
 * (num_experts, num_experts_per_tok, num_shared_experts, moe_intermediate_size,
 * route_scale, hidden_act) and "expert routing" / "shared experts"; MiniMax-M3
 * issue (mlxcel #763), "Architecture specification" (packed shared expert at
 * index E with score 1.0; clamp-SwiGLU x_glu*sigmoid(alpha*x_glu)*(x_linear+beta),
 * alpha 1.702, limit 7.0, beta 1.0).
 *
 * Conventions for every entry point:
 *   - Tensors are row-major and contiguous.  Device pointers must be 16-byte
 *     aligned.  Every pointer is BORROWED: the library never frees it.
 *   - Calls that take a stream are asynchronous on that stream (NULL = the
 *     legacy default stream); results are valid once the stream is synchronised.
 *   - Argument errors are detected on the host, before anything is launched,
 *     and return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED.
 *   - A failed device-side check (a bounded wait that ran out, an index out of
 *     range) sets a device error word; moe_sync_status() reports it as
 *     MOE_ERR_TIMEOUT / MOE_ERR_DEVICE_CHECK and clears it.
 *   - moe_last_error() returns a per-thread message for the last failure.
 *   - A handle is not thread-safe: calls on one handle must not overlap.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the runtime's stream handle), passed through unchanged. */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* a NULL, misaligned or out-of-range argument */
    MOE_ERR_UNSUPPORTED = 2,  /* a valid config outside what the kernels handle */
    MOE_ERR_CUDA = 3,         /* a CUDA runtime call failed; see moe_last_error() */
    MOE_ERR_OOM = 4,          /* workspace allocation failed */
    MOE_ERR_TIMEOUT = 5,      /* a bounded device wait ran out (device error word) */
    MOE_ERR_DEVICE_CHECK = 6  /* a device-side bounds check failed (device error word) */
} moe_status;

/* score_func: HF AFMoE docs list sigmoid or softmax routing; Trinity and M3 use
 * sigmoid ("Routing detail"; MiniMax-M3 "Architecture specification"). */
typedef enum { MOE_SCORE_SIGMOID = 0, MOE_SCORE_SOFTMAX = 1 } moe_score_func;

/* hidden_act: "silu" gives a = silu(g) * u (AfmoeConfig default); "swigluoai"
 * gives a = min(g,limit) * sigmoid(alpha*min(g,limit)) * (clamp(u,-limit,limit) + beta)
 * (MiniMax-M3, Activation bullet; the clamp placement follows the gpt-oss
 * convention that bullet names). */
typedef enum { MOE_ACT_SILU = 0, MOE_ACT_SWIGLU_OAI = 1 } moe_act;

/* dtype of X and Y.  Router weights and the expert bias are always fp32; the
 * expert weights are bf16 or block-scaled (moe_weight_format). */
typedef enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1 } moe_dtype;

/* Storage of the expert weights (routed, shared and dense-layer gate/up/down).
 * The Arcee AFMoE issue ("Checkpoint confirmed") lists 4-bit and MXFP8
 * checkpoints; the MX variants follow the OCP Microscaling Formats v1.0: every
 * 32 consecutive values along a row's input dimension K (H for gate/up, I or S
 * for down) share one E8M0 scale byte c, and a weight is element(code) * 2^(c - 127)
 * (c = 255 is NaN).  The activations stay bf16: the block multiplies bf16 tokens
 * by the exactly decoded weights (each decoded value is a bf16 number as long as
 * it lies in bf16's range; outside it rounds to nearest).
 *   MXFP8: one E4M3 code per byte, [rows, K] per weight slice.
 *   MXFP4: two E2M1 codes per byte, [rows, K / 2], element 2j in the low nibble.
 *   Scales: uint8 [K / 32, rows] per weight slice (block-major: for each
 *           32-value block, the scales of all rows).
 * MX weights run on the tensor-core paths: the grouped GEMM (the auto path; where
 * MOE_OPT_GEMM_PAIR picks 256-row tiles, one CTA runs both 128-row halves against
 * each decoded weight tile) or,
 * with moe_set_option MOE_OPT_PATH 3, the swapped-operand GEMM that decodes the
 * weights straight into tensor memory; MOE_OPT_PATH 1 is refused. */
typedef enum { MOE_WEIGHTS_BF16 = 0, MOE_WEIGHTS_MXFP8 = 1, MOE_WEIGHTS_MXFP4 = 2 } moe_weight_format;

/* Norms around the MLP (y = x / sqrt(mean(x^2) + eps) * g over the H values of a row). */
typedef enum {
    MOE_NORM_NONE = 0,  /* no norms: out = mlp(X) */
    MOE_NORM_RMS = 1,   /* g = weight */
    MOE_NORM_GEMMA = 2  /* g = 1 + weight */
} moe_norm;

typedef struct {
    int hidden_size;              /* H; multiple of 64 */
    int num_experts;              /* E routed experts; 1..256.  0: a dense MLP layer (the dense
                                     prefix layers: no router, the "shared" tensors are the
                                     layer's gate/up/down of width shared_intermediate_size, a
                                     multiple of 64 up to 16384; bf16 activations only) */
    int num_experts_per_tok;      /* k; 1..min(E, 16) (0 when E == 0) */
    int num_shared_experts;       /* 0, or the count of always-on shared experts */
    int moe_intermediate_size;    /* I, width of one routed expert; multiple of 64 */
    int shared_intermediate_size; /* S, total shared width; 0 => num_shared_experts * I */
    int shared_packed;            /* 1 => the shared expert is slice E of the stacked
                                     gate/up/down tensors (width I, score 1.0) */
    int score_func;               /* moe_score_func */
    int route_norm;               /* 1 => renormalise the k gathered weights */
    float route_scale;            /* multiplies the routed weights after route_norm */
    int hidden_act;               /* moe_act */
    float act_alpha, act_limit, act_beta; /* swigluoai constants (1.702, 7.0, 1.0) */
    int act_dtype;                /* moe_dtype of X and Y */
    int max_tokens;               /* largest T any later call may pass; sizes the workspace */
    int mlp_norm;                 /* moe_norm: the layer's sandwich norms, out = X +
                                     post_norm(mlp(pre_norm(X))) (Arcee AFMoE issue: four norms per
                                     layer; MiniMax-M3 issue: Gemma-style RMSNorm, weight + 1) */
    float rms_norm_eps;           /* eps of both norms (AfmoeConfig rms_norm_eps 1e-5) */
    int weight_format;            /* moe_weight_format of the expert weights (0: bf16) */
} moe_config;

/* Device pointers to the block's weights.  BORROWED: they must stay valid and
 * unchanged until moe_destroy().  E' = E + 1 when shared_packed, else E. */
typedef struct {
    const float *router_w;    /* [E, H] fp32 (mlp.router.gate) */
    const float *expert_bias; /* [E] fp32 (mlp.expert_bias); NULL => zeros */
    const void *gate;         /* [E', I, H] bf16 (experts.gate_proj, [out, in] per expert) */
    const void *up;           /* [E', I, H] bf16 (experts.up_proj) */
    const void *down;         /* [E', H, I] bf16 (experts.down_proj) */
    const void *sh_gate;      /* [S, H] bf16 (shared_experts.gate_proj); NULL when packed or S == 0 */
    const void *sh_up;        /* [S, H] bf16 */
    const void *sh_down;      /* [H, S] bf16 */
    const float *pre_norm_w;  /* [H] fp32 (pre_mlp_layernorm.weight); required when mlp_norm != 0 */
    const float *post_norm_w; /* [H] fp32 (post_mlp_layernorm.weight); required when mlp_norm != 0 */
    /* MX weight formats only (NULL otherwise): the E8M0 scales of the tensors
     * above, uint8, block-major per slice (see moe_weight_format), each required
     * exactly where its weight tensor is.  gate_scale, up_scale: [E', H/32, I];
     * down_scale: [E', I/32, H]; sh_gate_scale, sh_up_scale: [H/32, S];
     * sh_down_scale: [S/32, H].  The element tensors gate, up, down, sh_* then
     * hold the codes: MXFP8 [.., rows, K] uint8, MXFP4 [.., rows, K/2] uint8. */
    const uint8_t *gate_scale, *up_scale, *down_scale;
    const uint8_t *sh_gate_scale, *sh_up_scale, *sh_down_scale;
} moe_weights;

typedef struct moe_handle moe_handle;

/* Validate the config, record the borrowed weights, allocate the workspace
 * (sized by max_tokens) and build the TMA descriptors of the weight tensors on
 * the current CUDA device.  On success *out owns the handle (free it with
 * moe_destroy).  Errors: INVALID_ARG (NULL, misaligned, inconsistent keys),
 * UNSUPPORTED (sizes outside the kernels' limits above), OOM, CUDA. */
moe_status moe_create(const moe_config *config, const moe_weights *weights, moe_handle **out);

/* Router only: for X [T, H] (act_dtype, device) write topk_idx [T, k] int32
 * (experts in descending biased score, ties to the lower index) and topk_w
 * [T, k] fp32 (unbiased scores, renormalised and scaled).  T == 0 is a no-op.
 * Errors: INVALID_ARG (NULL pointer, T < 0 or T > max_tokens), CUDA. */
moe_status moe_route(moe_handle *h, const void *X, int T, int32_t *topk_idx, float *topk_w,
                     moe_stream_t stream);

/* The whole block: Y [T, H] (act_dtype, device) from X [T, H] (device).
 * X and Y must not overlap.  T == 0 is a no-op.
 * Errors: INVALID_ARG, CUDA. */
moe_status moe_forward(moe_handle *h, const void *X, int T, void *Y, moe_stream_t stream);

/* moe_forward with HOST buffers: copies X_host to the handle's device staging
 * buffer, runs the block and copies the result back to Y_host, all on
 * `stream`; the call returns once Y_host holds the result.  When both buffers
 * are page-locked (pinned) and 16-byte aligned, a copy kernel reads X_host over
 * the host link and the block's last kernel stores its rows into Y_host itself;
 * otherwise the copy engines move the bytes (pageable memory works but is
 * slower).  Errors: INVALID_ARG, CUDA. */
moe_status moe_forward_host(moe_handle *h, const void *X_host, int T, void *Y_host,
                            moe_stream_t stream);

/* Synchronise the handle's work and read (then clear) its device error word.
 * Returns MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_CHECK or MOE_ERR_CUDA. */
moe_status moe_sync_status(moe_handle *h);

/* Free the workspace and the handle.  NULL is a no-op.  Synchronises first. */
void moe_destroy(moe_handle *h);

/* Message of the last failure on the calling thread ("" if none). */
const char *moe_last_error(void);

/* ----------------------------------------------------------------------------
 * Options, statistics and inspection (tests and measurement).
 */
typedef enum {
    MOE_OPT_PATH = 0,          /* 0 auto (= 2 at every size), 1 weight-streaming decode kernels on
                                  the CUDA cores, 2 tcgen05 grouped GEMMs (tokens as M), 3 tcgen05
                                  swapped-operand GEMMs (weights as M).  Paths 1 and 3 are
                                  diagnostic alternatives kept for comparison and parity tests: on
                                  GB300 path 1 is slower than path 2 from T = 1 up and path 3 at
                                  best ties it, so the auto path never selects them */
    MOE_OPT_WAIT_LIMIT_NS = 1, /* bound of every device-side wait in ns (default 500000000);
                                  0 makes the first wait that finds its data not ready give up,
                                  which exercises the timeout path */
    MOE_OPT_STAGE_EVENTS = 2,  /* 1: record a CUDA event on the stream before the first and after
                                  every kernel of moe_forward, for moe_get_stage_times (default 0) */
    MOE_OPT_FUSE_EXPERTS = 3,  /* path 2: 1 (default) runs the gate/up and down GEMMs as one
                                  persistent launch whose down tiles wait for their gate/up rows;
                                  0 runs them as two launches */
    MOE_OPT_PREFETCH = 4,      /* 1 (default): when T*k >= 2E (nearly every expert is touched) and the
                                  expert-sorted copy of the T*k token rows is at most a quarter of L2, an
                                  internal side stream prefetches the first experts' gate/up weights
                                  into L2 while the routing kernels run (forked from and joined back
                                  into the caller's stream); 0: no prefetch.  A hint: results are
                                  unchanged */
    MOE_OPT_TRACE = 5,         /* 1: every kernel of moe_forward on the grouped path records, in a
                                  device buffer of the handle, when its first CTA started, when its
                                  first and last CTA passed the wait on the previous kernel, and when
                                  its first and last CTA finished (the GPU's global timer), for
                                  moe_get_trace.  Costs a memset and a few atomics per CTA; default 0 */
    MOE_OPT_GEMM_PAIR = 6,     /* path 2: expert GEMM tiles of 256 rows on CTA pairs (tcgen05 with
                                  cta_group::2: each CTA of a two-CTA cluster stages its 128 token rows
                                  and half of the weight tile; MX weights: one CTA per 256-row tile,
                                  two 128-row MMAs on each decoded weight tile); 0 never, 1 always,
                                  2 (default) when T*k >= 160*E with bf16 weights, 256*E with MX
                                  weights, and the expert width is at least 512; T >= 256 for
                                  a dense layer (tensor-bound sizes) */
    MOE_OPT_GRAPH = 8,         /* moe_forward_host: 1 (default) captures the copy in, the forward and the
                                  copy out into a CUDA graph on the second call with the same host
                                  buffers, T and options, and replays it on later such calls (host
                                  buffers must then be pinned: with pageable ones the capture fails
                                  and the call runs eagerly); 0 always runs eagerly.  Graphs are not
                                  used while stage events or the trace are on. */
    MOE_OPT_PAIR_SWAP = 9,     /* path 2 on CTA pairs with bf16 weights: 1 (default) runs an expert's
                                  last 256-row tile with the operands swapped when it holds at most
                                  128 rows (the pair's 256 weight rows as M, the tile's rows rounded
                                  up to 32 as N), so the MMA skips most of the padding rows; 0 runs
                                  every tile with the tokens as M.  Results are unchanged */
    MOE_OPT_COMBINE_OVERLAP = 10, /* path 2 without the post-MLP norm: 1 (default) launches the combine
                                  while the expert GEMM runs; the down tiles count each token's
                                  stored rows and the combine adds a token as soon as all of its
                                  rows are in (the same fixed-order sum); 0 waits for the whole GEMM
                                  first.  Results are unchanged */
    MOE_OPT_STAGED_STORES = 11 /* path 2, bf16 weights: 1 (default) stores the expert GEMM's outputs
                                  of tiles with the tokens as M through shared memory (TMA stores of
                                  32-row slices, coalesced stores of partial ones); 0 stores each
                                  row from registers.  Results are unchanged */
} moe_option;

/* Set an option.  Errors: INVALID_ARG (unknown option or value). */
moe_status moe_set_option(moe_handle *h, int option, long long value);

typedef struct {
    int path;              /* path of the last forward: 1 decode, 2 grouped, 3 swapped */
    int kernel_launches;   /* kernels the last forward (or route) launched */
    long long workspace_bytes;
} moe_stats;

/* Statistics of the last call on this handle (host-side; no synchronisation). */
moe_status moe_get_stats(const moe_handle *h, moe_stats *out);

/* With MOE_OPT_STAGE_EVENTS on: wait for the last moe_forward and write the
 * duration in ms of each of its kernels, in launch order (names from
 * moe_get_stage_name), to ms[0..*n).  At most `max` values are written.  Errors: INVALID_ARG (events off, no forward yet,
 * NULL argument), CUDA. */
moe_status moe_get_stage_times(moe_handle *h, float *ms, int max, int *n);

/* Name of kernel i (0-based, launch order) of the last call, e.g. "router_logits",
 * "router_topk", "dispatch_scatter", "experts_gemm" (or "gate_up_gemm", "down_gemm"),
 * "combine";
 * NULL when i is out of range.  The string is static. */
const char *moe_get_stage_name(const moe_handle *h, int i);

/* Fields of one kernel's entry in moe_get_trace, in us from the first kernel's first CTA start. */
#define MOE_TRACE_FIELDS 5
typedef enum {
    MOE_TRACE_FIRST_BEGIN = 0, /* first CTA started */
    MOE_TRACE_FIRST_READY = 1, /* first CTA passed the wait on the previous kernel */
    MOE_TRACE_LAST_READY = 2,  /* last CTA passed that wait */
    MOE_TRACE_FIRST_END = 3,   /* first CTA finished */
    MOE_TRACE_LAST_END = 4     /* last CTA finished */
} moe_trace_field;

/* With MOE_OPT_TRACE on: wait for the device to go idle and write, for each kernel of the
 * last moe_forward in launch order (names from moe_get_stage_name), MOE_TRACE_FIELDS times
 * to t_us[MOE_TRACE_FIELDS * i + field].  With programmatic dependent launch a kernel
 * begins before its predecessor ends; FIRST_READY minus the predecessor's LAST_END is the
 * hand-over gap.  A kernel that records nothing (the decode and swapped paths' GEMMs)
 * reads -1.  At most `max` kernels; *n = kernels written.  Errors: INVALID_ARG (trace off,
 * no forward, NULL argument), CUDA. */
moe_status moe_get_trace(moe_handle *h, double *t_us, int max, int *n);

typedef enum {
    MOE_BUF_TOPK_IDX = 0,     /* [T, k] int32, routing of the last forward */
    MOE_BUF_TOPK_W = 1,       /* [T, k] fp32 */
    MOE_BUF_EXPERT_OFFS = 2,  /* [E + 1] int32: rows of expert e are [offs[e], offs[e+1]) */
    MOE_BUF_SORTED_TOKEN = 3, /* [T * k] int32: token of each expert-sorted row */
    MOE_BUF_SLOT = 4,         /* [T * k] int32: sorted row of routing slot (t, j) */
    MOE_BUF_HIDDEN = 5,       /* [T * k, I] bf16: act(gate, up) of each sorted row */
    MOE_BUF_GEMM_STATS = 6,   /* [8] uint64, with MOE_OPT_TRACE on and the fused expert GEMM: ns
                                 summed over its CTAs of: producer waiting for a free stage,
                                 producer waiting for gate/up rows, MMA waiting for data, MMA
                                 waiting for an accumulator, epilogue waiting for an accumulator,
                                 epilogue working, CTA time past the dependency wait; then the
                                 number of tiles */
    MOE_BUF_ROUTER_STATS = 7, /* [8] uint64, with MOE_OPT_TRACE on and the tensor-core router: ns
                                 summed over its CTAs of: main loop, first cluster barrier,
                                 pushing the partial logits to the routing CTAs with the second
                                 barrier, adding them and routing, histogram; then the number of
                                 CTAs */
    MOE_BUF_NORMED_X = 8,     /* [T, H] in the activation dtype: pre_norm(X), the MLP's input
                                 (mlp_norm != 0 only) */
    MOE_BUF_SHARED_HIDDEN = 9 /* [T, S] bf16: act(gate, up) of the shared experts (of the dense
                                 MLP when num_experts == 0) */
} moe_buffer;

/* Copy `bytes` of an internal buffer, as the last forward left it, to the
 * device pointer dst (stream-ordered on `stream`).  Errors: INVALID_ARG
 * (unknown buffer, bytes beyond its size). */
moe_status moe_inspect(const moe_handle *h, int buffer, void *dst, size_t bytes, moe_stream_t stream);

/* ----------------------------------------------------------------------------
 * Dispatch sort without device allocation.  The pages have no counterpart of
 * this call; it is a library facility.
 *
 * Who it is for: callers that cannot allocate device memory at the point where
 * they route tokens -- an inference server whose memory pool owns the whole
 * device, a plugin handed a fixed memory budget, or a latency-critical loop
 * that cannot afford cudaMalloc's implicit device synchronisation.  This is
 * the dispatch step of moe_forward as a standalone call whose scratch (the
 * per-block expert histograms and their scan) lives in a static device array
 * inside libmoe.so: MOE_DISPATCH_NOALLOC_SCRATCH_INTS int32 values (1 MiB),
 * held by every GPU that loads the library until the process exits.  The call
 * allocates nothing; the caller passes the inputs and outputs.
 *
 * In:  topk_idx [T, k] int32 (device): expert ids, normally in [0, E).
 * Out (device): expert_offs [E + 1]: the rows of expert e are
 *      [expert_offs[e], expert_offs[e + 1]); sorted_token [T * k]: the token
 *      of each row, rows ordered by (expert, token, slot); slot [T * k]: the
 *      row of routing slot (t, j), or -1 when topk_idx[t, j] is out of range;
 *      bad_index [1] int: 1 when some index was out of range, else 0.
 * Limits: 1 <= k <= 16, 1 <= E <= 256 and ceil(T / 32) * E + 2 * (E + 1) <=
 *      MOE_DISPATCH_NOALLOC_SCRATCH_INTS (for E = 128: T <= 65440); larger
 *      sizes return MOE_ERR_UNSUPPORTED with a message, before any launch.
 *      T = 0 writes zeros to expert_offs[0 .. E] and bad_index (topk_idx,
 *      sorted_token and slot may then be NULL).
 * The first call on a device looks up the device address of the array (with
 * that device current), and again after the device's context was reset; make
 * that first call before any stream capture.  All
 * calls on one device share the array and it keeps the last call's contents
 * (every entry a call reads it writes first, so nothing needs clearing); calls
 * that overlap on the GPU race on it, so the caller must serialise them.
 * Asynchronous on `stream`.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
#define MOE_DISPATCH_NOALLOC_SCRATCH_INTS (1 << 18)
moe_status moe_dispatch_noalloc(const int32_t *topk_idx, int T, int k, int E, int32_t *expert_offs,
                                int32_t *sorted_token, int32_t *slot, int *bad_index, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
