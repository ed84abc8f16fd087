"""ctypes binding of libmoe.so (include/moe.h): argument marshalling only.

Every step of the block runs in the library's CUDA kernels; this module only
passes device pointers, sizes and the current torch stream.  There is no
fallback: if libmoe.so has not been built (``expert_routed_ffn_gb300.build``),
``load()`` raises.
"""

from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "_build", "libmoe.so")
HEADER = os.path.join(ROOT, "include", "moe.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_OOM, MOE_ERR_TIMEOUT, \
    MOE_ERR_DEVICE_CHECK = range(7)
STATUS_NAMES = ["MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_CUDA",
                "MOE_ERR_OOM", "MOE_ERR_TIMEOUT", "MOE_ERR_DEVICE_CHECK"]
MOE_SCORE_SIGMOID, MOE_SCORE_SOFTMAX = 0, 1
MOE_ACT_SILU, MOE_ACT_SWIGLU_OAI = 0, 1
MOE_DTYPE_BF16, MOE_DTYPE_F32 = 0, 1
MOE_NORM_NONE, MOE_NORM_RMS, MOE_NORM_GEMMA = 0, 1, 2
MOE_WEIGHTS_BF16, MOE_WEIGHTS_MXFP8, MOE_WEIGHTS_MXFP4 = 0, 1, 2
WEIGHT_FORMATS = {"bf16": MOE_WEIGHTS_BF16, "mxfp8": MOE_WEIGHTS_MXFP8, "mxfp4": MOE_WEIGHTS_MXFP4}
SCALE_KEYS = ("gate_scale", "up_scale", "down_scale", "sh_gate_scale", "sh_up_scale", "sh_down_scale")
MOE_OPT_PATH, MOE_OPT_WAIT_LIMIT_NS, MOE_OPT_STAGE_EVENTS, MOE_OPT_FUSE_EXPERTS, MOE_OPT_PREFETCH = 0, 1, 2, 3, 4
MOE_OPT_TRACE = 5
MOE_OPT_GEMM_PAIR = 6
MOE_OPT_GRAPH = 8
MOE_OPT_PAIR_SWAP = 9
MOE_OPT_COMBINE_OVERLAP = 10
MOE_OPT_STAGED_STORES = 11
MOE_BUF_GEMM_STATS = 6
MOE_BUF_ROUTER_STATS = 7
MOE_BUF_NORMED_X = 8
MOE_BUF_SHARED_HIDDEN = 9
TRACE_FIELDS = 5  # first begin, first ready, last ready, first end, last end
PATH_AUTO, PATH_DECODE, PATH_GROUPED, PATH_SWAPPED = 0, 1, 2, 3
(MOE_BUF_TOPK_IDX, MOE_BUF_TOPK_W, MOE_BUF_EXPERT_OFFS, MOE_BUF_SORTED_TOKEN, MOE_BUF_SLOT,
 MOE_BUF_HIDDEN) = range(6)


class MoeConfig(ctypes.Structure):
    _fields_ = [
        ("hidden_size", ctypes.c_int), ("num_experts", ctypes.c_int),
        ("num_experts_per_tok", ctypes.c_int), ("num_shared_experts", ctypes.c_int),
        ("moe_intermediate_size", ctypes.c_int), ("shared_intermediate_size", ctypes.c_int),
        ("shared_packed", ctypes.c_int), ("score_func", ctypes.c_int), ("route_norm", ctypes.c_int),
        ("route_scale", ctypes.c_float), ("hidden_act", ctypes.c_int), ("act_alpha", ctypes.c_float),
        ("act_limit", ctypes.c_float), ("act_beta", ctypes.c_float), ("act_dtype", ctypes.c_int),
        ("max_tokens", ctypes.c_int), ("mlp_norm", ctypes.c_int), ("rms_norm_eps", ctypes.c_float),
        ("weight_format", ctypes.c_int),
    ]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("router_w", "expert_bias", "gate", "up", "down", "sh_gate", "sh_up", "sh_down",
                 "pre_norm_w", "post_norm_w", "gate_scale", "up_scale", "down_scale", "sh_gate_scale",
                 "sh_up_scale", "sh_down_scale")]


class MoeStats(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("kernel_launches", ctypes.c_int),
                ("workspace_bytes", ctypes.c_longlong)]


def header_symbols() -> list:
    """Names of the functions include/moe.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:moe_status|void|const char \*)\s*(moe_\w+)\s*\(", text, re.M)))


_lib = None


def load():
    """Load libmoe.so (must already be built: expert_routed_ffn_gb300.build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libmoe.so is not built ({LIB_PATH}); run expert_routed_ffn_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, I, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    L.moe_create.argtypes = [ctypes.POINTER(MoeConfig), ctypes.POINTER(MoeWeights), ctypes.POINTER(P)]
    L.moe_route.argtypes = [P, P, I, P, P, P]
    L.moe_forward.argtypes = [P, P, I, P, P]
    L.moe_forward_host.argtypes = [P, P, I, P, P]
    L.moe_sync_status.argtypes = [P]
    L.moe_destroy.argtypes = [P]
    L.moe_destroy.restype = None
    L.moe_last_error.argtypes = []
    L.moe_last_error.restype = ctypes.c_char_p
    L.moe_set_option.argtypes = [P, I, LL]
    L.moe_get_stats.argtypes = [P, ctypes.POINTER(MoeStats)]
    L.moe_inspect.argtypes = [P, I, P, ctypes.c_size_t, P]
    L.moe_get_stage_times.argtypes = [P, ctypes.POINTER(ctypes.c_float), I, ctypes.POINTER(I)]
    L.moe_get_trace.argtypes = [P, ctypes.POINTER(ctypes.c_double), I, ctypes.POINTER(I)]
    L.moe_get_stage_name.argtypes = [P, I]
    L.moe_get_stage_name.restype = ctypes.c_char_p
    L.moe_dispatch_noalloc.argtypes = [P, I, I, I, P, P, P, P, P]
    for name in ("moe_create", "moe_route", "moe_forward", "moe_forward_host", "moe_sync_status", "moe_dispatch_noalloc",
                 "moe_set_option", "moe_get_stats", "moe_inspect", "moe_get_stage_times", "moe_get_trace"):
        getattr(L, name).restype = I
    _lib = L
    return L


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = load().moe_last_error().decode(errors="replace")
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{where}: {name}: {msg}")


def check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def config_from_shape(shape, max_tokens: int = None) -> MoeConfig:
    """C config from a workloads.MoeShape (the pages' config keys)."""
    return MoeConfig(
        hidden_size=shape.H, num_experts=shape.E, num_experts_per_tok=shape.k,
        num_shared_experts=shape.num_shared_experts, moe_intermediate_size=shape.I,
        shared_intermediate_size=0 if shape.shared_packed else shape.S,
        shared_packed=int(shape.shared_packed),
        score_func={"sigmoid": MOE_SCORE_SIGMOID, "softmax": MOE_SCORE_SOFTMAX}[shape.score_func],
        route_norm=int(shape.route_norm), route_scale=shape.route_scale,
        hidden_act={"silu": MOE_ACT_SILU, "swigluoai": MOE_ACT_SWIGLU_OAI}[shape.hidden_act],
        act_alpha=shape.act_alpha, act_limit=shape.act_limit, act_beta=shape.act_beta,
        act_dtype={"bf16": MOE_DTYPE_BF16, "f32": MOE_DTYPE_F32}[shape.dtype],
        max_tokens=max(1, shape.T if max_tokens is None else max_tokens),
        mlp_norm={"none": MOE_NORM_NONE, "rms": MOE_NORM_RMS, "gemma": MOE_NORM_GEMMA}[shape.mlp_norm],
        rms_norm_eps=shape.rms_norm_eps,
        weight_format=WEIGHT_FORMATS[getattr(shape, "weight_format", "bf16")])


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class MoeBlock:
    """One handle of libmoe.so over borrowed torch CUDA tensors.

    weights: dict with router_w [E,H] fp32, expert_bias [E] fp32 (or None),
    gate/up [E',I,H], down [E',H,I] bf16 and sh_gate/sh_up [S,H], sh_down [H,S]
    bf16 (or None), and pre_norm_w / post_norm_w [H] fp32 with the sandwich
    norms.  MX weight formats: the six expert tensors hold uint8 element codes
    and gate_scale ... sh_down_scale their uint8 E8M0 scales.  The tensors are
    kept referenced for the handle's lifetime.
    """

    def __init__(self, config: MoeConfig, weights: dict):
        import torch
        self._torch = torch
        self.cfg = config
        self._keep = {k: v for k, v in weights.items() if isinstance(v, torch.Tensor)}
        w = MoeWeights(**{k: (None if weights.get(k) is None else weights[k].data_ptr())
                          for k in ("router_w", "expert_bias", "gate", "up", "down", "sh_gate",
                                    "sh_up", "sh_down", "pre_norm_w", "post_norm_w") + SCALE_KEYS})
        h = ctypes.c_void_p()
        check(load().moe_create(ctypes.byref(config), ctypes.byref(w), ctypes.byref(h)), "moe_create")
        self.h = h
        self.x_dtype = torch.float32 if config.act_dtype == MOE_DTYPE_F32 else torch.bfloat16

    def close(self):
        if getattr(self, "h", None):
            load().moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def route(self, X, stream=None):
        T = X.shape[0]
        torch = self._torch
        idx = torch.empty((T, self.cfg.num_experts_per_tok), dtype=torch.int32, device=X.device)
        w = torch.empty((T, self.cfg.num_experts_per_tok), dtype=torch.float32, device=X.device)
        check(load().moe_route(self.h, _ptr(X), T, _ptr(idx), _ptr(w), _stream(stream)), "moe_route")
        return idx, w

    def forward(self, X, Y=None, stream=None):
        if Y is None:
            Y = self._torch.empty_like(X)
        check(load().moe_forward(self.h, _ptr(X), X.shape[0], _ptr(Y), _stream(stream)), "moe_forward")
        return Y

    def forward_host(self, X_host, Y_host, stream=None):
        check(load().moe_forward_host(self.h, _ptr(X_host), X_host.shape[0], _ptr(Y_host),
                                      _stream(stream)), "moe_forward_host")
        return Y_host

    def sync_status(self) -> int:
        return load().moe_sync_status(self.h)

    def set_option(self, option: int, value: int):
        check(load().moe_set_option(self.h, option, int(value)), "moe_set_option")

    def stats(self) -> MoeStats:
        s = MoeStats()
        check(load().moe_get_stats(self.h, ctypes.byref(s)), "moe_get_stats")
        return s

    def stage_times(self) -> list:
        buf = (ctypes.c_float * 8)()
        n = ctypes.c_int()
        check(load().moe_get_stage_times(self.h, buf, 8, ctypes.byref(n)), "moe_get_stage_times")
        return [buf[i] for i in range(n.value)]

    def trace(self) -> list:
        """(name, first_begin, first_ready, last_ready, first_end, last_end) in us per kernel
        of the last forward (MOE_OPT_TRACE on)."""
        buf = (ctypes.c_double * (TRACE_FIELDS * 8))()
        n = ctypes.c_int()
        check(load().moe_get_trace(self.h, buf, 8, ctypes.byref(n)), "moe_get_trace")
        names = self.stage_names()
        return [(names[i],) + tuple(buf[TRACE_FIELDS * i + f] for f in range(TRACE_FIELDS)) for i in range(n.value)]

    def stage_names(self) -> list:
        L = load()
        return [L.moe_get_stage_name(self.h, i).decode() for i in range(self.stats().kernel_launches)]

    def inspect(self, buffer: int, count: int, dtype, stream=None):
        torch = self._torch
        out = torch.empty(count, dtype=dtype, device="cuda")
        nbytes = count * out.element_size()
        check(load().moe_inspect(self.h, buffer, _ptr(out), nbytes, _stream(stream)), "moe_inspect")
        return out


def block_from_inputs(shape, inputs: dict, max_tokens: int = None) -> MoeBlock:
    """MoeBlock over a workloads.make_inputs() dict on the GPU (expert weights
    rounded to bf16 when the workload stores them in fp32)."""
    from .workloads import expert_weights_bf16
    w = dict(router_w=inputs["router_w"], expert_bias=inputs["expert_bias"], **expert_weights_bf16(inputs),
             pre_norm_w=inputs.get("pre_norm_w"), post_norm_w=inputs.get("post_norm_w"),
             **{k: inputs.get(k) for k in SCALE_KEYS})
    blk = MoeBlock(config_from_shape(shape, max_tokens), w)
    return blk
