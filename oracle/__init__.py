"""fp64 CPU oracle of the token-choice MoE FFN block (AFMoE / MiniMax-M3).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference leg of ``bench.py`` may import this package.  It shares no
code with the CUDA path; the arithmetic lives in ``moe_oracle.c`` (plain C,
double precision), which this module compiles with gcc on first use and calls
through ctypes.

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (brute force, closed forms, library routines and
the invariants the pages imply).  Where the clamp of clamp-SwiGLU is applied is
not printed on the MiniMax-M3 page; that reading is pinned only by its reduction
to plain SwiGLU and by hand-evaluated points.
"""

from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libmoe_oracle.so")

OR_F32, OR_BF16, OR_MXFP8, OR_MXFP4 = 0, 1, 2, 3
# expert weight formats of a workload -> the oracle's dtype code (None: as stored)
WEIGHT_FORMATS = {"bf16": None, "mxfp8": OR_MXFP8, "mxfp4": OR_MXFP4}
SCALE_KEYS = ("gate_scale", "up_scale", "down_scale", "sh_gate_scale", "sh_up_scale", "sh_down_scale")
OR_SIGMOID, OR_SOFTMAX = 0, 1
OR_SILU, OR_SWIGLU_OAI = 0, 1


class OracleCfg(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int), ("I", ctypes.c_int),
        ("S", ctypes.c_int), ("shared_packed", ctypes.c_int), ("score_func", ctypes.c_int),
        ("route_norm", ctypes.c_int), ("route_scale", ctypes.c_double), ("act", ctypes.c_int),
        ("alpha", ctypes.c_double), ("limit", ctypes.c_double), ("beta", ctypes.c_double),
    ]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (gcc, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _configure(L):
    P = ctypes.c_void_p
    L.oracle_route.argtypes = [ctypes.POINTER(OracleCfg), P, ctypes.c_int, P, P, ctypes.c_int,
                               P, P, P, P, P, P, P, ctypes.c_int]
    L.oracle_route.restype = ctypes.c_int
    L.oracle_forward.argtypes = [ctypes.POINTER(OracleCfg), P, ctypes.c_int, P, P, P, P, P,
                                 P, P, P, ctypes.c_int, P, ctypes.c_int, P, P, ctypes.c_int]
    L.oracle_forward.restype = ctypes.c_int
    L.oracle_expert.argtypes = [ctypes.POINTER(OracleCfg), P, ctypes.c_int, P, P, P,
                                ctypes.c_int, P, ctypes.c_int, P, P, P, P]
    L.oracle_expert.restype = ctypes.c_int
    L.oracle_act.argtypes = [ctypes.POINTER(OracleCfg), ctypes.c_double, ctypes.c_double]
    L.oracle_act.restype = ctypes.c_double
    L.oracle_dense.argtypes = [ctypes.POINTER(OracleCfg), P, ctypes.c_int, P, P, P, ctypes.c_int, P,
                               ctypes.c_int, P, P, ctypes.c_int]
    L.oracle_dense.restype = ctypes.c_int
    L.oracle_rmsnorm.argtypes = [P, ctypes.c_int, P, ctypes.c_double, ctypes.c_int, P]
    L.oracle_rmsnorm.restype = ctypes.c_int
    L.oracle_mx_value.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    L.oracle_mx_value.restype = ctypes.c_double
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Run the oracle from another build of moe_oracle.c (used by the mutation
    test, which plants mistakes in copies of the source)."""
    global _lib
    prev = lib()
    with _lock:
        _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = prev


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile a variant of moe_oracle.c's text with the same flags as build()."""
    c_path = out_path + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
                           "-ffp-contract=off", "-fno-fast-math", c_path, "-o", out_path, "-lm"])
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def make_cfg(H, E, k, I, S=0, shared_packed=False, score_func="sigmoid", route_norm=True,
             route_scale=1.0, act="silu", alpha=1.702, limit=7.0, beta=1.0) -> OracleCfg:
    return OracleCfg(H=H, E=E, k=k, I=I, S=S, shared_packed=int(bool(shared_packed)),
                     score_func={"sigmoid": OR_SIGMOID, "softmax": OR_SOFTMAX}[score_func],
                     route_norm=int(bool(route_norm)), route_scale=float(route_scale),
                     act={"silu": OR_SILU, "swigluoai": OR_SWIGLU_OAI}[act],
                     alpha=float(alpha), limit=float(limit), beta=float(beta))


def cfg_from_shape(shape) -> OracleCfg:
    """Oracle config from a workloads.MoeShape (E = 0: a dense MLP of width S)."""
    if shape.E == 0:
        return make_cfg(shape.H, 0, 0, 0, S=shape.S, act=shape.hidden_act, alpha=shape.act_alpha,
                        limit=shape.act_limit, beta=shape.act_beta)
    return make_cfg(shape.H, shape.E, shape.k, shape.I, S=(0 if shape.shared_packed else shape.S),
                    shared_packed=shape.shared_packed, score_func=shape.score_func,
                    route_norm=shape.route_norm, route_scale=shape.route_scale,
                    act=shape.hidden_act, alpha=shape.act_alpha, limit=shape.act_limit,
                    beta=shape.act_beta)


# ------------------------------------------------------------------ marshalling

def _as_host(a):
    """numpy array (or torch tensor) -> (contiguous numpy array, dtype code).

    bf16 tensors travel as their raw uint16 bit patterns."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            t = a.detach().contiguous().cpu()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), OR_BF16
            if t.dtype == torch.float32:
                return t.numpy(), OR_F32
            raise TypeError(f"unsupported tensor dtype {t.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, OR_BF16
    if a.dtype == np.float32:
        return a, OR_F32
    raise TypeError(f"unsupported array dtype {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u8(a):
    """uint8 array (or tensor) of MX element or scale codes."""
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().contiguous().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError("MX element and scale codes are uint8")
    return a


def _weights(tensors, wfmt, scales):
    """Expert weight tensors -> (host arrays, dtype code, ctypes array of the
    scale pointers or None, the scale arrays kept alive)."""
    code = WEIGHT_FORMATS[wfmt]
    if code is None:
        hs, ds = zip(*[(None, None) if t is None else _as_host(t) for t in tensors])
        used = {d for d in ds if d is not None}
        if len(used) != 1:
            raise TypeError("the expert tensors must share one dtype")
        return list(hs), used.pop(), None, None
    if scales is None or len(scales) != len(tensors):
        raise ValueError("MX weights need one scale tensor per weight tensor")
    hs = [_u8(t) for t in tensors]
    sc = [_u8(t) for t in scales]
    arr = (ctypes.c_void_p * len(sc))(*[None if a is None else a.ctypes.data for a in sc])
    return hs, code, arr, sc


def mx_value(wfmt: str, code: int, scale: int) -> float:
    """Decoded MX element (E4M3 byte or E2M1 nibble) times its E8M0 scale."""
    return lib().oracle_mx_value(WEIGHT_FORMATS[wfmt], int(code), int(scale))


def _f32(a):
    if a is None:
        return None
    h, d = _as_host(a)
    if d != OR_F32:
        raise TypeError("router weights and bias are fp32")
    return h


def _tokens(tokens, T):
    if tokens is None:
        return None, T
    tk = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    if tk.size and (tk.min() < 0 or tk.max() >= T):
        raise IndexError("token index out of range")
    return tk, int(tk.size)


def route(cfg: OracleCfg, X, Wr, bias=None, tokens=None, nthreads=0) -> dict:
    """Routing of the listed tokens: logits, scores, biased scores [n,E], idx [n,k],
    w [n,k] and margin [n] (k-th minus (k+1)-th biased score)."""
    Xh, xd = _as_host(X)
    T = Xh.shape[0]
    Wrh, bh = _f32(Wr), _f32(bias)
    tk, n = _tokens(tokens, T)
    E, k = cfg.E, cfg.k
    out = dict(logits=np.empty((n, E)), scores=np.empty((n, E)), biased=np.empty((n, E)),
               idx=np.empty((n, k), dtype=np.int32), w=np.empty((n, k)), margin=np.empty(n))
    if n == 0:
        return out
    r = lib().oracle_route(ctypes.byref(cfg), _ptr(Xh), xd, _ptr(Wrh), _ptr(bh), n, _ptr(tk),
                           _ptr(out["logits"]), _ptr(out["scores"]), _ptr(out["biased"]),
                           _ptr(out["idx"]), _ptr(out["w"]), _ptr(out["margin"]), int(nthreads))
    if r < 0:
        raise ValueError("oracle_route rejected its arguments")
    out["threads"] = r
    return out


def forward(cfg: OracleCfg, X, Wr, bias, Wg, Wu, Wd, Wgs=None, Wus=None, Wds=None,
            tokens=None, nthreads=0, wfmt="bf16", scales=None) -> np.ndarray:
    """Block output Y [n,H] (fp64) for the listed tokens.  wfmt "mxfp8" /
    "mxfp4": the six weight tensors hold uint8 element codes and ``scales`` the
    six block-major uint8 scale tensors (None where a tensor is unused)."""
    Xh, xd = _as_host(X)
    T = Xh.shape[0]
    Wrh, bh = _f32(Wr), _f32(bias)
    use_sh = not cfg.shared_packed and cfg.S > 0
    tensors = [Wg, Wu, Wd] + ([Wgs, Wus, Wds] if use_sh else [None, None, None])
    if scales is not None and not use_sh:
        scales = list(scales[:3]) + [None, None, None]
    hs, wd, sc_arr, _keep = _weights(tensors, wfmt, scales)
    tk, n = _tokens(tokens, T)
    Y = np.empty((n, cfg.H))
    if n == 0:
        return Y
    r = lib().oracle_forward(ctypes.byref(cfg), _ptr(Xh), xd, _ptr(Wrh), _ptr(bh), _ptr(hs[0]),
                             _ptr(hs[1]), _ptr(hs[2]), _ptr(hs[3]), _ptr(hs[4]), _ptr(hs[5]), wd,
                             sc_arr, n, _ptr(tk), _ptr(Y), int(nthreads))
    if r < 0:
        raise ValueError("oracle_forward rejected its arguments")
    return Y


def _scales(shape, inputs: dict):
    if shape.weight_format == "bf16":
        return None
    return [inputs.get(k) for k in SCALE_KEYS]


def forward_inputs(shape, inputs: dict, tokens=None, nthreads=0) -> np.ndarray:
    """Block output for a workloads.make_inputs() dict (the oracle sees the
    workload's own dtypes: fp32 expert weights stay fp32, MX codes are decoded)."""
    return forward(cfg_from_shape(shape), inputs["X"], inputs["router_w"], inputs["expert_bias"],
                   inputs["gate"], inputs["up"], inputs["down"], inputs["sh_gate"],
                   inputs["sh_up"], inputs["sh_down"], tokens=tokens, nthreads=nthreads,
                   wfmt=shape.weight_format, scales=_scales(shape, inputs))


def route_inputs(shape, inputs: dict, tokens=None, nthreads=0) -> dict:
    return route(cfg_from_shape(shape), inputs["X"], inputs["router_w"], inputs["expert_bias"],
                 tokens=tokens, nthreads=nthreads)


def expert(cfg: OracleCfg, x, Wg, Wu, Wd, width: int, wfmt="bf16", scales=None):
    """One expert MLP on one token: returns (g, u, a, y) in fp64 (MX weights:
    uint8 codes and the three scale tensors)."""
    xh, xd = _as_host(x)
    hs, wd, sc_arr, _keep = _weights([Wg, Wu, Wd], wfmt, scales)
    g, u, a, y = (np.empty(width), np.empty(width), np.empty(width), np.empty(cfg.H))
    r = lib().oracle_expert(ctypes.byref(cfg), _ptr(xh), xd, _ptr(hs[0]), _ptr(hs[1]), _ptr(hs[2]), wd,
                            sc_arr, int(width), _ptr(g), _ptr(u), _ptr(a), _ptr(y))
    if r < 0:
        raise ValueError("oracle_expert rejected its arguments")
    return g, u, a, y


def act(cfg: OracleCfg, g: float, u: float) -> float:
    return lib().oracle_act(ctypes.byref(cfg), float(g), float(u))


def dense(cfg: OracleCfg, X, Wg, Wu, Wd, tokens=None, nthreads=0, wfmt="bf16", scales=None) -> np.ndarray:
    """Dense MLP of width cfg.S (a dense prefix layer) for the listed tokens: [n,H] fp64."""
    Xh, xd = _as_host(X)
    T = Xh.shape[0]
    hs, wd, sc_arr, _keep = _weights([Wg, Wu, Wd], wfmt, scales)
    tk, n = _tokens(tokens, T)
    Y = np.empty((n, cfg.H))
    if n == 0:
        return Y
    r = lib().oracle_dense(ctypes.byref(cfg), _ptr(Xh), xd, _ptr(hs[0]), _ptr(hs[1]), _ptr(hs[2]), wd, sc_arr,
                           n, _ptr(tk), _ptr(Y), int(nthreads))
    if r < 0:
        raise ValueError("oracle_dense rejected its arguments")
    return Y


def to_f64(a) -> np.ndarray:
    """Exact fp64 values of an fp32 / bf16 array or tensor (bf16 from its bits)."""
    h, d = _as_host(a)
    if d == OR_BF16:
        return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return h.astype(np.float64)


def round_to(a: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 values rounded to the activation dtype: fp32 (round to nearest even),
    or bf16 as uint16 bits (fp32 first, then round to nearest even)."""
    f = np.ascontiguousarray(a, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return f
    b = f.view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def rmsnorm(X, w, eps: float, gemma: bool) -> np.ndarray:
    """Row-wise RMSNorm of X [n,H] in fp64: x / sqrt(mean(x^2) + eps) * g, g = w or 1 + w."""
    Xd = np.ascontiguousarray(to_f64(X) if not isinstance(X, np.ndarray) or X.dtype != np.float64 else X)
    wd = np.ascontiguousarray(to_f64(w) if not isinstance(w, np.ndarray) or w.dtype != np.float64 else w)
    n, H = Xd.shape
    Y = np.empty_like(Xd)
    for i in range(n):
        if lib().oracle_rmsnorm(_ptr(Xd[i]), H, _ptr(wd), float(eps), int(bool(gemma)), _ptr(Y[i])) < 0:
            raise ValueError("oracle_rmsnorm rejected its arguments")
    return Y


def normed_input(shape, X, w_pre) -> np.ndarray:
    """The block's input after pre_mlp_norm, rounded to the activation dtype (the
    MLP consumes it in that dtype): bf16 bits or fp32 values [T,H]."""
    return round_to(rmsnorm(X, w_pre, shape.rms_norm_eps, shape.mlp_norm == "gemma"), shape.dtype)


def block_output(shape, inputs: dict, tokens=None, nthreads=0) -> np.ndarray:
    """Output of the layer for the listed tokens, fp64 [n,H].  E > 0: the MoE
    block; E = 0: a dense MLP of width S.  With the sandwich norms
    (shape.mlp_norm "rms" or "gemma"): out = X + post_norm(mlp(pre_norm(X))),
    pre_norm's output rounded to the activation dtype."""
    X = inputs["X"]
    xin = X if shape.mlp_norm == "none" else normed_input(shape, X, inputs["pre_norm_w"])
    cfg = cfg_from_shape(shape)
    sc = _scales(shape, inputs)
    if shape.E == 0:
        y = dense(cfg, xin, inputs["sh_gate"], inputs["sh_up"], inputs["sh_down"], tokens=tokens,
                  nthreads=nthreads, wfmt=shape.weight_format, scales=None if sc is None else sc[3:])
    else:
        y = forward(cfg, xin, inputs["router_w"], inputs["expert_bias"], inputs["gate"], inputs["up"],
                    inputs["down"], inputs["sh_gate"], inputs["sh_up"], inputs["sh_down"], tokens=tokens,
                    nthreads=nthreads, wfmt=shape.weight_format, scales=sc)
    if shape.mlp_norm == "none":
        return y
    x = to_f64(X)
    if tokens is not None:
        x = x[np.asarray(tokens)]
    return x + rmsnorm(y, inputs["post_norm_w"], shape.rms_norm_eps, shape.mlp_norm == "gemma")


def margin_filter(shape, min_margin: float = 1e-3, nthreads: int = 0):
    """Row filter for workloads.make_inputs: True for tokens whose gap between
    the k-th and (k+1)-th biased scores is below ``min_margin`` (routing the
    pre_mlp_norm output when the workload has the sandwich norms)."""
    cfg = cfg_from_shape(shape)

    def _filter(X, Wr, b, w_pre=None):
        xin = X if shape.mlp_norm == "none" else normed_input(shape, X, w_pre)
        return route(cfg, xin, Wr, b, nthreads=nthreads)["margin"] < min_margin

    return _filter
