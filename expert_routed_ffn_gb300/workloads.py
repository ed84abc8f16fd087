"""Seeded synthetic workloads for the token-choice MoE FFN block.

This module only draws inputs: shapes, dtypes, seeds and value distributions.
It holds none of the block's arithmetic (no routing, no activation, no
combine), so both the CUDA path and the fp64 oracle can be fed from it.

Shapes follow the pages:
  * Arcee AFMoE issue (mlxcel #845), "Checkpoint confirmed": Trinity-Nano has
    hidden 1024 and 128 experts; "Routing detail": route_scale 2.826.
  * HF Transformers AFMoE docs, ``AfmoeConfig`` signature: hidden_size 2048,
    moe_intermediate_size 1408, num_experts 64, num_experts_per_tok 6,
    num_shared_experts 2, route_scale 1.0, initializer_range 0.02.
  * MiniMax-M3 issue (mlxcel #763), "Architecture specification": hidden 6144,
    128 experts of width 3072, top-4, routed_scaling_factor 2.0, one shared
    expert of width 3072 packed as expert index 128, clamp-SwiGLU.

Recipe (all workloads):
  * X ~ N(0, 1); router, expert and shared weights ~ N(0, 0.02);
  * expert_bias ~ U(-0.1, 0.1), or, for the load-skew sweep, a Zipf(s=1.2)
    profile r^-1.2 over ranks r = 1..E, min-max scaled to [0, 0.5] and assigned
    to experts through a seeded random permutation;
  * draw order: router, bias, gate, up, down (all E or E+1 slices), shared
    gate/up/down, then X from its own generator;
  * bf16 workloads round every drawn value to bf16 (round-to-nearest-even).
    Router weights are rounded to bf16 too but stored as fp32, so the router
    of both sides sees identical fp32 values;
  * the tiny workload keeps fp32 for X, router and expert weights;
  * dense layers (num_experts = 0: the dense prefix of the AFMoE issue, "Dense
    prefix", and the MiniMax-M3 issue, dense_intermediate_size 12288; width
    6144 is AfmoeConfig's intermediate_size) draw only their MLP weights, as
    the shared tensors;
  * with the sandwich norms (mlp_norm "rms" or "gemma": AFMoE issue, four norms
    per layer; MiniMax-M3 issue, Gemma-style RMSNorm weight + 1), the
    pre_mlp / post_mlp norm weights [H] fp32 are drawn after the MLP weights:
    1 + N(0, 0.1) for "rms", N(0, 0.1) for "gemma" (applied as 1 + w).

A caller may pass ``row_filter``: a function of the host copy of
(X, router_w, expert_bias) (and pre_mlp_norm's weight when the workload has the
sandwich norms) returning a boolean mask of token rows to redraw.
The parity tests use it to enforce a gap of at least 1e-3 between the k-th and
(k+1)-th biased router scores, so that top-k sets are unique.  Redrawn rows
come from a generator seeded with (x_seed, attempt).
"""

from __future__ import annotations

import dataclasses
from typing import Callable, Optional

import torch

WEIGHT_STD = 0.02
BIAS_HALF_RANGE = 0.1
ZIPF_S = 1.2
ZIPF_MAX = 0.5
NORM_STD = 0.1


@dataclasses.dataclass(frozen=True)
class MoeShape:
    """One workload: the MoE block's config keys plus the token count."""

    name: str
    T: int
    hidden_size: int
    num_experts: int
    num_experts_per_tok: int
    moe_intermediate_size: int
    num_shared_experts: int
    shared_intermediate_size: int  # total shared width S
    shared_packed: bool
    hidden_act: str  # "silu" | "swigluoai"
    score_func: str  # "sigmoid" | "softmax"
    route_norm: bool
    route_scale: float
    dtype: str  # "f32" | "bf16"
    bias_kind: str  # "uniform" | "zipf"
    seed: int
    x_seed: int
    act_alpha: float = 1.702
    act_limit: float = 7.0
    act_beta: float = 1.0
    mlp_norm: str = "none"  # "none" | "rms" | "gemma": pre_mlp / post_mlp RMSNorm around the MLP
    rms_norm_eps: float = 1e-5
    weight_format: str = "bf16"  # "bf16" | "mxfp8" | "mxfp4": storage of the expert weights

    @property
    def H(self) -> int:
        return self.hidden_size

    @property
    def E(self) -> int:
        return self.num_experts

    @property
    def k(self) -> int:
        return self.num_experts_per_tok

    @property
    def I(self) -> int:  # noqa: E743 - the pages' name for the expert width
        return self.moe_intermediate_size

    @property
    def S(self) -> int:
        return self.shared_intermediate_size

    @property
    def stacked_experts(self) -> int:
        """Slices of the stacked gate/up/down tensors (E, or E+1 when packed)."""
        return self.E + (1 if self.shared_packed else 0)

    def with_tokens(self, T: int, x_seed: Optional[int] = None) -> "MoeShape":
        return dataclasses.replace(self, T=T, x_seed=self.x_seed if x_seed is None else x_seed)

    def replace(self, **kw) -> "MoeShape":
        return dataclasses.replace(self, **kw)


def _afmoe_default(T: int, bias_kind: str, seed: int, x_seed: int, name: str) -> MoeShape:
    return MoeShape(
        name=name, T=T, hidden_size=2048, num_experts=64, num_experts_per_tok=6,
        moe_intermediate_size=1408, num_shared_experts=2, shared_intermediate_size=2 * 1408,
        shared_packed=False, hidden_act="silu", score_func="sigmoid", route_norm=True,
        route_scale=1.0, dtype="bf16", bias_kind=bias_kind, seed=seed, x_seed=x_seed)


TINY = MoeShape(
    name="tiny_f32_T64_H256_E16_k4", T=64, hidden_size=256, num_experts=16, num_experts_per_tok=4,
    moe_intermediate_size=128, num_shared_experts=1, shared_intermediate_size=128,
    shared_packed=False, hidden_act="silu", score_func="sigmoid", route_norm=True,
    route_scale=2.826, dtype="f32", bias_kind="uniform", seed=1001, x_seed=1101)

NANO_DECODE = MoeShape(
    name="nano_decode_T256_H1024_E128_k8", T=256, hidden_size=1024, num_experts=128,
    num_experts_per_tok=8, moe_intermediate_size=256, num_shared_experts=1,
    shared_intermediate_size=256, shared_packed=False, hidden_act="silu", score_func="sigmoid",
    route_norm=True, route_scale=2.826, dtype="bf16", bias_kind="uniform", seed=1002, x_seed=1102)

AFMOE_PREFILL = _afmoe_default(4096, "uniform", 1003, 1103, "afmoe_prefill_T4096_H2048_E64_k6")

M3 = MoeShape(
    name="m3_T2048_H6144_E128_k4_packed", T=2048, hidden_size=6144, num_experts=128,
    num_experts_per_tok=4, moe_intermediate_size=3072, num_shared_experts=1,
    shared_intermediate_size=3072, shared_packed=True, hidden_act="swigluoai",
    score_func="sigmoid", route_norm=False, route_scale=2.0, dtype="bf16", bias_kind="uniform",
    seed=1004, x_seed=1104)

ZIPF_TOKENS = (1, 8, 64, 512, 4096, 16384)


def zipf_sweep(T: int) -> MoeShape:
    return _afmoe_default(T, "zipf", 1005, 2000 + T, f"afmoe_zipf_T{T}")


def dense_layer(T: int, model: str) -> MoeShape:
    """A dense prefix layer: AFMoE (hidden 2048, intermediate_size 6144, silu) or
    MiniMax-M3 (hidden 6144, dense_intermediate_size 12288, clamp-SwiGLU)."""
    if model == "afmoe":
        return MoeShape(name=f"dense_afmoe_T{T}_H2048_I6144", T=T, hidden_size=2048, num_experts=0,
                        num_experts_per_tok=0, moe_intermediate_size=0, num_shared_experts=1,
                        shared_intermediate_size=6144, shared_packed=False, hidden_act="silu",
                        score_func="sigmoid", route_norm=True, route_scale=1.0, dtype="bf16",
                        bias_kind="uniform", seed=1006, x_seed=3000 + T, mlp_norm="rms")
    return MoeShape(name=f"dense_m3_T{T}_H6144_I12288", T=T, hidden_size=6144, num_experts=0,
                    num_experts_per_tok=0, moe_intermediate_size=0, num_shared_experts=1,
                    shared_intermediate_size=12288, shared_packed=False, hidden_act="swigluoai",
                    score_func="sigmoid", route_norm=True, route_scale=1.0, dtype="bf16",
                    bias_kind="uniform", seed=1007, x_seed=4000 + T, mlp_norm="gemma")


WORKLOADS = {
    "tiny": TINY,
    "nano_decode": NANO_DECODE,
    "afmoe_prefill": AFMOE_PREFILL,
    "m3": M3,
    **{f"zipf_T{t}": zipf_sweep(t) for t in ZIPF_TOKENS},
    # the layers around the block (next rows): sandwich norms, dense prefix
    "afmoe_prefill_sandwich": AFMOE_PREFILL.replace(name="afmoe_prefill_sandwich_T4096", mlp_norm="rms"),
    "nano_decode_sandwich": NANO_DECODE.replace(name="nano_decode_sandwich_T256", mlp_norm="rms"),
    "m3_sandwich": M3.replace(name="m3_sandwich_T2048_gemma", mlp_norm="gemma"),
    "dense_afmoe_prefill": dense_layer(4096, "afmoe"),
    "dense_afmoe_decode": dense_layer(256, "afmoe"),
    "dense_m3": dense_layer(2048, "m3"),
    # block-scaled expert weights (next row): the same draws, stored as MXFP8 / MXFP4
    "nano_decode_mxfp8": NANO_DECODE.replace(name="nano_decode_mxfp8_T256", weight_format="mxfp8"),
    "nano_decode_mxfp4": NANO_DECODE.replace(name="nano_decode_mxfp4_T256", weight_format="mxfp4"),
    "afmoe_prefill_mxfp8": AFMOE_PREFILL.replace(name="afmoe_prefill_mxfp8_T4096", weight_format="mxfp8"),
    "m3_mxfp8": M3.replace(name="m3_mxfp8_T2048", weight_format="mxfp8"),
}


def _torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _normal(gen: torch.Generator, shape, std: float, dtype: torch.dtype, device) -> torch.Tensor:
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        v.mul_(std)
    return v.to(dtype)


def _stacked(gen, n, rows, cols, dtype, device) -> torch.Tensor:
    out = torch.empty((n, rows, cols), dtype=dtype, device=device)
    for e in range(n):  # one slice at a time bounds the fp32 temporary
        out[e].copy_(_normal(gen, (rows, cols), WEIGHT_STD, dtype, device))
    return out


MX_BLOCK = 32
# largest exponent of the MX element types (E4M3: 448 = 1.75 * 2^8; E2M1: 6 = 1.5 * 2^2)
_MX_EMAX = {"mxfp8": 8, "mxfp4": 2}
_E2M1_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)  # between 0, .5, 1, 1.5, 2, 3, 4, 6


def mx_quantize(w: torch.Tensor, fmt: str):
    """[rows, cols] fp32 -> (element codes, block scales) in the OCP MX layout
    used by the block: blocks of 32 along cols share the E8M0 exponent
    floor(log2(max |w|)) - emax(element), elements rounded to nearest and
    saturated.  Codes: [rows, cols] uint8 (E4M3) or [rows, cols / 2] uint8
    (E2M1, element 2j in the low nibble); scales [cols / 32, rows] uint8
    (block-major)."""
    rows, cols = w.shape
    b = w.float().reshape(rows, cols // MX_BLOCK, MX_BLOCK)
    amax = b.abs().amax(-1)
    _, ex = torch.frexp(amax)  # amax = m * 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1
    e = torch.where(amax > 0, ex - 1 - _MX_EMAX[fmt], torch.full_like(ex, -127)).clamp(-127, 127)
    v = b * torch.exp2(-e.float())[..., None]
    if fmt == "mxfp8":
        codes = v.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).reshape(rows, cols)
    else:
        mids = torch.tensor(_E2M1_MIDPOINTS, dtype=torch.float32, device=w.device)
        mag = torch.bucketize(v.abs().clamp(max=6.0), mids).to(torch.uint8)  # code order = value order
        nib = (mag | ((v < 0).to(torch.uint8) << 3)).reshape(rows, cols)
        codes = nib[:, 0::2] | (nib[:, 1::2] << 4)
    return codes.contiguous(), (e + 127).to(torch.uint8).t().contiguous()


def _stacked_mx(gen, n, rows, cols, fmt, device):
    per = cols if fmt == "mxfp8" else cols // 2
    codes = torch.empty((n, rows, per), dtype=torch.uint8, device=device)
    scales = torch.empty((n, cols // MX_BLOCK, rows), dtype=torch.uint8, device=device)
    for e in range(n):  # the same draws as the bf16 tensors, quantized slice by slice
        codes[e], scales[e] = mx_quantize(_normal(gen, (rows, cols), WEIGHT_STD, torch.float32, device), fmt)
    return codes, scales


def _bias(shape: MoeShape, gen: torch.Generator, device) -> torch.Tensor:
    E = shape.E
    if shape.bias_kind == "uniform":
        u = torch.rand((E,), generator=gen, device=device, dtype=torch.float32)
        return (u * 2.0 - 1.0) * BIAS_HALF_RANGE
    if shape.bias_kind == "zipf":
        ranks = torch.arange(1, E + 1, dtype=torch.float64)
        z = ranks.pow(-ZIPF_S)
        z = ZIPF_MAX * (z - z.min()) / (z.max() - z.min())
        perm = torch.randperm(E, generator=gen, device=device).cpu()
        b = torch.empty(E, dtype=torch.float64)
        b[perm] = z  # expert perm[r-1] gets rank r
        return b.to(torch.float32).to(device)
    raise ValueError(shape.bias_kind)


def make_inputs(shape: MoeShape, device="cpu",
                row_filter: Optional[Callable[[torch.Tensor, torch.Tensor, torch.Tensor], torch.Tensor]] = None,
                max_attempts: int = 64) -> dict:
    """Draw every tensor of one workload on ``device``.

    Returns a dict with X [T,H], router_w [E,H] fp32, expert_bias [E] fp32,
    gate/up [E',I,H], down [E',H,I] (E' = E+1 when the shared expert is packed)
    and, for a separate shared expert, sh_gate/sh_up [S,H], sh_down [H,S].
    Expert tensors are fp32 for the f32 workload and bf16 otherwise.
    ``redraws`` counts the token rows that ``row_filter`` sent back.
    """
    device = torch.device(device)
    dt = _torch_dtype(shape.dtype)
    g = torch.Generator(device=device)
    g.manual_seed(shape.seed)
    E, H, I, S = shape.E, shape.H, shape.I, shape.S
    Ep = shape.stacked_experts

    wf = shape.weight_format
    scales = {}
    router_w = expert_bias = gate = up = down = None
    if E > 0:
        router_w = _normal(g, (E, H), WEIGHT_STD, dt, device).to(torch.float32)
        expert_bias = _bias(shape, g, device)
        if wf == "bf16":
            gate = _stacked(g, Ep, I, H, dt, device)
            up = _stacked(g, Ep, I, H, dt, device)
            down = _stacked(g, Ep, H, I, dt, device)
        else:
            gate, scales["gate_scale"] = _stacked_mx(g, Ep, I, H, wf, device)
            up, scales["up_scale"] = _stacked_mx(g, Ep, I, H, wf, device)
            down, scales["down_scale"] = _stacked_mx(g, Ep, H, I, wf, device)
    sh_gate = sh_up = sh_down = None
    if not shape.shared_packed and S > 0:
        if wf == "bf16":
            sh_gate = _normal(g, (S, H), WEIGHT_STD, dt, device)
            sh_up = _normal(g, (S, H), WEIGHT_STD, dt, device)
            sh_down = _normal(g, (H, S), WEIGHT_STD, dt, device)
        else:
            sh_gate, scales["sh_gate_scale"] = mx_quantize(_normal(g, (S, H), WEIGHT_STD, torch.float32, device), wf)
            sh_up, scales["sh_up_scale"] = mx_quantize(_normal(g, (S, H), WEIGHT_STD, torch.float32, device), wf)
            sh_down, scales["sh_down_scale"] = mx_quantize(_normal(g, (H, S), WEIGHT_STD, torch.float32, device),
                                                           wf)
    pre_norm_w = post_norm_w = None
    if shape.mlp_norm != "none":
        centre = 1.0 if shape.mlp_norm == "rms" else 0.0
        pre_norm_w = _normal(g, (H,), NORM_STD, torch.float32, device) + centre
        post_norm_w = _normal(g, (H,), NORM_STD, torch.float32, device) + centre

    gx = torch.Generator(device=device)
    gx.manual_seed(shape.x_seed)
    X = _normal(gx, (shape.T, H), 1.0, dt, device)

    redraws = 0
    if row_filter is not None and shape.T > 0 and E > 0:
        for attempt in range(max_attempts):
            extra = () if pre_norm_w is None else (pre_norm_w.cpu(),)
            bad = row_filter(X.cpu(), router_w.cpu(), expert_bias.cpu(), *extra)
            bad = torch.as_tensor(bad, dtype=torch.bool)
            n_bad = int(bad.sum())
            if n_bad == 0:
                break
            redraws += n_bad
            gr = torch.Generator(device=device)
            gr.manual_seed(shape.x_seed * 1_000_003 + attempt + 1)
            rows = bad.nonzero().flatten().to(device)
            X[rows] = _normal(gr, (n_bad, H), 1.0, dt, device)
        else:
            raise RuntimeError(f"{shape.name}: rows still rejected after {max_attempts} redraws")

    return dict(X=X, router_w=router_w, expert_bias=expert_bias, gate=gate, up=up, down=down,
                sh_gate=sh_gate, sh_up=sh_up, sh_down=sh_down, pre_norm_w=pre_norm_w,
                post_norm_w=post_norm_w, redraws=redraws, **scales)


def expert_weights_bf16(inputs: dict) -> dict:
    """bf16 (round-to-nearest-even) copies of the expert tensors, for the CUDA path.

    The f32 workload stores fp32 expert weights; the CUDA path takes bf16 expert
    weights, so they are rounded once here.  bf16 workloads pass through.
    """
    out = {}
    for key in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        t = inputs[key]
        # MX element codes (uint8) pass through, like bf16 tensors
        out[key] = None if t is None else (t if t.dtype == torch.uint8 else t.to(torch.bfloat16).contiguous())
    return out
