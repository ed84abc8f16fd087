"""Helpers of the GPU parity tests: seeded inputs with the top-k margin
enforced by the oracle, a handle over them, and the comparisons.

Tolerances:
  * top-k: the per-token SETS of expert ids are compared bit-exactly; the
    order inside a set is compared where neighbouring biased scores differ by
    more than 1e-5 (closer scores may legitimately swap between fp32 and fp64);
  * routing weights: per expert id, |w_gpu - w_ref| <= 1e-5 |w_ref| + 1e-7;
  * outputs: max |Y_gpu - Y_ref| <= 2e-2 * rms(Y_ref), element-wise, with
    Y_ref the fp64 oracle's output (bf16 storage of the activations between
    the two projections, fp32 accumulation).  Two ratios are recorded per
    check: that literal one, and max |Y_gpu - rne_bf16(Y_ref)| / rms(Y_ref)
    against the oracle's output rounded once to the output dtype, with the
    number of elements that land on the other bf16 neighbour of Y_ref.  The
    second is recorded, not asserted: one bf16 ulp is 2^-5 rms at |Y| in
    [4, 8) rms, so any disagreement in the last bit of such an element exceeds
    2e-2 rms, and the bf16 hidden activations alone move Y by ~1e-3 rms.

The oracle reads the same stored buffers as the CUDA path: the block takes
bf16 expert weights, so a workload drawn in fp32 hands both sides the same
bf16-rounded expert tensors (X and the router stay fp32 on both sides), except
where a test asks for the fp32 originals (``host_inputs(..., as_drawn=True)``)
to measure the rounding of the expert weights as well.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from expert_routed_ffn_gb300 import capi
from expert_routed_ffn_gb300 import workloads as wl

Y_TOL = 2e-2
W_RTOL = 1e-5
MARGIN = 1e-3


def make_case(shape, max_tokens=None, device="cuda"):
    inputs = wl.make_inputs(shape, device, row_filter=oracle.margin_filter(shape, MARGIN))
    blk = capi.block_from_inputs(shape, inputs, max_tokens=max_tokens)
    return inputs, blk


# every output check: (test id, max|Y - Y_ref| / rms, max|Y - rne_bf16(Y_ref)| / rms,
# elements on the other bf16 neighbour of Y_ref, elements compared)
RESULTS = []


def host_inputs(inputs, as_drawn=False):
    """Host copies of what the CUDA path reads (expert weights as stored: bf16),
    or, with ``as_drawn``, of the tensors as the workload drew them (fp32 expert
    weights of the fp32 workload)."""
    if as_drawn:
        return {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}
    experts = wl.expert_weights_bf16(inputs)
    out = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inputs.items() if k not in experts}
    for k, v in experts.items():
        out[k] = None if v is None else v.cpu()
    return out


def bf16_half_ulp(y):
    """Half the bf16 spacing at |y| (8 significant bits): 2^(floor(log2|y|) - 8)."""
    a = np.abs(y)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def check_route(shape, inputs_h, idx_gpu, w_gpu, tokens=None, w_rtol=W_RTOL):
    """``w_rtol``: a scalar, or one relative tolerance per token."""
    ref = oracle.route_inputs(shape, inputs_h, tokens=tokens)
    rtol = np.broadcast_to(np.asarray(w_rtol, dtype=np.float64), (ref["idx"].shape[0],))
    idx_gpu = np.asarray(idx_gpu, dtype=np.int64)
    w_gpu = np.asarray(w_gpu, dtype=np.float64)
    ridx = ref["idx"].astype(np.int64)
    assert ref["margin"].min() >= MARGIN - 1e-12
    assert np.array_equal(np.sort(idx_gpu, 1), np.sort(ridx, 1)), "top-k sets differ"
    c = ref["biased"]
    for t in range(ridx.shape[0]):
        cs = c[t, ridx[t]]
        for j in range(ridx.shape[1]):
            lo_ok = j == 0 or cs[j - 1] - cs[j] > 1e-5
            hi_ok = j == ridx.shape[1] - 1 or cs[j] - cs[j + 1] > 1e-5
            if lo_ok and hi_ok:
                assert idx_gpu[t, j] == ridx[t, j], f"order of token {t} slot {j}"
        wg = dict(zip(idx_gpu[t].tolist(), w_gpu[t].tolist()))
        for e, wr in zip(ridx[t].tolist(), ref["w"][t].tolist()):
            assert abs(wg[e] - wr) <= rtol[t] * abs(wr) + 1e-7, f"weight of token {t} expert {e}"
    return ref


def rne_bf16(y):
    """fp64 values rounded to the nearest bf16 (ties to even), via fp32 (exact for
    the magnitudes here: the fp32 rounding cannot create a bf16 tie)."""
    f = np.ascontiguousarray(np.asarray(y, dtype=np.float64).astype(np.float32))
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def check_output(Y_gpu, Y_ref, out_bf16=True, tol=Y_TOL, tag=""):
    """Asserts max |Y_gpu - Y_ref| <= tol * rms(Y_ref); returns that ratio."""
    Yg = np.asarray(Y_gpu, dtype=np.float64)
    rms = float(np.sqrt(np.mean(Y_ref ** 2)))
    assert np.isfinite(Yg).all(), "non-finite output"
    diff = np.abs(Yg - Y_ref)
    literal = float(diff.max()) / rms
    if out_bf16:
        R = rne_bf16(Y_ref)
        rounded = float(np.abs(Yg - R).max()) / rms
        other = int((Yg != R).sum())
    else:
        rounded, other = literal, 0
    RESULTS.append((tag, literal, rounded, other, int(Yg.size)))
    assert literal <= tol, f"max|Y-Yref|/rms(Yref) = {literal:.4f} exceeds {tol}"
    return literal


def to_np(t):
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


def normed_error(shape, x_gpu, inputs_h):
    """Checks the GPU's pre_norm(X) against the oracle's and returns
    (oracle's rounded normed input, per-token bound D_t on how far any router
    logit of the GPU's normed row can sit from the oracle's).

    bf16: every element equals the oracle's rounding of the fp64 value or is the
    other bf16 neighbour of a value within 1e-5 (relative) of a rounding
    midpoint: |x_gpu - x64| <= half a bf16 ulp + 1e-5 |x64|.  fp32: within
    1e-5 |x64| + 1e-30.  A router logit is sum_i x_i Wr[e, i], so a row that
    differs by dx moves every logit by at most D_t = sum_i |dx_i| max_e |Wr[e, i]|.
    """
    gemma = shape.mlp_norm == "gemma"
    x64 = oracle.rmsnorm(inputs_h["X"], inputs_h["pre_norm_w"], shape.rms_norm_eps, gemma)
    xin = oracle.normed_input(shape, inputs_h["X"], inputs_h["pre_norm_w"])
    xg = oracle.to_f64(x_gpu)
    xr = oracle.to_f64(xin)
    if shape.dtype == "bf16":
        bound = bf16_half_ulp(x64) + 1e-5 * np.abs(x64)
    else:
        bound = 1e-5 * np.abs(x64) + 1e-30
    diff = np.abs(xg - x64)
    assert np.all(diff[bound == 0] == 0), "an exact zero of the normed input is not zero"
    worst = float(np.max(diff[bound > 0] / bound[bound > 0], initial=0.0))
    assert worst <= 1.0, f"normed input off by x{worst:.3f} of its bound"
    if shape.E == 0:
        return xin, np.zeros(xg.shape[0])
    wmax = np.abs(oracle.to_f64(inputs_h["router_w"])).max(axis=0)
    return xin, np.abs(xg - xr) @ wmax


def route_rtol(D):
    """Relative tolerance of the routing weights when every logit may move by D:
    a sigmoid score's log moves by at most D, a softmax probability's by 2D, and
    renormalising the k selected weights at most doubles that, so |dw / w| <= 4D
    to first order (4.5 D covers the second-order term for D < 0.01)."""
    assert np.all(D < 1e-2)
    return W_RTOL + 4.5 * np.asarray(D)
