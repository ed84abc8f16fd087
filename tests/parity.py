"""Helpers of the GPU parity tests: seeded inputs with the top-k margin
enforced by the oracle, a handle over them, and the comparisons.

Tolerances:
  * top-k: the per-token SETS of expert ids are compared bit-exactly; the
    order inside a set is compared where neighbouring biased scores differ by
    more than 1e-5 (closer scores may legitimately swap between fp32 and fp64);
  * routing weights: per expert id, |w_gpu - w_ref| <= 1e-5 |w_ref| + 1e-7;
  * outputs: |Y_gpu - Y_ref| <= 2e-2 * rms(Y_ref) + (half a bf16 ulp of Y_ref
    when Y is stored in bf16), element-wise.  A bf16 output cannot be closer to
    the fp64 value than half an ulp, and at |Y| ~ 5 rms that alone is up to
    ~1.9% of rms, so the storage rounding of Y is added to the 2e-2 * rms budget
    of the computation (bf16 expert weights and activations, fp32 accumulation).
    The literal ratio max|Y_gpu - Y_ref| / rms(Y_ref) is recorded as well.

The oracle reads the same stored buffers as the CUDA path: the block takes
bf16 expert weights, so a workload drawn in fp32 hands both sides the same
bf16-rounded expert tensors (X and the router stay fp32 on both sides).
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


RESULTS = []  # (test id, literal max|dY|/rms, bound-normalised error) of every output check


def host_inputs(inputs):
    """Host copies of what the CUDA path reads (expert weights as stored: bf16)."""
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


def check_route(shape, inputs_h, idx_gpu, w_gpu, tokens=None):
    ref = oracle.route_inputs(shape, inputs_h, tokens=tokens)
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
            assert abs(wg[e] - wr) <= W_RTOL * abs(wr) + 1e-7, f"weight of token {t} expert {e}"
    return ref


def check_output(Y_gpu, Y_ref, out_bf16=True, tol=Y_TOL, tag=""):
    Yg = np.asarray(Y_gpu, dtype=np.float64)
    rms = float(np.sqrt(np.mean(Y_ref ** 2)))
    assert np.isfinite(Yg).all(), "non-finite output"
    diff = np.abs(Yg - Y_ref)
    bound = tol * rms + (bf16_half_ulp(Y_ref) if out_bf16 else 0.0)
    worst = float((diff / bound).max())
    literal = float(diff.max()) / rms
    RESULTS.append((tag, literal, worst))
    assert worst <= 1.0, (f"|Y-Yref| exceeds {tol}*rms(+half bf16 ulp) by x{worst:.3f}; "
                          f"max|Y-Yref|/rms = {literal:.4f}")
    return literal


def to_np(t):
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
