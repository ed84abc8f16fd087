"""GPU parity of the layers around the MoE block and of the dense prefix layers,
through the C ABI, against the fp64 oracle.

* Sandwich norms (Arcee AFMoE: RMSNorm before and after the MLP, residual add;
  MiniMax-M3: the same with Gemma-style RMSNorm, scale 1 + weight): the GPU's
  normed input is checked element-wise against the oracle's, the routing of it
  on every token, and out = X + post_norm(mlp(pre_norm(X))) on every token, on
  every expert path, as a whole and with the residual taken out.
* Dense prefix layers (num_experts 0; AFMoE: SiLU-gated, width 6144; M3:
  clamp-SwiGLU, width 12288): hidden activations and outputs on every token
  for small widths on one CTA per tile and on CTA pairs; sampled tokens at the
  full sizes in the launch configuration the benchmark times.
"""

import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_gb300 import capi
from expert_routed_ffn_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

PATHS = {"decode": (capi.PATH_DECODE, 0), "grouped": (capi.PATH_GROUPED, 0), "pair": (capi.PATH_GROUPED, 1),
         "swapped": (capi.PATH_SWAPPED, 0)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routed_ffn_gb300 import build
    build.build()
    capi.load()


def _run(shape, path=None, inputs=None, blk=None, max_tokens=None):
    if inputs is None:
        inputs, blk = P.make_case(shape, max_tokens=max_tokens)
    if path is not None:
        blk.set_option(capi.MOE_OPT_PATH, path[0])
        blk.set_option(capi.MOE_OPT_GEMM_PAIR, path[1])
    Y = blk.forward(inputs["X"])
    torch.cuda.synchronize()
    assert blk.sync_status() == capi.MOE_OK
    return inputs, blk, Y


def _normed(blk, shape, T):
    dt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    x = blk.inspect(capi.MOE_BUF_NORMED_X, T * shape.H, dt).view(T, shape.H)
    torch.cuda.synchronize()
    return x.cpu()


def _topk(blk, T, k):
    idx = blk.inspect(capi.MOE_BUF_TOPK_IDX, T * k, torch.int32).view(T, k)
    w = blk.inspect(capi.MOE_BUF_TOPK_W, T * k, torch.float32).view(T, k)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def _check_layer(shape, inputs, blk, Y, tokens=None, tag=""):
    """Normed input (every token), routing (every token) and output (the listed
    tokens, or all), with and without the residual."""
    ih = P.host_inputs(inputs)
    T = shape.T
    if shape.mlp_norm != "none":
        xin, D = P.normed_error(shape, _normed(blk, shape, T), ih)
        if shape.E > 0:
            idx, w = _topk(blk, T, shape.k)
            P.check_route(shape, dict(ih, X=xin), idx, w, w_rtol=P.route_rtol(D))
    elif shape.E > 0:
        idx, w = _topk(blk, T, shape.k)
        P.check_route(shape, ih, idx, w)
    Yref = oracle.block_output(shape, ih, tokens=tokens)
    Yg = P.to_np(Y) if tokens is None else P.to_np(Y)[tokens]
    out_bf16 = shape.dtype == "bf16"
    P.check_output(Yg, Yref, out_bf16, tag=tag)
    if shape.mlp_norm != "none":
        # the normed MLP output alone, recovered as Y - X: the residual X is exact on
        # both sides, and what is stored is the sum, so its bf16 rounding (half an
        # ulp of Y, not of the MLP part) is part of this difference
        x = oracle.to_f64(ih["X"])
        if tokens is not None:
            x = x[tokens]
        post_ref, post_gpu = Yref - x, Yg.astype(np.float64) - x
        bound = P.Y_TOL * np.sqrt(np.mean(post_ref ** 2)) + (P.bf16_half_ulp(Yref) if out_bf16 else 0.0)
        worst = float((np.abs(post_gpu - post_ref) / bound).max())
        assert worst <= 1.0, f"post_norm(mlp) part off by x{worst:.3f} of its bound"


# ------------------------------------------------------------ sandwich norms

SANDWICH = {
    "afmoe_ragged_rms": wl.AFMOE_PREFILL.replace(name="afmoe_ragged_rms", T=333, hidden_size=512,
                                                 moe_intermediate_size=192, shared_intermediate_size=384,
                                                 mlp_norm="rms"),
    "m3_small_gemma": wl.M3.replace(name="m3_small_gemma", T=96, hidden_size=512, num_experts=8,
                                    num_experts_per_tok=2, moe_intermediate_size=256,
                                    shared_intermediate_size=256, mlp_norm="gemma"),
    "nano_rms": wl.NANO_DECODE.replace(name="nano_rms", mlp_norm="rms"),
    "tiny_f32_rms": wl.TINY.replace(name="tiny_f32_rms", mlp_norm="rms"),
    "nano_T1_gemma": wl.NANO_DECODE.replace(name="nano_T1_gemma", T=1, mlp_norm="gemma"),
}


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("name", list(SANDWICH))
def test_sandwich_every_token(name, path):
    shape = SANDWICH[name]
    inputs, blk, Y = _run(shape, PATHS[path])
    _check_layer(shape, inputs, blk, Y, tag=f"{name}-{path}")
    names = blk.stage_names()
    assert names[0] == "pre_norm" and names[-1] == "combine"
    assert blk.stats().path == PATHS[path][0]


def test_sandwich_route_entry_point_routes_the_normed_input():
    shape = SANDWICH["afmoe_ragged_rms"]
    inputs, blk, _ = _run(shape)
    idx_f, w_f = _topk(blk, shape.T, shape.k)
    idx_r, w_r = blk.route(inputs["X"])
    torch.cuda.synchronize()
    assert np.array_equal(idx_r.cpu().numpy(), idx_f)
    assert np.array_equal(w_r.cpu().numpy(), w_f)
    assert blk.stage_names() == ["pre_norm", "router"]


def test_gemma_norm_with_zero_weight_equals_plain_norm_with_unit_weight():
    """Scale 1 + 0 and scale 1 are the same fp32 number: the two layers agree
    bit for bit (both norms, every path)."""
    shape = SANDWICH["m3_small_gemma"]
    inputs = wl.make_inputs(shape, "cuda", row_filter=oracle.margin_filter(shape, P.MARGIN))
    zero = dict(inputs, pre_norm_w=torch.zeros_like(inputs["pre_norm_w"]),
                post_norm_w=torch.zeros_like(inputs["post_norm_w"]))
    one = dict(inputs, pre_norm_w=torch.ones_like(inputs["pre_norm_w"]),
               post_norm_w=torch.ones_like(inputs["post_norm_w"]))
    rms_shape = shape.replace(mlp_norm="rms")
    for path in PATHS.values():
        _, _, Yg = _run(shape, path, zero, capi.block_from_inputs(shape, zero))
        _, _, Yr = _run(rms_shape, path, one, capi.block_from_inputs(rms_shape, one))
        assert torch.equal(Yg, Yr)


def test_sandwich_fused_equals_two_launches_and_is_deterministic():
    for name in ("afmoe_ragged_rms", "m3_small_gemma"):
        shape = SANDWICH[name]
        for path in (PATHS["grouped"], PATHS["pair"]):
            inputs, blk, Y1 = _run(shape, path)
            Y2 = blk.forward(inputs["X"])
            blk.set_option(capi.MOE_OPT_FUSE_EXPERTS, 0)
            Y3 = blk.forward(inputs["X"])
            torch.cuda.synchronize()
            assert blk.sync_status() == capi.MOE_OK
            assert torch.equal(Y1, Y2) and torch.equal(Y1, Y3)


def test_sandwich_forward_host_matches_forward():
    shape = SANDWICH["nano_rms"]
    inputs, blk, Y = _run(shape, max_tokens=shape.T)
    Xh = inputs["X"].cpu().pin_memory()
    Yh = torch.empty_like(Xh).pin_memory()
    blk.forward_host(Xh, Yh)
    assert torch.equal(Yh, Y.cpu())


# ------------------------------------------------------------- dense layers

DENSE = {
    "dense_afmoe_ragged": wl.dense_layer(333, "afmoe").replace(name="dense_afmoe_ragged", hidden_size=512,
                                                             shared_intermediate_size=384),
    "dense_m3_small": wl.dense_layer(96, "m3").replace(name="dense_m3_small", hidden_size=512,
                                                      shared_intermediate_size=640),
    "dense_plain": wl.dense_layer(200, "afmoe").replace(name="dense_plain", hidden_size=256,
                                                       shared_intermediate_size=192, mlp_norm="none"),
    "dense_T1": wl.dense_layer(1, "m3").replace(name="dense_T1", hidden_size=1024,
                                                shared_intermediate_size=2048),
    # K of the down projection in 16 ranges (8 with T = 1 above, 2 for dense_m3_small
    # on one CTA per tile): partial outputs summed by the combine
    "dense_split16": wl.dense_layer(100, "afmoe").replace(name="dense_split16", hidden_size=512,
                                                        shared_intermediate_size=4096),
}


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("name", list(DENSE))
def test_dense_every_token(name, pair):
    shape = DENSE[name]
    inputs, blk, Y = _run(shape, (capi.PATH_GROUPED, pair))
    _check_layer(shape, inputs, blk, Y, tag=f"{name}-pair{pair}")
    names = blk.stage_names()
    assert "router" not in names and "dispatch_scatter" not in names
    assert names[-2:] == ["experts_gemm", "combine"]
    assert blk.stats().path == capi.PATH_GROUPED


def test_dense_hidden_activations_match_oracle():
    shape = DENSE["dense_m3_small"]
    cfg = oracle.cfg_from_shape(shape)
    for pair in (0, 1):
        inputs, blk, _ = _run(shape, (capi.PATH_GROUPED, pair))
        ih = P.host_inputs(inputs)
        S = shape.shared_intermediate_size
        hid = blk.inspect(capi.MOE_BUF_SHARED_HIDDEN, shape.T * S, torch.bfloat16).view(shape.T, S)
        hid = hid.float().cpu().numpy()
        xin = oracle.normed_input(shape, ih["X"], ih["pre_norm_w"])
        for t in (0, 1, shape.T // 2, shape.T - 1):
            _, _, a, _ = oracle.expert(cfg, xin[t], ih["sh_gate"], ih["sh_up"], ih["sh_down"], S)
            err = np.abs(hid[t] - a).max()
            assert err <= 2e-2 * np.sqrt(np.mean(a ** 2)) + 1e-6, (pair, t, err)


def test_dense_fused_equals_two_launches_and_has_no_router():
    shape = DENSE["dense_afmoe_ragged"]
    for pair in (0, 1):
        inputs, blk, Y1 = _run(shape, (capi.PATH_GROUPED, pair))
        blk.set_option(capi.MOE_OPT_FUSE_EXPERTS, 0)
        Y2 = blk.forward(inputs["X"])
        torch.cuda.synchronize()
        assert blk.sync_status() == capi.MOE_OK
        assert torch.equal(Y1, Y2)
        assert blk.stage_names()[-3:] == ["gate_up_gemm", "down_gemm", "combine"]
    with pytest.raises(capi.MoeError):
        blk.route(inputs["X"])
    with pytest.raises(capi.MoeError):
        blk.inspect(capi.MOE_BUF_TOPK_IDX, 4, torch.int32)


@pytest.mark.parametrize("name", ["dense_afmoe_ragged", "dense_split16", "dense_T1"])
def test_dense_staged_stores_are_bit_identical(name):
    """Hidden activations and K-split partial outputs stored through shared memory (TMA
    stores of full 32-row slices, coalesced stores of partial ones) equal the rows stored
    from registers: the same hidden rows and the same block output, bit for bit."""
    shape = DENSE[name]
    S = shape.shared_intermediate_size
    for pair in (0, 1):
        inputs, blk, _ = _run(shape, (capi.PATH_GROUPED, pair))
        outs = []
        for staged in (1, 0):
            blk.set_option(capi.MOE_OPT_STAGED_STORES, staged)
            Y = blk.forward(inputs["X"]).clone()
            torch.cuda.synchronize()
            assert blk.sync_status() == capi.MOE_OK
            outs.append((Y, blk.inspect(capi.MOE_BUF_SHARED_HIDDEN, shape.T * S, torch.bfloat16)))
        assert torch.equal(outs[0][1], outs[1][1]), (name, pair)
        assert torch.equal(outs[0][0], outs[1][0]), (name, pair)


def test_dense_token_permutation_equivariance():
    shape = DENSE["dense_afmoe_ragged"]
    inputs, blk, Y = _run(shape)
    perm = torch.randperm(shape.T, generator=torch.Generator().manual_seed(11)).cuda()
    Yp = blk.forward(inputs["X"][perm].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(Yp, Y[perm])


# ---------------------------------------------------- full sizes, sampled

def _sample(T, n=16):
    return sorted(set([0, T - 1] + np.linspace(0, T - 1, n).astype(int).tolist()))


@pytest.mark.parametrize("name", ["afmoe_prefill_sandwich", "nano_decode_sandwich", "m3_sandwich",
                                  "dense_afmoe_prefill", "dense_afmoe_decode", "dense_m3"])
def test_full_size_layers(name):
    shape = wl.WORKLOADS[name]
    inputs, blk, Y = _run(shape, max_tokens=shape.T)
    toks = _sample(shape.T, 10 if shape.H > 4096 else 16)
    _check_layer(shape, inputs, blk, Y, tokens=toks, tag=shape.name)
