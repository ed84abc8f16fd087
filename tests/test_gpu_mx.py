"""GPU parity of the block on block-scaled (MX) expert weights.

The Arcee AFMoE issue ("Checkpoint confirmed") lists 4-bit and MXFP8
checkpoints.  The block stores each weight as an OCP microscaling element code
(E4M3 or E2M1) with one E8M0 scale per 32 consecutive input values of its row;
activations stay bf16.  Checks:

  * against the fp64 oracle (which decodes the same codes): routing of every
    token, outputs of every token on small shapes, sampled tokens at full size,
    with the bf16 tolerance (decoding is exact, so the arithmetic is the bf16
    path's);
  * bit-for-bit against the bf16 path on the decoded weights: both MX GEMMs (the
    grouped one, tokens as M, with 128-row tiles or 256-row tiles (against the bf16
    CTA-pair path), and the swapped one, weights decoded into tensor memory as M)
    multiply the same operand values in the same order as their bf16 counterparts, so
    Y must be identical, which pins the decoders (byte and nibble order, scale index,
    operand layouts, the tile halves) independently of any tolerance;
  * the options the MX path refuses.
"""

import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_gb300 import capi
from expert_routed_ffn_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

E2M1 = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0],
                    dtype=torch.float64)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routed_ffn_gb300 import build
    build.build()
    capi.load()


def mx_decode(codes, scales, fmt):
    """[..., rows, K or K/2] uint8 codes and [..., K/32, rows] uint8 scales ->
    [..., rows, K] float64 (OCP MX definitions; torch's float8_e4m3fn for E4M3)."""
    c = codes.cpu()
    if fmt == "mxfp8":
        v = c.view(torch.float8_e4m3fn).to(torch.float64)
    else:
        lo, hi = (c & 0xF).long(), (c >> 4).long()
        v = torch.stack([E2M1[lo], E2M1[hi]], dim=-1).flatten(-2)
    sc = scales.cpu().to(torch.float64)
    e = torch.where(sc == 255, torch.full_like(sc, float("nan")), torch.exp2(sc - 127.0))
    e = e.transpose(-1, -2).repeat_interleave(32, dim=-1)  # [..., rows, K]
    return v * e


def decoded_bf16_inputs(shape, inputs):
    """The same workload with the MX weights decoded into bf16 tensors (exact)."""
    out = {k: v for k, v in inputs.items() if k not in capi.SCALE_KEYS}
    for key, skey in zip(("gate", "up", "down", "sh_gate", "sh_up", "sh_down"), capi.SCALE_KEYS):
        t = inputs[key]
        if t is None:
            continue
        d = mx_decode(t, inputs[skey], shape.weight_format)
        b = d.to(torch.bfloat16)
        assert torch.equal(b.to(torch.float64), d), f"{key}: a decoded weight is not a bf16 value"
        out[key] = b.to(t.device)
    return out


def _forward(blk, X):
    Y = blk.forward(X)
    torch.cuda.synchronize()
    assert blk.sync_status() == capi.MOE_OK
    return Y


def _oracle_check(shape, inputs, Y, tokens=None, tag=""):
    host = P.host_inputs(inputs)
    ref = oracle.block_output(shape, host, tokens=tokens)
    Yg = P.to_np(Y) if tokens is None else P.to_np(Y[tokens])
    P.check_output(Yg, ref, out_bf16=shape.dtype == "bf16", tag=tag)


SMALL = {
    "nano": wl.NANO_DECODE,
    "nano_T1": wl.NANO_DECODE.replace(name="nano_T1", T=1),
    "tiny_f32": wl.TINY,
    "m3_small_packed": wl.M3.replace(name="m3_small", T=96, hidden_size=512, num_experts=8,
                                     num_experts_per_tok=2, moe_intermediate_size=256,
                                     shared_intermediate_size=256),
    "afmoe_ragged": wl.AFMOE_PREFILL.replace(name="afmoe_ragged", T=333, hidden_size=512,
                                             moe_intermediate_size=192, shared_intermediate_size=384),
    "nano_sandwich": wl.NANO_DECODE.replace(name="nano_sw", T=64, mlp_norm="rms"),
    "afmoe_T4": wl.AFMOE_PREFILL.replace(name="afmoe_T4", T=4, hidden_size=512, moe_intermediate_size=1024,
                                                shared_intermediate_size=512),
    "dense_small": wl.dense_layer(200, "afmoe").replace(name="dense_small", hidden_size=512,
                                                         shared_intermediate_size=1024),
    # >= 32 routed rows per expert on 128-row tiles: the kernel with sixteen converter warps
    "afmoe_rows48": wl.AFMOE_PREFILL.replace(name="afmoe_rows48", T=512, hidden_size=512,
                                             moe_intermediate_size=192, shared_intermediate_size=384),
}
FORMATS = ["mxfp8", "mxfp4"]


PATHS = {"grouped": capi.PATH_GROUPED, "swapped": capi.PATH_SWAPPED}
# GEMM variants: (path, MOE_OPT_GEMM_PAIR)
GEMMS = {"grouped": (capi.PATH_GROUPED, 0), "grouped_pairs": (capi.PATH_GROUPED, 1),
         "swapped": (capi.PATH_SWAPPED, 0)}


@pytest.mark.parametrize("gemm", list(GEMMS))
@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("name", list(SMALL))
def test_mx_small_every_token(name, fmt, gemm):
    shape = SMALL[name].replace(name=f"{SMALL[name].name}_{fmt}", weight_format=fmt)
    path, pair = GEMMS[gemm]
    inputs, blk = P.make_case(shape)
    blk.set_option(capi.MOE_OPT_GEMM_PAIR, pair)
    if shape.E > 0:
        blk.set_option(capi.MOE_OPT_PATH, path)
    elif path == capi.PATH_SWAPPED:
        pytest.skip("a dense layer runs on the grouped GEMM only")
    Y = _forward(blk, inputs["X"])
    if shape.E > 0 and shape.mlp_norm == "none":
        idx, w = (blk.inspect(b, shape.T * shape.k, dt).view(shape.T, shape.k).cpu().numpy()
                  for b, dt in ((capi.MOE_BUF_TOPK_IDX, torch.int32), (capi.MOE_BUF_TOPK_W, torch.float32)))
        P.check_route(shape, P.host_inputs(inputs), idx, w)
    _oracle_check(shape, inputs, Y, tag=f"mx_small[{name},{fmt},{gemm}]")
    blk.close()


@pytest.mark.parametrize("gemm", list(GEMMS))
@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("name", ["nano", "m3_small_packed", "afmoe_ragged", "dense_small", "nano_T1",
                                  "afmoe_T4", "afmoe_rows48"])
def test_mx_bit_identical_to_bf16_path_on_decoded_weights(name, fmt, gemm):
    shape = SMALL[name].replace(name=f"{SMALL[name].name}_{fmt}", weight_format=fmt)
    path, pair = GEMMS[gemm]
    if shape.E == 0 and path == capi.PATH_SWAPPED:
        pytest.skip("a dense layer runs on the grouped GEMM only")
    inputs, blk = P.make_case(shape)
    if shape.E > 0:
        blk.set_option(capi.MOE_OPT_PATH, path)
    blk.set_option(capi.MOE_OPT_GEMM_PAIR, pair)
    Y = _forward(blk, inputs["X"])
    dec = decoded_bf16_inputs(shape, inputs)
    bshape = shape.replace(weight_format="bf16")
    ref_blk = capi.block_from_inputs(bshape, dec)
    if shape.E > 0:
        ref_blk.set_option(capi.MOE_OPT_PATH, path)
    ref_blk.set_option(capi.MOE_OPT_GEMM_PAIR, pair)  # the same tile shape and MMAs
    Yb = _forward(ref_blk, dec["X"])
    assert torch.equal(Y, Yb), "MX path differs from the bf16 path on the decoded weights"
    ref_blk.close()
    blk.close()


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("fmt", FORMATS)
def test_mx_two_launches_and_repeat_are_bit_identical(fmt, pair):
    shape = wl.NANO_DECODE.replace(name=f"nano_{fmt}", T=200, weight_format=fmt)
    inputs, blk = P.make_case(shape)
    blk.set_option(capi.MOE_OPT_PATH, capi.PATH_GROUPED)  # the fused launch is the grouped kernel's
    blk.set_option(capi.MOE_OPT_GEMM_PAIR, pair)
    Y1 = _forward(blk, inputs["X"]).clone()
    Y2 = _forward(blk, inputs["X"]).clone()
    blk.set_option(capi.MOE_OPT_FUSE_EXPERTS, 0)
    Y3 = _forward(blk, inputs["X"])
    assert torch.equal(Y1, Y2) and torch.equal(Y1, Y3)
    blk.close()


def test_mx_refuses_other_paths():
    shape = wl.NANO_DECODE.replace(name="nano_mx8", T=16, weight_format="mxfp8")
    inputs, blk = P.make_case(shape)
    with pytest.raises(capi.MoeError) as ei:
        blk.set_option(capi.MOE_OPT_PATH, capi.PATH_DECODE)
    assert ei.value.status == capi.MOE_ERR_UNSUPPORTED
    blk.set_option(capi.MOE_OPT_PATH, capi.PATH_GROUPED)
    blk.set_option(capi.MOE_OPT_GEMM_PAIR, 1)  # CTA pairs at a decode size (T = 16)
    _oracle_check(shape, inputs, _forward(blk, inputs["X"]), tag="mx_pair_opt")
    blk.close()


FULL = [("nano_decode_mxfp8", 2), ("nano_decode_mxfp4", 2), ("afmoe_prefill_mxfp8", 2), ("m3_mxfp8", 2),
        ("afmoe_prefill_mxfp8", 1)]


@pytest.mark.parametrize("name,pair", FULL)
def test_mx_full_size_sampled(name, pair):
    """The bench's launch configuration (pair 2: automatic), and CTA pairs forced."""
    shape = wl.WORKLOADS[name]
    inputs, blk = P.make_case(shape, max_tokens=shape.T)
    blk.set_option(capi.MOE_OPT_GEMM_PAIR, pair)
    Y = _forward(blk, inputs["X"])
    T = shape.T
    idx, w = (blk.inspect(b, T * shape.k, dt).view(T, shape.k).cpu().numpy()
              for b, dt in ((capi.MOE_BUF_TOPK_IDX, torch.int32), (capi.MOE_BUF_TOPK_W, torch.float32)))
    P.check_route(shape, P.host_inputs(inputs), idx, w)
    tokens = sorted(set([0, T - 1] + np.linspace(0, T - 1, 24).astype(int).tolist()))
    _oracle_check(shape, inputs, Y, tokens=tokens, tag=f"mx_full[{name}]")
    blk.close()


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("fmt", FORMATS)
def test_mx_scales_outside_the_fast_decoder_range(fmt, path):
    """Scale codes above 142 (2^15) put the fast decoder's bf16 multiplier
    2^(scale - 15) out of bf16's normal range, so the converters take the fp32
    products for those rows; codes near 0 give bf16 subnormal products.  Both
    decoders must give the exactly decoded weights: bit-identity with the bf16 path
    on the decoded weights, and the oracle."""
    shape = SMALL["nano"].replace(name=f"nano_scales_{fmt}", T=64, weight_format=fmt)
    inputs = wl.make_inputs(shape, "cuda", row_filter=oracle.margin_filter(shape, P.MARGIN))
    g = torch.Generator().manual_seed(11)
    # 3 is the smallest code whose products stay exact in bf16 (E4M3's 2^-9 times
    # 2^-124 is bf16's smallest subnormal)
    for key, code in (("gate_scale", 145), ("up_scale", 150), ("down_scale", 3)):
        sc = inputs[key]
        u = torch.rand(sc.shape, generator=g)
        sc[(u < 0.02).to(sc.device)] = code
        sc[(u > 0.99).to(sc.device)] = code + 1
    blk = capi.block_from_inputs(shape, inputs)
    blk.set_option(capi.MOE_OPT_PATH, PATHS[path])
    Y = _forward(blk, inputs["X"])
    dec = decoded_bf16_inputs(shape, inputs)
    ref_blk = capi.block_from_inputs(shape.replace(weight_format="bf16"), dec)
    ref_blk.set_option(capi.MOE_OPT_PATH, PATHS[path])
    ref_blk.set_option(capi.MOE_OPT_GEMM_PAIR, 0)
    Yb = _forward(ref_blk, dec["X"])
    assert torch.isfinite(Y.float()).all()
    assert torch.equal(Y, Yb), "MX path differs from the bf16 path on the decoded weights"
    _oracle_check(shape, inputs, Y, tag=f"mx_scales[{fmt},{path}]")
    ref_blk.close()
    blk.close()
