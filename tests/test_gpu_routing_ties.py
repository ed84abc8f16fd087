"""GPU routing with exact ties of the biased score.

The routing rule chooses, k times, the largest biased score among the experts
not chosen yet, equal values going to the lower expert index (Arcee AFMoE
issue, "Routing detail": top-k over score + bias, the bias selection-only).
Random weights almost never tie, so these cases build ties on purpose:

  * router rows and biases duplicated in pairs (expert 2j+1 a copy of 2j): every
    expert ties with its partner in every token, on both sides bit-exactly (the
    same row through the same arithmetic), so the lower index of each pair must
    come first, and with an odd k the pair cut at the k-th slot must give up its
    upper expert;
  * a zero router and zero bias: every expert scores 0.5 (or 1/E under softmax),
    so the choice is experts 0 .. k-1 in that order.

Both routers are covered (the tensor-core one for bf16 X, the CUDA-core one for
fp32 X), sigmoid and softmax scores, and k on both sides of 8.
"""

import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_gb300 import capi
from expert_routed_ffn_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routed_ffn_gb300 import build
    build.build()
    capi.load()


CASES = {
    "nano_k8": wl.NANO_DECODE.replace(name="nano_k8", T=200),
    "nano_k7": wl.NANO_DECODE.replace(name="nano_k7", T=200, num_experts_per_tok=7),
    "nano_k11": wl.NANO_DECODE.replace(name="nano_k11", T=200, num_experts_per_tok=11),
    "nano_softmax_k5": wl.NANO_DECODE.replace(name="nano_sm_k5", T=130, num_experts_per_tok=5,
                                              score_func="softmax"),
    "afmoe_E64_k3": wl.AFMOE_PREFILL.replace(name="afmoe_k3", T=160, hidden_size=512, num_experts_per_tok=3,
                                             moe_intermediate_size=128, shared_intermediate_size=128),
    "tiny_f32_k3": wl.TINY.replace(name="tiny_k3", num_experts_per_tok=3),
    "tiny_f32_k10": wl.TINY.replace(name="tiny_k10", num_experts_per_tok=10),
    "m3_E256_k9": wl.M3.replace(name="m3_k9", T=96, hidden_size=512, num_experts=256, num_experts_per_tok=9,
                                moe_intermediate_size=128, shared_intermediate_size=128),
}


def _route(shape, inputs):
    blk = capi.block_from_inputs(shape, inputs)
    idx, w = blk.route(inputs["X"])
    torch.cuda.synchronize()
    assert blk.sync_status() == capi.MOE_OK
    # the forward's own routing (the fused router of the forward path)
    blk.forward(inputs["X"])
    torch.cuda.synchronize()
    assert blk.sync_status() == capi.MOE_OK
    T, k = shape.T, shape.k
    fidx = blk.inspect(capi.MOE_BUF_TOPK_IDX, T * k, torch.int32).view(T, k).cpu().numpy()
    fw = blk.inspect(capi.MOE_BUF_TOPK_W, T * k, torch.float32).view(T, k).cpu().numpy()
    blk.close()
    idx, w = idx.cpu().numpy(), w.cpu().numpy()
    assert np.array_equal(idx, fidx) and np.array_equal(w, fw)
    return idx, w


@pytest.mark.parametrize("name", list(CASES))
def test_paired_experts_tie_to_the_lower_index(name):
    shape = CASES[name]
    inputs = wl.make_inputs(shape, "cuda")
    Wr, b = inputs["router_w"], inputs["expert_bias"]
    Wr[1::2] = Wr[0::2]
    if b is not None:
        b[1::2] = b[0::2]
    idx, w = _route(shape, inputs)
    ref = oracle.route_inputs(shape, P.host_inputs(inputs))
    k, E = shape.k, shape.E
    # tokens whose pair values (biased scores of the even experts) are apart by more
    # than fp32 rounding over the pairs that decide the choice
    c = ref["biased"][:, 0::2]
    cs = -np.sort(-c, axis=1)[:, : (k + 1) // 2 + 1]
    clear = np.all(cs[:, :-1] - cs[:, 1:] > 1e-5, axis=1)
    assert clear.mean() > 0.9, "too few tokens with separated pairs"
    assert np.array_equal(idx[clear], ref["idx"][clear].astype(idx.dtype))
    # within every chosen pair the lower index comes first, in every token
    for t in range(shape.T):
        for j in range(k):
            e = int(idx[t, j])
            if e % 2 == 1:
                assert j > 0 and idx[t, j - 1] == e - 1, f"token {t}: expert {e} chosen before its partner"
        assert len(set(idx[t].tolist())) == k and idx[t].min() >= 0 and idx[t].max() < E
    if k % 2 == 1:  # the last slot is always the lower half of a split pair
        assert np.all(idx[:, k - 1] % 2 == 0)
    assert np.allclose(w[clear], ref["w"][clear], rtol=P.W_RTOL, atol=1e-7)


@pytest.mark.parametrize("name", ["nano_k8", "nano_k11", "nano_softmax_k5", "tiny_f32_k3", "m3_E256_k9"])
def test_all_equal_scores_choose_the_first_k_experts(name):
    shape = CASES[name]
    inputs = wl.make_inputs(shape, "cuda")
    inputs["router_w"].zero_()
    if inputs["expert_bias"] is not None:
        inputs["expert_bias"].zero_()
    idx, w = _route(shape, inputs)
    k = shape.k
    assert np.array_equal(idx, np.tile(np.arange(k, dtype=idx.dtype), (shape.T, 1)))
    ref = oracle.route_inputs(shape, P.host_inputs(inputs))
    assert np.array_equal(ref["idx"].astype(idx.dtype), idx)
    assert np.allclose(w, ref["w"], rtol=P.W_RTOL, atol=1e-7)
