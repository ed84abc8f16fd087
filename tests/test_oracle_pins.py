"""Pins of the fp64 oracle against things other than itself.

Each test ties one step of the oracle to brute force, a closed form, a library
routine (numpy matmul, scipy expit/softmax) on a special case, or an invariant
the pages imply.  Shapes use H != I != S so a transposed operand fails.
"""

import itertools
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit, softmax

import oracle
from expert_routed_ffn_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _tiny(seed, T=7, H=24, E=8, k=3, I=40, S=0, packed=False, f32=True):
    r = _rng(seed)
    X = r.standard_normal((T, H)).astype(np.float32)
    Wr = (r.standard_normal((E, H)) * 0.3).astype(np.float32)
    b = r.uniform(-0.1, 0.1, E).astype(np.float32)
    Ep = E + (1 if packed else 0)
    Wg = (r.standard_normal((Ep, I, H)) * 0.2).astype(np.float32)
    Wu = (r.standard_normal((Ep, I, H)) * 0.2).astype(np.float32)
    Wd = (r.standard_normal((Ep, H, I)) * 0.2).astype(np.float32)
    sh = (None, None, None)
    if S:
        sh = ((r.standard_normal((S, H)) * 0.2).astype(np.float32),
              (r.standard_normal((S, H)) * 0.2).astype(np.float32),
              (r.standard_normal((H, S)) * 0.2).astype(np.float32))
    return X, Wr, b, Wg, Wu, Wd, sh


def _silu_glu(g, u):
    return g * expit(g) * u


def _mlp_np(x, Wg, Wu, Wd, act=_silu_glu):
    """Library-routine expert MLP: matmuls of numpy fp64."""
    g = x.astype(np.float64) @ Wg.astype(np.float64).T
    u = x.astype(np.float64) @ Wu.astype(np.float64).T
    return act(g, u) @ Wd.astype(np.float64).T


# ----------------------------------------------------------------- routing

def test_logits_scores_biased_against_library_routines():
    X, Wr, b, *_ = _tiny(1)
    cfg = oracle.make_cfg(24, 8, 3, 40)
    r = oracle.route(cfg, X, Wr, b)
    l = X.astype(np.float64) @ Wr.astype(np.float64).T
    np.testing.assert_allclose(r["logits"], l, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(r["scores"], expit(l), rtol=1e-13)
    # the bias is added to the score, not the logit
    np.testing.assert_allclose(r["biased"] - r["scores"], np.broadcast_to(b.astype(np.float64), l.shape),
                               atol=1e-15)


def test_softmax_variant_against_scipy():
    X, Wr, b, *_ = _tiny(2)
    cfg = oracle.make_cfg(24, 8, 3, 40, score_func="softmax")
    r = oracle.route(cfg, X, Wr, b)
    l = X.astype(np.float64) @ Wr.astype(np.float64).T
    np.testing.assert_allclose(r["scores"], softmax(l, axis=1), rtol=1e-13)
    np.testing.assert_allclose(r["scores"].sum(1), 1.0, rtol=1e-14)


@pytest.mark.parametrize("E,k", [(5, 1), (6, 2), (8, 3), (10, 4), (7, 7)])
def test_topk_set_is_brute_force_maximiser(E, k):
    X, Wr, b, *_ = _tiny(10 + E * k, T=12, E=E, k=k)
    r = oracle.route(oracle.make_cfg(24, E, k, 40), X, Wr, b)
    for t in range(X.shape[0]):
        c = r["biased"][t]
        best = max(itertools.combinations(range(E), k), key=lambda s: sum(c[list(s)]))
        assert sorted(r["idx"][t].tolist()) == sorted(best)
        # returned in descending biased score
        assert np.all(np.diff(c[r["idx"][t]]) <= 0)


def test_tie_break_lowest_index():
    H, E, k = 24, 8, 3
    X = np.zeros((2, H), np.float32)  # logits 0 -> every score 0.5
    Wr = np.ones((E, H), np.float32)
    cfg = oracle.make_cfg(H, E, k, 40)
    r = oracle.route(cfg, X, Wr, np.zeros(E, np.float32))
    assert r["idx"].tolist() == [[0, 1, 2]] * 2
    b = np.array([0, .1, .1, 0, .1, .1, 0, 0], np.float32)
    r = oracle.route(cfg, X, Wr, b)
    assert r["idx"].tolist() == [[1, 2, 4]] * 2


def test_route_norm_and_scale():
    X, Wr, b, *_ = _tiny(3, T=16)
    cfg = oracle.make_cfg(24, 8, 3, 40, route_norm=True, route_scale=2.826)
    r = oracle.route(cfg, X, Wr, b)
    np.testing.assert_allclose(r["w"].sum(1), 2.826, rtol=1e-15)
    s_sel = np.take_along_axis(r["scores"], r["idx"].astype(np.int64), 1)
    np.testing.assert_allclose(r["w"], 2.826 * s_sel / s_sel.sum(1, keepdims=True), rtol=1e-14)
    cfg_off = oracle.make_cfg(24, 8, 3, 40, route_norm=False, route_scale=2.0)
    r2 = oracle.route(cfg_off, X, Wr, b)
    np.testing.assert_allclose(r2["w"], 2.0 * expit(np.take_along_axis(r2["logits"], r2["idx"].astype(np.int64), 1)),
                               rtol=1e-14)


def test_bias_changes_selection_never_weights():
    X, Wr, b, *_ = _tiny(4, T=10)
    cfg = oracle.make_cfg(24, 8, 3, 40)
    r0 = oracle.route(cfg, X, Wr, b)
    # shift every bias by a constant: nothing changes
    r1 = oracle.route(cfg, X, Wr, (b + np.float32(0.25)).astype(np.float32))
    assert np.array_equal(r0["idx"], r1["idx"])
    assert np.array_equal(r0["w"], r1["w"])
    # raise the bias of already-selected experts of token 0: same set, same weights
    b2 = b.copy()
    b2[r0["idx"][0]] += np.float32(0.05)
    r2 = oracle.route(cfg, X[:1], Wr, b2)
    assert sorted(r2["idx"][0]) == sorted(r0["idx"][0])
    w_by_e0 = dict(zip(r0["idx"][0].tolist(), r0["w"][0].tolist()))
    w_by_e2 = dict(zip(r2["idx"][0].tolist(), r2["w"][0].tolist()))
    assert w_by_e0 == w_by_e2
    # a large bias on an unselected expert pulls it in; its weight is its UNBIASED score
    out = [e for e in range(8) if e not in r0["idx"][0]][0]
    b3 = b.copy()
    b3[out] = np.float32(5.0)
    r3 = oracle.route(cfg, X[:1], Wr, b3)
    assert r3["idx"][0][0] == out
    s = r3["scores"][0]
    sel = r3["idx"][0]
    np.testing.assert_allclose(r3["w"][0][0], s[out] / s[sel].sum(), rtol=1e-14)


def test_margin_definition():
    X, Wr, b, *_ = _tiny(5, T=9)
    r = oracle.route(oracle.make_cfg(24, 8, 3, 40), X, Wr, b)
    srt = -np.sort(-r["biased"], axis=1)
    np.testing.assert_allclose(r["margin"], srt[:, 2] - srt[:, 3], rtol=1e-15)
    rk = oracle.route(oracle.make_cfg(24, 8, 8, 40), X, Wr, b)
    assert np.all(np.isinf(rk["margin"]))


# ------------------------------------------------------------- activations

def test_swigluoai_hand_points():
    cfg = oracle.make_cfg(4, 1, 1, 4, act="swigluoai", alpha=1.702, limit=7.0, beta=1.0)
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))  # noqa: E731
    # gate above the limit clamps to 7; up below -limit clamps to -7
    assert oracle.act(cfg, 10.0, -9.0) == pytest.approx(7.0 * sig(1.702 * 7.0) * (-7.0 + 1.0), rel=1e-15)
    # inside the limits nothing is clamped
    assert oracle.act(cfg, 2.0, 3.0) == pytest.approx(2.0 * sig(1.702 * 2.0) * 4.0, rel=1e-15)
    # the gate is clamped from above only
    assert oracle.act(cfg, -12.0, 0.5) == pytest.approx(-12.0 * sig(-1.702 * 12.0) * 1.5, rel=1e-15)
    # up clamps from above too
    assert oracle.act(cfg, 1.0, 8.0) == pytest.approx(1.0 * sig(1.702) * 8.0, rel=1e-15)


def test_swigluoai_reduces_to_silu_glu():
    silu = oracle.make_cfg(4, 1, 1, 4, act="silu")
    oai = oracle.make_cfg(4, 1, 1, 4, act="swigluoai", alpha=1.0, limit=float("inf"), beta=0.0)
    r = _rng(6)
    for g, u in r.standard_normal((50, 2)) * 6:
        assert oracle.act(oai, g, u) == oracle.act(silu, g, u)
        assert oracle.act(silu, g, u) == pytest.approx(g * expit(g) * u, rel=1e-14, abs=1e-300)


def test_page_constants_match_workloads():
    vals = {}
    with open(os.path.join(GOLDEN, "page_constants.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, val, _cite = line.split()
                vals[key] = float(val)
    assert wl.NANO_DECODE.route_scale == vals["trinity_route_scale"] == wl.TINY.route_scale
    assert wl.NANO_DECODE.H == vals["trinity_nano_hidden"] and wl.NANO_DECODE.E == vals["trinity_nano_experts"]
    a = wl.AFMOE_PREFILL
    assert (a.H, a.I, a.E, a.k, a.num_shared_experts, a.route_scale) == (
        vals["afmoe_hidden_size"], vals["afmoe_moe_intermediate_size"], vals["afmoe_num_experts"],
        vals["afmoe_num_experts_per_tok"], vals["afmoe_num_shared_experts"], vals["afmoe_route_scale"])
    assert wl.WEIGHT_STD == vals["afmoe_initializer_range"]
    m = wl.M3
    assert (m.H, m.E, m.k, m.route_scale, m.S) == (
        vals["m3_hidden_size"], vals["m3_num_local_experts"], vals["m3_num_experts_per_tok"],
        vals["m3_routed_scaling_factor"], vals["m3_shared_intermediate_size"])
    assert m.shared_packed and m.stacked_experts - 1 == vals["m3_packed_shared_index"]
    assert (m.act_alpha, m.act_limit, m.act_beta) == (
        vals["swigluoai_alpha"], vals["swigluoai_limit"], vals["swigluoai_beta"])
    da, dm = wl.WORKLOADS["dense_afmoe_prefill"], wl.WORKLOADS["dense_m3"]
    assert (da.H, da.S, da.E) == (vals["afmoe_hidden_size"], vals["afmoe_intermediate_size"], 0)
    assert (dm.H, dm.S, dm.E) == (vals["m3_hidden_size"], vals["m3_dense_intermediate_size"], 0)
    assert dm.hidden_act == "swigluoai" and dm.mlp_norm == wl.WORKLOADS["m3_sandwich"].mlp_norm == "gemma"
    assert da.rms_norm_eps == wl.WORKLOADS["afmoe_prefill_sandwich"].rms_norm_eps == vals["afmoe_rms_norm_eps"]
    # Gemma-style: weight + 1 (the oracle's offset, on a unit input of one element)
    assert oracle.rmsnorm(np.ones((1, 1)), np.zeros(1), 0.0, True)[0, 0] == vals["m3_gemma_norm_offset"]


# ------------------------------------------------------------ expert MLPs

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_expert_reduces_to_plain_swiglu_mlp(dtype):
    """E = 1, k = 1, norm on, scale 1, no shared: Y is one SwiGLU MLP."""
    X, Wr, b, Wg, Wu, Wd, _ = _tiny(7, T=5, E=1, k=1)
    cfg = oracle.make_cfg(24, 1, 1, 40, route_norm=True, route_scale=1.0)
    if dtype == "bf16":
        Wg, Wu, Wd = (torch.from_numpy(a).to(torch.bfloat16) for a in (Wg, Wu, Wd))
        ref = _mlp_np(X, Wg[0].double().numpy(), Wu[0].double().numpy(), Wd[0].double().numpy())
    else:
        ref = _mlp_np(X, Wg[0], Wu[0], Wd[0])
    Y = oracle.forward(cfg, X, Wr, b, Wg, Wu, Wd)
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-14)


def test_expert_intermediates_against_numpy():
    X, Wr, b, Wg, Wu, Wd, _ = _tiny(8, T=1)
    cfg = oracle.make_cfg(24, 8, 3, 40, act="swigluoai", alpha=1.702, limit=0.5, beta=1.0)
    g, u, a, y = oracle.expert(cfg, X[0], Wg[2], Wu[2], Wd[2], 40)
    x = X[0].astype(np.float64)
    np.testing.assert_allclose(g, Wg[2].astype(np.float64) @ x, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(u, Wu[2].astype(np.float64) @ x, rtol=1e-13, atol=1e-15)
    assert (np.abs(u) > 0.5).any() and (g > 0.5).any()  # the clamp fires at limit 0.5
    gc, uc = np.minimum(g, 0.5), np.clip(u, -0.5, 0.5)
    np.testing.assert_allclose(a, gc * expit(1.702 * gc) * (uc + 1.0), rtol=1e-14)
    np.testing.assert_allclose(y, Wd[2].astype(np.float64) @ a, rtol=1e-12, atol=1e-15)


def _dense_mask_reference(X, Wr, b, Wg, Wu, Wd, sh, E, k, route_norm, scale, packed=False):
    """Every expert on every token, masked by a brute-force top-k set."""
    l = X.astype(np.float64) @ Wr.astype(np.float64).T
    s = expit(l)
    c = s + b.astype(np.float64)
    Y = np.zeros((X.shape[0], X.shape[1]))
    ys = np.stack([_mlp_np(X, Wg[e], Wu[e], Wd[e]) for e in range(E)], 1)  # [T,E,H]
    for t in range(X.shape[0]):
        sel = list(max(itertools.combinations(range(E), k), key=lambda q: sum(c[t, list(q)])))
        m = np.zeros(E)
        m[sel] = 1.0
        w = s[t] * m
        if route_norm:
            w = w / w.sum()
        Y[t] = (scale * w) @ ys[t]
    if packed:
        Y += _mlp_np(X, Wg[E], Wu[E], Wd[E])
    elif sh[0] is not None:
        Y += _mlp_np(X, *sh)
    return Y


@pytest.mark.parametrize("route_norm,scale", [(True, 2.826), (False, 2.0)])
def test_forward_equals_dense_mask_formulation(route_norm, scale):
    X, Wr, b, Wg, Wu, Wd, sh = _tiny(9, T=9, E=6, k=2, S=56)
    cfg = oracle.make_cfg(24, 6, 2, 40, S=56, route_norm=route_norm, route_scale=scale)
    Y = oracle.forward(cfg, X, Wr, b, Wg, Wu, Wd, *sh)
    ref = _dense_mask_reference(X, Wr, b, Wg, Wu, Wd, sh, 6, 2, route_norm, scale)
    np.testing.assert_allclose(Y, ref, rtol=1e-11, atol=1e-13)


def test_topk_equals_E_zero_bias_is_dense_weighted_sum():
    E = 5
    X, Wr, _, Wg, Wu, Wd, sh = _tiny(11, T=6, E=E, k=E, S=32)
    cfg = oracle.make_cfg(24, E, E, 40, S=32, route_norm=True, route_scale=1.7)
    Y = oracle.forward(cfg, X, Wr, np.zeros(E, np.float32), Wg, Wu, Wd, *sh)
    s = expit(X.astype(np.float64) @ Wr.astype(np.float64).T)
    ref = sum((1.7 * s[:, e] / s.sum(1))[:, None] * _mlp_np(X, Wg[e], Wu[e], Wd[e]) for e in range(E))
    ref = ref + _mlp_np(X, *sh)
    np.testing.assert_allclose(Y, ref, rtol=1e-11, atol=1e-13)


def test_packed_shared_equals_separate_shared_mlp():
    E = 6
    X, Wr, b, Wg, Wu, Wd, _ = _tiny(12, T=8, E=E, k=2, packed=True)
    packed = oracle.make_cfg(24, E, 2, 40, shared_packed=True, route_norm=False, route_scale=2.0)
    sep = oracle.make_cfg(24, E, 2, 40, S=40, route_norm=False, route_scale=2.0)
    Yp = oracle.forward(packed, X, Wr, b, Wg, Wu, Wd)
    Ys = oracle.forward(sep, X, Wr, b, Wg[:E], Wu[:E], Wd[:E], Wg[E], Wu[E], Wd[E])
    assert np.array_equal(Yp, Ys)
    # and the packed slice never enters top-k: routing sees only E experts
    r = oracle.route(packed, X, Wr, b)
    assert r["idx"].max() < E
    ref = _dense_mask_reference(X, Wr, b, Wg, Wu, Wd, None, E, 2, False, 2.0, packed=True)
    np.testing.assert_allclose(Yp, ref, rtol=1e-11, atol=1e-13)


def test_two_shared_experts_equal_one_of_double_width():
    X, Wr, b, Wg, Wu, Wd, sh = _tiny(13, T=5, S=40)
    X2, _, _, _, _, _, sh2 = _tiny(14, T=5, S=40)
    cfg1 = oracle.make_cfg(24, 8, 3, 40, S=80)
    cat = (np.concatenate([sh[0], sh2[0]]), np.concatenate([sh[1], sh2[1]]),
           np.concatenate([sh[2], sh2[2]], axis=1))
    Y = oracle.forward(cfg1, X, Wr, b, Wg, Wu, Wd, *cat)
    cfg0 = oracle.make_cfg(24, 8, 3, 40, S=0)
    Yr = oracle.forward(cfg0, X, Wr, b, Wg, Wu, Wd)
    for t in range(X.shape[0]):
        _, _, _, y1 = oracle.expert(cfg1, X[t], *sh, 40)
        _, _, _, y2 = oracle.expert(cfg1, X[t], *sh2, 40)
        np.testing.assert_allclose(Y[t], Yr[t] + y1 + y2, rtol=1e-12, atol=1e-14)


def test_token_permutation_equivariance_and_thread_independence():
    X, Wr, b, Wg, Wu, Wd, sh = _tiny(15, T=11, S=24)
    cfg = oracle.make_cfg(24, 8, 3, 40, S=24, route_scale=2.826)
    Y = oracle.forward(cfg, X, Wr, b, Wg, Wu, Wd, *sh, nthreads=3)
    perm = _rng(16).permutation(11)
    Yp = oracle.forward(cfg, X[perm], Wr, b, Wg, Wu, Wd, *sh, nthreads=1)
    assert np.array_equal(Yp, Y[perm])
    Ysub = oracle.forward(cfg, X, Wr, b, Wg, Wu, Wd, *sh, tokens=[7, 2, 7])
    assert np.array_equal(Ysub, Y[[7, 2, 7]])


def test_margin_filter_drives_generator_redraws():
    shape = wl.TINY.replace(T=48)
    inp = wl.make_inputs(shape, "cpu", row_filter=oracle.margin_filter(shape))
    r = oracle.route_inputs(shape, inp)
    assert r["margin"].min() >= 1e-3
    # same seed, same draws
    inp2 = wl.make_inputs(shape, "cpu", row_filter=oracle.margin_filter(shape))
    assert torch.equal(inp["X"], inp2["X"]) and inp["redraws"] == inp2["redraws"]


# ------------------------------------------------ layers around the block

def test_dense_mlp_equals_numpy_swiglu_and_a_zero_scaled_block():
    """A dense prefix layer is a plain MLP: numpy matmuls of the same weights; and
    the MoE block with route_scale 0 (routed experts contribute nothing) and the
    dense weights as its shared expert gives the same output."""
    X, Wr, b, Wg, Wu, Wd, sh = _tiny(11, S=56)
    cfg = oracle.make_cfg(24, 0, 0, 0, S=56)
    Y = oracle.dense(cfg, X, *sh)
    ref = _mlp_np(X, *sh)
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)
    blk = oracle.make_cfg(24, 8, 3, 40, S=56, route_scale=0.0)
    Yb = oracle.forward(blk, X, Wr, b, Wg, Wu, Wd, *sh)
    assert np.allclose(Y, Yb, rtol=1e-12, atol=1e-12)
    # a subset of tokens gives the same rows
    assert np.array_equal(oracle.dense(cfg, X, *sh, tokens=[5, 0, 2]), Y[[5, 0, 2]])


def test_dense_swigluoai_against_hand_activation():
    X, *_rest, sh = _tiny(12, S=32)
    cfg = oracle.make_cfg(24, 0, 0, 0, S=32, act="swigluoai")

    def clamp_glu(g, u):
        gg = np.minimum(g, 7.0)
        uu = np.clip(u, -7.0, 7.0)
        return gg * expit(1.702 * gg) * (uu + 1.0)

    Xs = X * 20  # drive the clamps
    Y = oracle.dense(cfg, Xs, *sh)
    assert np.allclose(Y, _mlp_np(Xs, *sh, act=clamp_glu), rtol=1e-12, atol=1e-10)


def test_rmsnorm_closed_forms():
    H = 48
    w = _rng(13).uniform(0.5, 1.5, H)
    # a constant row a * 1: mean square a^2, so y = a / sqrt(a^2 + eps) * w
    for a, eps in ((0.7, 1e-5), (-3.0, 1e-6), (2.0, 0.0)):
        y = oracle.rmsnorm(np.full((1, H), a), w, eps, False)[0]
        assert np.allclose(y, a / math.sqrt(a * a + eps) * w, rtol=1e-15, atol=0)
    # with unit weights and eps = 0 the output has mean square exactly 1
    x = _rng(14).standard_normal((5, H))
    y = oracle.rmsnorm(x, np.ones(H), 0.0, False)
    assert np.allclose((y * y).mean(axis=1), 1.0, rtol=1e-14)
    # sign and direction are kept: y is a positive multiple of x per row
    ratio = y / x
    assert np.allclose(ratio, ratio[:, :1], rtol=1e-13) and (ratio > 0).all()


def test_rmsnorm_scale_invariance_and_gemma_offset():
    x = _rng(15).standard_normal((4, 40))
    w = _rng(16).standard_normal(40) * 0.1
    # eps = 0: multiplying a row by 4 leaves the output unchanged (exact in binary)
    assert np.array_equal(oracle.rmsnorm(4 * x, w, 0.0, False), oracle.rmsnorm(x, w, 0.0, False))
    # Gemma style scales by 1 + w: the plain form with weight 1 + w
    g = oracle.rmsnorm(x, w, 1e-5, True)
    assert np.allclose(g, oracle.rmsnorm(x, 1.0 + w, 1e-5, False), rtol=1e-15, atol=1e-15)
    # Gemma with w = 0 is the unweighted norm
    assert np.array_equal(oracle.rmsnorm(x, np.zeros(40), 1e-5, True), oracle.rmsnorm(x, np.ones(40), 1e-5, False))


def test_round_to_bf16_is_nearest_even():
    # bf16 keeps 8 significant bits: the spacing above 1 is 2^-7
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 1.0 + 2 ** -7],
                 dtype=np.float64)
    back = oracle.to_f64(oracle.round_to(v, "bf16"))
    # ties go to the even significand: 1 + 2^-8 -> 1, 1 + 3*2^-8 -> 1 + 2^-6;
    # 1 + 3*2^-9 is nearer 1 + 2^-7; exact bf16 values stay
    assert np.array_equal(back, [1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -2.5, 1.0 + 2 ** -7])


def _sandwich_shape(mlp_norm, E=8):
    base = wl.TINY.replace(name="sw", T=9, hidden_size=64, num_experts=E, num_experts_per_tok=min(3, E),
                           moe_intermediate_size=32, shared_intermediate_size=48, dtype="bf16",
                           mlp_norm=mlp_norm)
    if E == 0:
        base = base.replace(num_experts_per_tok=0, moe_intermediate_size=0)
    return base


@pytest.mark.parametrize("mlp_norm", ["rms", "gemma"])
@pytest.mark.parametrize("E", [8, 0])
def test_sandwich_identity_when_the_mlp_outputs_zero(mlp_norm, E):
    """out = X + post_norm(mlp(pre_norm(X))): with zero down weights the MLP
    output is 0, post_norm(0) = 0 (eps > 0), so out equals X exactly."""
    shape = _sandwich_shape(mlp_norm, E)
    inputs = wl.make_inputs(shape)
    inputs["sh_down"] = torch.zeros_like(inputs["sh_down"])
    if E:
        inputs["down"] = torch.zeros_like(inputs["down"])
    out = oracle.block_output(shape, inputs)
    assert np.array_equal(out, oracle.to_f64(inputs["X"]))


@pytest.mark.parametrize("mlp_norm", ["rms", "gemma"])
@pytest.mark.parametrize("E", [8, 0])
def test_sandwich_residual_and_input_scale_invariance(mlp_norm, E):
    """With eps = 0, scaling X by 4 scales the residual term by 4 and leaves the
    normalised branch unchanged: out(4X) - 4X == out(X) - X (up to the rounding
    of adding and removing the residual in fp64).  And the branch is the post
    norm of the plain layer on the rounded pre-norm output (the layer without
    norms, fed pre_norm(X) as its input)."""
    shape = _sandwich_shape(mlp_norm, E).replace(rms_norm_eps=0.0)
    inputs = wl.make_inputs(shape)
    out = oracle.block_output(shape, inputs)
    x = oracle.to_f64(inputs["X"])
    scaled = dict(inputs, X=(inputs["X"].float() * 4).to(torch.bfloat16))
    out4 = oracle.block_output(shape, scaled)
    assert np.allclose(out4 - 4 * x, out - x, rtol=0, atol=1e-13)
    plain = shape.replace(mlp_norm="none")
    xn_bits = oracle.normed_input(shape, inputs["X"], inputs["pre_norm_w"])
    xn = torch.from_numpy(xn_bits.view(np.int16)).view(torch.bfloat16)
    y = oracle.block_output(plain, dict(inputs, X=xn))
    g = mlp_norm == "gemma"
    assert np.allclose(out - x, oracle.rmsnorm(y, oracle.to_f64(inputs["post_norm_w"]), 0.0, g), rtol=0, atol=1e-13)


# ---------------------------------------------------- block-scaled weights

# OCP Microscaling Formats (MX) v1.0: the eight E2M1 magnitudes by code
E2M1_VALUES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def test_e4m3_decoding_matches_torch_float8_and_hand_values():
    """All 256 E4M3 codes against PyTorch's float8_e4m3fn (a library routine),
    at scale 2^0 and 2^3; hand values of the format's edges."""
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    for scale, mul in ((127, 1.0), (130, 8.0)):
        got = np.array([oracle.mx_value("mxfp8", c, scale) for c in range(256)])
        assert np.array_equal(np.isnan(got), np.isnan(ref))
        fin = ~np.isnan(ref)
        assert np.array_equal(got[fin], ref[fin] * mul)
    hand = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5,
            0xB8: -1.0, 0x7E: 448.0, 0xFE: -448.0}
    for c, v in hand.items():
        assert oracle.mx_value("mxfp8", c, 127) == v
    assert math.isnan(oracle.mx_value("mxfp8", 0x7F, 127)) and math.isnan(oracle.mx_value("mxfp8", 0xFF, 127))


def test_e2m1_and_e8m0_decoding():
    for c in range(16):
        v = E2M1_VALUES[c & 7] * (-1.0 if c & 8 else 1.0)
        assert oracle.mx_value("mxfp4", c, 127) == v
        assert oracle.mx_value("mxfp4", c, 125) == v / 4
    assert oracle.mx_value("mxfp8", 0x38, 0) == 2.0 ** -127
    assert oracle.mx_value("mxfp8", 0x38, 254) == 2.0 ** 127
    assert math.isnan(oracle.mx_value("mxfp8", 0x38, 255))


def _dequant(codes, scales, fmt):
    """Library-routine decode of stored MX tensors [..., rows, cols'] with
    block-major scales [..., cols / 32, rows]: E4M3 through PyTorch's
    float8_e4m3fn, E2M1 through the format's value table, times 2^(s - 127)."""
    codes = codes.cpu()
    if fmt == "mxfp8":
        v = codes.view(torch.float8_e4m3fn).double()
    else:
        lo, hi = (codes & 15).long(), (codes >> 4).long()
        nib = torch.stack([lo, hi], -1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
        table = torch.tensor([E2M1_VALUES[c & 7] * (-1.0 if c & 8 else 1.0) for c in range(16)], dtype=torch.float64)
        v = table[nib]
    s = torch.exp2(scales.cpu().double() - 127.0).transpose(-1, -2)  # [..., rows, cols / 32]
    return (v * s.repeat_interleave(32, dim=-1)).float()


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("packed", [False, True])
def test_mx_forward_equals_forward_on_the_decoded_weights(fmt, packed):
    """The block on MX weights equals, bit for bit, the block on the same values
    decoded by library routines and stored in fp32 (every MX value is exact in
    fp32).  Distinct H, I, S so that a transposed scale index reads the wrong
    blocks; several blocks per row in every projection."""
    base = wl.TINY.replace(T=9, hidden_size=128, num_experts=6, num_experts_per_tok=2, moe_intermediate_size=96,
                           shared_intermediate_size=64, dtype="bf16", weight_format=fmt)
    if packed:
        base = base.replace(shared_packed=True, shared_intermediate_size=96)
    inputs = wl.make_inputs(base)
    Ymx = oracle.forward_inputs(base, inputs)
    keys = ("gate", "up", "down") + (() if packed else ("sh_gate", "sh_up", "sh_down"))
    dec = dict(inputs, **{k: _dequant(inputs[k], inputs[k + "_scale"], fmt) for k in keys})
    Yf = oracle.forward_inputs(base.replace(weight_format="bf16"), dec)
    assert np.array_equal(Ymx, Yf)
    # and the decoded weights are the fp32 draws to within the format's precision
    # (the relative spacing of E4M3 is 2^-3, of E2M1 2^-1, plus saturation)
    assert np.isfinite(Ymx).all()


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_mx_dense_and_expert_equal_decoded(fmt):
    shape = wl.dense_layer(5, "afmoe").replace(hidden_size=128, shared_intermediate_size=192, weight_format=fmt,
                                               mlp_norm="none")
    inputs = wl.make_inputs(shape)
    Y = oracle.block_output(shape, inputs)
    dec = {k: _dequant(inputs[k], inputs[k + "_scale"], fmt) for k in ("sh_gate", "sh_up", "sh_down")}
    Yf = oracle.block_output(shape.replace(weight_format="bf16"), dict(inputs, **dec))
    assert np.array_equal(Y, Yf)
    cfg = oracle.cfg_from_shape(shape)
    sc = [inputs[k + "_scale"] for k in ("sh_gate", "sh_up", "sh_down")]
    g, u, a, y = oracle.expert(cfg, inputs["X"][2], inputs["sh_gate"], inputs["sh_up"], inputs["sh_down"], 192,
                               wfmt=fmt, scales=sc)
    gf, uf, af, yf = oracle.expert(cfg, inputs["X"][2], dec["sh_gate"], dec["sh_up"], dec["sh_down"], 192)
    assert np.array_equal(g, gf) and np.array_equal(y, yf) and np.array_equal(Y[2], y)


def test_mx_scale_moves_one_block_only():
    """Raising one E8M0 scale code by 1 doubles exactly the 32 weights of its
    block: the gate pre-activation of that row changes by the block's own
    partial dot product, and no other row changes."""
    shape = wl.dense_layer(3, "afmoe").replace(hidden_size=128, shared_intermediate_size=64, weight_format="mxfp8",
                                               mlp_norm="none")
    inputs = wl.make_inputs(shape)
    cfg = oracle.cfg_from_shape(shape)
    sc = [inputs[k + "_scale"].clone() for k in ("sh_gate", "sh_up", "sh_down")]
    x = inputs["X"][1]
    g0, _, _, _ = oracle.expert(cfg, x, inputs["sh_gate"], inputs["sh_up"], inputs["sh_down"], 64, wfmt="mxfp8",
                                scales=sc)
    row, blk = 5, 2
    sc2 = [t.clone() for t in sc]
    sc2[0][blk, row] += 1
    g1, _, _, _ = oracle.expert(cfg, x, inputs["sh_gate"], inputs["sh_up"], inputs["sh_down"], 64, wfmt="mxfp8",
                                scales=sc2)
    w = _dequant(inputs["sh_gate"], sc[0], "mxfp8").double().numpy()
    part = float(np.dot(w[row, 32 * blk:32 * blk + 32], oracle.to_f64(x)[32 * blk:32 * blk + 32]))
    changed = np.nonzero(g1 != g0)[0]
    assert list(changed) == [row]
    assert abs((g1[row] - g0[row]) - part) <= 1e-12 * (abs(part) + abs(g0[row]))
