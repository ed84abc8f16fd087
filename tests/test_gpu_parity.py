"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Small workloads are checked on every token and on both expert paths
(weight-streaming decode kernels and tcgen05 grouped GEMMs).  The full-size
workloads run in the launch configuration the benchmark times (auto path,
max_tokens = T) and are checked on every token's routing and on sampled
tokens' outputs (first, last and spread-out tokens).
"""

import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_gb300 import capi
from expert_routed_ffn_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

# (MOE_OPT_PATH, MOE_OPT_GEMM_PAIR): "grouped" runs one CTA per tile, "pair" the
# CTA-pair (cta_group::2) expert GEMM on the same path
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
        path, pair = path if isinstance(path, tuple) else (path, 0)
        blk.set_option(capi.MOE_OPT_PATH, path)
        blk.set_option(capi.MOE_OPT_GEMM_PAIR, pair)
    Y = blk.forward(inputs["X"])
    torch.cuda.synchronize()
    assert blk.sync_status() == capi.MOE_OK
    return inputs, blk, Y


def _topk(blk, T, k):
    idx = blk.inspect(capi.MOE_BUF_TOPK_IDX, T * k, torch.int32).view(T, k)
    w = blk.inspect(capi.MOE_BUF_TOPK_W, T * k, torch.float32).view(T, k)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def _sample(T, n=16):
    return sorted(set([0, T - 1] + np.linspace(0, T - 1, n).astype(int).tolist()))


# ------------------------------------------------------- small, every token

SMALL = {
    "tiny_f32": wl.TINY,
    "nano_decode": wl.NANO_DECODE,
    "tiny_softmax": wl.TINY.replace(name="tiny_softmax", score_func="softmax"),
    "tiny_no_shared": wl.TINY.replace(name="tiny_noshared", num_shared_experts=0, shared_intermediate_size=0),
    "tiny_k_equals_E": wl.TINY.replace(name="tiny_kE", num_experts_per_tok=16),
    "m3_small_packed": wl.M3.replace(name="m3_small", T=96, hidden_size=512, num_experts=8,
                                     num_experts_per_tok=2, moe_intermediate_size=256,
                                     shared_intermediate_size=256),
    "afmoe_ragged": wl.AFMOE_PREFILL.replace(name="afmoe_ragged", T=333, hidden_size=512,
                                             moe_intermediate_size=192, shared_intermediate_size=384),
    "nano_T1": wl.NANO_DECODE.replace(name="nano_T1", T=1),
    # a few tokens with a wide expert (I = 1024, 16 k-blocks)
    "afmoe_T4": wl.AFMOE_PREFILL.replace(name="afmoe_T4", T=4, hidden_size=512, moe_intermediate_size=1024,
                                                shared_intermediate_size=512),
    "afmoe_T1": wl.AFMOE_PREFILL.replace(name="afmoe_T1", T=1, hidden_size=512, moe_intermediate_size=1024,
                                                shared_intermediate_size=1024),
    "nano_T129": wl.NANO_DECODE.replace(name="nano_T129", T=129),
}


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("name", list(SMALL))
def test_small_workload_every_token(name, path):
    shape = SMALL[name]
    inputs, blk, Y = _run(shape, PATHS[path])
    ih = P.host_inputs(inputs)
    idx, w = _topk(blk, shape.T, shape.k)
    P.check_route(shape, ih, idx, w)
    P.check_output(P.to_np(Y), oracle.forward_inputs(shape, ih), shape.dtype == "bf16", tag=f"{name}-{path}")
    assert blk.stats().path == PATHS[path][0]


@pytest.mark.parametrize("path", list(PATHS))
def test_tiny_fp32_against_fp32_expert_weights(path):
    """The tiny workload as drawn: fp32 X, router and expert weights.  The block
    stores its expert weights in bf16 and its GEMMs read X in bf16; the oracle
    here runs on the fp32 originals, so the output error includes the rounding
    of every expert weight and of X, and still meets 2e-2 rms.  The routing
    stays fp32 on both sides, so the top-k is compared as everywhere else."""
    shape = wl.TINY
    inputs, blk, Y = _run(shape, PATHS[path])
    assert inputs["gate"].dtype == torch.float32 and inputs["X"].dtype == torch.float32
    drawn = P.host_inputs(inputs, as_drawn=True)
    idx, w = _topk(blk, shape.T, shape.k)
    P.check_route(shape, drawn, idx, w)
    P.check_output(P.to_np(Y), oracle.forward_inputs(shape, drawn), out_bf16=False, tag=f"tiny_fp32_drawn-{path}")


def test_clamp_swiglu_fires_and_matches():
    """Scaled gate/up weights push |gate| and |up| past limit 7 on many entries."""
    shape = SMALL["m3_small_packed"]
    inputs = wl.make_inputs(shape, "cuda", row_filter=oracle.margin_filter(shape))
    inputs["gate"] = inputs["gate"] * 12
    inputs["up"] = inputs["up"] * 12
    ih = P.host_inputs(inputs)
    # the clamp really fires on the oracle's own intermediates
    cfg = oracle.cfg_from_shape(shape)
    g, u, _, _ = oracle.expert(cfg, ih["X"][0], ih["gate"][3], ih["up"][3], ih["down"][3], shape.I)
    assert (g > 7).mean() > 0.1 and (np.abs(u) > 7).mean() > 0.1
    for path in PATHS.values():
        blk = capi.block_from_inputs(shape, inputs)
        _, blk, Y = _run(shape, path, inputs, blk)
        P.check_output(P.to_np(Y), oracle.forward_inputs(shape, ih), tag=f"clamp-{path}")


def test_hidden_activations_match_oracle_expert():
    shape = SMALL["afmoe_ragged"]
    for path in PATHS.values():
        inputs, blk, _ = _run(shape, path)
        ih = P.host_inputs(inputs)
        T, k, E, I = shape.T, shape.k, shape.E, shape.I
        offs = blk.inspect(capi.MOE_BUF_EXPERT_OFFS, E + 1, torch.int32).cpu().numpy()
        tok = blk.inspect(capi.MOE_BUF_SORTED_TOKEN, T * k, torch.int32).cpu().numpy()
        hid = blk.inspect(capi.MOE_BUF_HIDDEN, T * k * I, torch.bfloat16).view(T * k, I).float().cpu().numpy()
        cfg = oracle.cfg_from_shape(shape)
        for e in (0, E // 2, E - 1):
            for row in range(offs[e], min(offs[e + 1], offs[e] + 3)):
                x = ih["X"][tok[row]]
                _, _, a, _ = oracle.expert(cfg, x, ih["gate"][e], ih["up"][e], ih["down"][e], I)
                err = np.abs(hid[row] - a).max()
                assert err <= 2e-2 * np.sqrt(np.mean(a ** 2)) + 1e-6, (e, row, err)


def test_dispatch_is_a_stable_sort_by_expert():
    shape = SMALL["nano_T129"]
    inputs, blk, _ = _run(shape, capi.PATH_GROUPED)
    T, k, E = shape.T, shape.k, shape.E
    idx, _ = _topk(blk, T, k)
    offs = blk.inspect(capi.MOE_BUF_EXPERT_OFFS, E + 1, torch.int32).cpu().numpy()
    tok = blk.inspect(capi.MOE_BUF_SORTED_TOKEN, T * k, torch.int32).cpu().numpy()
    slot = blk.inspect(capi.MOE_BUF_SLOT, T * k, torch.int32).view(T, k).cpu().numpy()
    assert offs[0] == 0 and offs[E] == T * k and np.all(np.diff(offs) >= 0)
    counts = np.bincount(idx.ravel(), minlength=E)
    assert np.array_equal(np.diff(offs), counts)
    # brute-force stable order: (expert, token, slot)
    order = sorted(((idx[t, j], t, j) for t in range(T) for j in range(k)))
    for row, (e, t, j) in enumerate(order):
        assert tok[row] == t and slot[t, j] == row and offs[e] <= row < offs[e + 1]


def test_route_entry_point_matches_forward_routing():
    shape = SMALL["nano_decode"]
    inputs, blk, _ = _run(shape)
    idx_f, w_f = _topk(blk, shape.T, shape.k)
    idx_r, w_r = blk.route(inputs["X"])
    torch.cuda.synchronize()
    assert np.array_equal(idx_r.cpu().numpy(), idx_f)
    assert np.array_equal(w_r.cpu().numpy(), w_f)
    assert blk.stage_names() == ["router"]


def test_packed_shared_equals_separate_shared_on_gpu():
    shape = SMALL["m3_small_packed"]
    inputs = wl.make_inputs(shape, "cuda", row_filter=oracle.margin_filter(shape))
    E = shape.E
    sep_shape = shape.replace(shared_packed=False)
    sep = dict(inputs, gate=inputs["gate"][:E].contiguous(), up=inputs["up"][:E].contiguous(),
               down=inputs["down"][:E].contiguous(), sh_gate=inputs["gate"][E].contiguous(),
               sh_up=inputs["up"][E].contiguous(), sh_down=inputs["down"][E].contiguous())
    for path in PATHS.values():
        _, _, Yp = _run(shape, path, inputs, capi.block_from_inputs(shape, inputs))
        _, _, Ys = _run(sep_shape, path, sep, capi.block_from_inputs(sep_shape, sep))
        assert torch.equal(Yp, Ys)


def test_fused_expert_gemm_equals_two_launches():
    """One persistent launch (down tiles wait for their gate/up rows) and two
    launches compute the same tiles with the same arithmetic: bit-identical."""
    for name in ("afmoe_ragged", "m3_small_packed", "nano_decode"):
        shape = SMALL[name]
        inputs, blk, Y1 = _run(shape, capi.PATH_GROUPED)
        names = blk.stage_names()
        g = names.index("dispatch_scatter") + 1
        assert names[g:] == ["experts_gemm", "combine"]
        blk.set_option(capi.MOE_OPT_FUSE_EXPERTS, 0)
        Y2 = blk.forward(inputs["X"])
        torch.cuda.synchronize()
        assert blk.sync_status() == capi.MOE_OK
        assert blk.stage_names()[g:] == ["gate_up_gemm", "down_gemm", "combine"]
        assert torch.equal(Y1, Y2)


def test_device_trace_orders_the_kernels_and_leaves_results_unchanged():
    """With the trace on, each kernel of the grouped path reports first start <=
    first ready <= last ready <= last end and first ready <= first end, and a
    kernel passes its dependency wait only after its predecessor's last CTA
    ended (the global timer ticks in about 1 us steps, hence the slack)."""
    for name in ("nano_decode", "tiny_f32"):
        shape = SMALL[name]
        inputs, blk, Y1 = _run(shape, capi.PATH_GROUPED)
        blk.set_option(capi.MOE_OPT_TRACE, 1)
        Y2 = blk.forward(inputs["X"])
        tr = blk.trace()
        assert blk.sync_status() == capi.MOE_OK
        assert torch.equal(Y1, Y2)
        assert [t[0] for t in tr] == blk.stage_names()
        assert min(t[1] for t in tr) == 0.0
        for name_i, b, r, rl, e0, e in tr:
            assert 0.0 <= b <= r <= rl <= e < 1e5 and r <= e0 <= e, (name_i, b, r, rl, e0, e)
        for prev, cur in zip(tr, tr[1:]):
            assert cur[2] >= prev[5] - 1.5, (prev, cur)
        blk.set_option(capi.MOE_OPT_TRACE, 0)
        with pytest.raises(capi.MoeError):
            blk.trace()


def test_pair_gemm_fused_equals_two_launches_and_oracle():
    """The CTA-pair expert GEMM in one launch and in two launches: bit-identical,
    and within tolerance of the oracle on every token."""
    for name in ("afmoe_ragged", "m3_small_packed"):
        shape = SMALL[name]
        inputs, blk, Y1 = _run(shape, PATHS["pair"])
        names = blk.stage_names()
        assert names[names.index("dispatch_scatter") + 1:] == ["experts_gemm", "combine"]
        blk.set_option(capi.MOE_OPT_FUSE_EXPERTS, 0)
        Y2 = blk.forward(inputs["X"])
        torch.cuda.synchronize()
        assert blk.sync_status() == capi.MOE_OK
        assert torch.equal(Y1, Y2)
        ih = P.host_inputs(inputs)
        P.check_output(P.to_np(Y1), oracle.forward_inputs(shape, ih), shape.dtype == "bf16", tag=f"{name}-pair-fused")


def test_pair_swapped_remainder_tiles_match_unswapped_and_oracle():
    """CTA pairs: m-tiles of at most 128 rows run with the weights as M and the tokens
    as N.  A mix of experts (full 256-row tiles, remainders of <= 128 and of > 128
    rows) against the same forward with every tile unswapped (bit-identical: each
    output is the same K-ordered sum of the same products) and against the oracle on
    every token."""
    shape = wl.AFMOE_PREFILL.replace(name="afmoe_mixed", T=1500, hidden_size=512, moe_intermediate_size=192,
                                     shared_intermediate_size=384)
    inputs, blk = P.make_case(shape)
    blk.set_option(capi.MOE_OPT_PATH, capi.PATH_GROUPED)
    blk.set_option(capi.MOE_OPT_GEMM_PAIR, 1)
    Y1 = blk.forward(inputs["X"]).clone()
    torch.cuda.synchronize()
    assert blk.sync_status() == capi.MOE_OK
    blk.set_option(capi.MOE_OPT_PAIR_SWAP, 0)
    Y0 = blk.forward(inputs["X"])
    torch.cuda.synchronize()
    assert blk.sync_status() == capi.MOE_OK
    assert torch.equal(Y1, Y0), "swapped remainder tiles differ from unswapped ones"
    ih = P.host_inputs(inputs)
    P.check_output(P.to_np(Y1), oracle.forward_inputs(shape, ih), True, tag="afmoe_mixed-pair-swap")
    blk.close()


@pytest.mark.parametrize("name", ["nano_decode", "afmoe_ragged", "m3_small_packed", "nano_T1"])
def test_combine_overlapped_with_gemm_is_bit_identical(name):
    """The combine that starts while the expert GEMM runs (each token once its rows
    are counted in) adds the same terms in the same order as the combine that waits
    for the whole GEMM: bit-identical, with one and with two GEMM launches."""
    shape = SMALL[name]
    inputs, blk = P.make_case(shape)
    blk.set_option(capi.MOE_OPT_PATH, capi.PATH_GROUPED)
    ys = []
    for fuse in (1, 0):
        blk.set_option(capi.MOE_OPT_FUSE_EXPERTS, fuse)
        for ovl in (1, 0):
            blk.set_option(capi.MOE_OPT_COMBINE_OVERLAP, ovl)
            ys.append(blk.forward(inputs["X"]).clone())
            torch.cuda.synchronize()
            assert blk.sync_status() == capi.MOE_OK
    assert all(torch.equal(ys[0], y) for y in ys[1:])
    blk.close()


@pytest.mark.parametrize("name,pair", [("nano_decode", 2), ("nano_T1", 2), ("nano_T129", 2), ("afmoe_ragged", 0),
                                       ("afmoe_ragged", 1), ("m3_small_packed", 2)])
def test_staged_stores_are_bit_identical(name, pair):
    """The expert GEMM's outputs stored through shared memory (a TMA store per full
    32-row slice, coalesced stores of the rows of a partial one) equal the rows each
    lane stores from registers, bit for bit: routed hidden activations, the shared
    expert's hidden activations and the block output; 32-row (decode), 128-row and
    256-row (CTA pair) tiles, ragged experts, one token."""
    shape = SMALL[name]
    inputs, blk = P.make_case(shape)
    blk.set_option(capi.MOE_OPT_PATH, capi.PATH_GROUPED)
    blk.set_option(capi.MOE_OPT_GEMM_PAIR, pair)
    T, k, I, S = shape.T, shape.k, shape.I, shape.S
    outs = []
    for staged in (1, 0):
        blk.set_option(capi.MOE_OPT_STAGED_STORES, staged)
        Y = blk.forward(inputs["X"]).clone()
        torch.cuda.synchronize()
        assert blk.sync_status() == capi.MOE_OK
        hid = blk.inspect(capi.MOE_BUF_HIDDEN, T * k * I, torch.bfloat16)
        sh = blk.inspect(capi.MOE_BUF_SHARED_HIDDEN, T * S, torch.bfloat16) if S else None
        outs.append((Y, hid, sh))
    (Y1, h1, s1), (Y0, h0, s0) = outs
    assert torch.equal(h1, h0), "routed hidden rows differ"
    if S:
        assert torch.equal(s1, s0), "shared hidden rows differ"
    assert torch.equal(Y1, Y0), "block output differs"
    ih = P.host_inputs(inputs)
    P.check_output(P.to_np(Y1), oracle.forward_inputs(shape, ih), True, tag=f"{name}-staged")
    blk.close()


def test_set_option_takes_only_documented_values():
    """Every option accepts only its documented values and an unknown option id is
    refused, before anything runs; a refused call leaves the handle as it was."""
    shape = SMALL["nano_T1"]
    inputs, blk = P.make_case(shape)
    Y0 = blk.forward(inputs["X"]).clone()
    binary = [capi.MOE_OPT_GRAPH, capi.MOE_OPT_PREFETCH, capi.MOE_OPT_FUSE_EXPERTS, capi.MOE_OPT_COMBINE_OVERLAP,
              capi.MOE_OPT_STAGED_STORES, capi.MOE_OPT_PAIR_SWAP, capi.MOE_OPT_TRACE, capi.MOE_OPT_STAGE_EVENTS]
    for opt in binary:
        for bad in (-1, 2):
            with pytest.raises(capi.MoeError):
                blk.set_option(opt, bad)
    for opt, bad in ((capi.MOE_OPT_GEMM_PAIR, 3), (capi.MOE_OPT_PATH, 4), (capi.MOE_OPT_PATH, -1),
                     (capi.MOE_OPT_WAIT_LIMIT_NS, -1), (7, 0), (12, 0)):
        with pytest.raises(capi.MoeError):
            blk.set_option(opt, bad)
    Y1 = blk.forward(inputs["X"])
    torch.cuda.synchronize()
    assert blk.sync_status() == capi.MOE_OK
    assert torch.equal(Y0, Y1)
    blk.close()


def test_token_permutation_equivariance_and_determinism():
    shape = SMALL["afmoe_ragged"]
    for path in PATHS.values():
        inputs, blk, Y = _run(shape, path)
        Y2 = blk.forward(inputs["X"])
        torch.cuda.synchronize()
        assert torch.equal(Y, Y2), "two runs differ"
        perm = torch.randperm(shape.T, generator=torch.Generator().manual_seed(7)).cuda()
        Yp = blk.forward(inputs["X"][perm].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(Yp, Y[perm])


def test_forward_host_matches_forward_and_edge_sizes():
    shape = SMALL["nano_decode"]
    inputs, blk, Y = _run(shape, max_tokens=shape.T)
    Xh = inputs["X"].cpu().pin_memory()
    Yh = torch.empty_like(Xh).pin_memory()
    blk.forward_host(Xh, Yh)
    assert torch.equal(Yh, Y.cpu())
    # T = 0 is a no-op; T above max_tokens is rejected without launching
    empty = inputs["X"][:0]
    assert capi.load().moe_forward(blk.h, capi._ptr(inputs["X"]), 0, capi._ptr(Y), None) == capi.MOE_OK
    assert blk.stats().kernel_launches == 0
    big = capi.load().moe_forward(blk.h, capi._ptr(inputs["X"]), shape.T + 1, capi._ptr(Y), None)
    assert big == capi.MOE_ERR_INVALID_ARG
    assert empty.shape[0] == 0


def test_forward_host_pinned_pageable_and_fp32_buffers():
    """Pinned host buffers are read and written by the GPU itself; pageable ones (or a
    pinned one paired with a pageable one) go through the copy engines; fp32 tokens
    move 4 bytes per value.  Every combination equals moe_forward bit for bit."""
    for name in ("nano_decode", "tiny_f32"):
        shape = SMALL[name]
        inputs, blk, Y = _run(shape, max_tokens=shape.T)
        ref = Y.cpu()
        Xp, Xg = inputs["X"].cpu().pin_memory(), inputs["X"].cpu()
        for xh, pinned_y in ((Xp, True), (Xg, False), (Xp, False), (Xg, True)):
            Yh = torch.empty_like(Xg)
            if pinned_y:
                Yh = Yh.pin_memory()
            for _ in range(3):  # eager, then (pinned pairs) capture and replay
                Yh.zero_()
                blk.forward_host(xh, Yh)
                assert torch.equal(Yh, ref), (name, xh.is_pinned(), pinned_y)
        assert blk.sync_status() == capi.MOE_OK
        blk.close()


def test_forward_host_graph_replay_matches_forward():
    """moe_forward_host runs eagerly, then captures a CUDA graph on the second call with
    the same buffers and T, then replays it: every call equals moe_forward bit for bit,
    on the legacy stream and on a caller's stream; new inputs in the same pinned buffer
    are picked up by the replay; an option change or another T goes back to eager runs."""
    for name in ("nano_decode", "afmoe_ragged", "m3_small_packed"):
        shape = SMALL[name]
        inputs, blk, Y = _run(shape, max_tokens=shape.T)
        Xh = inputs["X"].cpu().pin_memory()
        Yh = torch.empty_like(Xh).pin_memory()
        ref = Y.cpu()
        for _ in range(4):  # eager, capture, replay, replay
            Yh.zero_()
            blk.forward_host(Xh, Yh)
            assert torch.equal(Yh, ref)
        side = torch.cuda.Stream()
        for _ in range(3):
            Yh.zero_()
            blk.forward_host(Xh, Yh, stream=side)
            assert torch.equal(Yh, ref)
        # new token values in the captured buffer
        X2 = torch.roll(inputs["X"], 1, 0).contiguous()
        Xh.copy_(X2.cpu())
        Y2 = blk.forward(X2)
        torch.cuda.synchronize()
        for _ in range(2):
            blk.forward_host(Xh, Yh)
            assert torch.equal(Yh, Y2.cpu())
        blk.set_option(capi.MOE_OPT_PREFETCH, 0)  # a changed option: eager, then a new capture
        for _ in range(3):
            blk.forward_host(Xh, Yh)
            assert torch.equal(Yh, Y2.cpu())
        blk.set_option(capi.MOE_OPT_GRAPH, 0)
        blk.forward_host(Xh, Yh)
        assert torch.equal(Yh, Y2.cpu())
        half = shape.T // 2  # another T
        Yh2 = torch.empty_like(Xh[:half]).pin_memory()
        blk.set_option(capi.MOE_OPT_GRAPH, 1)
        Yd = blk.forward(X2[:half].contiguous())
        torch.cuda.synchronize()
        for _ in range(3):  # every call writes this call's output buffer
            Yh2.zero_()
            blk.forward_host(Xh[:half], Yh2)
            assert torch.equal(Yh2, Yd.cpu())
        for _ in range(3):  # and back to the first buffers: a new capture, not the old graph
            Yh.zero_()
            blk.forward_host(Xh, Yh)
            assert torch.equal(Yh, Y2.cpu())
        assert blk.sync_status() == capi.MOE_OK
        blk.close()


# ---------------------------------------------------- full sizes, sampled

def _full(shape, n_sample=16):
    inputs, blk, Y = _run(shape, max_tokens=shape.T)
    ih = P.host_inputs(inputs)
    idx, w = _topk(blk, shape.T, shape.k)
    P.check_route(shape, ih, idx, w)
    toks = _sample(shape.T, n_sample)
    Yref = oracle.forward_inputs(shape, ih, tokens=toks)
    rel = P.check_output(P.to_np(Y)[toks], Yref, shape.dtype == "bf16", tag=shape.name)
    return rel, blk


def test_full_afmoe_prefill():
    _full(wl.AFMOE_PREFILL)


def test_full_m3_packed_clamp_swiglu():
    _full(wl.M3, n_sample=10)


@pytest.mark.parametrize("T", wl.ZIPF_TOKENS)
def test_full_zipf_sweep(T):
    _, blk = _full(wl.zipf_sweep(T), n_sample=12)
    assert blk.stats().path in (capi.PATH_DECODE, capi.PATH_GROUPED, capi.PATH_SWAPPED)
