"""moe_dispatch_noalloc: the dispatch sort for callers that cannot allocate.

Callers whose device memory is owned by another pool, who run on a fixed
budget, or who cannot accept cudaMalloc's implicit synchronisation get the
dispatch step of moe_forward as a call that allocates nothing: its scratch
sits in a static device array inside libmoe.so, shared by every call on the
device.  This test runs it through the C ABI twice in a row (the second call
finds the first call's contents in the array) and checks that both calls
reproduce exactly the dispatch that moe_forward computed for the same
routing (integer results: bit-exact).  The file is named to be collected last.
"""

import ctypes

import pytest
import torch

from expert_routed_ffn_gb300 import capi
from expert_routed_ffn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routed_ffn_gb300 import build
    build.build()
    capi.load()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _forward_dispatch(shape):
    inputs = wl.make_inputs(shape, "cuda")
    blk = capi.block_from_inputs(shape, inputs)
    blk.forward(inputs["X"])
    T, k, E = shape.T, shape.k, shape.E
    idx = blk.inspect(capi.MOE_BUF_TOPK_IDX, T * k, torch.int32)
    offs = blk.inspect(capi.MOE_BUF_EXPERT_OFFS, E + 1, torch.int32)
    tok = blk.inspect(capi.MOE_BUF_SORTED_TOKEN, T * k, torch.int32)
    slot = blk.inspect(capi.MOE_BUF_SLOT, T * k, torch.int32)
    torch.cuda.synchronize()
    assert blk.sync_status() == capi.MOE_OK
    blk.close()
    return idx, offs, tok, slot


def _noalloc(idx, T, k, E):
    lib = capi.load()
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    slot = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    bad = torch.full((1,), 5, dtype=torch.int32, device="cuda")
    st = lib.moe_dispatch_noalloc(_ptr(idx), T, k, E, _ptr(offs), _ptr(tok), _ptr(slot), _ptr(bad),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == capi.MOE_OK, lib.moe_last_error().decode()
    torch.cuda.synchronize()
    return offs, tok, slot, int(bad.item())


def test_noalloc_dispatch_matches_forward_on_two_calls_in_a_row():
    big = wl.NANO_DECODE                                   # T 256, E 128, k 8
    small = wl.AFMOE_PREFILL.replace(T=333, hidden_size=512, moe_intermediate_size=192,
                                     shared_intermediate_size=384)  # ragged T, E 64, k 6
    for shape in (big, small):
        ref_idx, ref_offs, ref_tok, ref_slot = _forward_dispatch(shape)
        for _ in range(2):  # the second call sees the first call's scratch contents
            offs, tok, slot, bad = _noalloc(ref_idx, shape.T, shape.k, shape.E)
            assert bad == 0
            assert torch.equal(offs, ref_offs)
            assert torch.equal(tok, ref_tok)
            assert torch.equal(slot, ref_slot)


def test_noalloc_dispatch_rejects_sizes_beyond_its_scratch():
    lib = capi.load()
    idx = torch.zeros(8, dtype=torch.int32, device="cuda")
    out = torch.zeros(8, dtype=torch.int32, device="cuda")
    T = 32 * ((1 << 18) // 128 + 1)  # ceil(T/32) * E alone exceeds the array for E = 128
    st = lib.moe_dispatch_noalloc(_ptr(idx), T, 1, 128, _ptr(out), _ptr(out), _ptr(out), _ptr(out), None)
    assert st == capi.MOE_ERR_UNSUPPORTED
    assert "scratch" in lib.moe_last_error().decode()


def test_noalloc_dispatch_out_of_range_ids_and_empty_batch():
    """Ids outside [0, E) get slot -1 and raise bad_index; the valid slots keep
    the stable (expert, token, slot) order and the offsets count only them.
    An empty batch writes zero offsets and a clear bad_index."""
    T, k, E = 70, 3, 16
    g = torch.Generator().manual_seed(7)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    idx[0, 0] = -1
    idx[33, 2] = E
    idx[69, 1] = -1
    offs, tok, slot, bad = _noalloc(idx.cuda(), T, k, E)
    assert bad == 1
    valid = [(int(idx[t, j]), t, j) for t in range(T) for j in range(k) if 0 <= idx[t, j] < E]
    order = sorted(valid)
    offs, tok, slot = offs.cpu(), tok.cpu(), slot.cpu().view(T, k)
    assert int(offs[E]) == len(valid) and int(offs[0]) == 0
    counts = torch.bincount(torch.tensor([e for e, _, _ in valid]), minlength=E)
    assert torch.equal(offs[1:] - offs[:-1], counts.to(torch.int32))
    for row, (e, t, j) in enumerate(order):
        assert int(tok[row]) == t and int(slot[t, j]) == row
    assert int(slot[0, 0]) == -1 and int(slot[33, 2]) == -1 and int(slot[69, 1]) == -1

    lib = capi.load()
    offs0 = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    bad0 = torch.full((1,), 5, dtype=torch.int32, device="cuda")
    st = lib.moe_dispatch_noalloc(None, 0, k, E, _ptr(offs0), None, None, _ptr(bad0),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == capi.MOE_OK, lib.moe_last_error().decode()
    torch.cuda.synchronize()
    assert int(bad0.item()) == 0 and bool((offs0 == 0).all())
