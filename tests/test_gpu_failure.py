"""Failure detection on the GPU without a fault: every device wait is bounded.
With the bound set to 0 the first wait that finds its data not ready gives up;
the kernel records the timeout in the device error word, drains its copies,
frees its tensor memory and returns, so the context stays usable."""

import pytest
import torch

from expert_routed_ffn_gb300 import capi
from expert_routed_ffn_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pair", [0, 1])
def test_wait_bound_reports_timeout_and_context_survives(pair):
    """pair = 1: the CTA-pair expert GEMM, whose abort also stops the other CTA."""
    from expert_routed_ffn_gb300 import build
    build.build()
    shape = wl.NANO_DECODE.replace(T=512)
    inputs, blk = P.make_case(shape)
    blk.set_option(capi.MOE_OPT_PATH, capi.PATH_GROUPED)
    blk.set_option(capi.MOE_OPT_GEMM_PAIR, pair)
    Y0 = blk.forward(inputs["X"]).clone()
    assert blk.sync_status() == capi.MOE_OK
    blk.set_option(capi.MOE_OPT_WAIT_LIMIT_NS, 0)
    blk.forward(inputs["X"])
    assert blk.sync_status() == capi.MOE_ERR_TIMEOUT
    assert "bound" in capi.load().moe_last_error().decode()
    blk.set_option(capi.MOE_OPT_WAIT_LIMIT_NS, 500_000_000)
    Y1 = blk.forward(inputs["X"])
    assert blk.sync_status() == capi.MOE_OK
    assert torch.equal(Y0, Y1)
