"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every entry point include/moe.h declares, and rejects
bad arguments before touching the device."""

import ctypes
import subprocess

import pytest

from expert_routed_ffn_gb300 import build as moe_build
from expert_routed_ffn_gb300 import capi
from expert_routed_ffn_gb300 import workloads as wl


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return capi.load()


def test_exports_every_declared_symbol(lib):
    names = capi.header_symbols()
    for expected in ("moe_create", "moe_route", "moe_forward", "moe_destroy", "moe_last_error"):
        assert expected in names
    out = subprocess.run(["nm", "-D", "--defined-only", capi.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(lib, n)


def _weights():
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: validation fails first
    return capi.MoeWeights(router_w=fake, expert_bias=None, gate=fake, up=fake, down=fake,
                           sh_gate=fake, sh_up=fake, sh_down=fake)


@pytest.mark.parametrize("field,value,status", [
    ("hidden_size", 100, capi.MOE_ERR_UNSUPPORTED),
    ("hidden_size", 0, capi.MOE_ERR_UNSUPPORTED),
    ("num_experts", 0, capi.MOE_ERR_INVALID_ARG),  # a dense layer needs num_experts_per_tok 0
    ("num_experts", -1, capi.MOE_ERR_UNSUPPORTED),
    ("num_experts", 300, capi.MOE_ERR_UNSUPPORTED),
    ("num_experts_per_tok", 0, capi.MOE_ERR_INVALID_ARG),
    ("num_experts_per_tok", 129, capi.MOE_ERR_INVALID_ARG),
    ("moe_intermediate_size", 96, capi.MOE_ERR_UNSUPPORTED),
    ("score_func", 7, capi.MOE_ERR_INVALID_ARG),
    ("hidden_act", 5, capi.MOE_ERR_INVALID_ARG),
    ("act_dtype", 3, capi.MOE_ERR_INVALID_ARG),
    ("max_tokens", 0, capi.MOE_ERR_INVALID_ARG),
    ("shared_intermediate_size", 100, capi.MOE_ERR_UNSUPPORTED),
    ("mlp_norm", 3, capi.MOE_ERR_INVALID_ARG),
])
def test_create_rejects_bad_config(lib, field, value, status):
    cfg = capi.config_from_shape(wl.NANO_DECODE)
    setattr(cfg, field, value)
    h = ctypes.c_void_p()
    assert lib.moe_create(ctypes.byref(cfg), ctypes.byref(_weights()), ctypes.byref(h)) == status
    assert h.value is None
    assert lib.moe_last_error().decode()


def test_create_rejects_bad_weights(lib):
    cfg = capi.config_from_shape(wl.NANO_DECODE)
    h = ctypes.c_void_p()
    w = _weights()
    w.gate = None
    assert lib.moe_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    w = _weights()
    w.up = ctypes.c_void_p((1 << 20) + 2)  # misaligned
    assert lib.moe_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    assert "aligned" in lib.moe_last_error().decode()
    w = _weights()
    w.sh_down = None  # a separate shared expert needs all three tensors
    assert lib.moe_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    packed = capi.config_from_shape(wl.M3)
    packed.shared_intermediate_size = 1024  # packed width must equal the routed width
    assert lib.moe_create(ctypes.byref(packed), ctypes.byref(_weights()), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_create(None, ctypes.byref(_weights()), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_create(ctypes.byref(cfg), ctypes.byref(_weights()), None) == capi.MOE_ERR_INVALID_ARG


def test_create_rejects_bad_dense_and_norm_configs(lib):
    h = ctypes.c_void_p()
    dense = capi.config_from_shape(wl.WORKLOADS["dense_afmoe_decode"])
    w = _weights()
    w.pre_norm_w = w.post_norm_w = ctypes.c_void_p(1 << 20)
    bad = capi.config_from_shape(wl.WORKLOADS["dense_afmoe_decode"])
    bad.shared_intermediate_size = 6100  # not a multiple of 64
    assert lib.moe_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_UNSUPPORTED
    bad = capi.config_from_shape(wl.WORKLOADS["dense_afmoe_decode"])
    bad.shared_packed = 1  # nothing to pack into
    assert lib.moe_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    bad = capi.config_from_shape(wl.WORKLOADS["dense_afmoe_decode"])
    bad.act_dtype = capi.MOE_DTYPE_F32  # the dense layers run bf16 activations
    assert lib.moe_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_UNSUPPORTED
    bad = capi.config_from_shape(wl.WORKLOADS["dense_afmoe_decode"])
    bad.rms_norm_eps = -1.0
    assert lib.moe_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    w.post_norm_w = None  # the sandwich needs both norm weights
    assert lib.moe_create(ctypes.byref(dense), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    assert "norm" in lib.moe_last_error().decode()
    assert h.value is None


def test_create_rejects_bad_mx_configs(lib):
    """Block-scaled weights: the format must be known, every used weight tensor needs
    its scale tensor, and scale pointers must be 16-byte aligned."""
    h = ctypes.c_void_p()
    fake = ctypes.c_void_p(1 << 20)
    bad = capi.config_from_shape(wl.NANO_DECODE)
    bad.weight_format = 3
    assert lib.moe_create(ctypes.byref(bad), ctypes.byref(_weights()), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    cfg = capi.config_from_shape(wl.WORKLOADS["nano_decode_mxfp8"])
    assert cfg.weight_format == capi.MOE_WEIGHTS_MXFP8
    w = _weights()  # no scales at all
    assert lib.moe_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    assert "scale" in lib.moe_last_error().decode()
    w.gate_scale = w.up_scale = w.down_scale = fake
    assert lib.moe_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    assert "sh_gate_scale" in lib.moe_last_error().decode()  # the separate shared expert's scales
    w.sh_gate_scale = w.sh_up_scale = fake
    w.sh_down_scale = ctypes.c_void_p((1 << 20) + 8)  # misaligned
    assert lib.moe_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    assert "aligned" in lib.moe_last_error().decode()
    packed = capi.config_from_shape(wl.WORKLOADS["m3_mxfp8"])  # packed shared expert: routed scales suffice
    w = _weights()
    w.sh_gate = w.sh_up = w.sh_down = None
    w.gate_scale = w.up_scale = None
    w.down_scale = fake
    assert lib.moe_create(ctypes.byref(packed), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    assert h.value is None


def test_null_handle_calls_fail_cleanly(lib):
    assert lib.moe_forward(None, None, 4, None, None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_route(None, None, 4, None, None, None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_host(None, None, 4, None, None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_sync_status(None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_set_option(None, 0, 0) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_get_stats(None, None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_inspect(None, 0, None, 0, None) == capi.MOE_ERR_INVALID_ARG
    lib.moe_destroy(None)


def test_config_keys_follow_the_pages():
    names = [f[0] for f in capi.MoeConfig._fields_]
    for key in ("num_experts", "num_experts_per_tok", "num_shared_experts", "moe_intermediate_size",
                "route_scale", "score_func", "route_norm", "hidden_act", "shared_intermediate_size"):
        assert key in names
