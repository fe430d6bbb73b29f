"""CPU checks of the C-ABI library: it builds for sm_103a, loads, exports
every entry point declared in include/moe_layer.h, and its host-only entry
points (sizes, validation, error reporting) behave. No GPU compute."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from oracle import moe_oracle as O
from w4a16_routed_expert_gb300 import build as B
from w4a16_routed_expert_gb300 import capi, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return capi.lib()


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_entry_point_is_exported(lib):
    names = _declared_functions()
    assert "moe_layer_forward" in names and "moe_layer_create" in names
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (moe_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(lib, n)
    assert set(names) <= set(capi.PROTOTYPES), "binding lacks a prototype"


def test_abi_version(lib):
    assert lib.moe_abi_version() == 3


@pytest.mark.parametrize("H,I,G", [(256, 128, 64), (2048, 1024, 128), (2048, 512, 128), (2880, 2880, 128)])
def test_record_layout_agrees_with_oracle_and_generator(lib, H, I, G):
    offs, rb = O.record_layout(H, I, G)
    assert capi.record_bytes(H, I, G) == rb == synth.record_bytes(H, I, G)
    for i, name in enumerate(("gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s")):
        assert capi.record_section(H, I, G, i) == offs[name]


@pytest.mark.parametrize("H,I,G", [(2048, 1024, 32), (2880, 2880, 128), (256, 512, 64)])
def test_zero_point_record_layout_matches_generator(lib, H, I, G):
    offs = synth.section_layout(H, I, G, zero_points=True)
    assert lib.moe_record_bytes_zp(H, I, G, 1) == offs["record_bytes"]
    assert lib.moe_record_bytes_zp(H, I, G, 0) == synth.record_bytes(H, I, G) == lib.moe_record_bytes(H, I, G)
    names = ("gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s", "gate_z", "up_z", "down_z")
    for i, name in enumerate(names):
        assert capi.record_section(H, I, G, i) == offs[name]


def test_host_side_validation_and_errors(lib):
    assert lib.moe_layer_destroy(None) == capi.MOE_OK
    assert lib.moe_record_bytes(0, 128, 64) == 0
    h = ctypes.c_void_p()
    assert lib.moe_layer_create(None, None, ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    assert "NULL" in capi.last_error()
    cfg = capi.moe_layer_config_t(hidden=100, intermediate=128, num_experts=8, top_k=2, group_size=64,
                                  renormalize=1, has_shared_expert=0, max_tokens=4, num_slots=8,
                                  residency=0, add_residual=0)
    w = capi.moe_layer_weights_t(router_w=1, router_bias=None, slot_pool=256, expert_to_slot=1, host_backing=None)
    assert lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_UNSUPPORTED
    assert h.value is None
    cfg.hidden = 256
    cfg.top_k = 9
    assert lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    cfg.top_k = 2
    cfg.group_size = 48
    assert lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_UNSUPPORTED
    cfg.group_size = 64
    cfg.zero_points = 2
    assert lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    cfg.zero_points = 0
    w.slot_pool = 100  # not 256-byte aligned
    assert lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == capi.MOE_ERR_INVALID_ARG
    # partial residency with too few slots for one token's experts
    cfg.residency, cfg.num_slots = 1, 1
    w2 = capi.moe_layer_weights_t(router_w=1, router_bias=None, slot_pool=None, expert_to_slot=None,
                                  host_backing=1)
    assert lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(w2), ctypes.byref(h)) == capi.MOE_ERR_CAPACITY
    assert lib.moe_layer_forward(None, None, 1, None, None, None, None) == capi.MOE_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(capi, "_lib", None)
    monkeypatch.setattr(capi, "LIB_PATH", "/nonexistent/libmoe_w4a16.so")
    with pytest.raises(RuntimeError, match="not built"):
        capi.lib()


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "w4a16_routed_expert_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", text, flags=re.M), fn
                assert "moe_oracle" not in text, fn
