"""The C-ABI library builds, loads without a GPU, exports every symbol that
include/kda.h declares, and rejects invalid arguments on the host before any
CUDA call."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import linear_attention_decode_03_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(kda_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    kda.build()
    return kda.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    assert names == sorted(["kda_prepare", "kda_step", "kda_check", "kda_destroy", "kda_strerror",
                            "kda_launch_info", "kda_set_gate_mode", "kda_set_state_dtype", "kda_set_v_split",
                            "kda_plan_create",
                            "kda_plan_launch", "kda_plan_destroy", "kda_linear", "kda_linear_check",
                            "kda_layer_plan_create"])


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(kda.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_host_validation_without_gpu(lib):
    h = ctypes.c_void_p()
    # prepare: bad sizes are rejected before any CUDA call
    assert lib.kda_prepare(0, 4, 1, None, 1, 1, 1, 1, -5.0, 1e-6, ctypes.byref(h)) == -1
    assert lib.kda_prepare(2, 5, 1, None, 1, 1, 1, 1, -5.0, 1e-6, ctypes.byref(h)) == -1
    assert lib.kda_prepare(2, 4, 1, None, 1, 1, 1, 1, -5.0, 0.0, ctypes.byref(h)) == -1
    assert lib.kda_prepare(2, 4, None, None, 16, 16, 16, 16, -5.0, 1e-6, ctypes.byref(h)) == -1
    assert lib.kda_prepare(2, 4, 16, None, 16, 16, 16, 16, -5.0, 1e-6, None) == -1
    # step / check with no handle
    assert lib.kda_step(None, 16, 1, 1154, 16, 1, 16, 4, 16, 1, None, 16, None) == -1
    assert lib.kda_check(None, None, None) == -1
    assert lib.kda_set_v_split(None, 1) == -1
    lib.kda_destroy(None)
    assert lib.kda_launch_info(0, None, None, None) == -1
    assert lib.kda_launch_info(9, None, None, None) == -1
    assert lib.kda_set_gate_mode(None, 0) == -1
    assert lib.kda_set_state_dtype(None, 1) == -1
    # kda_linear: bad shapes rejected before any CUDA call
    assert lib.kda_linear(None, 4, 64, None, 8, 60, None, 8, None) == -1    # K not a multiple of 8
    assert lib.kda_linear(None, 4, 64, None, 0, 64, None, 8, None) == -1    # N < 1
    assert lib.kda_linear(None, 4, 64, None, 8, 64, None, 8, None) == -1    # null pointers
    assert lib.kda_linear(None, 0, 64, None, 8, 64, None, 8, None) == 0     # rows = 0: nothing
    assert lib.kda_linear_check(None, None) == -1                            # null flags pointer
    # (argument types as set by the binding)
    assert lib.kda_layer_plan_create(None, None, 1, 7168, 7168, None, None, 1154, None, 1, None, 4, None, 1,
                                     None, None, None, None, 7168, 1, None) == -1  # no plan out-pointer / handle
    p = ctypes.c_void_p()
    assert lib.kda_plan_create(None, None, 16, 1154, None, 1, None, 16, None, 1, None, None, ctypes.byref(p)) == -1
    assert lib.kda_plan_create(None, None, 16, 1154, None, 1, None, 16, None, 1, None, None, None) == -1
    assert lib.kda_plan_launch(None, None) == -1
    lib.kda_plan_destroy(None)
    assert kda.kda_strerror(0) == "ok"
    assert kda.kda_strerror(-1) == "invalid argument"
    assert kda.kda_strerror(-2) == "CUDA error"


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(kda, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        kda.load_library(str(tmp_path / "nope.so"))
