"""CPU oracle for the KDA decode / spec-verify core.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library (`linear_attention_decode_03_gb300`), and the CUDA library
never imports it.

Two independent implementations of the same definition:

* ``kda_oracle.c`` -- plain sequential fp64 C, built here with gcc into
  ``oracle/_build/libkda_oracle.so`` and called through ctypes
  (:func:`step`).  This is the oracle the GPU path is compared with.
* ``oracle_np.py`` -- the same steps written with NumPy (:func:`oracle_np.step`),
  used to cross-check the C oracle on small inputs.

The definition follows the vLLM documentation pages for the Kimi-K3 KDA
layer: "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.kda"
(K1 kda_pre, module docstring) and
"vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.prepared"
(PreparedKda: _operands, __init__, run).

Parity pins: every function here is pinned by the invariant tests in
``tests/test_oracle_pins.py`` (verify = chained decode, beta = 0 decay only,
the delta property, identity / shifted conv, unit RMS, the zero-state closed
form, the gate's limits, the l2-norm norms, the rounding rule).  Absolute
values beyond those invariants are not printed on the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

HEAD_DIM = 128
ERR_SLOT = 1
ERR_ACCEPTED = 2
DIAG_WIDTH = 5 * HEAD_DIM + 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libkda_oracle.so")
# A test that plants a mistake in the oracle (tests/test_oracle_mutations.py)
# points this variable at a mutated build; nothing else sets it.
_LIB_OVERRIDE = os.environ.get("KDA_ORACLE_LIB_OVERRIDE")
_lib = None


GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off"]


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no vectorisation flags), with
    OpenMP over the (request, head) tasks where the compiler has it (the
    results do not depend on the thread count)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    res = subprocess.run(["gcc", *GCC_FLAGS, "-fopenmp", "-o", tmp, _SRC, "-lm"], capture_output=True, text=True)
    if res.returncode != 0:  # no OpenMP runtime: the same source, serial
        subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def max_threads() -> int:
    """Threads the oracle can run its (request, head) tasks on (1 without OpenMP)."""
    return int(_load().kda_oracle_max_threads())


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_LIB_OVERRIDE or build())
        lib.kda_oracle_step.restype = ctypes.c_int
        lib.kda_oracle_bf16_round.restype = ctypes.c_uint16
        lib.kda_oracle_bf16_round.argtypes = [ctypes.c_double]
        lib.kda_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


@dataclass
class Weights:
    """Layer parameters as the model holds them (host arrays).

    conv_w  [3D, 1, W] uint16 (bf16 bits);  bias [3D] uint16 or None
    f_b     [D, 128] uint16;  A_log [H] f32;  dt_bias [D] f32;  o_norm [128] f32
    """

    heads: int
    conv_w: np.ndarray
    bias: Optional[np.ndarray]
    f_b: np.ndarray
    A_log: np.ndarray
    dt_bias: np.ndarray
    o_norm: np.ndarray
    gate_lower_bound: float = -5.0
    eps: float = 1e-6

    @property
    def width(self) -> int:
        return int(self.conv_w.shape[-1])


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def bf16_round(x: float) -> int:
    """The C oracle's fp64 -> bf16 (ties to even) rounding, as a bit pattern."""
    return int(_load().kda_oracle_bf16_round(float(x)))


def step(w: Weights, projected, conv_state, state_pool, slots, L: int, accepted=None, *,
         dim_first: bool = True, act: str = "silu", gate_mode: int = 0, state_dtype: str = "f32",
         diag: bool = False, threads: int = 1):
    """One decode (accepted None, L = 1) or verify step of the C oracle.

    gate_mode 0: g = lb * sigmoid(e^A (z + dt)); 1: g = max(-e^A softplus(z + dt), lb).
    state_dtype "f32" (state_pool fp32) or "bf16" (state_pool uint16 bf16 bits,
    each stored state rounded to nearest even).
    threads: OpenMP threads over the step's (request, head) tasks; each task
    runs in the same order whatever the count, so the results are the same.

    conv_state and state_pool are copied, not modified.  Returns
    ``(out, conv_state, state_pool, err[, diag])`` where ``diag`` is
    [rows, H, 5*128 + 1] fp64: q^, k^, v, g, bf16 o, beta per token-head.
    """
    lib = _load()
    projected = np.ascontiguousarray(projected, dtype=np.uint16)
    rows, pitch = projected.shape
    heads = w.heads
    D = HEAD_DIM * heads
    conv_state = np.array(conv_state, dtype=np.uint16, copy=True, order="C")
    bf16_state = state_dtype == "bf16"
    state_pool = np.array(state_pool, dtype=np.uint16 if bf16_state else np.float32, copy=True, order="C")
    pool = state_pool.shape[0]
    slots = np.ascontiguousarray(np.asarray(slots, dtype=np.int32).reshape(-1))
    acc = None if accepted is None else np.ascontiguousarray(np.asarray(accepted, dtype=np.int32))
    out = np.zeros((rows, D), dtype=np.uint16)
    err = ctypes.c_uint32(0)
    dg = np.zeros((rows, heads, DIAG_WIDTH), dtype=np.float64) if diag else None
    conv_w = np.ascontiguousarray(w.conv_w, dtype=np.uint16)
    bias = None if w.bias is None else np.ascontiguousarray(w.bias, dtype=np.uint16)
    f_b = np.ascontiguousarray(w.f_b, dtype=np.uint16)
    A_log = np.ascontiguousarray(w.A_log, dtype=np.float32)
    dt_bias = np.ascontiguousarray(w.dt_bias, dtype=np.float32)
    o_norm = np.ascontiguousarray(w.o_norm, dtype=np.float32)
    rc = lib.kda_oracle_step(
        ctypes.c_int(heads), ctypes.c_int(w.width), _ptr(conv_w), _ptr(bias), _ptr(f_b),
        _ptr(A_log), _ptr(dt_bias), _ptr(o_norm), ctypes.c_float(w.gate_lower_bound),
        ctypes.c_float(w.eps), ctypes.c_int(1 if act == "silu" else 0), ctypes.c_int(int(gate_mode)), _ptr(projected),
        ctypes.c_int64(rows), ctypes.c_int64(pitch), _ptr(conv_state), ctypes.c_int(1 if dim_first else 0),
        _ptr(state_pool), ctypes.c_int64(pool), ctypes.c_int(1 if bf16_state else 0), _ptr(slots), ctypes.c_int(L),
        _ptr(acc), _ptr(out),
        ctypes.byref(err), _ptr(dg), ctypes.c_int(int(threads)),
    )
    if rc != 0:
        raise ValueError(f"kda_oracle_step rejected its arguments (rc={rc})")
    if diag:
        return out, conv_state, state_pool, int(err.value), dg
    return out, conv_state, state_pool, int(err.value)
