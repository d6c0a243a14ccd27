"""Oracle for the layer's projections around the KDA core: y = x . W^T.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.  It shares nothing
with the CUDA library.

Sources: the K1 page ("vllm.models.kimi_k3.amd.specialized_decode.mono.
attention.kda") puts an in_proj GEMV in front of the KDA core (x [rows, 7168]
to the packed projection row) and the K2a page ("vllm.models.kimi_k3.amd.
specialized_decode.mono.attention.back", module docstring: K2a attn_post) an
o_proj GEMV after it (core_out [rows, D] to [rows, 7168]).  A GEMV has a plain
definition, so the oracle is that definition: the exact product of the bf16
inputs in fp64, rounded once to bf16 (nearest even).  W is [out, in] (a torch
Linear weight).
"""
from __future__ import annotations

import numpy as np

from .oracle_np import bf16_to_f64, f64_to_bf16


def linear(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """bf16 bits x [rows, K], W [N, K] -> bf16 bits of round(x . W^T).

    fp64 holds each bf16 x bf16 product exactly and the K-term sums to far
    below a bf16 half ulp, so the single rounding is the correctly rounded one
    but for values within fp64 noise of a rounding boundary."""
    x = bf16_to_f64(x_bits)
    w = bf16_to_f64(w_bits)
    return f64_to_bf16(x @ w.T)


def abs_products(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """sum_k |x_k w_k| per output: the scale of the accumulation error of any
    summation order (for a tolerance on an fp32-accumulated product)."""
    return np.abs(bf16_to_f64(x_bits)) @ np.abs(bf16_to_f64(w_bits)).T
