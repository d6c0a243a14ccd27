"""Small helpers shared by the tests: ad-hoc workloads and bf16 bit views.

Nothing here computes any step of the method; it only builds inputs (through
the seeded generator module) and views bit patterns.
"""
from __future__ import annotations

import numpy as np

from linear_attention_decode_03_gb300 import inputs as I

HEAD_DIM = 128
BF16_POS_INF = np.uint16(0x7F80)
BF16_NEG_INF = np.uint16(0xFF80)


def bf16_value(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def case(heads=2, requests=2, L=1, pool=8, width=4, seed=7, with_bias=False, verify=None, accepted=None):
    """A small seeded step: returns (StepInputs, oracle-style weights dict)."""
    if verify is None:
        verify = L > 1
    w = I.Workload(f"case_h{heads}_r{requests}_l{L}", heads=heads, requests=requests, L=L,
                   pool=pool, verify=verify, width=width, seed=seed)
    si = I.make_step_inputs(w, with_bias=with_bias, accepted=accepted)
    return si


def oracle_weights(si, **override):
    import oracle

    d = si.weights.as_dict()
    d.update(override)
    return oracle.Weights(**d)


def head_cols(D, which, h):
    """Column slice of block `which` (0 = q, 1 = k, 2 = v) for head h in the projected row."""
    return slice(which * D + h * HEAD_DIM, which * D + (h + 1) * HEAD_DIM)
