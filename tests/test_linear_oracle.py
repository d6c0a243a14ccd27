"""The projection oracle (oracle/linear.py) against what fixes it: identity and
permutation weights return x's columns exactly, a scaled identity scales
exactly, a pure-Python loop on tiny shapes gives the same bits, and the one
rounding is to nearest even (ties checked on constructed exact ties)."""
from __future__ import annotations

import numpy as np

from linear_attention_decode_03_gb300.inputs import to_bf16_bits
from oracle import linear as OL
from oracle.oracle_np import bf16_to_f64, f64_to_bf16


def _rand_bits(rng, shape, scale=1.0):
    return to_bf16_bits(rng.normal(0.0, scale, size=shape).astype(np.float32))


def test_identity_and_permutation_weights():
    rng = np.random.default_rng(1)
    x = _rand_bits(rng, (5, 64))
    eye = to_bf16_bits(np.eye(64, dtype=np.float32))
    assert np.array_equal(OL.linear(x, eye), x)
    perm = rng.permutation(64)
    w = to_bf16_bits(np.eye(64, dtype=np.float32)[perm])     # y[:, n] = x[:, perm[n]]
    assert np.array_equal(OL.linear(x, w), x[:, perm])
    two = to_bf16_bits(2.0 * np.eye(64, dtype=np.float32))
    assert np.array_equal(bf16_to_f64(OL.linear(x, two)), 2.0 * bf16_to_f64(x))


def test_matches_a_python_loop_on_tiny_shapes():
    rng = np.random.default_rng(2)
    x, w = _rand_bits(rng, (3, 64)), _rand_bits(rng, (5, 64), 0.1)
    xv, wv = bf16_to_f64(x), bf16_to_f64(w)
    for r in range(3):
        for n in range(5):
            s = 0.0
            for k in range(64):
                s += xv[r, k] * wv[n, k]
            assert OL.linear(x, w)[r, n] == f64_to_bf16(np.array(s))


def test_single_rounding_ties_to_even():
    # 1 + 2^-8 lies halfway between the bf16 values 1 and 1 + 2^-7: even is 1;
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6... even is 1 + 2^-6
    x = to_bf16_bits(np.array([[1.0, 2.0 ** -8, 0.0, 0.0] + [0.0] * 60], dtype=np.float32))
    w = to_bf16_bits(np.ones((1, 64), dtype=np.float32))
    assert bf16_to_f64(OL.linear(x, w))[0, 0] == 1.0
    x3 = to_bf16_bits(np.array([[1.0, 2.0 ** -7, 2.0 ** -8, 0.0] + [0.0] * 60], dtype=np.float32))
    assert bf16_to_f64(OL.linear(x3, w))[0, 0] == 1.0 + 2.0 ** -6
    assert np.all(OL.abs_products(x3, w) >= np.abs(bf16_to_f64(OL.linear(x3, w))) * (1 - 2.0 ** -8))
