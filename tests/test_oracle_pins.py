"""Pins of the CPU oracle against what the definition itself fixes.

The pages print no worked example, so the oracle is pinned by invariants and
closed forms of the KDA decode / spec-verify core (K1 kda_pre module
docstring on the "...amd.specialized_decode.mono.attention.kda" page; the
PreparedKda page for the column split and scalars), each chosen so that a
plausible slip -- a dropped term, a wrong sign, a transposed state, the decay
on the wrong axis, o taken before the update, a wrong tap order or slot index
-- fails at least one of them.  Both oracles (C and NumPy) are pinned.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import oracle_np
from linear_attention_decode_03_gb300.inputs import to_bf16_bits as I_to_bf16
from tests.helpers import (BF16_NEG_INF, BF16_POS_INF, HEAD_DIM, bf16_value, case, head_cols,
                           oracle_weights)

IMPLS = {"c": oracle.step, "np": oracle_np.step}


@pytest.fixture(params=sorted(IMPLS))
def run(request):
    return IMPLS[request.param]


def _decode_case(heads=2, requests=3, pool=6, seed=11, **kw):
    si = case(heads=heads, requests=requests, L=1, pool=pool, seed=seed, **kw)
    return si, si.full_state_pool(), si.full_conv_state()


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rounding_closed_forms():
    one = 1.0
    table = [
        (one, 0x3F80),
        (one + 2.0 ** -8, 0x3F80),                 # tie -> even (down)
        (one + 3 * 2.0 ** -8, 0x3F82),             # tie -> even (up)
        (one + 2.0 ** -8 + 2.0 ** -40, 0x3F81),    # just above the tie: rounded once from fp64
        (-2.5, 0xC020),
        (-0.0, 0x8000),
        (1.5 * 2.0 ** -133, 0x0002),               # subnormal tie -> even
        (2.0 ** -134, 0x0000),                     # half the smallest subnormal -> 0 (even)
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),    # largest finite
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),    # max + half ulp -> inf (tie to even)
        (float("inf"), 0x7F80),
    ]
    for x, bits in table:
        assert oracle.bf16_round(x) == bits, (x, hex(oracle.bf16_round(x)))
        assert int(oracle_np.f64_to_bf16(x)) == bits, x
    assert oracle.bf16_round(float("nan")) & 0x7F80 == 0x7F80


def test_bf16_rounding_matches_torch_on_fp32_values():
    """For values already in fp32, fp64->bf16 must equal torch's fp32->bf16 (RNE)."""
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 1e-38, 500), rng.normal(0, 1e30, 500)])
    x32 = x.astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got_np = oracle_np.f64_to_bf16(x32.astype(np.float64))
    got_c = np.array([oracle.bf16_round(float(v)) for v in x32], dtype=np.uint16)
    assert np.array_equal(got_np, ref)
    assert np.array_equal(got_c, ref)


# ------------------------------------------------------------------- recurrence

def test_verify_equals_chained_decode(run):
    """An L-token verify equals L single-token decodes chained through the
    slots: token t starts from slots[r, t-1] (token 0 from the start slot
    slots[r, accepted-1]) and leaves its state and window in slots[r, t]."""
    R, L, H = 3, 3, 2
    si = case(heads=H, requests=R, L=L, pool=12, seed=21, accepted=[2, 3, 1])
    W = oracle_weights(si)
    pool, conv = si.full_state_pool(), si.full_conv_state()
    out_v, conv_v, pool_v, err = run(W, si.projected, conv, pool, si.slots, L, si.accepted)
    assert err == 0

    slots = si.slots.reshape(R, L)
    pool_d, conv_d = pool.copy(), conv.copy()
    out_d = np.zeros_like(out_v)
    for r in range(R):
        src = slots[r, si.accepted[r] - 1]
        for t in range(L):
            dst = slots[r, t]
            if dst != src:
                pool_d[dst] = pool_d[src]
                conv_d[dst] = conv_d[src]
            row = r * L + t
            o, conv_d, pool_d, e = run(W, si.projected[row:row + 1], conv_d, pool_d,
                                       np.array([dst], np.int32), 1, None)
            assert e == 0
            out_d[row] = o[0]
            src = dst
    written = np.unique(slots)
    np.testing.assert_allclose(pool_v[written], pool_d[written], rtol=0, atol=2e-6)
    assert np.array_equal(conv_v, conv_d)
    a, b = bf16_value(out_v), bf16_value(out_d)
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.abs(b) + 1e-6)


def test_beta_zero_is_decay_only(run):
    """beta = sigmoid(-inf) = 0: S' = diag(e^g) S (decay along k) and o = S'^T q^."""
    si, pool, conv = _decode_case(seed=12)
    H, D = si.workload.heads, si.workload.dim
    si.projected[:, 4 * D + HEAD_DIM:4 * D + HEAD_DIM + H] = BF16_NEG_INF
    W = oracle_weights(si)
    out, _, newpool, err, dg = run(W, si.projected, conv, pool, si.slots, 1, None, diag=True)
    assert err == 0
    for b, slot in enumerate(si.slots):
        for h in range(H):
            g = dg[b, h, 3 * HEAD_DIM:4 * HEAD_DIM]
            qh = dg[b, h, :HEAD_DIM]
            assert dg[b, h, -1] == 0.0
            assert np.ptp(g) > 1e-3                     # a per-channel decay, not a constant
            S = pool[slot, h].astype(np.float64)        # [v, k]
            expect = S * np.exp(g)[None, :]
            np.testing.assert_allclose(newpool[slot, h], expect, rtol=2e-7, atol=1e-12)
            o_exact = expect @ qh
            o = dg[b, h, 4 * HEAD_DIM:5 * HEAD_DIM]
            assert np.all(np.abs(o - o_exact) <= 2.0 ** -8 * np.abs(o_exact) + 1e-12)


def test_bf16_state_storage(run):
    """bf16 state pool: the start state is the bf16 values widened exactly, the
    step carries it in fp64 and each stored state is rounded once to bf16
    (nearest even).  With beta = 0 the stored state is bf16(e^g S) exactly."""
    si, _, conv = _decode_case(seed=13)
    H, D = si.workload.heads, si.workload.dim
    si.projected[:, 4 * D + HEAD_DIM:4 * D + HEAD_DIM + H] = BF16_NEG_INF
    pool16 = si.full_state_pool_bf16()
    out, _, newpool, err, dg = run(oracle_weights(si), si.projected, conv, pool16, si.slots, 1, None,
                                   state_dtype="bf16", diag=True)
    assert err == 0 and newpool.dtype == np.uint16
    for b, slot in enumerate(si.slots):
        for h in range(H):
            g = dg[b, h, 3 * HEAD_DIM:4 * HEAD_DIM]
            S = bf16_value(pool16[slot, h])                          # [v, k], exact
            assert np.array_equal(newpool[slot, h], oracle_np.f64_to_bf16(S * np.exp(g)[None, :]))
    untouched = np.setdiff1d(np.arange(si.workload.pool), si.slots)
    assert np.array_equal(newpool[untouched], pool16[untouched])


def test_delta_property(run):
    """g = 0 (lower bound 0), beta = 1 (+inf logit): S'^T k^ = v up to the
    l2norm eps, i.e. the delta rule stores v exactly under key k^."""
    si, pool, conv = _decode_case(seed=13)
    H, D = si.workload.heads, si.workload.dim
    si.projected[:, 4 * D + HEAD_DIM:4 * D + HEAD_DIM + H] = BF16_POS_INF
    W = oracle_weights(si, gate_lower_bound=0.0)
    _, _, newpool, err, dg = run(W, si.projected, conv, pool, si.slots, 1, None, diag=True)
    assert err == 0
    for b, slot in enumerate(si.slots):
        for h in range(H):
            kh = dg[b, h, HEAD_DIM:2 * HEAD_DIM]
            v = dg[b, h, 2 * HEAD_DIM:3 * HEAD_DIM]
            assert np.all(dg[b, h, 3 * HEAD_DIM:4 * HEAD_DIM] == 0.0)
            assert dg[b, h, -1] == 1.0
            S = pool[slot, h].astype(np.float64)
            delta = 1.0 - kh @ kh                          # l2norm eps leaves |k^| just below 1
            resid = np.abs(newpool[slot, h].astype(np.float64) @ kh - v)
            bound = abs(delta) * np.abs(v - S @ kh) + 2e-6 * (1 + np.abs(v))
            assert np.all(resid <= bound)
            assert np.max(np.abs(S @ kh)) > 1e-2           # the old read-out was not already v


def test_zero_state_closed_form(run):
    """S0 = 0, one token, beta_logit = 0 (beta = 1/2): S' = k^ v^T / 2 and
    o = (k^ . q^) v / 2 -- o comes from the updated state."""
    si, pool, conv = _decode_case(seed=14)
    H, D = si.workload.heads, si.workload.dim
    si.projected[:, 4 * D + HEAD_DIM:4 * D + HEAD_DIM + H] = 0
    pool[si.slots] = 0.0
    W = oracle_weights(si)
    _, _, newpool, err, dg = run(W, si.projected, conv, pool, si.slots, 1, None, diag=True)
    assert err == 0
    for b, slot in enumerate(si.slots):
        for h in range(H):
            qh, kh = dg[b, h, :HEAD_DIM], dg[b, h, HEAD_DIM:2 * HEAD_DIM]
            v = dg[b, h, 2 * HEAD_DIM:3 * HEAD_DIM]
            assert dg[b, h, -1] == 0.5
            np.testing.assert_allclose(newpool[slot, h], 0.5 * np.outer(v, kh), rtol=1e-7, atol=1e-30)
            o_exact = 0.5 * (kh @ qh) * v
            o = dg[b, h, 4 * HEAD_DIM:5 * HEAD_DIM]
            assert np.all(np.abs(o - o_exact) <= 2.0 ** -8 * np.abs(o_exact) + 1e-12)


def test_gate_limits(run):
    """g = lb * sigmoid(e^A (z + dt)): z + dt = 0 gives lb/2; z + dt -> +inf
    gives lb; -> -inf gives 0; otherwise g lies in (lb, 0)."""
    si, pool, conv = _decode_case(seed=15)
    lb = -5.0
    zero_fb = np.zeros_like(si.weights.f_b)
    for dt, expect in [(0.0, lb / 2), (1e4, lb), (-1e4, 0.0)]:
        W = oracle_weights(si, f_b=zero_fb, dt_bias=np.full_like(si.weights.dt_bias, dt),
                           gate_lower_bound=lb)
        *_, err, dg = run(W, si.projected, conv, pool, si.slots, 1, None, diag=True)
        g = dg[:, :, 3 * HEAD_DIM:4 * HEAD_DIM]
        assert err == 0 and np.all(np.abs(g - expect) <= 1e-12)
    W = oracle_weights(si)
    *_, dg = run(W, si.projected, conv, pool, si.slots, 1, None, diag=True)
    g = dg[:, :, 3 * HEAD_DIM:4 * HEAD_DIM]
    assert np.all((g > lb) & (g < 0))


def _zero_gate_weights(si, f_b):
    """A_log = 0 and dt_bias = 0, so that the sigmoid gate is g = lb * sigmoid(z)."""
    return oracle_weights(si, f_b=f_b, A_log=np.zeros_like(si.weights.A_log),
                          dt_bias=np.zeros_like(si.weights.dt_bias), gate_lower_bound=-5.0)


def _gates(run, si, W):
    *_, err, dg = run(W, si.projected, si.full_conv_state(), si.full_state_pool(), si.slots, 1, None, diag=True)
    assert err == 0
    return dg[:, :, 3 * HEAD_DIM:4 * HEAD_DIM].reshape(si.workload.rows, -1)  # [rows, D], channel c = 128 h + i


def _bf16_of_f32(x) -> np.ndarray:
    """torch's fp32 -> bf16 (nearest even) of values exactly representable in fp32, as fp64."""
    x32 = np.asarray(x, dtype=np.float32)
    assert np.array_equal(x32.astype(np.float64), np.asarray(x, dtype=np.float64)), "not exact in fp32"
    return torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()


def test_z_one_hot_rows_pick_f_a(run):
    """z = f_b . f_a over the f_a columns [4D, 4D + 128) of the packed row
    (PreparedKda._operands; K1 "f_b MFMA + lower-bound gate"): with row c of
    f_b the unit vector e_{pi(c)} (pi a permutation per head), z[c] =
    f_a[pi(c)] exactly, so with A_log = dt_bias = 0 the gate is
    g[c] = lb * sigmoid(f_a[pi(c)]) in closed form.  A transposed f_b, another
    column offset for f_a or a dropped product fails this."""
    si, _, _ = _decode_case(heads=2, requests=3, seed=31)
    D, H = si.workload.dim, si.workload.heads
    rng = np.random.default_rng(31)
    perm = np.concatenate([rng.permutation(HEAD_DIM) for _ in range(H)])   # pi(c) for c < D
    f_b = np.zeros((D, HEAD_DIM), np.uint16)
    f_b[np.arange(D), perm] = 0x3F80                                        # bf16 1.0
    g = _gates(run, si, _zero_gate_weights(si, f_b))
    f_a = bf16_value(si.projected[:, 4 * D:4 * D + HEAD_DIM])              # [rows, 128]
    expect = -5.0 / (1.0 + np.exp(-f_a[:, perm]))
    np.testing.assert_allclose(g, expect, rtol=1e-13, atol=0)


def test_z_two_taps_rounded_once_to_bf16(run):
    """Two taps a row, f_b[c, pi(c)] = 1 and f_b[c, pi'(c)] = 1/8, and f_a
    entries of magnitude in [1, 2): z = f_a[pi(c)] + f_a[pi'(c)] / 8 is exact
    in fp32 and is handed on rounded once to bf16 (nearest even; the hand-offs
    of the unfused path, K1 rounding statement).  Most sums are not bf16
    values, so a z kept unrounded, or rounded another way, fails."""
    si, _, _ = _decode_case(heads=2, requests=4, seed=32)
    D, H = si.workload.dim, si.workload.heads
    rng = np.random.default_rng(32)
    fa = rng.uniform(1.0, 2.0, size=(si.workload.rows, HEAD_DIM)) * rng.choice([-1.0, 1.0], size=(si.workload.rows, HEAD_DIM))
    si.projected[:, 4 * D:4 * D + HEAD_DIM] = I_to_bf16(fa)
    perm = np.concatenate([rng.permutation(HEAD_DIM) for _ in range(H)])
    perm2 = np.concatenate([np.roll(perm[h * HEAD_DIM:(h + 1) * HEAD_DIM], 1) for h in range(H)])
    f_b = np.zeros((D, HEAD_DIM), np.uint16)
    f_b[np.arange(D), perm] = 0x3F80                                        # 1.0
    f_b[np.arange(D), perm2] = 0x3E00                                       # 0.125
    g = _gates(run, si, _zero_gate_weights(si, f_b))
    f_a = bf16_value(si.projected[:, 4 * D:4 * D + HEAD_DIM])
    z_exact = f_a[:, perm] + f_a[:, perm2] / 8.0
    z = _bf16_of_f32(z_exact)
    assert np.mean(z != z_exact) > 0.5                                      # the rounding is exercised
    np.testing.assert_allclose(g, -5.0 / (1.0 + np.exp(-z)), rtol=1e-13, atol=0)


def test_z_full_row_sum(run):
    """Every tap nonzero: f_b[c, j] = 2^-(c mod 8) for all j and integer f_a
    in [-8, 8], so z[c] = 2^-(c mod 8) * sum_j f_a[j] exactly before the bf16
    rounding: the whole 128-term contraction is summed."""
    si, _, _ = _decode_case(heads=1, requests=3, seed=33)
    D = si.workload.dim
    rng = np.random.default_rng(33)
    fa = rng.integers(-8, 9, size=(si.workload.rows, HEAD_DIM)).astype(np.float64)
    si.projected[:, 4 * D:4 * D + HEAD_DIM] = I_to_bf16(fa)
    scale = 2.0 ** -(np.arange(D) % 8)
    f_b = np.repeat(I_to_bf16(scale)[:, None], HEAD_DIM, axis=1)
    g = _gates(run, si, _zero_gate_weights(si, f_b))
    z = _bf16_of_f32(fa.sum(axis=1)[:, None] * scale[None, :])
    np.testing.assert_allclose(g, -5.0 / (1.0 + np.exp(-z)), rtol=1e-13, atol=0)


def test_gate_limits_softplus_form(run):
    """gate_mode 1, g = max(-e^A softplus(z + dt), lb): z + dt = 0 gives
    -e^A ln 2 (per head); z + dt -> +inf is clamped to lb; -> -inf gives 0;
    otherwise g lies in [lb, 0)."""
    si, pool, conv = _decode_case(seed=17)
    lb = -5.0
    zero_fb = np.zeros_like(si.weights.f_b)
    A = si.weights.A_log.astype(np.float64)
    for dt, expect in [(0.0, -np.exp(A) * np.log(2.0)), (1e4, np.full(A.shape, lb)), (-1e4, np.zeros(A.shape))]:
        W = oracle_weights(si, f_b=zero_fb, dt_bias=np.full_like(si.weights.dt_bias, dt), gate_lower_bound=lb)
        *_, err, dg = run(W, si.projected, conv, pool, si.slots, 1, None, gate_mode=1, diag=True)
        g = dg[:, :, 3 * HEAD_DIM:4 * HEAD_DIM]                       # [rows, H, 128]
        assert err == 0 and np.all(np.abs(g - expect[None, :, None]) <= 1e-12)
    *_, dg = run(oracle_weights(si, gate_lower_bound=lb), si.projected, conv, pool, si.slots, 1, None,
                 gate_mode=1, diag=True)
    g = dg[:, :, 3 * HEAD_DIM:4 * HEAD_DIM]
    assert np.all((g >= lb) & (g < 0))


def test_l2norm_and_q_scale(run):
    si, pool, conv = _decode_case(seed=16)
    *_, dg = run(oracle_weights(si), si.projected, conv, pool, si.slots, 1, None, diag=True)
    for row in dg.reshape(-1, dg.shape[-1]):
        qh, kh = row[:HEAD_DIM], row[HEAD_DIM:2 * HEAD_DIM]
        assert abs(np.linalg.norm(kh) - 1.0) < 1e-6
        assert abs(np.linalg.norm(qh) - HEAD_DIM ** -0.5) < 1e-6


# ------------------------------------------------------------------------ conv

@pytest.mark.parametrize("dim_first", [True, False])
def test_identity_and_shifted_conv(run, dim_first):
    """Taps (0,0,0,1), no activation: the conv passes the current token
    through; taps (0,0,1,0): it returns the previous token (the window's
    newest entry for token 0).  The window after token t holds the last W-1
    inputs, oldest first, in slots[r, t]."""
    R, L, H = 2, 3, 1
    si = case(heads=H, requests=R, L=L, pool=8, seed=17, accepted=[1, 3])
    D = si.workload.dim
    C = 3 * D
    for taps, shift in [((0, 0, 0, 1), 0), ((0, 0, 1, 0), 1)]:
        cw = np.zeros_like(si.weights.conv_w)
        cw[:, 0, :] = np.array([0x3F80 if t else 0 for t in taps], dtype=np.uint16)
        W = oracle_weights(si, conv_w=cw)
        conv = si.full_conv_state(dim_first)
        out, newconv, _, err, dg = run(W, si.projected, conv, si.full_state_pool(), si.slots, L,
                                       si.accepted, dim_first=dim_first, act="none", diag=True)
        assert err == 0
        win = conv if dim_first else conv.transpose(0, 2, 1)
        nwin = newconv if dim_first else newconv.transpose(0, 2, 1)
        slots = si.slots.reshape(R, L)
        for r in range(R):
            start = slots[r, si.accepted[r] - 1]
            seq = np.concatenate([win[start].T, si.projected[r * L:(r + 1) * L, :C]], axis=0)
            for t in range(L):
                cur = seq[2 + t + 1 - shift]               # x_t (shift 0) or x_{t-1} (shift 1)
                v = dg[r * L + t, 0, 2 * HEAD_DIM:3 * HEAD_DIM]
                assert np.array_equal(v, bf16_value(cur[2 * D:2 * D + HEAD_DIM]))
                assert np.array_equal(nwin[slots[r, t]].T, seq[t + 1:t + 4])


def test_silu_activation(run):
    si, pool, conv = _decode_case(heads=1, seed=18)
    cw = np.zeros_like(si.weights.conv_w)
    cw[:, 0, 3] = 0x3F80
    W = oracle_weights(si, conv_w=cw)
    *_, dg = run(W, si.projected, conv, pool, si.slots, 1, None, diag=True)
    D = si.workload.dim
    x = bf16_value(si.projected[:, 2 * D:2 * D + HEAD_DIM])
    silu = x / (1.0 + np.exp(-x))
    v = dg[:, 0, 2 * HEAD_DIM:3 * HEAD_DIM]
    assert np.all(np.abs(v - silu) <= 2.0 ** -8 * np.abs(silu) + 1e-30)


def test_conv_bias_and_layouts_agree(run):
    si = case(heads=2, requests=2, L=2, pool=6, seed=19, with_bias=True)
    W = oracle_weights(si)
    a = run(W, si.projected, si.full_conv_state(True), si.full_state_pool(), si.slots, 2, si.accepted,
            dim_first=True)
    b = run(W, si.projected, si.full_conv_state(False), si.full_state_pool(), si.slots, 2, si.accepted,
            dim_first=False)
    assert np.array_equal(a[0], b[0])
    assert np.array_equal(a[1], b[1].transpose(0, 2, 1))
    assert np.array_equal(a[2].view(np.uint32), b[2].view(np.uint32))
    nb = run(oracle_weights(si, bias=None), si.projected, si.full_conv_state(True), si.full_state_pool(),
             si.slots, 2, si.accepted)
    assert not np.array_equal(a[0], nb[0])


# ------------------------------------------------------------------------ norm

def test_unit_rms(run):
    """o_norm = 1 and out-gate = +inf (sigmoid = 1): each head's output row has
    RMS sqrt(ms / (ms + eps)), ms = mean(o^2) of the bf16 o."""
    si, pool, conv = _decode_case(seed=20)
    D, H = si.workload.dim, si.workload.heads
    si.projected[:, 3 * D:4 * D] = BF16_POS_INF
    out, *_, dg = run(oracle_weights(si), si.projected, conv, pool, si.slots, 1, None, diag=True)
    y = bf16_value(out)
    for b in range(si.workload.rows):
        for h in range(H):
            o = dg[b, h, 4 * HEAD_DIM:5 * HEAD_DIM]
            ms = np.mean(o * o)
            rms = np.sqrt(np.mean(y[b, h * HEAD_DIM:(h + 1) * HEAD_DIM] ** 2))
            assert abs(rms - np.sqrt(ms / (ms + 1e-6))) < 4e-3
            assert np.all(np.sign(y[b, h * HEAD_DIM:(h + 1) * HEAD_DIM]) == np.sign(o))


def test_output_gate_and_weight(run):
    """out-gate = -inf gives exactly zero output; o_norm scales channel-wise."""
    si, pool, conv = _decode_case(seed=22)
    D = si.workload.dim
    p = si.projected.copy()
    p[:, 3 * D:4 * D] = BF16_NEG_INF
    out, *_ = run(oracle_weights(si), p, conv, pool, si.slots, 1, None)
    assert np.all(bf16_value(out) == 0.0)
    si.projected[:, 3 * D:4 * D] = BF16_POS_INF
    base, *_ = run(oracle_weights(si), si.projected, conv, pool, si.slots, 1, None)
    wgt = np.ones(HEAD_DIM, np.float32)
    wgt[::2] = 2.0
    scaled, *_ = run(oracle_weights(si, o_norm=wgt), si.projected, conv, pool, si.slots, 1, None)
    assert np.array_equal(bf16_value(scaled), bf16_value(base) * np.tile(wgt, si.workload.heads))


# --------------------------------------------------------------- slot indexing

def test_written_slots_padding_and_errors(run):
    """Only slots[r, t] are written; a request whose first slot is -1 is
    padding (zero output, caches untouched); accepted outside 1..L or a slot
    outside the pool sets the error bit and skips that request."""
    R, L = 4, 2
    si = case(heads=1, requests=R, L=L, pool=16, seed=23, accepted=[2, 1, 1, 2])
    slots = si.slots.reshape(R, L).copy()
    slots[1, 0] = -1                # padding request 1
    acc = si.accepted.copy()
    acc[2] = 0                      # bad accepted -> request 2 skipped
    slots[3, 1] = 16                # slot out of range -> request 3 skipped
    pool, conv = si.full_state_pool(), si.full_conv_state()
    for s in slots.reshape(-1):
        if 0 <= s < 16:
            pool[s] = 0.01
            conv[s] = 0x3F80
    out, nconv, npool, err = run(oracle_weights(si), si.projected, conv, pool, slots.reshape(-1), L, acc)
    assert err == oracle.ERR_ACCEPTED | oracle.ERR_SLOT
    changed = {s for s in range(16) if not np.array_equal(npool[s].view(np.uint32), pool[s].view(np.uint32))}
    assert changed == set(int(s) for s in slots[0])
    changed_conv = {s for s in range(16) if not np.array_equal(nconv[s], conv[s])}
    assert changed_conv == set(int(s) for s in slots[0])
    assert np.all(out[2:] == 0) and np.any(out[:2] != 0)   # rows of requests 1..3 stay zero


def test_column_split_per_head(run):
    """The packed row: beta logits at 4D + 128 + h, one per head; q and k of
    head h at blocks 0 and 1 (PreparedKda._operands column split)."""
    si, pool, conv = _decode_case(heads=3, seed=24)
    D, H = si.workload.dim, si.workload.heads
    logits = [BF16_NEG_INF, BF16_POS_INF, np.uint16(0)]
    for h in range(H):
        si.projected[:, 4 * D + HEAD_DIM + h] = logits[h]
    cw = np.zeros_like(si.weights.conv_w)
    cw[:, 0, 3] = 0x3F80                                   # identity taps
    *_, dg = run(oracle_weights(si, conv_w=cw), si.projected, conv, pool, si.slots, 1, None, act="none", diag=True)
    assert np.array_equal(dg[:, :, -1], np.tile([0.0, 1.0, 0.5], (si.workload.rows, 1)))
    for h in range(H):
        xq = bf16_value(si.projected[:, head_cols(D, 0, h)])
        xk = bf16_value(si.projected[:, head_cols(D, 1, h)])
        qh, kh = dg[:, h, :HEAD_DIM], dg[:, h, HEAD_DIM:2 * HEAD_DIM]
        np.testing.assert_allclose(qh, xq / np.linalg.norm(xq, axis=1, keepdims=True) * HEAD_DIM ** -0.5,
                                   rtol=1e-6, atol=1e-9)
        np.testing.assert_allclose(kh, xk / np.linalg.norm(xk, axis=1, keepdims=True), rtol=1e-6, atol=1e-9)


def test_padding_alone_sets_no_error(run):
    """A padding request (slot -1 first) is not an error: no error bits, zero
    output rows, no cache written; the other requests run normally."""
    R, L = 3, 2
    si = case(heads=1, requests=R, L=L, pool=10, seed=25, accepted=[1, 2, 2])
    slots = si.slots.reshape(R, L).copy()
    slots[1, :] = -1
    pool, conv = si.full_state_pool(), si.full_conv_state()
    out, nconv, npool, err = run(oracle_weights(si), si.projected, conv, pool, slots.reshape(-1), L, si.accepted)
    assert err == 0
    assert np.all(out[L:2 * L] == 0) and np.all(out[:L] != 0) and np.all(out[2 * L:] != 0)
    written = {s for s in range(10) if not np.array_equal(npool[s].view(np.uint32), pool[s].view(np.uint32))}
    assert written == set(int(s) for s in slots[[0, 2]].reshape(-1))


def test_c_matches_numpy_on_random_shapes():
    rng = np.random.default_rng(5)
    for trial in range(6):
        H = int(rng.integers(1, 3))
        L = int(rng.integers(1, 4))
        Wd = int(rng.integers(2, 5))
        R = int(rng.integers(1, 4))
        si = case(heads=H, requests=R, L=L, pool=R * L + 2, width=Wd, seed=100 + trial,
                  with_bias=bool(trial % 2), verify=L > 1 or trial % 3 == 0)
        W = oracle_weights(si)
        dim_first = bool(trial % 2 == 0)
        args = (W, si.projected, si.full_conv_state(dim_first), si.full_state_pool(), si.slots, L, si.accepted)
        gm = trial % 2  # both gate forms
        a = oracle.step(*args, dim_first=dim_first, gate_mode=gm, diag=True)
        b = oracle_np.step(*args, dim_first=dim_first, gate_mode=gm, diag=True)
        assert a[3] == b[3] == 0
        da, db = bf16_value(a[0]), bf16_value(b[0])
        assert np.mean(a[0] != b[0]) < 0.01
        assert np.all(np.abs(da - db) <= 2.0 ** -7 * np.abs(db) + 1e-6)
        assert np.array_equal(a[1], b[1])
        np.testing.assert_allclose(np.nan_to_num(a[2]), np.nan_to_num(b[2]), rtol=0, atol=1e-7)
        np.testing.assert_allclose(a[4], b[4], rtol=1e-9, atol=1e-9)
        # the bf16 state pool: the two oracles' fp64 states round to the same bf16
        # but where one sits within fp64 noise of a rounding boundary
        pool16 = si.full_state_pool_bf16()
        args16 = (W, si.projected, si.full_conv_state(dim_first), pool16, si.slots, L, si.accepted)
        a16 = oracle.step(*args16, dim_first=dim_first, gate_mode=gm, state_dtype="bf16")
        b16 = oracle_np.step(*args16, dim_first=dim_first, gate_mode=gm, state_dtype="bf16")
        assert a16[3] == b16[3] == 0
        fin = ~np.isnan(bf16_value(b16[2]))
        assert np.array_equal(np.isnan(bf16_value(a16[2])), ~fin)
        assert np.mean(a16[2][fin] != b16[2][fin]) < 1e-4


def test_threaded_oracle_equals_serial():
    """The C oracle's OpenMP path over (request, head) tasks gives the same bits
    as one thread: every task runs its steps in the same order either way."""
    n = max(2, oracle.max_threads())
    for trial, (H, R, L) in enumerate([(3, 4, 1), (2, 5, 3), (4, 3, 8)]):
        si = case(heads=H, requests=R, L=L, pool=R * L + 3, seed=200 + trial, with_bias=bool(trial % 2),
                  verify=L > 1)
        W = oracle_weights(si)
        for sd in ("f32", "bf16"):
            pool = si.full_state_pool_bf16() if sd == "bf16" else si.full_state_pool()
            args = (W, si.projected, si.full_conv_state(), pool, si.slots, L, si.accepted)
            a = oracle.step(*args, state_dtype=sd, diag=True, threads=1)
            b = oracle.step(*args, state_dtype=sd, diag=True, threads=n)
            assert a[3] == b[3] == 0
            assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
            assert np.array_equal(a[2].view(np.uint8), b[2].view(np.uint8))
            assert np.array_equal(a[4].view(np.uint64), b[4].view(np.uint64))
