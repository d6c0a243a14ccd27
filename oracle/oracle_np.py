"""NumPy restatement of the KDA decode / spec-verify core (fp64).

TEST INFRASTRUCTURE ONLY: a second, independent oracle written with NumPy
array operations, used to cross-check the C oracle (``kda_oracle.c``) on small
inputs.  It imports nothing from the C oracle or from the CUDA library.

Definition sources: the vLLM documentation pages
"vllm.models.kimi_k3.amd.specialized_decode.mono.attention.kda" (K1 kda_pre,
module docstring: conv update, f_b . f_a with the lower-bound gate, l2norm,
the recurrence with one state written per token, gated RMSNorm over the
head's 128; bf16 rounding at every hand-off of the unfused path) and
"vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.prepared"
(PreparedKda._operands column split; __init__ scalars and fp32 o_norm).
The readings taken where the pages are silent are the C oracle's, listed in
its header.
"""
from __future__ import annotations

import numpy as np

HEAD_DIM = 128
ERR_SLOT = 1
ERR_ACCEPTED = 2


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """fp64 -> nearest bf16 bit pattern, ties to even, rounded once from fp64."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    _, e = np.frexp(ax)                       # ax = m 2^e, m in [0.5, 1)
    qexp = np.maximum(e.astype(np.int64) - 8, -133)
    quantum = np.ldexp(np.ones_like(ax), qexp)
    with np.errstate(over="ignore", invalid="ignore"):
        r = np.rint(ax / quantum) * quantum       # rint: round half to even
    r = np.where((ax == 0) | np.isinf(ax), ax, r)
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    r = np.copysign(r, x)
    bits = (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    return np.where(np.isnan(x), np.uint16(0x7FC0), bits).astype(np.uint16)


def _bf16_round_value(x) -> np.ndarray:
    return bf16_to_f64(f64_to_bf16(x))


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def step(w, projected, conv_state, state_pool, slots, L, accepted=None, *, dim_first=True,
         act="silu", gate_mode=0, state_dtype="f32", diag=False):
    """Same contract as ``oracle.step`` (the C oracle); inputs are not modified."""
    projected = np.asarray(projected, dtype=np.uint16)
    rows, pitch = projected.shape
    H = w.heads
    D = HEAD_DIM * H
    C = 3 * D
    W = int(w.conv_w.shape[-1])
    SL = W - 1
    if rows % L or (accepted is None and L != 1) or pitch < 4 * D + HEAD_DIM + H:
        raise ValueError("arguments make the step undefined")
    conv = np.array(conv_state, dtype=np.uint16, copy=True)
    # work on a [pool, C, SL] view whatever the storage order
    conv_v = conv if dim_first else conv.transpose(0, 2, 1)
    bf16_state = state_dtype == "bf16"
    pool_arr = np.array(state_pool, dtype=np.uint16 if bf16_state else np.float32, copy=True)
    npool = pool_arr.shape[0]
    slots = np.asarray(slots, dtype=np.int64).reshape(-1)
    out = np.zeros((rows, D), dtype=np.uint16)
    dg = np.zeros((rows, H, 5 * HEAD_DIM + 1)) if diag else None
    err = 0

    taps = bf16_to_f64(w.conv_w).reshape(C, W)
    bias = np.zeros(C) if w.bias is None else bf16_to_f64(w.bias)
    f_b = bf16_to_f64(w.f_b)                       # [D, 128]
    A = np.asarray(w.A_log, dtype=np.float64)
    dt = np.asarray(w.dt_bias, dtype=np.float64)
    onorm = np.asarray(w.o_norm, dtype=np.float64)
    lb = float(np.float32(w.gate_lower_bound))
    eps = float(np.float32(w.eps))

    for r in range(rows // L):
        rws = np.arange(r * L, r * L + L)
        if slots[rws[0]] == -1:                   # padding request
            continue                              # out rows stay zero
        a = 1 if accepted is None else int(accepted[r])
        if not 1 <= a <= L:
            err |= ERR_ACCEPTED
            continue
        req_slots = slots[rws]
        if np.any((req_slots < 0) | (req_slots >= npool)):
            err |= ERR_SLOT
            continue
        start = req_slots[a - 1]
        P = bf16_to_f64(projected[rws])           # [L, pitch]

        # conv over the L tokens: sequence = window (oldest first) then the tokens
        seq = np.concatenate([bf16_to_f64(conv_v[start]).T, P[:, :C]], axis=0)  # [SL + L, C]
        y = np.stack([(seq[t:t + W] * taps.T).sum(axis=0) for t in range(L)]) + bias  # [L, C]
        if act == "silu":
            y = y * _sigmoid(y)
        qkv = _bf16_round_value(y)
        for t in range(L):
            conv_v[req_slots[t]] = f64_to_bf16(seq[t + 1:t + 1 + SL].T)

        z = _bf16_round_value(P[:, 4 * D:4 * D + HEAD_DIM] @ f_b.T)          # [L, D]
        if gate_mode == 0:
            g = lb * _sigmoid(np.repeat(np.exp(A), HEAD_DIM) * (z + dt))      # [L, D]
        else:
            g = np.maximum(-np.repeat(np.exp(A), HEAD_DIM) * np.logaddexp(0.0, z + dt), lb)
        beta = _sigmoid(P[:, 4 * D + HEAD_DIM:4 * D + HEAD_DIM + H])          # [L, H]
        gate = P[:, 3 * D:4 * D]

        for h in range(H):
            cs = slice(h * HEAD_DIM, (h + 1) * HEAD_DIM)
            S = (bf16_to_f64(pool_arr[start, h]) if bf16_state else pool_arr[start, h].astype(np.float64)).T  # S[k, v]
            for t in range(L):
                q = qkv[t, 0 * D:1 * D][cs]
                k = qkv[t, 1 * D:2 * D][cs]
                v = qkv[t, 2 * D:3 * D][cs]
                qh = q / np.sqrt(q @ q + 1e-6) * HEAD_DIM ** -0.5
                kh = k / np.sqrt(k @ k + 1e-6)
                S = np.exp(g[t, cs])[:, None] * S
                u = v - S.T @ kh
                S = S + beta[t, h] * np.outer(kh, u)
                o = _bf16_round_value(S.T @ qh)
                pool_arr[req_slots[t], h] = f64_to_bf16(S.T) if bf16_state else S.T.astype(np.float32)
                rstd = 1.0 / np.sqrt(np.mean(o * o) + eps)
                out[rws[t], cs] = f64_to_bf16(o * rstd * onorm * _sigmoid(gate[t, cs]))
                if diag:
                    dg[rws[t], h] = np.concatenate([qh, kh, v, g[t, cs], o, [beta[t, h]]])
    if diag:
        return out, conv, pool_arr, err, dg
    return out, conv, pool_arr, err
