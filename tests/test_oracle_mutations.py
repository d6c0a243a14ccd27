"""The pins catch plausible mistakes: each case plants one mistake in a copy of
the C oracle (on the CPU), builds it, and runs the pin suite against it with
the C-versus-NumPy cross-check switched off, so only the pins can notice.
Every planted mistake must make at least one pin fail.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kda_oracle.c")

# (name, original text, planted mistake)
MUTATIONS = [
    ("delta_sign", "u[v] = vr[v] - s;", "u[v] = vr[v] + s;"),
    ("state_transposed", "S[k * HEAD_DIM + v] = (double)src[v * HEAD_DIM + k];",
     "S[k * HEAD_DIM + v] = (double)src[k * HEAD_DIM + v];"),
    ("decay_on_v_axis", "for (int v = 0; v < HEAD_DIM; ++v) S[k * HEAD_DIM + v] *= decay;",
     "for (int v = 0; v < HEAD_DIM; ++v) S[k * HEAD_DIM + v] *= exp(gr[v]);"),
    ("readout_with_k", "for (int k = 0; k < HEAD_DIM; ++k) s += S[k * HEAD_DIM + v] * qh[k];",
     "for (int k = 0; k < HEAD_DIM; ++k) s += S[k * HEAD_DIM + v] * kh[k];"),
    ("readout_before_update", "for (int k = 0; k < HEAD_DIM; ++k) s += S[k * HEAD_DIM + v] * qh[k];",
     "for (int k = 0; k < HEAD_DIM; ++k) s += (S[k * HEAD_DIM + v] - bt * kh[k] * u[v]) * qh[k];"),
    ("beta_dropped", "S[k * HEAD_DIM + v] += bt * kh[k] * u[v];", "S[k * HEAD_DIM + v] += kh[k] * u[v];"),
    ("tap_order_reversed", "y += bf16_value(conv_w[c * W + j]) * x;",
     "y += bf16_value(conv_w[c * W + (W - 1 - j)]) * x;"),
    ("window_newest_first", "if (SL > 0) window[SL - 1] = x_t;", "if (SL > 0) window[0] = x_t;"),
    ("start_slot_first", "start_of[r] = slots[row0 + acc - 1];", "start_of[r] = slots[row0];"),
    ("window_slot_first", "const int64_t dst = a->slots[row0 + t];", "const int64_t dst = a->slots[row0];"),
    ("q_scale_dropped", "qh[i] = qr[i] * qn * q_scale;", "qh[i] = qr[i] * qn;"),
    ("gate_dt_sign", "(z + (double)a->dt_bias[c])", "(z - (double)a->dt_bias[c])"),
    ("gate_bound_ignored", "(double)lb * sigmoid(", "-1.0 * sigmoid("),
    ("softplus_gate_unclamped", "softplus(z + a->dt_bias[c]), (double)lb)", "softplus(z + a->dt_bias[c]), -1e300)"),
    ("softplus_gate_no_scale", "fmax(-exp((double)a->A_log[h]) * softplus(", "fmax(-1.0 * softplus("),
    ("bf16_state_truncated", "dst16[v * HEAD_DIM + k] = bf16_round(S[k * HEAD_DIM + v]);",
     "dst16[v * HEAD_DIM + k] = (uint16_t)(bf16_round(S[k * HEAD_DIM + v]) & 0xFFFEu);"),
    ("bf16_state_transposed", "bf16_value(src16[v * HEAD_DIM + k])", "bf16_value(src16[k * HEAD_DIM + v])"),
    ("gate_one_token", "const double *gr = b->g + t * HEAD_DIM;", "const double *gr = b->g;"),
    ("rms_sum_not_mean", "ms /= HEAD_DIM;", "ms /= 1;"),
    ("rms_eps_dropped", "const double rstd = 1.0 / sqrt(ms + a->eps);", "const double rstd = 1.0 / sqrt(ms);"),
    ("silu_dropped", "if (a->act) y = y * sigmoid(y);", "if (a->act) y = y;"),
    ("bias_ignored", "double y = bias ? bf16_value(bias[c]) : 0.0;", "double y = 0.0;"),
    ("beta_of_head0", "b->beta[t] = sigmoid(bf16_value(prow[4 * D + HEAD_DIM + h]));",
     "b->beta[t] = sigmoid(bf16_value(prow[4 * D + HEAD_DIM]));"),
    ("out_gate_dropped", "* sigmoid(bf16_value(gate[v]));", ";"),
    ("padding_not_detected", "if (slots[row0] == -1) {", "if (0) {"),
    ("fb_transposed", "bf16_value(f_b[c * HEAD_DIM + j])", "bf16_value(f_b[j * D + c])"),
    ("fa_offset_outgate", "bf16_value(prow[4 * D + j])", "bf16_value(prow[3 * D + j])"),
    ("fa_offset_shifted", "bf16_value(prow[4 * D + j])", "bf16_value(prow[4 * D + (j + 1) % HEAD_DIM])"),
    ("z_unrounded", "z = bf16_rounded(z);", "z = z + 0.0;"),
    ("no_round_to_even", "r = nearbyint(ax / quantum) * quantum;", "r = floor(ax / quantum + 0.5) * quantum;"),
]


@pytest.fixture(scope="module")
def source():
    return open(SRC).read()


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(source, tmp_path, name, old, new):
    assert source.count(old) == 1, f"mutation site for {name} not unique"
    mutated = tmp_path / "kda_oracle_mut.c"
    mutated.write_text(source.replace(old, new))
    lib = tmp_path / "libkda_oracle_mut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
                    "-o", str(lib), str(mutated), "-lm"], check=True)
    env = dict(os.environ, KDA_ORACLE_LIB_OVERRIDE=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                          "-k", "not np and not c_matches_numpy"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"no pin caught the planted mistake {name}:\n{res.stdout[-2000:]}"
