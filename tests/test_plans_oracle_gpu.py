"""Launch plans against the oracle (not only against the direct calls).

A step plan (kda_plan_*: one kda_step recorded as a CUDA graph on fixed
buffers) is launched three times, the third time on new projected rows
written into its buffer; after every launch its out, conv windows and states
are compared with the oracle applied to the same buffers in the same order
(the PreparedKda page's prepare_caches / run: a prepared executable run on
the caches step after step).  The layer plan (in_proj -> step -> o_proj) is
compared stage by stage with the oracles on the inputs each stage consumed,
and end to end with the oracles chained on the host."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_decode_03_gb300 as kda
import oracle
from linear_attention_decode_03_gb300 import inputs as I
from oracle import linear as OL
from tests import gpu_harness as G
from tests.helpers import case

pytestmark = pytest.mark.gpu

HIDDEN = 7168


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.load_library()


def _state_close(gpu: np.ndarray, ref: np.ndarray):
    """States of slots that hold a sentinel on both sides compare by bits; the
    rest within the state tolerances."""
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(gpu), nan)
    G.assert_state_close(gpu[~nan], ref[~nan])


@pytest.mark.parametrize("v_split", [1, 2])
@pytest.mark.parametrize("L", [1, 4])
def test_plan_replays_match_oracle(L, v_split):
    # v_split = 2: the recorded launch is a cluster launch of two CTAs a (request, head)
    si = case(heads=2, requests=4, L=L, pool=4 * L + 3, seed=180 + L, verify=L > 1)
    W = oracle.Weights(**si.weights.as_dict())
    ds = G.DeviceStep(si, v_split=v_split)
    plan = ds.prep.plan(ds.projected, ds.out, caches=(ds.conv, ds.state), slots=ds.slots, accepted=ds.accepted)
    conv, pool = si.full_conv_state(), si.full_state_pool()
    proj = si.projected.copy()
    rng = np.random.default_rng(L)
    for launch in range(3):
        if launch == 2:  # new inputs into the plan's buffer
            proj = I.to_bf16_bits(rng.normal(0.0, 1.0, size=proj.shape).astype(np.float32))
            ds.projected.copy_(G.bf16_np_to_torch(proj, ds.device))
        plan.launch()
        assert ds.prep.check() == 0
        out_ref, conv, pool, err = oracle.step(W, proj, conv, pool, si.slots, L, si.accepted)
        assert err == 0
        G.assert_out_close(G.torch_bf16_to_np(ds.out), out_ref)
        assert np.array_equal(G.torch_bf16_to_np(ds.conv), conv)
        _state_close(ds.state.cpu().numpy(), pool)
    plan.close()
    ds.close()


def test_bf16_decode_plan_replays_match_oracle():
    # bf16 state pool, decode: the recorded launch is the two-row kernel (five rows, so its
    # last CTA serves one).  Each launch is compared with the oracle applied to the caches
    # the GPU held before it: two bf16 pools rounded from fp32 and fp64 may drift by more
    # than one step when each is chained on its own.
    si = case(heads=2, requests=5, L=1, pool=9, seed=187)
    W = oracle.Weights(**si.weights.as_dict())
    ds = G.DeviceStep(si, state_dtype="bf16")
    plan = ds.prep.plan(ds.projected, ds.out, caches=(ds.conv, ds.state), slots=ds.slots, accepted=None)
    proj = si.projected.copy()
    rng = np.random.default_rng(187)
    written = np.unique(si.slots)
    rest = np.setdiff1d(np.arange(si.workload.pool), written)
    for launch in range(3):
        if launch == 2:  # new inputs into the plan's buffer
            proj = I.to_bf16_bits(rng.normal(0.0, 1.0, size=proj.shape).astype(np.float32))
            ds.projected.copy_(G.bf16_np_to_torch(proj, ds.device))
        conv_in, pool_in = G.torch_bf16_to_np(ds.conv), G.torch_bf16_to_np(ds.state)
        plan.launch()
        assert ds.prep.check() == 0
        out_ref, conv_ref, pool_ref, err = oracle.step(W, proj, conv_in, pool_in, si.slots, 1, None,
                                                       state_dtype="bf16")
        assert err == 0
        G.assert_out_close(G.torch_bf16_to_np(ds.out), out_ref)
        assert np.array_equal(G.torch_bf16_to_np(ds.conv), conv_ref)
        st = G.torch_bf16_to_np(ds.state)
        G.assert_state_close_bf16(st[written], pool_ref[written])
        assert np.array_equal(st[rest], pool_ref[rest])
    plan.close()
    ds.close()


def _linear_close(y_bits, x_bits, w_bits):
    """kda_linear's criterion: one bf16 step of the correctly rounded product
    plus the fp32 accumulation's share, 2^-14 sum |x_k w_k|."""
    ref = OL.linear(x_bits, w_bits)
    g, r = G.bf16_value(y_bits), G.bf16_value(ref)
    bound = np.maximum(np.abs(r), 1e-30) * 2.0 ** -7 + 2.0 ** -14 * OL.abs_products(x_bits, w_bits)
    assert np.all(np.abs(g - r) <= bound)


@pytest.mark.parametrize("w", [I.WORKLOADS["tiny_decode"],
                               I.Workload("verify_80_rows_o", heads=2, requests=20, L=4, pool=96, verify=True,
                                          seed=3080)], ids=lambda w: w.name)
def test_layer_plan_matches_oracle(w):
    si = I.make_step_inputs(w)
    W = oracle.Weights(**si.weights.as_dict())
    ds = G.DeviceStep(si)
    rng = np.random.default_rng(w.seed)
    xb = I.to_bf16_bits(rng.normal(0.0, 1.0, size=(w.rows, HIDDEN)).astype(np.float32))
    wib = I.to_bf16_bits(rng.normal(0.0, 0.02, size=(w.pitch, HIDDEN)).astype(np.float32))
    wob = I.to_bf16_bits(rng.normal(0.0, 0.05, size=(HIDDEN, w.dim)).astype(np.float32))
    x, w_in, w_o = (G.bf16_np_to_torch(a, ds.device) for a in (xb, wib, wob))
    proj = torch.empty((w.rows, w.pitch), dtype=torch.bfloat16, device=ds.device)
    core = torch.empty((w.rows, w.dim), dtype=torch.bfloat16, device=ds.device)
    y = torch.empty((w.rows, HIDDEN), dtype=torch.bfloat16, device=ds.device)
    plan = ds.prep.layer_plan(x, w_in, proj, core, w_o, y, caches=(ds.conv, ds.state), slots=ds.slots,
                              accepted=ds.accepted, pdl=True)
    plan.launch()
    torch.cuda.synchronize()
    assert ds.prep.check() == 0 and kda.kda_linear_check() == 0
    proj_g, core_g, y_g = (G.torch_bf16_to_np(t) for t in (proj, core, y))
    # stage by stage, each against the oracle on the inputs the GPU stage consumed
    _linear_close(proj_g, xb, wib)
    out_ref, conv_ref, pool_ref, err = oracle.step(W, proj_g, si.full_conv_state(), si.full_state_pool(), si.slots,
                                                   w.L, si.accepted)
    assert err == 0
    G.assert_out_close(core_g, out_ref)
    assert np.array_equal(G.torch_bf16_to_np(ds.conv), conv_ref)
    _state_close(ds.state.cpu().numpy(), pool_ref)
    _linear_close(y_g, core_g, wob)
    # end to end: the oracles chained on the host (in_proj -> step -> o_proj); y within the
    # product's own criterion plus the core's tolerance carried through o_proj
    p_ref = OL.linear(xb, wib)
    c_ref, *_ = oracle.step(W, p_ref, si.full_conv_state(), si.full_state_pool(), si.slots, w.L, si.accepted)
    y_ref = OL.linear(c_ref, wob)
    g, r = G.bf16_value(y_g), G.bf16_value(y_ref)
    carried = (G.OUT_ATOL + G.OUT_RTOL * np.abs(G.bf16_value(c_ref))) @ np.abs(G.bf16_value(wob)).T
    bound = np.abs(r) * 2.0 ** -7 + 2.0 ** -14 * OL.abs_products(c_ref, wob) + carried
    assert np.all(np.abs(g - r) <= bound)
    plan.close()
    ds.close()
