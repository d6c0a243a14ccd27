"""The layer plan (in_proj -> KDA step -> o_proj recorded as one CUDA graph,
with and without programmatic dependent launch) against the same three calls
made one after another: every output, intermediate and cache bit-identical
(the kernels are deterministic, so the composition must not change a bit),
on a 1-row decode, a 24-row verify (the 64-row projection tiles) and an 80-row
verify (tcgen05 projection tiles); and a plan replayed on new x."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_decode_03_gb300 as kda
from linear_attention_decode_03_gb300 import inputs as I
from tests import gpu_harness as G

pytestmark = pytest.mark.gpu

HIDDEN = 7168


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.load_library()


def _bits(t):
    return t.view(torch.int16)


def _rand(gen, shape, scale):
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16).cuda()


WORKLOADS = [
    I.WORKLOADS["tiny_decode"],
    I.Workload("verify_24_rows", heads=2, requests=6, L=4, pool=32, verify=True, seed=2024),
    I.Workload("verify_80_rows", heads=2, requests=20, L=4, pool=96, verify=True, seed=2080),
]


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_layer_plan_equals_the_three_calls(w):
    si = I.make_step_inputs(w)
    ds = G.DeviceStep(si)
    conv0, state0 = ds.conv.clone(), ds.state.clone()
    gen = torch.Generator().manual_seed(w.seed)
    x = _rand(gen, (w.rows, HIDDEN), 1.0)
    w_in = _rand(gen, (w.pitch, HIDDEN), 0.02)
    w_o = _rand(gen, (HIDDEN, w.dim), 0.05)
    caches = (ds.conv, ds.state)

    def separate(xin):
        proj = kda.linear(xin, w_in)
        core = torch.empty((w.rows, w.dim), dtype=torch.bfloat16, device="cuda")
        ds.prep.run(proj, core, caches=caches, slots=ds.slots, accepted=ds.accepted)
        y = kda.linear(core, w_o)
        torch.cuda.synchronize()
        return proj, core, y, ds.conv.clone(), ds.state.clone()

    ref = separate(x)
    assert ds.prep.check() == 0 and kda.kda_linear_check() == 0
    for pdl in (0, kda.KDA_PDL_STEP, kda.KDA_PDL_O_PROJ, True):
        ds.conv.copy_(conv0)
        ds.state.copy_(state0)
        proj = torch.empty((w.rows, w.pitch), dtype=torch.bfloat16, device="cuda")
        core = torch.empty((w.rows, w.dim), dtype=torch.bfloat16, device="cuda")
        y = torch.empty((w.rows, HIDDEN), dtype=torch.bfloat16, device="cuda")
        xb = x.clone()
        plan = ds.prep.layer_plan(xb, w_in, proj, core, w_o, y, caches=caches, slots=ds.slots,
                                  accepted=ds.accepted, pdl=pdl)
        plan.launch()
        torch.cuda.synchronize()
        assert ds.prep.check() == 0 and kda.kda_linear_check() == 0
        got = (proj, core, y, ds.conv, ds.state)
        for name, a, b in zip(("projected", "core_out", "y", "conv_state", "state"), got, ref):
            va = a.view(torch.int32) if a.dtype == torch.float32 else _bits(a)
            vb = b.view(torch.int32) if b.dtype == torch.float32 else _bits(b)
            assert torch.equal(va, vb), f"pdl={pdl}: {name} differs from the three separate calls"
        if pdl is True:
            # the plan reads its buffers at each launch: new x, caches back to the start
            x2 = _rand(gen, (w.rows, HIDDEN), 1.0)
            ds.conv.copy_(conv0)
            ds.state.copy_(state0)
            ref2 = separate(x2)
            ds.conv.copy_(conv0)
            ds.state.copy_(state0)
            xb.copy_(x2)
            plan.launch()
            torch.cuda.synchronize()
            for name, a, b in zip(("projected", "core_out", "y"), (proj, core, y), ref2[:3]):
                assert torch.equal(_bits(a), _bits(b)), f"replay: {name} differs"
        plan.close()
    ds.close()


@pytest.mark.parametrize("variant", ["bf16_state", "bf16_state_decode", "softplus_gate", "conv_transposed"])
def test_layer_plan_variants(variant):
    # the layer graph on the core's variants (bf16 state pool -- for decode the two-row
    # kernel, an odd row count leaving its last CTA one row --, the second gate form, the
    # [pool, W-1, 3D] conv layout), PDL on both edges, against the three separate calls
    if variant == "bf16_state_decode":
        w = I.Workload("decode_9_rows_v", heads=2, requests=9, L=1, pool=16, verify=False, seed=2125)
    else:
        w = I.Workload("verify_24_rows_v", heads=2, requests=6, L=4, pool=32, verify=True, seed=2124)
    si = I.make_step_inputs(w)
    kw = {"bf16_state": dict(state_dtype="bf16"), "bf16_state_decode": dict(state_dtype="bf16"),
          "softplus_gate": dict(gate_mode=1), "conv_transposed": dict(dim_first=False)}[variant]
    ds = G.DeviceStep(si, **kw)
    conv0, state0 = ds.conv.clone(), ds.state.clone()
    gen = torch.Generator().manual_seed(w.seed)
    x = _rand(gen, (w.rows, HIDDEN), 1.0)
    w_in = _rand(gen, (w.pitch, HIDDEN), 0.02)
    w_o = _rand(gen, (HIDDEN, w.dim), 0.05)
    caches = (ds.conv, ds.state)
    proj_r = kda.linear(x, w_in)
    core_r = torch.empty((w.rows, w.dim), dtype=torch.bfloat16, device="cuda")
    ds.prep.run(proj_r, core_r, caches=caches, slots=ds.slots, accepted=ds.accepted)
    y_r = kda.linear(core_r, w_o)
    torch.cuda.synchronize()
    conv_r, state_r = ds.conv.clone(), ds.state.clone()
    ds.conv.copy_(conv0)
    ds.state.copy_(state0)
    proj = torch.empty_like(proj_r)
    core = torch.empty_like(core_r)
    y = torch.empty_like(y_r)
    plan = ds.prep.layer_plan(x, w_in, proj, core, w_o, y, caches=caches, slots=ds.slots, accepted=ds.accepted,
                              pdl=True)
    plan.launch()
    torch.cuda.synchronize()
    assert ds.prep.check() == 0 and kda.kda_linear_check() == 0
    for name, a, b in (("projected", proj, proj_r), ("core_out", core, core_r), ("y", y, y_r),
                       ("conv_state", ds.conv, conv_r), ("state", ds.state, state_r)):
        va = a.view(torch.int32) if a.dtype == torch.float32 else _bits(a)
        vb = b.view(torch.int32) if b.dtype == torch.float32 else _bits(b)
        assert torch.equal(va, vb), f"{variant}: {name} differs"
    plan.close()
    ds.close()


def test_layer_plan_rejects_inconsistent_shapes():
    w = I.WORKLOADS["tiny_decode"]
    si = I.make_step_inputs(w)
    ds = G.DeviceStep(si)
    x = torch.zeros((w.rows, HIDDEN), dtype=torch.bfloat16, device="cuda")
    w_in = torch.zeros((w.pitch, HIDDEN), dtype=torch.bfloat16, device="cuda")
    w_o = torch.zeros((HIDDEN, w.dim + 8), dtype=torch.bfloat16, device="cuda")  # wrong in_features
    proj = torch.empty((w.rows, w.pitch), dtype=torch.bfloat16, device="cuda")
    core = torch.empty((w.rows, w.dim), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((w.rows, HIDDEN), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        ds.prep.layer_plan(x, w_in, proj, core, w_o, y, caches=(ds.conv, ds.state), slots=ds.slots)
    ds.close()
