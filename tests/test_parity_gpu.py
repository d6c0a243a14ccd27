"""GPU parity: libkda.so (through the C ABI) against the CPU oracle.

Criteria: slot / accepted indexing and the set of cache rows written are
bit-exact (unwritten slots keep their sentinel bits; conv windows are copies
of inputs, compared bit for bit); bf16 out within |d| <= 2e-2 + 1e-2 |ref|;
fp32 state within max-abs 1e-3.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_attention_decode_03_gb300 import inputs as I
from tests import gpu_harness as G
from tests.helpers import case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_decode_03_gb300 as kda

    kda.build()
    kda.load_library()


def _check_full(si: I.StepInputs, dim_first=True, reqs=None, gate_mode=0, v_split=1):
    """Run the whole step on the GPU; compare requests `reqs` (default all)
    with the oracle and check the untouched part of every pool."""
    w = si.workload
    ds = G.DeviceStep(si, dim_first=dim_first, gate_mode=gate_mode, v_split=v_split)
    flags = ds.run()
    if reqs is None:
        reqs = np.arange(w.requests)
    out_ref, rows, used, pool_ref, conv_ref, err = G.oracle_requests(si, reqs, dim_first=dim_first,
                                                                      gate_mode=gate_mode)
    assert flags == err == 0
    out = G.torch_bf16_to_np(ds.out[torch.from_numpy(rows).to(ds.device)])
    G.assert_out_close(out, out_ref)
    if len(used):
        uidx = torch.from_numpy(used).to(ds.device)
        G.assert_state_close(ds.state[uidx].cpu().numpy(), pool_ref)
        conv_gpu = G.torch_bf16_to_np(ds.conv[uidx])
        assert np.array_equal(conv_gpu, conv_ref)
    # every slot outside slots[] still holds the sentinel bits, state and conv
    written = np.zeros(w.pool, dtype=bool)
    written[si.slots[si.slots >= 0]] = True
    untouched = torch.from_numpy(np.nonzero(~written)[0]).to(ds.device)
    if untouched.numel():
        st = ds.state[untouched].view(torch.int32)
        assert bool((st == int(I.STATE_SENTINEL.view(np.int32))).all())
        cv = ds.conv[untouched].view(torch.int16)
        assert bool((cv == int(np.array(I.CONV_SENTINEL).view(np.int16))).all())
    # every written slot holds finite values, every out row was written
    widx = torch.from_numpy(np.nonzero(written)[0]).to(ds.device)
    assert bool(torch.isfinite(ds.state[widx]).all())
    assert bool(torch.isfinite(ds.out.float()).all())
    ds.close()


@pytest.mark.parametrize("name", ["tiny_decode", "batched_decode", "spec_verify"])
def test_workload_full_parity(name):
    _check_full(I.make_step_inputs(I.WORKLOADS[name]))


def test_large_decode_full_parity():
    _check_full(I.make_step_inputs(I.WORKLOADS["large_decode"]))


def test_full_width_verify_full_parity():
    """96 heads, R = 128 x L = 8 on a 2048-slot pool (12.9 GB of state): the
    whole step runs on the GPU and every request is recomputed by the oracle,
    streamed 8 requests at a time so that host memory holds one chunk's
    caches; the untouched slots of the whole pool are checked on the device."""
    si = I.make_step_inputs(I.WORKLOADS["full_width_verify"])
    w = si.workload
    ds = G.DeviceStep(si)
    assert ds.run() == 0
    G.compare_streamed(ds, si, chunk=8)
    written = np.zeros(w.pool, dtype=bool)
    written[si.slots[si.slots >= 0]] = True
    untouched = torch.from_numpy(np.nonzero(~written)[0]).to(ds.device)
    st = ds.state[untouched].view(torch.int32)
    assert bool((st == int(I.STATE_SENTINEL.view(np.int32))).all())
    cv = ds.conv[untouched].view(torch.int16)
    assert bool((cv == int(np.array(I.CONV_SENTINEL).view(np.int16))).all())
    ds.close()


@pytest.mark.parametrize("v_split", [1, 2])
@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 6, 7, 8])
def test_every_token_count(L, v_split):
    # one CTA a (request, head), or two in a cluster (64 v rows each, o halves swapped)
    si = case(heads=2, requests=5, L=L, pool=5 * L + 3, seed=40 + L, verify=L > 1)
    _check_full(si, v_split=v_split)


@pytest.mark.parametrize("name", ["batched_decode", "spec_verify"])
def test_two_ctas_per_head_on_many_waves(name):
    # the split forced where the automatic choice keeps one CTA: 2 x 768 or 2 x 384 CTAs,
    # clusters of two in more than one wave
    _check_full(I.make_step_inputs(I.WORKLOADS[name]), v_split=2)


@pytest.mark.parametrize("L", [1, 3])
@pytest.mark.parametrize("width", [2, 3])
def test_conv_widths(width, L):
    _check_full(case(heads=2, requests=3, L=L, pool=12, width=width, seed=50 + width, verify=L > 1))


def test_transposed_conv_state_and_bias():
    _check_full(case(heads=3, requests=4, L=4, pool=20, seed=60, with_bias=True), dim_first=False)
    _check_full(case(heads=1, requests=7, L=1, pool=9, seed=61, with_bias=True), dim_first=True)
    # the two-CTA split is built for the window-first layout: asked for on the other, the step runs one CTA
    _check_full(case(heads=3, requests=4, L=4, pool=20, seed=60, with_bias=True), dim_first=False, v_split=2)


def test_v_split_rejects_other_values():
    import linear_attention_decode_03_gb300 as kda

    ds = G.DeviceStep(case(heads=2, requests=2, L=1, pool=4, seed=65))
    for bad in (0, 3, -1):
        with pytest.raises(kda.KdaError):
            kda.kda_set_v_split(ds.prep.handle, bad)
    kda.kda_set_v_split(ds.prep.handle, 2)
    kda.kda_set_v_split(ds.prep.handle, 1)
    ds.close()


@pytest.mark.parametrize("L", [1, 4])
def test_softplus_gate_mode(L):
    """The clamped-softplus gate (kda_set_gate_mode), decode and verify, against
    the oracle run with the same gate form."""
    _check_full(case(heads=3, requests=5, L=L, pool=5 * L + 4, seed=70 + L, verify=L > 1), gate_mode=1)


@pytest.mark.parametrize("L", [1, 4])
def test_plan_replays_equal_steps(L):
    """A launch plan (one step recorded as a CUDA graph on fixed buffers) gives
    the bits kda_step gives, and each launch is a step on what the buffers
    then hold (new projected rows written between launches)."""
    si = case(heads=2, requests=4, L=L, pool=4 * L + 3, seed=80 + L, verify=L > 1)
    a, b = G.DeviceStep(si), G.DeviceStep(si)
    plan = b.prep.plan(b.projected, b.out, caches=(b.conv, b.state), slots=b.slots, accepted=b.accepted)
    gen = torch.Generator(device="cpu").manual_seed(L)
    for step in range(3):
        if step == 2:  # the same new inputs into both sets of buffers
            fresh = torch.randn(a.projected.shape, generator=gen).to(torch.bfloat16).to(a.device)
            a.projected.copy_(fresh)
            b.projected.copy_(fresh)
        assert a.run() == 0
        plan.launch()
        assert b.prep.check() == 0
        assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
        assert torch.equal(a.state.view(torch.int32), b.state.view(torch.int32))
        assert torch.equal(a.conv.view(torch.int16), b.conv.view(torch.int16))
    plan.close()
    a.close()
    b.close()


def _check_bf16_state(si: I.StepInputs, reqs=None, v_split=1):
    """The bf16 state pool (kda_set_state_dtype): outputs and windows as in
    fp32, each stored state within one bf16 step of the oracle's, untouched
    slots keep their bf16 sentinel."""
    w = si.workload
    ds = G.DeviceStep(si, state_dtype="bf16", v_split=v_split)
    flags = ds.run()
    if reqs is None:
        reqs = np.arange(w.requests)
    out_ref, rows, used, pool_ref, conv_ref, err = G.oracle_requests(si, reqs, state_dtype="bf16")
    assert flags == err == 0
    G.assert_out_close(G.torch_bf16_to_np(ds.out[torch.from_numpy(rows).to(ds.device)]), out_ref)
    uidx = torch.from_numpy(used).to(ds.device)
    G.assert_state_close_bf16(G.torch_bf16_to_np(ds.state[uidx]), pool_ref)
    assert np.array_equal(G.torch_bf16_to_np(ds.conv[uidx]), conv_ref)
    written = np.zeros(w.pool, dtype=bool)
    written[si.slots[si.slots >= 0]] = True
    untouched = torch.from_numpy(np.nonzero(~written)[0]).to(ds.device)
    if untouched.numel():
        sentinel = int(np.array(I.STATE_SENTINEL_BF16).view(np.int16))
        assert bool((ds.state[untouched].view(torch.int16) == sentinel).all())
    ds.close()


@pytest.mark.parametrize("name", ["batched_decode", "spec_verify"])
def test_bf16_state_workloads(name):
    _check_bf16_state(I.make_step_inputs(I.WORKLOADS[name]))


def test_bf16_state_large_decode_sampled():
    si = I.make_step_inputs(I.WORKLOADS["large_decode"])
    _check_bf16_state(si, reqs=np.array([0, 1, 77, 300, 511]))


@pytest.mark.parametrize("v_split", [1, 2])
@pytest.mark.parametrize("L", [1, 3, 8])
def test_bf16_state_token_counts(L, v_split):
    _check_bf16_state(case(heads=2, requests=4, L=L, pool=4 * L + 3, seed=90 + L, verify=L > 1), v_split=v_split)


def test_verify_with_one_token_accepted_array():
    _check_full(case(heads=2, requests=6, L=1, pool=8, seed=62, verify=True))


def _full_pool_oracle(si, slots, acc, dim_first=True):
    W = oracle.Weights(**si.weights.as_dict())
    return oracle.step(W, si.projected, si.full_conv_state(dim_first), si.full_state_pool(), slots, si.workload.L,
                       acc, dim_first=dim_first)


@pytest.mark.parametrize("v_split", [1, 2])
def test_padding_and_bad_values(v_split):
    """slot -1 first = padding (zero out, no cache I/O); accepted outside 1..L
    and slots outside the pool set their error bits and skip the request,
    exactly as the oracle does (one or two CTAs a (request, head))."""
    R, L = 6, 3
    si = case(heads=2, requests=R, L=L, pool=24, seed=63, accepted=[3, 1, 2, 2, 1, 3])
    slots = si.slots.reshape(R, L).copy()
    acc = si.accepted.copy()
    slots[1, 0] = -1        # padding request
    acc[2] = 0              # bad accepted
    acc[3] = L + 1          # bad accepted
    slots[4, 2] = 24        # out of the pool
    si.slots = slots.reshape(-1).copy()
    out_ref, conv_ref, pool_ref, err = _full_pool_oracle(si, si.slots, acc)
    assert err == oracle.ERR_ACCEPTED | oracle.ERR_SLOT
    ds = G.DeviceStep(si, v_split=v_split)
    ds.accepted = torch.from_numpy(acc).to(ds.device)
    flags = ds.run()
    assert flags == err
    out = G.torch_bf16_to_np(ds.out)
    ok_rows = np.r_[0:L, 5 * L:6 * L]
    G.assert_out_close(out[ok_rows], out_ref[ok_rows])
    assert np.all(out[L:2 * L] == 0)                            # padding rows zeroed
    assert np.all(out[2 * L:5 * L] == G.OUT_SENTINEL)           # skipped rows untouched
    st = ds.state.cpu().numpy()
    assert np.array_equal(np.isnan(st), np.isnan(pool_ref))
    fin = ~np.isnan(pool_ref)
    assert np.abs(st[fin] - pool_ref[fin]).max() <= G.STATE_ATOL
    assert np.array_equal(G.torch_bf16_to_np(ds.conv), conv_ref)
    # the error word was cleared by the check
    assert ds.prep.check() == 0
    ds.close()


@pytest.mark.parametrize("v_split", [1, 2])
def test_decode_padding_rows(v_split):
    si = case(heads=2, requests=5, L=1, pool=8, seed=64)
    si.slots[[1, 3]] = -1
    out_ref, conv_ref, pool_ref, err = _full_pool_oracle(si, si.slots, None)
    ds = G.DeviceStep(si, v_split=v_split)
    assert ds.run() == err == 0
    out = G.torch_bf16_to_np(ds.out)
    G.assert_out_close(out, out_ref)
    assert np.all(out[[1, 3]] == 0)
    assert np.array_equal(G.torch_bf16_to_np(ds.conv), conv_ref)
    ds.close()


def test_verify_equals_chained_decode_on_gpu():
    """The GPU's L-token verify equals L chained GPU decodes (slot copies in
    between done with torch), to the state tolerance."""
    R, L = 3, 4
    si = case(heads=2, requests=R, L=L, pool=16, seed=65, accepted=[4, 1, 2])
    ds = G.DeviceStep(si)
    assert ds.run() == 0
    dd = G.DeviceStep(si)
    slots = si.slots.reshape(R, L)
    one = torch.zeros(1, dtype=torch.int32, device=dd.device)
    out_d = torch.empty_like(dd.out)
    for r in range(R):
        src = int(slots[r, si.accepted[r] - 1])
        for t in range(L):
            dst = int(slots[r, t])
            if dst != src:
                dd.state[dst] = dd.state[src]
                dd.conv[dst] = dd.conv[src]
            one.fill_(dst)
            row = r * L + t
            dd.prep.run(dd.projected[row:row + 1], out_d[row:row + 1], caches=(dd.conv, dd.state), slots=one)
            src = dst
    assert dd.prep.check() == 0
    used = torch.from_numpy(np.unique(slots)).to(dd.device)
    assert (ds.state[used] - dd.state[used]).abs().max().item() <= 1e-5
    assert torch.equal(ds.conv[used], dd.conv[used])
    diff = (ds.out.float() - out_d.float()).abs()
    assert bool((diff <= 2.0 ** -7 * out_d.float().abs() + 1e-6).all())
    ds.close()
    dd.close()


def test_deterministic_and_empty():
    si = case(heads=2, requests=4, L=2, pool=10, seed=66)
    a, b = G.DeviceStep(si), G.DeviceStep(si)
    assert a.run() == 0 and b.run() == 0
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.state.view(torch.int32), b.state.view(torch.int32))
    # rows = 0: nothing enqueued, nothing changed
    before = a.state.clone()
    a.prep.run(a.projected[:0], a.out[:0], caches=(a.conv, a.state), slots=a.slots[:0], accepted=a.accepted[:0])
    assert a.prep.check() == 0
    assert torch.equal(before.view(torch.int32), a.state.view(torch.int32))
    a.close()
    b.close()


def test_two_consecutive_decode_steps():
    """In-place decode twice on the same slots equals the oracle applied twice."""
    si = case(heads=2, requests=4, L=1, pool=6, seed=67)
    ds = G.DeviceStep(si)
    assert ds.run() == 0
    assert ds.run() == 0
    W = oracle.Weights(**si.weights.as_dict())
    o1, c1, p1, e1 = oracle.step(W, si.projected, si.full_conv_state(), si.full_state_pool(), si.slots, 1, None)
    o2, c2, p2, e2 = oracle.step(W, si.projected, c1, p1, si.slots, 1, None)
    G.assert_out_close(G.torch_bf16_to_np(ds.out), o2)
    used = np.unique(si.slots)
    G.assert_state_close(ds.state.cpu().numpy()[used], p2[used])
    assert np.array_equal(G.torch_bf16_to_np(ds.conv), c2)
    ds.close()


def test_invalid_arguments_rejected():
    import linear_attention_decode_03_gb300 as kda

    si = case(heads=2, requests=2, L=2, pool=6, seed=68)
    ds = G.DeviceStep(si)
    h = ds.prep.handle
    w = si.workload
    p = ds.projected
    common = dict(projected=p.data_ptr(), rows=w.rows, pitch=p.stride(0), conv_state=ds.conv.data_ptr(),
                  conv_dim_first=True, state_pool=ds.state.data_ptr(), pool_slots=w.pool,
                  slots=ds.slots.data_ptr(), L=w.L, accepted=ds.accepted.data_ptr(), out=ds.out.data_ptr(), stream=0)
    bad = [dict(L=9), dict(L=0), dict(rows=3), dict(pitch=w.pitch - 1), dict(accepted=None),
           dict(state_pool=ds.state.data_ptr() + 4), dict(out=ds.out.data_ptr() + 2), dict(slots=0),
           dict(rows=-2)]
    for change in bad:
        args = dict(common)
        args.update(change)
        with pytest.raises(kda.KdaError) as ei:
            kda.kda_step(h, **args)
        assert ei.value.code == -1, change
    with pytest.raises(kda.KdaError):
        kda.kda_step(0, **common)
    assert ds.prep.check() == 0
    ds.close()


def test_launch_info():
    import linear_attention_decode_03_gb300 as kda

    for L in range(1, 9):
        threads, smem, per_sm = kda.kda_launch_info(L)
        # one CTA of 8 warps per (request, head) with its 64 KiB state in shared
        # memory: three resident per SM up to L = 4, two above
        assert threads == 256 and smem >= 65536
        assert per_sm == (3 if L <= 4 else 2), (L, per_sm)
