"""The binding's argument handling (PreparedKda.run): slots and accepted longer
than the batch are read in place (the step reads their first rows only),
strided ones are copied to the layout the C ABI takes, and buffers too small
for the step are rejected on the host before anything is enqueued.  Each
passing case is compared bit for bit with the same step on exact-size
contiguous inputs, which the parity tests compare with the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

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


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def _same(a: G.DeviceStep, b: G.DeviceStep):
    for name in ("out", "conv", "state"):
        assert torch.equal(_bits(getattr(a, name)), _bits(getattr(b, name))), name


def test_decode_slots_longer_than_the_batch():
    si = case(heads=2, requests=6, L=1, pool=12, seed=301)
    ref, ds = G.DeviceStep(si), G.DeviceStep(si)
    assert ref.run() == 0
    # five more entries that name no valid slot: read, they would set KDA_ERR_SLOT
    longer = torch.full((6 + 5,), 1 << 20, dtype=torch.int32, device=ds.device)
    longer[:6] = ds.slots
    ds.prep.run(ds.projected, ds.out, caches=(ds.conv, ds.state), slots=longer)
    assert ds.prep.check() == 0
    _same(ref, ds)
    ref.close()
    ds.close()


def test_verify_slots_and_accepted_longer_than_the_batch():
    R, L = 5, 3
    si = case(heads=2, requests=R, L=L, pool=20, seed=302)
    ref, ds = G.DeviceStep(si), G.DeviceStep(si)
    assert ref.run() == 0
    slots = torch.full((R + 3, L), 1 << 20, dtype=torch.int32, device=ds.device)
    slots[:R] = ds.slots.view(R, L)
    acc = torch.full((R + 3,), 99, dtype=torch.int32, device=ds.device)  # out of 1..L past the batch
    acc[:R] = ds.accepted
    ds.prep.run(ds.projected, ds.out, caches=(ds.conv, ds.state), slots=slots, accepted=acc)
    assert ds.prep.check() == 0
    _same(ref, ds)
    ref.close()
    ds.close()


def test_strided_verify_slots_and_accepted_are_copied():
    R, L = 4, 4
    si = case(heads=2, requests=R, L=L, pool=20, seed=303)
    ref, ds = G.DeviceStep(si), G.DeviceStep(si)
    assert ref.run() == 0
    wide = torch.full((R, 2 * L), -5, dtype=torch.int32, device=ds.device)
    wide[:, ::2] = ds.slots.view(R, L)
    acc_wide = torch.zeros(2 * R, dtype=torch.int32, device=ds.device)
    acc_wide[::2] = ds.accepted
    strided_slots, strided_acc = wide[:, ::2], acc_wide[::2]
    assert strided_slots.stride() == (2 * L, 2) and not strided_acc.is_contiguous()
    ds.prep.run(ds.projected, ds.out, caches=(ds.conv, ds.state), slots=strided_slots, accepted=strided_acc)
    assert ds.prep.check() == 0
    _same(ref, ds)
    ref.close()
    ds.close()


def test_buffers_too_small_are_rejected_before_launch():
    R, L = 3, 2
    si = case(heads=2, requests=R, L=L, pool=10, seed=304)
    ds = G.DeviceStep(si)
    before = {n: getattr(ds, n).clone() for n in ("out", "conv", "state")}
    caches = (ds.conv, ds.state)
    slots = ds.slots.view(R, L)
    with pytest.raises(ValueError):  # one request short
        ds.prep.run(ds.projected, ds.out, caches=caches, slots=slots[:R - 1], accepted=ds.accepted)
    with pytest.raises(ValueError):
        ds.prep.run(ds.projected, ds.out, caches=caches, slots=slots, accepted=ds.accepted[:R - 1])
    with pytest.raises(ValueError):  # out one row short
        ds.prep.run(ds.projected, ds.out[:-1], caches=caches, slots=slots, accepted=ds.accepted)
    with pytest.raises(ValueError):  # projected without its beta columns
        ds.prep.run(ds.projected[:, :4 * 256 + 128], ds.out, caches=caches, slots=slots, accepted=ds.accepted)
    with pytest.raises(ValueError):  # conv windows for fewer slots than the state pool
        ds.prep.run(ds.projected, ds.out, caches=(ds.conv[:-1], ds.state), slots=slots, accepted=ds.accepted)
    with pytest.raises(ValueError):  # a state pool of another head count
        ds.prep.run(ds.projected, ds.out, caches=(ds.conv, ds.state.view(-1)[:-128 * 128]), slots=slots,
                    accepted=ds.accepted)
    d1 = G.DeviceStep(case(heads=2, requests=4, L=1, pool=6, seed=305))
    with pytest.raises(ValueError):  # decode slots one row short
        d1.prep.run(d1.projected, d1.out, caches=(d1.conv, d1.state), slots=d1.slots[:3])
    assert ds.prep.check() == 0 and d1.prep.check() == 0
    for n, t in before.items():
        assert torch.equal(_bits(getattr(ds, n)), _bits(t)), n
    ds.close()
    d1.close()
