"""The KDA_DEBUG build (libkda_debug.so, -DKDA_DEBUG): a device check flags a
step whose rows write the same slot twice (KDA_ERR_DUPLICATE; the step itself
is undefined then, and still runs in bounds); steps with distinct slots set no
bit and match the oracle as the release build does."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_decode_03_gb300 as kda
from linear_attention_decode_03_gb300 import inputs as I
from tests import gpu_harness as G
from tests.helpers import case

pytestmark = pytest.mark.gpu


@pytest.fixture()
def debug_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    path = kda.build(debug=True)
    saved = kda._lib
    kda._lib = None
    kda.load_library(path)
    try:
        yield
    finally:
        kda._lib = saved


@pytest.mark.parametrize("L", [1, 4])
def test_distinct_slots_pass_and_match_the_oracle(debug_build, L):
    si = case(heads=2, requests=5, L=L, pool=5 * L + 3, seed=120 + L, verify=L > 1)
    ds = G.DeviceStep(si)
    assert ds.run() == 0
    out_ref, rows, used, pool_ref, conv_ref, err = G.oracle_requests(si, np.arange(si.workload.requests))
    assert err == 0
    G.assert_out_close(G.torch_bf16_to_np(ds.out[torch.from_numpy(rows).to(ds.device)]), out_ref)
    G.assert_state_close(ds.state[torch.from_numpy(used).to(ds.device)].cpu().numpy(), pool_ref)
    ds.close()


def test_duplicate_decode_slots_are_flagged(debug_build):
    si = case(heads=2, requests=4, L=1, pool=8, seed=130)
    si.slots[:] = np.array([3, 5, 3, 7], dtype=np.int32)
    si.read_slots = np.array([3, 5, 7], dtype=np.int64)
    si.states = si.states[:3]
    si.windows = si.windows[:3]
    ds = G.DeviceStep(si)
    assert ds.run() == kda.KDA_ERR_DUPLICATE
    ds.close()


def test_duplicate_verify_slots_are_flagged_but_not_in_padding(debug_build):
    R, L = 3, 2
    si = case(heads=2, requests=R, L=L, pool=10, seed=131, accepted=[1, 1, 1])
    slots = si.slots.reshape(R, L)
    # request 2 writes a slot request 0 writes: flagged
    dup = si.slots.copy().reshape(R, L)
    dup[2, 1] = dup[0, 1]
    si_dup = case(heads=2, requests=R, L=L, pool=10, seed=131, accepted=[1, 1, 1])
    si_dup.slots = dup.reshape(-1).copy()
    ds = G.DeviceStep(si_dup)
    assert ds.run() == kda.KDA_ERR_DUPLICATE
    ds.close()
    # the same slot in a padding request (slot -1 first) writes nothing: not flagged
    pad = slots.copy()
    pad[2, 0] = -1
    pad[2, 1] = slots[0, 1]
    si.slots = pad.reshape(-1).copy()
    ds = G.DeviceStep(si)
    assert ds.run() == 0
    ds.close()
