"""Decode with a bf16 state pool runs rows 2p and 2p + 1 of one head in one CTA.
Parity with the oracle (run on the whole pool) for row counts that leave the
last CTA a single row, several head counts, both conv cache layouts, conv
widths 2-4 with a bias, and padding rows, bad slots and good rows mixed inside
one CTA's pair: outputs within the output tolerance, each stored state element
within one bf16 step, windows bit-exact, and every slot the step must not write
left bit-identical."""
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


def _check(si: I.StepInputs, dim_first: bool = True, slots=None):
    """One bf16-pool decode step on the device against the oracle on the full pool."""
    w = si.workload
    if slots is not None:
        si.slots = np.asarray(slots, dtype=np.int32)
    W = oracle.Weights(**si.weights.as_dict())
    out_ref, conv_ref, pool_ref, err = oracle.step(W, si.projected, si.full_conv_state(dim_first),
                                                   si.full_state_pool_bf16(), si.slots, 1, None,
                                                   dim_first=dim_first, state_dtype="bf16")
    ds = G.DeviceStep(si, dim_first=dim_first, state_dtype="bf16")
    flags = ds.run()
    assert flags == err
    out = G.torch_bf16_to_np(ds.out)
    ok = (si.slots >= 0) & (si.slots < w.pool)
    pad = si.slots == -1
    if ok.any():
        G.assert_out_close(out[ok], out_ref[ok])
    assert np.all(out[pad] == 0)                                # padding rows zeroed
    assert np.all(out[~ok & ~pad] == G.OUT_SENTINEL)            # skipped rows untouched
    st = G.torch_bf16_to_np(ds.state)
    written = np.unique(si.slots[ok])
    if len(written):
        G.assert_state_close_bf16(st[written], pool_ref[written])
    rest = np.setdiff1d(np.arange(w.pool), written)
    assert np.array_equal(st[rest], pool_ref[rest])             # unwritten slots bit-identical
    assert np.array_equal(G.torch_bf16_to_np(ds.conv), conv_ref)
    ds.close()


@pytest.mark.parametrize("requests", [1, 2, 3, 5, 8])
def test_row_counts(requests):
    _check(case(heads=2, requests=requests, L=1, pool=requests + 3, seed=400 + requests))


@pytest.mark.parametrize("heads", [1, 3, 5])
def test_head_counts(heads):
    _check(case(heads=heads, requests=3, L=1, pool=7, seed=410 + heads))


@pytest.mark.parametrize("dim_first", [True, False])
@pytest.mark.parametrize("width", [2, 3, 4])
def test_layouts_widths_and_bias(dim_first, width):
    _check(case(heads=2, requests=5, L=1, pool=9, width=width, with_bias=True, seed=420 + width), dim_first=dim_first)


def test_padding_bad_slots_and_good_rows_in_one_pair():
    si = case(heads=2, requests=8, L=1, pool=12, seed=430)
    slots = si.slots.copy()
    slots[1] = -1           # pair 0: a good row, then padding
    slots[2] = 12           # pair 1: a slot outside the pool, then a good row
    slots[4] = slots[5] = -1  # pair 2: both padding
    slots[6] = -7           # pair 3: a negative slot other than -1, then a good row
    _check(si, slots=slots)
