"""Decode of two rows or more runs rows 2p and 2p + 1 of one head in one CTA
(with an fp32 pool, the second row's halves are loaded into the one state
buffer as the first row's passes free them).  Parity with the oracle (run on
the whole pool), for both pool types, for row counts that leave the last CTA a
single row, several head counts, both conv cache layouts, conv widths 2-4 with
a bias, and padding rows, bad slots and good rows mixed inside one CTA's pair:
outputs within the output tolerance, stored states within the state tolerance
(bf16: one bf16 step), windows bit-exact, and every slot the step must not
write left bit-identical."""
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


def _check(si: I.StepInputs, dim_first: bool = True, slots=None, state_dtype: str = "bf16"):
    """One decode step on the device against the oracle on the full pool."""
    w = si.workload
    if slots is not None:
        si.slots = np.asarray(slots, dtype=np.int32)
    W = oracle.Weights(**si.weights.as_dict())
    bf16 = state_dtype == "bf16"
    pool0 = si.full_state_pool_bf16() if bf16 else si.full_state_pool()
    out_ref, conv_ref, pool_ref, err = oracle.step(W, si.projected, si.full_conv_state(dim_first), pool0, si.slots,
                                                   1, None, dim_first=dim_first, state_dtype=state_dtype)
    ds = G.DeviceStep(si, dim_first=dim_first, state_dtype=state_dtype)
    flags = ds.run()
    assert flags == err
    out = G.torch_bf16_to_np(ds.out)
    ok = (si.slots >= 0) & (si.slots < w.pool)
    pad = si.slots == -1
    if ok.any():
        G.assert_out_close(out[ok], out_ref[ok])
    assert np.all(out[pad] == 0)                                # padding rows zeroed
    assert np.all(out[~ok & ~pad] == G.OUT_SENTINEL)            # skipped rows untouched
    written = np.unique(si.slots[ok])
    rest = np.setdiff1d(np.arange(w.pool), written)
    if bf16:
        st = G.torch_bf16_to_np(ds.state)
        if len(written):
            G.assert_state_close_bf16(st[written], pool_ref[written])
        assert np.array_equal(st[rest], pool_ref[rest])         # unwritten slots bit-identical
    else:
        st = ds.state.cpu().numpy()
        if len(written):
            G.assert_state_close(st[written], pool_ref[written])
        assert np.array_equal(st[rest].view(np.uint32), pool_ref[rest].view(np.uint32))
    assert np.array_equal(G.torch_bf16_to_np(ds.conv), conv_ref)
    ds.close()


DTYPES = ["f32", "bf16"]


@pytest.mark.parametrize("state_dtype", DTYPES)
@pytest.mark.parametrize("requests", [1, 2, 3, 5, 8])
def test_row_counts(requests, state_dtype):
    _check(case(heads=2, requests=requests, L=1, pool=requests + 3, seed=400 + requests), state_dtype=state_dtype)


@pytest.mark.parametrize("state_dtype", DTYPES)
@pytest.mark.parametrize("heads", [1, 3, 5])
def test_head_counts(heads, state_dtype):
    _check(case(heads=heads, requests=3, L=1, pool=7, seed=410 + heads), state_dtype=state_dtype)


@pytest.mark.parametrize("state_dtype", DTYPES)
@pytest.mark.parametrize("dim_first", [True, False])
@pytest.mark.parametrize("width", [2, 3, 4])
def test_layouts_widths_and_bias(dim_first, width, state_dtype):
    _check(case(heads=2, requests=5, L=1, pool=9, width=width, with_bias=True, seed=420 + width), dim_first=dim_first,
           state_dtype=state_dtype)


@pytest.mark.parametrize("state_dtype", DTYPES)
def test_padding_bad_slots_and_good_rows_in_one_pair(state_dtype):
    # fp32: where the first row of a pair is padding or a bad slot, the second row's
    # state is loaded at once instead of behind the first row's passes
    si = case(heads=2, requests=10, L=1, pool=14, seed=430)
    slots = si.slots.copy()
    slots[1] = -1           # pair 0: a good row, then padding
    slots[2] = 14           # pair 1: a slot outside the pool, then a good row
    slots[4] = slots[5] = -1  # pair 2: both padding
    slots[6] = -7           # pair 3: a negative slot other than -1, then a good row
    slots[8] = -1           # pair 4: padding, then a good row
    _check(si, slots=slots, state_dtype=state_dtype)
