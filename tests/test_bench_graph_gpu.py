"""The benchmark's timed blocks -- steps recorded once as a CUDA graph and
replayed, stepping through independent copies of the caches in turn -- do the
same work as the same steps launched one by one: every copy's out rows, conv
windows and state pool come out bit-identical.  Uses bench.py's own set-up
(make_copies) and recording (record_block)."""
from __future__ import annotations

import types

import pytest
import torch

import bench
import linear_attention_decode_03_gb300 as kda
from linear_attention_decode_03_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.load_library()


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


@pytest.mark.parametrize("w,state_dtype", [
    (I.Workload("graph_decode", heads=2, requests=24, L=1, pool=32, verify=False, seed=3101), "f32"),
    (I.Workload("graph_verify", heads=2, requests=8, L=4, pool=40, verify=True, seed=3104), "f32"),
    (I.Workload("graph_verify_bf16", heads=2, requests=8, L=4, pool=40, verify=True, seed=3105), "bf16"),
], ids=lambda v: v.name if isinstance(v, I.Workload) else v)
def test_recorded_block_equals_direct_steps(w, state_dtype):
    device = torch.device("cuda", 0)
    si = I.make_step_inputs(w)
    args = types.SimpleNamespace(gate_mode="sigmoid", launch="graph", state_dtype=state_dtype)
    n_copies, steps = 3, 7  # every copy is stepped more than once: its caches evolve
    direct = bench.make_copies(si, device, args, n_copies)
    graphed = bench.make_copies(si, device, args, n_copies)
    for i in range(steps):
        direct[i % n_copies].step()
    torch.cuda.synchronize()
    assert direct[0].prep.check() == 0
    g = bench.record_block(graphed, steps, device)
    g.replay()
    torch.cuda.synchronize()
    assert graphed[0].prep.check() == 0
    for c, (a, b) in enumerate(zip(direct, graphed)):
        for name in ("out", "conv", "state"):
            assert torch.equal(_bits(getattr(a, name)), _bits(getattr(b, name))), f"copy {c}: {name} differs"
    # a second replay continues from the caches the first one left, as direct steps would
    for i in range(steps):
        direct[i % n_copies].step()
    g.replay()
    torch.cuda.synchronize()
    for c, (a, b) in enumerate(zip(direct, graphed)):
        for name in ("out", "conv", "state"):
            assert torch.equal(_bits(getattr(a, name)), _bits(getattr(b, name))), f"replay 2, copy {c}: {name}"
    del g
