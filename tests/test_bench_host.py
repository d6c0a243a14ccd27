"""Host-side accounting of the benchmark, on the CPU: the algorithmic bytes that
the roofline divides by, written out from the method's units (a decode
token-head moves its 64 KiB state in and out; a verify request-head reads one
state and writes one per token; a projected row, an out row and a conv window
move their bf16 elements), and the rule that decides how a workload is kept
out of L2 between timed steps."""
from __future__ import annotations

import pytest

import bench
from linear_attention_decode_03_gb300 import inputs as I

STATE = 128 * 128 * 4  # one (slot, head) fp32 state


def _by_hand(w: I.Workload):
    reads = w.requests * w.heads * STATE  # one start state a (request, head)
    writes = w.requests * w.L * w.heads * STATE  # one state a token
    d = 128 * w.heads
    pitch = 4 * d + 128 + w.heads
    window = 3 * d * (w.width - 1) * 2  # q, k, v channels x (W - 1) bf16
    other = (w.requests * w.L * pitch * 2  # projected rows in
             + w.requests * w.L * d * 2  # out rows
             + w.requests * window  # one start window read a request
             + w.requests * w.L * window)  # one window written a token
    return reads + writes, other


@pytest.mark.parametrize("name,state", [
    ("tiny_decode", 262_144),
    ("batched_decode", 100_663_296),
    ("spec_verify", 125_829_120),
    ("large_decode", 805_306_368),
    ("full_width_verify", 7_247_757_312),
])
def test_state_bytes_per_workload(name, state):
    w = I.WORKLOADS[name]
    s, a = bench.algorithmic_bytes(w)
    assert s == state
    hs, ho = _by_hand(w)
    assert s == hs and a == hs + ho


def test_large_decode_all_bytes():
    # 512 rows, 12 heads: projected 512 x 6284 x 2, out 512 x 1536 x 2, and 512 + 512
    # windows of 3 x 1536 x 3 bf16
    s, a = bench.algorithmic_bytes(I.WORKLOADS["large_decode"])
    assert a - s == 6_434_816 + 1_572_864 + 1024 * 27_648 == 36_319_232


def test_bf16_state_halves_only_the_state():
    w = I.WORKLOADS["spec_verify"]
    s32, a32 = bench.algorithmic_bytes(w, "f32")
    s16, a16 = bench.algorithmic_bytes(w, "bf16")
    assert s16 * 2 == s32 and a32 - s32 == a16 - s16


@pytest.mark.parametrize("name", sorted(I.WORKLOADS))
def test_rotation_keeps_each_step_out_of_l2(name):
    w = I.WORKLOADS[name]
    t = bench.touched_bytes(w)
    n = bench.rotation_copies(w)
    if t > bench.L2_BYTES or t < bench.L2_BYTES // 8:
        assert n == 0  # larger than L2 already, or a latency case timed after a flush
    else:
        # between two uses of one copy the other copies touch at least 3x L2
        assert (n - 1) * t >= 3 * bench.L2_BYTES
        assert (n - 2) * t < 3 * bench.L2_BYTES  # and no more copies than that needs


def test_rotation_applies_to_the_mid_sized_workloads():
    assert bench.rotation_copies(I.WORKLOADS["batched_decode"]) > 0
    assert bench.rotation_copies(I.WORKLOADS["spec_verify"]) > 0
    assert bench.rotation_copies(I.WORKLOADS["large_decode"]) == 0
    assert bench.rotation_copies(I.WORKLOADS["tiny_decode"]) == 0


def test_reference_arm_line():
    # the reference arm (the fp64 oracle on the host's cores) prints the contract's line
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload",
                          "batched_decode", "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                         timeout=600, cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["config"]["workload"] == "batched_decode" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["gpu_launches"] == 0


def test_traffic_is_filed_by_state_type_and_launch_shape(tmp_path, monkeypatch):
    # a bf16-state line must not carry the fp32 capture's bytes, nor a two-CTA line either
    f = tmp_path / "traffic.txt"
    f.write_text(f"source_sha256 {bench.kernel_source_hash()}\n"
                 "traffic large_decode 100\ntraffic large_decode_bf16 60\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.measured_traffic("large_decode") == 100
    assert bench.measured_traffic("large_decode", "bf16") == 60
    assert bench.measured_traffic("large_decode", "f32", 2) is None
    assert bench.measured_traffic("spec_verify", "bf16") is None
    f.write_text("source_sha256 0123\ntraffic large_decode 100\n")  # another source: no figure
    assert bench.measured_traffic("large_decode") is None


def test_committed_traffic_matches_the_kernel_source():
    # the committed captures were taken on the kernel as it stands
    assert bench.measured_traffic("large_decode") is not None
    assert bench.measured_traffic("large_decode", "bf16") is not None


def test_roofline_names_the_kernel_that_runs():
    # decode of two rows or more runs two rows of one head a CTA, whatever the pool type
    W = I.WORKLOADS
    for sd in ("f32", "bf16"):
        assert bench.step_kernel_name(W["large_decode"], sd) == "kda_decode_pair_kernel"
        assert bench.step_kernel_name(W["batched_decode"], sd) == "kda_decode_pair_kernel"
        assert bench.step_kernel_name(W["tiny_decode"], sd) == "kda_step_kernel"  # one row
        assert bench.step_kernel_name(W["large_decode"], sd, 2) == "kda_step_kernel"  # two CTAs a head
        assert bench.step_kernel_name(W["spec_verify"], sd) == "kda_step_kernel"
        assert bench.step_kernel_name(W["full_width_verify"], sd) == "kda_step_kernel"
