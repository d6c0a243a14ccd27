"""Seeded synthetic inputs for the KDA decode / spec-verify workloads.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle are
fed from it, so the two sides see bit-identical inputs.

Shapes follow the pages' workloads: 12 heads x 128 per tensor-parallel rank
slice (o_proj's local K = 1536 on the K2a attn_post page), 96 heads unsharded,
conv width 4, spec-verify with up to 8 tokens per request.  Distributions:
projected rows bf16 N(0,1); f_b N(0,0.02); A_log U(-1,1); dt_bias N(0,0.1);
o_norm ones; conv_w N(0,0.3); conv bias absent (optional N(0,0.1) for tests);
fp32 states N(0,0.02); conv windows bf16 N(0,1).

Cache slots that a step does not read are filled with sentinel bit patterns
(a quiet NaN for states and conv windows), so a wrongly indexed read shows up
as NaN and a stray write shows up as a changed sentinel.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

HEAD_DIM = 128
STATE_SENTINEL = np.uint32(0x7FEDBEEF)  # quiet NaN, fp32
CONV_SENTINEL = np.uint16(0x7FDB)       # quiet NaN, bf16
STATE_SENTINEL_BF16 = np.uint16(0x7FED)  # quiet NaN, bf16 (state pool stored as bf16)


def to_bf16_bits(x) -> np.ndarray:
    """float32 samples -> bf16 bit patterns (round to nearest even); finite inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)


@dataclass(frozen=True)
class Workload:
    """One step's shape: `requests` x `L` rows (decode: L = 1, no accepted)."""

    name: str
    heads: int
    requests: int
    L: int
    pool: int
    verify: bool
    width: int = 4
    seed: int = 1000

    @property
    def rows(self) -> int:
        return self.requests * self.L

    @property
    def dim(self) -> int:
        return HEAD_DIM * self.heads

    @property
    def pitch(self) -> int:
        return 4 * self.dim + HEAD_DIM + self.heads

    @property
    def state_bytes(self) -> int:
        """Algorithmic fp32 state bytes one step reads and writes."""
        per_block = HEAD_DIM * HEAD_DIM * 4
        reads = self.requests * self.heads * per_block
        writes = self.rows * self.heads * per_block
        return reads + writes

    @property
    def other_bytes(self) -> int:
        """Algorithmic bytes besides the state: projected rows read, out rows
        written, conv windows read (one per request) and written (one per row)."""
        win = 3 * self.dim * (self.width - 1) * 2
        return (self.rows * self.pitch * 2 + self.rows * self.dim * 2
                + self.requests * win + self.rows * win)


# The five workloads: tiny decode, batched decode, spec-verify, large decode,
# full-width verify.  Seeds are 1000 + the workload's number.
WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_decode", heads=2, requests=1, L=1, pool=4, verify=False, seed=1001),
        Workload("batched_decode", heads=12, requests=64, L=1, pool=64, verify=False, seed=1002),
        Workload("spec_verify", heads=12, requests=32, L=4, pool=256, verify=True, seed=1003),
        Workload("large_decode", heads=12, requests=512, L=1, pool=1024, verify=False, seed=1004),
        Workload("full_width_verify", heads=96, requests=128, L=8, pool=2048, verify=True, seed=1005),
    ]
}


@dataclass
class LayerWeights:
    """Layer parameters in the model's own layouts (host arrays, bf16 as uint16)."""

    heads: int
    conv_w: np.ndarray            # [3D, 1, W] bf16
    bias: Optional[np.ndarray]    # [3D] bf16 or None
    f_b: np.ndarray               # [D, 128] bf16
    A_log: np.ndarray             # [H] f32
    dt_bias: np.ndarray           # [D] f32
    o_norm: np.ndarray            # [128] f32
    gate_lower_bound: float = -5.0
    eps: float = 1e-6

    def as_dict(self):
        return dict(heads=self.heads, conv_w=self.conv_w, bias=self.bias, f_b=self.f_b,
                    A_log=self.A_log, dt_bias=self.dt_bias, o_norm=self.o_norm,
                    gate_lower_bound=self.gate_lower_bound, eps=self.eps)


def make_weights(heads: int, width: int = 4, seed: int = 1000, with_bias: bool = False) -> LayerWeights:
    rng = np.random.Generator(np.random.PCG64(seed))
    D = HEAD_DIM * heads
    conv_w = to_bf16_bits(rng.normal(0.0, 0.3, size=(3 * D, 1, width)))
    f_b = to_bf16_bits(rng.normal(0.0, 0.02, size=(D, HEAD_DIM)))
    A_log = rng.uniform(-1.0, 1.0, size=heads).astype(np.float32)
    dt_bias = rng.normal(0.0, 0.1, size=D).astype(np.float32)
    o_norm = np.ones(HEAD_DIM, dtype=np.float32)
    bias = to_bf16_bits(rng.normal(0.0, 0.1, size=3 * D)) if with_bias else None
    return LayerWeights(heads, conv_w, bias, f_b, A_log, dt_bias, o_norm)


@dataclass
class StepInputs:
    """Everything one step consumes.

    Only the slots the step reads carry random content (`read_slots`,
    `states`, `windows`); every other pool slot holds the sentinels.  Use
    :meth:`full_state_pool` / :meth:`full_conv_state` to materialise whole
    pools on the host when they are small.
    """

    workload: Workload
    weights: LayerWeights
    projected: np.ndarray              # [rows, pitch] bf16
    slots: np.ndarray                  # [rows] int32 (request-major for verify)
    accepted: Optional[np.ndarray]     # [R] int32 or None
    read_slots: np.ndarray             # distinct slots whose caches the step reads
    states: np.ndarray                 # [n_read, H, 128, 128] f32
    windows: np.ndarray                # [n_read, 3D, W-1] bf16 (dim-first)
    extra: dict = field(default_factory=dict)

    def full_state_pool(self) -> np.ndarray:
        w = self.workload
        pool = np.empty((w.pool, w.heads, HEAD_DIM, HEAD_DIM), dtype=np.float32)
        pool.view(np.uint32)[...] = STATE_SENTINEL
        pool[self.read_slots] = self.states
        return pool

    def states_bf16(self) -> np.ndarray:
        """The read states as bf16 bit patterns (nearest even), for a bf16 state pool."""
        return to_bf16_bits(self.states)

    def full_state_pool_bf16(self) -> np.ndarray:
        w = self.workload
        pool = np.full((w.pool, w.heads, HEAD_DIM, HEAD_DIM), STATE_SENTINEL_BF16, dtype=np.uint16)
        pool[self.read_slots] = self.states_bf16()
        return pool

    def full_conv_state(self, dim_first: bool = True) -> np.ndarray:
        w = self.workload
        sl = w.width - 1
        conv = np.full((w.pool, 3 * w.dim, sl), CONV_SENTINEL, dtype=np.uint16)
        conv[self.read_slots] = self.windows
        return conv if dim_first else np.ascontiguousarray(conv.transpose(0, 2, 1))


def make_step_inputs(w: Workload, *, with_bias: bool = False, seed: Optional[int] = None,
                     weights: Optional[LayerWeights] = None, accepted=None) -> StepInputs:
    """Draw one step's inputs; `accepted` (verify only) overrides the drawn counts."""
    seed = w.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    if weights is None:
        weights = make_weights(w.heads, w.width, seed=seed + 7919, with_bias=with_bias)
    projected = to_bf16_bits(rng.normal(0.0, 1.0, size=(w.rows, w.pitch)).astype(np.float32))
    if w.verify:
        slots = rng.choice(w.pool, size=w.rows, replace=False).astype(np.int32)
        drawn = rng.integers(1, w.L + 1, size=w.requests).astype(np.int32)
        accepted = drawn if accepted is None else np.asarray(accepted, dtype=np.int32).copy()
        start = slots.reshape(w.requests, w.L)[np.arange(w.requests), accepted - 1]
    else:
        slots = rng.permutation(w.pool)[: w.rows].astype(np.int32)
        accepted = None
        start = slots
    read_slots = np.array(sorted(set(int(s) for s in start)), dtype=np.int64)
    n = len(read_slots)
    states = rng.normal(0.0, 0.02, size=(n, w.heads, HEAD_DIM, HEAD_DIM)).astype(np.float32)
    windows = to_bf16_bits(rng.normal(0.0, 1.0, size=(n, 3 * w.dim, w.width - 1)).astype(np.float32))
    return StepInputs(w, weights, projected, slots, accepted, read_slots, states, windows)
