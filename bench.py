"""Benchmark of the KDA decode / spec-verify step on GB300.

One step = one kda_step over one batch of the workload (default: large
decode, B = 512 rows x 12 heads x 128, conv width 4, a 1024-slot pool;
805 MB of fp32 state read and written per step, larger than L2).

Prints ONE JSON line:
  value      tokens/s with every input resident in HBM: blocks of exactly
             --steps steps (CUDA events on the launching stream) repeated
             until --min-timed-s seconds of timed work; ms_per_step is the
             median block.  By default (--launch graph) a block is recorded
             once as a CUDA graph of the same kda_step launches and replayed;
             the same blocks launched one step at a time are reported beside
             it (`direct`)
  e2e        the same metric through the public API with host buffers:
             each step copies its projected rows, slots (and accepted) from
             pinned host memory and reads `out` back
  roofline   the step kernel's algorithmic bytes / its average launch time
             against the measured HBM copy bandwidth
  per_workload  the other workloads (tiny decode, batched decode, spec-verify,
             full-width verify), each timed the same way in the same process:
             step time, tokens/s, and the fractions of the HBM peak for the
             state bytes and for all algorithmic bytes
  cpu_baseline  the CPU oracle (plain fp64 C) on a bounded sample of the same
             workload, on every host core (OpenMP over (request, head)) and on
             one thread (one_thread)
  clocks     nvidia-smi samples taken during the timed region

`--impl reference` times the CPU oracle as the reference arm instead.
With torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step); value = all ranks' tokens / the slowest rank.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from linear_attention_decode_03_gb300 import inputs as I  # noqa: E402

METRIC = "KDA tokens/s and achieved HBM GB/s (state R+W) vs GB300 peak, 1 GPU"
L2_BYTES = 129 * 1024 * 1024
E2E_BLOCK = 128  # steps a recorded e2e graph holds (each replay refills the copy pipeline)
HEAD_DIM = 128


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "kda_step_kernel_dram_traffic.txt")
KERNEL_SOURCES = [os.path.join(ROOT, "linear_attention_decode_03_gb300", "csrc", "kda_step.cu")]


def kernel_source_hash() -> str:
    import hashlib

    h = hashlib.sha256()
    for path in KERNEL_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_key(workload: str, state_dtype: str = "f32", v_split: int = 1):
    """The name a capture is filed under: the workload, `_bf16` for a bf16 state
    pool; None for launch shapes that no capture covers (two CTAs a head)."""
    if v_split != 1:
        return None
    return workload if state_dtype == "f32" else f"{workload}_{state_dtype}"


def step_kernel_name(w: I.Workload, state_dtype: str = "f32", v_split: int = 1) -> str:
    """The kernel kda_step launches for this workload: decode of two rows or more
    runs two rows of one head a CTA."""
    if not w.verify and w.L == 1 and v_split == 1 and w.rows >= 2:
        return "kda_decode_pair_kernel"
    return "kda_step_kernel"


def measured_traffic(workload: str, state_dtype: str = "f32", v_split: int = 1):
    """DRAM bytes (read + write) per launch that an ncu capture recorded for
    this workload and state type, or None when there is none or the kernel
    source changed since (the summary stores the hash of the sources it was
    taken on)."""
    key = traffic_key(workload, state_dtype, v_split)
    if key is None or not os.path.exists(TRAFFIC_FILE):
        return None
    src_hash, per_wl = None, {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 2 and parts[0] == "source_sha256":
                src_hash = parts[1]
            elif len(parts) == 3 and parts[0] == "traffic":
                per_wl[parts[1]] = int(parts[2])
    if src_hash != kernel_source_hash():
        return None
    return per_wl.get(key)


def max_over_ranks(values, dist=None, device=None):
    """Element-wise max of per-rank values (identity on one process)."""
    if dist is None:
        return list(values)
    import torch

    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(world: int, rows: int, steps: int, elapsed_ms: float) -> float:
    """Tokens per second of all replicas, timed by the slowest rank."""
    return world * rows * steps / (elapsed_ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 100 ms) with host timestamps."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu_index = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        used = inside
        if not used:  # region shorter than the sampling period: nearest samples after its start
            used = [s for t, s in self.samples if t >= t0][:2]
        sm = [float(s[0]) for s in used if s[0].replace(".", "").isdigit()]
        smax = [float(s[1]) for s in used if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in used for n, v in zip(names, s[4:8]) if v.lower() == "active"})
        power = [float(s[2]) for s in used if s[2].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(used), "samples_in_region": len(inside),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------ device setup
class DeviceWorkload:
    """One workload's inputs resident on the device (pools sentinel-filled,
    read slots filled from the seeded generator)."""

    def __init__(self, si: I.StepInputs, device, gate_mode: int = 0, plan: bool = False, state_dtype: str = "f32",
                 prep=None, v_split: int = 1):
        import torch
        import linear_attention_decode_03_gb300 as kda

        self.si, self.w = si, si.workload
        w = self.w
        self.device = device

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

        wt = si.weights
        self.own_prep = prep is None
        self.prep = prep if prep is not None else kda.PreparedKda(
            bf16(wt.conv_w), None if wt.bias is None else bf16(wt.bias), bf16(wt.f_b),
            torch.from_numpy(wt.A_log).to(device), torch.from_numpy(wt.dt_bias).to(device),
            torch.from_numpy(wt.o_norm).to(device), gate_lower_bound=wt.gate_lower_bound,
            eps=wt.eps, conv_dim_first=True, gate_mode=gate_mode, state_dtype=state_dtype, v_split=v_split)
        self.projected = bf16(si.projected)
        idx = torch.from_numpy(si.read_slots).to(device)
        if state_dtype == "bf16":
            self.state = torch.empty((w.pool, w.heads, HEAD_DIM, HEAD_DIM), dtype=torch.bfloat16, device=device)
            self.state.view(torch.int16).fill_(int(np.array(I.STATE_SENTINEL_BF16).view(np.int16)))
            self.state[idx] = bf16(si.states_bf16())
        else:
            self.state = torch.empty((w.pool, w.heads, HEAD_DIM, HEAD_DIM), dtype=torch.float32, device=device)
            self.state.view(torch.int32).fill_(int(I.STATE_SENTINEL.view(np.int32)))
            self.state[idx] = torch.from_numpy(si.states).to(device)
        self.conv = torch.empty((w.pool, 3 * w.dim, w.width - 1), dtype=torch.bfloat16, device=device)
        self.conv.view(torch.int16).fill_(int(np.array(I.CONV_SENTINEL).view(np.int16)))
        self.conv[idx] = bf16(si.windows)
        self.slots = torch.from_numpy(si.slots.copy()).to(device)
        if w.verify:
            self.slots = self.slots.view(w.requests, w.L)
        self.accepted = None if si.accepted is None else torch.from_numpy(si.accepted.copy()).to(device)
        self.out = torch.empty((w.rows, w.dim), dtype=torch.bfloat16, device=device)
        self.plan = None
        if plan:  # the step recorded once as a CUDA graph (PreparedKda.plan)
            self.plan = self.prep.plan(self.projected, self.out, caches=(self.conv, self.state), slots=self.slots,
                                       accepted=self.accepted)

    def step(self):
        if self.plan is not None:
            self.plan.launch()
            return
        self.prep.run(self.projected, self.out, caches=(self.conv, self.state), slots=self.slots,
                      accepted=self.accepted)


def algorithmic_bytes(w: I.Workload, state_dtype: str = "f32"):
    """(state bytes, all bytes) per step; a bf16 state pool moves half the state bytes."""
    state = w.state_bytes // 2 if state_dtype == "bf16" else w.state_bytes
    return state, state + w.other_bytes


# ----------------------------------------------------------- CPU oracle arm
def oracle_sample_inputs(si: I.StepInputs, reqs, state_dtype: str = "f32"):
    """Inputs of requests `reqs` with the pools compacted to the slots they touch."""
    w = si.workload
    L = w.L
    slots2 = si.slots.reshape(w.requests, L)[reqs]
    used = np.unique(slots2)
    pos = {int(s): i for i, s in enumerate(used)}
    read_pos = {int(s): i for i, s in enumerate(si.read_slots)}
    if state_dtype == "bf16":
        cpool = np.full((len(used), w.heads, HEAD_DIM, HEAD_DIM), I.STATE_SENTINEL_BF16, dtype=np.uint16)
        states = si.states_bf16()
    else:
        cpool = np.empty((len(used), w.heads, HEAD_DIM, HEAD_DIM), dtype=np.float32)
        cpool.view(np.uint32)[...] = I.STATE_SENTINEL
        states = si.states
    cconv = np.full((len(used), 3 * w.dim, w.width - 1), I.CONV_SENTINEL, dtype=np.uint16)
    for s, i in pos.items():
        if s in read_pos:
            cpool[i] = states[read_pos[s]]
            cconv[i] = si.windows[read_pos[s]]
    cslots = np.array([pos[int(s)] for s in slots2.reshape(-1)], dtype=np.int32)
    rows = (np.asarray(reqs)[:, None] * L + np.arange(L)[None, :]).reshape(-1)
    acc = None if si.accepted is None else si.accepted[reqs]
    return si.projected[rows], cconv, cpool, cslots, acc


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def time_oracle(si: I.StepInputs, n_requests: int, repeats: int = 1, state_dtype: str = "f32", threads: int = 1):
    """Seconds and tokens of the C oracle over the first `n_requests` requests,
    `repeats` passes, on `threads` OpenMP threads over (request, head)."""
    import oracle

    W = oracle.Weights(**si.weights.as_dict())
    reqs = np.arange(min(n_requests, si.workload.requests))
    proj, cconv, cpool, cslots, acc = oracle_sample_inputs(si, reqs, state_dtype)
    t0 = time.perf_counter()
    for _ in range(repeats):
        oracle.step(W, proj, cconv, cpool, cslots, si.workload.L, acc, state_dtype=state_dtype, threads=threads)
    dt = time.perf_counter() - t0
    return dt, len(reqs) * si.workload.L * repeats


def oracle_sample_size(si: I.StepInputs, budget_s: float, state_dtype: str, threads: int):
    """Whole requests (in order) whose oracle pass takes about `budget_s`,
    measured on a calibration pass of enough requests to give every thread a
    (request, head) task; and the passes that fill the budget."""
    w = si.workload
    n0 = min(w.requests, max(1, -(-threads // w.heads)))
    dt0, _ = time_oracle(si, n0, state_dtype=state_dtype, threads=threads)
    n = int(max(1, min(w.requests, n0 * budget_s / max(dt0, 1e-6))))
    repeats = int(max(1, budget_s / max(dt0 * n / n0, 1e-6)))
    return n, repeats


def cpu_baseline(si: I.StepInputs, budget_s: float = 10.0, state_dtype: str = "f32"):
    """The oracle on a bounded sample of the workload (about `budget_s` of CPU
    work each): on every host core (OpenMP over (request, head); the
    headline), and on one thread."""
    import oracle

    w = si.workload
    res = {}
    for threads in sorted({host_cores(), 1}, reverse=True):
        used = min(threads, oracle.max_threads()) if threads > 1 else 1
        n, repeats = oracle_sample_size(si, budget_s, state_dtype, used)
        dt, tok = time_oracle(si, n, repeats, state_dtype, used)
        res[used] = {"value": tok / dt, "unit": "tokens/s", "cores": used, "kind": "oracle",
                     "sample": f"first {n} of {w.requests} requests of the {w.name} workload x {repeats} passes "
                               f"({tok} tokens x {w.heads} heads), fp64 C oracle, {used} thread(s), {dt:.1f} s"}
    top = res[max(res)]
    if 1 in res and max(res) != 1:
        top = dict(top, one_thread=res[1])
    return top


def run_reference(args, w: I.Workload):
    """The reference arm: the oracle, as it stands, on every host core (OpenMP
    over (request, head)), each step a bounded sample of the workload."""
    import oracle

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    si = I.make_step_inputs(w)
    sd = args.state_dtype
    threads = min(host_cores(), oracle.max_threads())
    per_step_budget = 150.0 / max(args.steps + args.warmup, 1)
    n, _ = oracle_sample_size(si, per_step_budget, sd, threads)
    for _ in range(args.warmup):
        time_oracle(si, n, state_dtype=sd, threads=threads)
    total_t, total_tok = 0.0, 0
    for _ in range(args.steps):
        dt, tok = time_oracle(si, n, state_dtype=sd, threads=threads)
        total_t += dt
        total_tok += tok
    value = total_tok / total_t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: first {n} of {w.requests} requests of {w.name} "
                                   f"({n * w.L} tokens x {w.heads} heads), fp64 C oracle, {threads} thread(s)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def workload_config(w: I.Workload, args):
    state, allb = algorithmic_bytes(w, getattr(args, "state_dtype", "f32"))
    big = state > L2_BYTES
    n_copies = getattr(args, "rotation_copies", 0)
    if n_copies:
        l2 = (f"inputs larger than L2: {n_copies} independent copies of the workload's caches and inputs "
              f"({n_copies * allb / 1e6:.0f} MB touched a round), stepped through in turn back to back")
    elif big:
        l2 = "inputs larger than L2 (%.0f MB of state per step)" % (state / 1e6)
    else:
        l2 = "L2 flushed between timed steps (256 MiB write, then 256 MiB read; outside the per-step events)"
    return {"workload": w.name, "heads": w.heads, "head_dim": HEAD_DIM, "requests": w.requests, "tokens_per_request": w.L,
            "rows": w.rows, "pool_slots": w.pool, "conv_width": w.width, "state_bytes_per_step": state,
            "algorithmic_bytes_per_step": allb, "l2": l2,
            "parallelism": "replicas" if args.gpus > 1 else "single GPU",
            "gate": getattr(args, "gate_mode", "sigmoid"),
            "launch": getattr(args, "launch", "direct"),
            "v_split": getattr(args, "v_split", 1),
            "state_storage": getattr(args, "state_dtype", "f32")}


# ------------------------------------------------------ the layer's projections
PROJ_METRIC = "projection tokens/s (kda_linear: in_proj or o_proj of the KDA layer) vs GB300 peak, 1 GPU"
HIDDEN = 7168  # the model width the projections map from / to


def bf16_tflops_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def overlapped_e2e(device, steps, upload, compute, download, nb=2, graph=True):
    """End-to-end time per step (ms) of `steps` steps, each: upload(b) (host -> device
    copies of buffer set b) on a stream of its own, compute(b) on the compute stream,
    download(b) (device -> host) on a third stream; two buffer sets, so step i+1's inputs
    go up and step i-1's outputs come back while step i computes.  With `graph`, blocks
    of E2E_BLOCK steps are recorded once as a CUDA graph and replayed, so the host does
    not pace short steps; else the blocks are issued directly."""
    import torch

    up, down, cap = torch.cuda.Stream(device), torch.cuda.Stream(device), torch.cuda.Stream(device)
    in_ready = [torch.cuda.Event() for _ in range(nb)]
    done = [torch.cuda.Event() for _ in range(nb)]
    out_back = [torch.cuda.Event() for _ in range(nb)]

    def block(n):
        up.wait_stream(cap)
        down.wait_stream(cap)
        for i in range(n):
            b = i % nb
            with torch.cuda.stream(up):
                if i >= nb:
                    up.wait_event(done[b])  # the compute that read buffer set b is done
                upload(b)
                in_ready[b].record(up)
            cap.wait_event(in_ready[b])
            if i >= nb:
                cap.wait_event(out_back[b])  # buffer set b's last output is home
            with torch.cuda.stream(cap):
                compute(b)
            done[b].record(cap)
            with torch.cuda.stream(down):
                down.wait_event(done[b])
                download(b)
                out_back[b].record(down)
        cap.wait_stream(up)
        cap.wait_stream(down)

    block(E2E_BLOCK)  # warm: allocations, first launches
    torch.cuda.synchronize(device)
    reps = max(1, -(-steps // E2E_BLOCK))
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            block(E2E_BLOCK)
        with torch.cuda.stream(cap):  # replay() launches on the current stream
            g.replay()
        torch.cuda.synchronize(device)
        run = g.replay
    else:
        def run():
            block(E2E_BLOCK)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cap):
        e0.record(cap)
        for _ in range(reps):
            run()
        e1.record(cap)
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1) / (reps * E2E_BLOCK), reps * E2E_BLOCK


def run_linear(args, w: I.Workload):
    """--op in_proj / o_proj: kda_linear on the layer's shape for the workload's
    rows (in_proj: x [rows, 7168] . W [pitch, 7168]^T; o_proj: core [rows, D] .
    W [7168, D]^T), one launch a step, L2 flushed between steps (the weight fits
    L2 but would not stay there across a model's layers)."""
    import torch
    import linear_attention_decode_03_gb300 as kda
    from oracle import linear as OL

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    kda.build()
    kda.load_library()
    rows = w.rows
    K, N = (HIDDEN, w.pitch) if args.op == "in_proj" else (w.dim, HIDDEN)
    rng = np.random.Generator(np.random.PCG64(w.seed + 17))
    xb = I.to_bf16_bits(rng.normal(0.0, 1.0, size=(rows, K)).astype(np.float32))
    wb = I.to_bf16_bits(rng.normal(0.0, 0.02, size=(N, K)).astype(np.float32))

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    x, W = dev(xb), dev(wb)
    y = torch.empty((rows, N), dtype=torch.bfloat16, device=device)
    nbytes = N * K * 2 + rows * K * 2 + rows * N * 2
    flops = 2 * rows * N * K
    hbm, hbm_src = load_peaks()
    tf, tf_src = bf16_tflops_peak()
    tensor_bound = flops / nbytes > tf * 1e12 / (hbm * 1e9)
    scratch = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    scratch_rd = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        kda.linear(x, W, y)
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    t_host0 = time.time()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        scratch.fill_(float(i))
        scratch_rd.sum()
        starts[i].record(stream)
        kda.linear(x, W, y)
        ends[i].record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = sum(step_ms) / args.steps
    median_ms = statistics.median(step_ms)
    # e2e: x up from pinned host memory and y back every step (the weight is resident),
    # copies overlapped with the products on streams of their own
    hx = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16).pin_memory()
    hy = torch.empty((rows, N), dtype=torch.bfloat16).pin_memory()
    dx = [torch.empty_like(x) for _ in range(2)]
    dy = [torch.empty_like(y) for _ in range(2)]
    e2e_ms, e2e_steps = overlapped_e2e(
        device, args.e2e_steps or max(3, min(args.steps, 200)),
        upload=lambda b: dx[b].copy_(hx, non_blocking=True),
        compute=lambda b: kda.linear(dx[b], W, dy[b]),
        download=lambda b: hy.copy_(dy[b], non_blocking=True))
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": flops / (ms / 1e3) / 1e12, "peak": tf, "unit": "TFLOP/s",
                "peak_source": f"{tf_src} bf16_tflops (MEASURED_PEAKS.json)"}
    else:
        roof = {"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                "peak_source": f"{hbm_src} hbm_gbs (MEASURED_PEAKS.json)"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = None
    roof["kernel"] = "kda_linear_kernel"
    line = {
        "metric": PROJ_METRIC, "value": rows / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": median_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 x bf16 -> f32 accumulate", "data": "synthetic",
        "config": {"workload": f"{args.op} for {w.name}", "op": args.op, "rows": rows, "in_features": K,
                   "out_features": N, "weight_bytes": N * K * 2, "algorithmic_bytes_per_step": nbytes,
                   "flops_per_step": flops,
                   "l2": "L2 flushed between timed steps (256 MiB write, then 256 MiB read; outside the events)"},
        "roofline": roof,
        "e2e": {"value": rows / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": rows * K * 2,
                "d2h_bytes_per_step": rows * N * 2, "steps": e2e_steps,
                "overlap": f"uploads and downloads on streams of their own, two buffer sets; blocks of {E2E_BLOCK} "
                           "steps recorded as a CUDA graph"},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(t_host0, t_host1),
    }
    if not args.no_cpu_baseline:
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 5.0 or reps == 0:
            OL.linear(xb, wb)
            reps += 1
        dt = (time.perf_counter() - t0) / reps
        line["cpu_baseline"] = {"value": rows / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"the whole step ({rows} rows), fp64 NumPy product (BLAS threads), "
                                          f"{reps} runs in {time.perf_counter() - t0:.1f} s"}
    print(json.dumps(line), flush=True)


LAYER_METRIC = "KDA layer tokens/s (in_proj -> KDA core -> o_proj as one CUDA graph) vs GB300 peak, 1 GPU"


def _timed_launches(fn, steps, stream, flush_w, flush_r):
    """Per-call device times (ms) of `fn`, L2 flushed (outside the events) before each."""
    import torch

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush_w.fill_(float(i))
        flush_r.sum()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def run_layer(args, w: I.Workload):
    """--op layer: one step of the whole layer -- in_proj (x [rows, 7168] -> the packed
    projection row), the KDA core, o_proj (core_out -> [rows, 7168]) -- recorded once as
    a CUDA graph (PreparedKda.layer_plan, programmatic dependent launches between the
    kernels) and replayed every step, L2 flushed between steps. Also timed: the same graph
    without dependent launches, and the three calls made one by one."""
    import torch
    import linear_attention_decode_03_gb300 as kda
    from oracle import linear as OL

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    kda.build()
    kda.load_library()
    si = I.make_step_inputs(w)
    dw = DeviceWorkload(si, device, gate_mode=0 if args.gate_mode == "sigmoid" else 1,
                        state_dtype=args.state_dtype, v_split=args.v_split)
    rng = np.random.Generator(np.random.PCG64(w.seed + 29))
    xb = I.to_bf16_bits(rng.normal(0.0, 1.0, size=(w.rows, HIDDEN)).astype(np.float32))
    wib = I.to_bf16_bits(rng.normal(0.0, 0.02, size=(w.pitch, HIDDEN)).astype(np.float32))
    wob = I.to_bf16_bits(rng.normal(0.0, 0.05, size=(HIDDEN, w.dim)).astype(np.float32))

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    x, w_in, w_o = dev(xb), dev(wib), dev(wob)
    y = torch.empty((w.rows, HIDDEN), dtype=torch.bfloat16, device=device)
    caches = (dw.conv, dw.state)
    masks = {"both": 3, "none": 0, "step_edge": 1, "o_proj_edge": 2}
    plans = {k: dw.prep.layer_plan(x, w_in, dw.projected, dw.out, w_o, y, caches=caches, slots=dw.slots,
                                   accepted=dw.accepted, pdl=m) for k, m in masks.items()}
    head = args.layer_pdl
    stream = torch.cuda.current_stream(device)
    flush_w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    flush_r = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    def separate():
        kda.linear(x, w_in, dw.projected)
        dw.prep.run(dw.projected, dw.out, caches=caches, slots=dw.slots, accepted=dw.accepted)
        kda.linear(dw.out, w_o, y)

    for _ in range(args.warmup):
        for p in plans.values():
            p.launch()
        separate()
    torch.cuda.synchronize()
    if dw.prep.check() != 0 or kda.kda_linear_check() != 0:
        raise RuntimeError("device error bits set during warm-up")
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    t_host0 = time.time()
    t_head = _timed_launches(plans[head].launch, args.steps, stream, flush_w, flush_r)
    t_host1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    others = {k: sum(_timed_launches(p.launch, args.steps, stream, flush_w, flush_r)) / args.steps
              for k, p in plans.items() if k != head}
    t_sep = _timed_launches(separate, args.steps, stream, flush_w, flush_r)
    if dw.prep.check() != 0 or kda.kda_linear_check() != 0:
        raise RuntimeError("device error bits set during the timed steps")
    ms = sum(t_head) / args.steps
    median_ms = statistics.median(t_head)

    # e2e: x up from pinned host memory and y back every step, copies overlapped with the
    # layer on streams of their own: two buffer sets, a layer plan on each (the caches are
    # shared, so the steps stay in order on the compute stream)
    hx = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16).pin_memory()
    hy = torch.empty((w.rows, HIDDEN), dtype=torch.bfloat16).pin_memory()
    sets = [(torch.empty_like(x), torch.empty_like(dw.projected), torch.empty_like(dw.out), torch.empty_like(y))
            for _ in range(2)]
    e2e_plans = [dw.prep.layer_plan(bx, w_in, bp, bc, w_o, by, caches=caches, slots=dw.slots, accepted=dw.accepted,
                                    pdl=masks[head]) for bx, bp, bc, by in sets]
    e2e_ms, e2e_steps = overlapped_e2e(
        device, args.e2e_steps or max(3, min(args.steps, 200)),
        upload=lambda b: sets[b][0].copy_(hx, non_blocking=True),
        compute=lambda b: e2e_plans[b].launch(),
        download=lambda b: hy.copy_(sets[b][3], non_blocking=True), graph=False)

    state_b, step_b = algorithmic_bytes(w, args.state_dtype)
    proj_b = (w.pitch * HIDDEN + HIDDEN * w.dim) * 2 + w.rows * (HIDDEN * 2 + w.pitch + w.dim) * 2
    layer_b = step_b + proj_b
    flops = 2 * w.rows * HIDDEN * (w.pitch + w.dim)
    peak, peak_kind = load_peaks()
    achieved = layer_b / (ms / 1e3) / 1e9
    line = {
        "metric": LAYER_METRIC, "value": w.rows / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": median_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 projections (fp32 accumulate), f32 core", "data": "synthetic",
        "config": dict(workload_config(w, args), workload=f"layer for {w.name}", op="layer", hidden=HIDDEN,
                       dependent_launch_edges=head,
                       weight_bytes=(w.pitch * HIDDEN + HIDDEN * w.dim) * 2, algorithmic_bytes_per_step=layer_b,
                       projection_flops_per_step=flops,
                       l2="L2 flushed between timed steps (256 MiB write, then 256 MiB read; outside the events)"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "kernel": "layer graph (kda_linear, kda_step_kernel, kda_linear)",
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)"},
        "layer_ms": dict({f"graph_pdl_{head}": ms}, **{f"graph_pdl_{k}": v for k, v in others.items()},
                         three_calls=sum(t_sep) / args.steps),
        "e2e": {"value": w.rows / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": w.rows * HIDDEN * 2,
                "d2h_bytes_per_step": w.rows * HIDDEN * 2, "steps": e2e_steps,
                "overlap": "uploads and downloads on streams of their own, two buffer sets, each with a layer "
                           "plan (a CUDA graph)"},
        "gpu_launches": 3 * args.steps,
        "clocks": sampler.summary(t_host0, t_host1),
    }
    if not args.no_cpu_baseline:
        cb = cpu_baseline(si, budget_s=8.0, state_dtype=args.state_dtype)
        t0 = time.perf_counter()
        OL.linear(xb, wib)
        OL.linear(xb[:, :w.dim], wob)  # o_proj's shape: rows x D . (hidden x D)^T
        t_proj = time.perf_counter() - t0
        per_tok = 1.0 / cb["value"] + t_proj / w.rows
        line["cpu_baseline"] = {"value": 1.0 / per_tok, "unit": "tokens/s", "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": cb["sample"] + f"; plus both projections of all {w.rows} rows in fp64 "
                                                         f"NumPy ({t_proj:.2f} s, BLAS threads)"}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- step timing
MIN_TIMED_S = 0.5
PER_WORKLOAD = ["tiny_decode", "batched_decode", "spec_verify", "large_decode", "full_width_verify"]


def make_flush(device):
    """Two 256 MiB buffers: writing one and reading the other between timed
    steps leaves L2 holding neither the step's data nor dirty lines."""
    import torch

    return (torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device),
            torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device))


def time_blocks(step, steps, stream, flush_bufs, min_s=MIN_TIMED_S):
    """Blocks of `steps` steps, repeated until `min_s` seconds of timed work.
    With flush_bufs each step is timed alone (CUDA events on `stream`) after an
    L2 flush outside the events; otherwise a block is `steps` back-to-back
    steps between two events (inputs larger than L2).  Returns the ms per step
    of every block and the single-step times (flushed case only)."""
    import torch

    blocks, step_ms, total = [], [], 0.0
    while total < min_s * 1e3 or not blocks:
        if flush_bufs is not None:
            fw, fr = flush_bufs
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            for i in range(steps):
                fw.fill_(float(i))
                fr.sum()
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            torch.cuda.synchronize()
            ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
            step_ms.extend(ms)
            block = sum(ms)
        else:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                step()
            e1.record(stream)
            torch.cuda.synchronize()
            block = e0.elapsed_time(e1)
        blocks.append(block / steps)
        total += block
    return blocks, step_ms


def touched_bytes(w: I.Workload, state_dtype: str = "f32") -> int:
    """Bytes one step reads or writes (state, projected rows, out, conv windows)."""
    return algorithmic_bytes(w, state_dtype)[1]


def rotation_copies(w: I.Workload, state_dtype: str = "f32") -> int:
    """Independent copies of a workload's caches and inputs that a run steps
    through in turn so that each step finds none of its data in L2: the other
    copies' steps in between touch at least three times the L2 size.  0 when
    one step's own bytes already exceed L2 (no copies needed) or are too few
    for copies to be sensible (a latency case: its steps are flushed)."""
    t = touched_bytes(w, state_dtype)
    if t > L2_BYTES or t < L2_BYTES // 8:
        return 0
    return 1 + -(-3 * L2_BYTES // t)


def make_copies(si: I.StepInputs, device, args, n: int):
    """n device copies of one workload's caches and inputs sharing one prepared
    weight handle (the layer's weights are the same for every copy)."""
    plan = args.launch == "plan"
    first = DeviceWorkload(si, device, gate_mode=0 if args.gate_mode == "sigmoid" else 1, plan=plan,
                           state_dtype=args.state_dtype, v_split=getattr(args, "v_split", 1))
    return [first] + [DeviceWorkload(si, device, plan=plan, state_dtype=args.state_dtype, prep=first.prep)
                      for _ in range(n - 1)]


def time_rotating(copies, steps, stream, min_s=MIN_TIMED_S):
    """Blocks of `steps` back-to-back steps, step i on copy i mod len(copies),
    launched one by one between two CUDA events; repeated until `min_s`
    seconds of timed work.  Returns the ms per step of every block."""
    import torch

    blocks, total, i = [], 0.0, 0
    while total < min_s * 1e3 or not blocks:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            copies[i % len(copies)].step()
            i += 1
        e1.record(stream)
        torch.cuda.synchronize()
        block = e0.elapsed_time(e1)
        blocks.append(block / steps)
        total += block
    return blocks


def record_block(copies, steps, device):
    """One CUDA graph holding a block of `steps` steps, step i on copy
    i mod len(copies): the same kernel launches, with the same arguments, that
    the direct loop makes, so that a replay runs them with no host in between."""
    import torch

    cur = torch.cuda.current_stream(device)
    cap = torch.cuda.Stream(device)
    cap.wait_stream(cur)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for i in range(steps):
            copies[i % len(copies)].step()
    cur.wait_stream(cap)
    torch.cuda.synchronize(device)
    return g


def time_graph(graph, steps, stream, min_s=MIN_TIMED_S):
    """Replays of a recorded block of `steps` steps between two CUDA events on
    `stream`, repeated until `min_s` seconds of timed work.  Returns the ms per
    step of every replay."""
    import torch

    blocks, total = [], 0.0
    while total < min_s * 1e3 or not blocks:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        block = e0.elapsed_time(e1)
        blocks.append(block / steps)
        total += block
    return blocks


def time_steps(copies, steps, stream, flush_bufs, launch, device, min_s=MIN_TIMED_S):
    """The step time of one workload under the chosen launch mode.

    Steps back to back (on rotating copies, or on one copy whose inputs exceed
    L2): with launch == "graph" each block is one replay of the block recorded
    as a CUDA graph, and the same blocks launched one step at a time are timed
    too (returned as `direct`); otherwise the steps are launched one by one
    (kda_step calls, or plan launches).  Flushed single steps are always
    launched one by one.  Returns (blocks, single-step times, direct blocks)."""
    if flush_bufs is not None:
        blocks, step_ms = time_blocks(copies[0].step, steps, stream, flush_bufs, min_s)
        return blocks, step_ms, None
    if launch != "graph":
        return time_rotating(copies, steps, stream, min_s), [], None
    graph = record_block(copies, steps, device)
    graph.replay()  # first replay uploads the graph
    blocks = time_graph(graph, steps, stream, min_s)
    del graph
    direct = time_rotating(copies, steps, stream, min_s)
    return blocks, [], direct


def launch_rule(args, flushed: bool) -> str:
    if flushed:
        return "each step launched directly (kda_step) between its own CUDA events"
    if args.launch == "graph":
        return (f"each block of {args.steps} steps recorded once as a CUDA graph and replayed "
                "(the same kda_step launches, no host between them)")
    if args.launch == "plan":
        return "every step launched through a launch plan (the step recorded once as a CUDA graph)"
    return "every step launched directly (kda_step)"


def direct_record(direct, w: I.Workload, state_b: int, all_b: int, peak: float) -> dict:
    """The same blocks launched one step at a time, for comparison."""
    ms = statistics.median(direct)
    return {"ms_per_step": ms, "tokens_per_s": w.rows / (ms / 1e3), "blocks": len(direct),
            "state_frac_of_peak": state_b / (ms / 1e3) / 1e9 / peak, "frac": all_b / (ms / 1e3) / 1e9 / peak,
            "rule": "the same blocks, every step launched directly (kda_step) from the host loop"}


def measure_workload(w: I.Workload, device, args):
    """One more workload in the same process: step time (median block), tokens/s
    and the fractions of the measured HBM peak, for the state bytes alone and
    for all algorithmic bytes."""
    import torch

    si = I.make_step_inputs(w)
    state_b, all_b = algorithmic_bytes(w, args.state_dtype)
    n_copies = rotation_copies(w, args.state_dtype)
    copies = make_copies(si, device, args, max(n_copies, 1))
    dw = copies[0]
    stream = torch.cuda.current_stream(device)
    for _ in range(max(args.warmup, 3)):
        for c in copies:
            c.step()
    if dw.prep.check() != 0:
        raise RuntimeError(f"device error bits set during warm-up ({w.name})")
    flush_rec = None
    flush_bufs = None if (n_copies or state_b > L2_BYTES) else make_flush(device)
    blocks, step_ms, direct = time_steps(copies, args.steps, stream, flush_bufs, args.launch, device,
                                         args.min_timed_s)
    if n_copies:
        # the same steps one at a time after an L2 flush, for comparison
        flush_bufs = make_flush(device)
        fb, fms = time_blocks(dw.step, args.steps, stream, flush_bufs, args.min_timed_s)
        flush_rec = {"ms_per_step": statistics.median(fb), "ms_per_step_median_single_step": statistics.median(fms),
                     "rule": "each step alone, launched directly, L2 flushed before it (256 MiB write, then "
                             "256 MiB read), CUDA events around the step"}
    if dw.prep.check() != 0:
        raise RuntimeError(f"device error bits set during the timed steps ({w.name})")
    ms = statistics.median(blocks)
    peak, _ = load_peaks()
    rec = {"ms_per_step": ms, "tokens_per_s": w.rows / (ms / 1e3), "rows": w.rows, "heads": w.heads, "L": w.L,
           "state_bytes_per_step": state_b, "algorithmic_bytes_per_step": all_b,
           "state_gbs": state_b / (ms / 1e3) / 1e9, "state_frac_of_peak": state_b / (ms / 1e3) / 1e9 / peak,
           "achieved_gbs": all_b / (ms / 1e3) / 1e9, "frac": all_b / (ms / 1e3) / 1e9 / peak,
           "blocks": len(blocks), "launches": args.steps * len(blocks),
           "launch": launch_rule(args, flush_bufs is not None and not n_copies),
           "ms_per_step_median_single_step": statistics.median(step_ms) if step_ms else None,
           "l2": (f"inputs larger than L2: {n_copies} independent copies of the workload's caches and inputs "
                  f"({n_copies * touched_bytes(w, args.state_dtype) / 1e6:.0f} MB touched a round), stepped "
                  "through in turn back to back" if n_copies else
                  "inputs larger than L2" if flush_bufs is None else "L2 flushed between timed steps"),
           "traffic": measured_traffic(w.name, args.state_dtype, getattr(args, "v_split", 1))}
    if direct is not None:
        rec["direct_launch"] = direct_record(direct, w, state_b, all_b, peak)
    if flush_rec is not None:
        flush_rec["tokens_per_s"] = w.rows / (flush_rec["ms_per_step"] / 1e3)
        flush_rec["state_frac_of_peak"] = state_b / (flush_rec["ms_per_step"] / 1e3) / 1e9 / peak
        flush_rec["frac"] = all_b / (flush_rec["ms_per_step"] / 1e3) / 1e9 / peak
        rec["flushed_single_step"] = flush_rec
    del dw, copies, flush_bufs
    torch.cuda.empty_cache()
    return rec


# -------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["kda", "reference"], default="kda")
    ap.add_argument("--workload", default="large_decode", choices=sorted(I.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--min-timed-s", type=float, default=MIN_TIMED_S,
                    help="blocks of --steps steps are repeated until this much timed work; "
                         "ms_per_step is the median block")
    ap.add_argument("--l2-flush", action="store_true",
                    help="time a workload whose step fits L2 as single steps after an L2 flush instead of on "
                         "independent copies stepped through in turn")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the other workloads (per_workload) measured after the main one")
    ap.add_argument("--launch", choices=["graph", "direct", "plan"], default="graph",
                    help="graph: each timed block of --steps steps recorded once as a CUDA graph and replayed "
                         "(the direct launches are timed too and reported beside); direct: every step launched "
                         "from the host loop; plan: every step launched through a launch plan")
    ap.add_argument("--state-dtype", choices=["f32", "bf16"], default="f32",
                    help="state pool storage type (kda_set_state_dtype); the step computes in fp32 either way")
    ap.add_argument("--op", choices=["step", "in_proj", "o_proj", "layer"], default="step",
                    help="step: the KDA core (default); in_proj / o_proj: the layer's projections (kda_linear) "
                         "for the workload's rows; layer: in_proj -> core -> o_proj as one CUDA graph")
    ap.add_argument("--layer-pdl", choices=["none", "step_edge", "o_proj_edge", "both"], default="both",
                    help="--op layer: the edges of the timed graph launched as programmatic dependents "
                         "(the others are timed too and reported under layer_ms)")
    ap.add_argument("--v-split", type=int, choices=[1, 2], default=1,
                    help="CTAs a (request, head) (kda_set_v_split); 2 splits the v rows over a cluster of two")
    ap.add_argument("--gate-mode", choices=["sigmoid", "softplus"], default="sigmoid",
                    help="decay gate form (kda_set_gate_mode); the default is the reading the step follows")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = I.WORKLOADS[args.workload]

    if args.impl == "reference":
        run_reference(args, w)
        return
    if args.op == "layer":
        run_layer(args, w)
        return
    if args.op != "step":
        run_linear(args, w)
        return

    import torch
    import linear_attention_decode_03_gb300 as kda

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist = dist_mod
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    kda.build()
    kda.load_library()

    si = I.make_step_inputs(w)
    state_b, all_b = algorithmic_bytes(w, args.state_dtype)
    # a workload whose step fits L2 is timed on independent copies stepped through in
    # turn (inputs larger than L2), unless --l2-flush asks for flushed single steps
    n_copies = 0 if args.l2_flush else rotation_copies(w, args.state_dtype)
    args.rotation_copies = n_copies
    copies = make_copies(si, device, args, max(n_copies, 1))
    dw = copies[0]
    flush_bufs = make_flush(device) if (not n_copies and state_b <= L2_BYTES) else None
    stream = torch.cuda.current_stream(device)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(device)

    for _ in range(args.warmup):
        for c in copies:
            c.step()
    if dw.prep.check() != 0:
        raise RuntimeError("device error bits set during warm-up")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier()
    t_host0 = time.time()
    blocks, step_ms, direct = time_steps(copies, args.steps, stream, flush_bufs, args.launch, device,
                                         args.min_timed_s)
    barrier()
    t_host1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    # the median block (each block is --steps steps) is the step time; the mean is kept beside it
    block_ms = statistics.median(blocks)
    elapsed_ms = block_ms * args.steps
    median_ms = statistics.median(step_ms) if step_ms else None
    flags = dw.prep.check()
    if flags != 0:
        raise RuntimeError(f"device error bits {flags} during the timed steps")

    # e2e through the public API with host buffers (pinned), every step's copies inside the
    # timed region.  Uploads and downloads run on streams of their own with two buffer
    # sets, so that step i+1's inputs go up and step i-1's output comes back while step
    # i's kernel runs (the kernels stay in order on the compute stream: the caches chain
    # them).
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 500))
    h_proj = torch.from_numpy(np.ascontiguousarray(si.projected).view(np.int16)).view(torch.bfloat16).pin_memory()
    h_slots = torch.from_numpy(si.slots.copy()).pin_memory()
    h_acc = None if si.accepted is None else torch.from_numpy(si.accepted.copy()).pin_memory()
    h_out = torch.empty((w.rows, w.dim), dtype=torch.bfloat16).pin_memory()
    h2d = h_proj.numel() * 2 + h_slots.numel() * 4 + (0 if h_acc is None else h_acc.numel() * 4)
    d2h = h_out.numel() * 2
    nb = 2
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    d_proj = [torch.empty_like(dw.projected) for _ in range(nb)]
    d_slots = [torch.empty_like(dw.slots) for _ in range(nb)]
    d_acc = [None if h_acc is None else torch.empty_like(dw.accepted) for _ in range(nb)]
    d_out = [torch.empty_like(dw.out) for _ in range(nb)]
    in_ready = [torch.cuda.Event() for _ in range(nb)]
    done = [torch.cuda.Event() for _ in range(nb)]
    out_back = [torch.cuda.Event() for _ in range(nb)]

    def e2e_block(n, compute):
        """n steps; kernels on `compute`, copies forked onto `up` / `down` and joined back."""
        up.wait_stream(compute)
        down.wait_stream(compute)
        for i in range(n):
            b = i % nb
            with torch.cuda.stream(up):
                if i >= nb:
                    up.wait_event(done[b])  # the kernel that read buffer set b is done
                d_proj[b].copy_(h_proj, non_blocking=True)
                d_slots[b].view(-1).copy_(h_slots, non_blocking=True)
                if d_acc[b] is not None:
                    d_acc[b].copy_(h_acc, non_blocking=True)
                in_ready[b].record(up)
            compute.wait_event(in_ready[b])
            if i >= nb:
                compute.wait_event(out_back[b])  # buffer set b's last output is home
            with torch.cuda.stream(compute):
                dw.prep.run(d_proj[b], d_out[b], caches=(dw.conv, dw.state), slots=d_slots[b], accepted=d_acc[b])
            done[b].record(compute)
            with torch.cuda.stream(down):
                down.wait_event(done[b])
                h_out.copy_(d_out[b], non_blocking=True)
                out_back[b].record(down)
        compute.wait_stream(up)
        compute.wait_stream(down)

    # the host side of a step (copies, event waits, the launch) would pace small batches,
    # so blocks of E2E_BLOCK steps are recorded once as a CUDA graph and replayed
    cap = torch.cuda.Stream(device)
    e2e_block(E2E_BLOCK, cap)
    barrier()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        e2e_block(E2E_BLOCK, cap)
    reps = max(1, -(-e2e_steps // E2E_BLOCK))
    e2e_steps = reps * E2E_BLOCK
    with torch.cuda.stream(cap):  # replay() launches on the current stream
        graph.replay()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cap):
        e0.record(cap)
        for _ in range(reps):
            graph.replay()
        e1.record(cap)
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    if dw.prep.check() != 0:
        raise RuntimeError("device error bits set during the e2e steps")

    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e_ms], dist, device)

    if rank != 0:
        dist.destroy_process_group()
        return

    ms_step = elapsed_ms / args.steps
    tokens_per_s = whole_job_rate(world, w.rows, args.steps, elapsed_ms)
    timing = {"blocks": len(blocks), "steps_per_block": args.steps, "timed_s": sum(blocks) * args.steps / 1e3,
              "block_ms_per_step_min": min(blocks), "block_ms_per_step_max": max(blocks),
              "ms_per_step_mean_over_blocks": statistics.mean(blocks),
              "launch": launch_rule(args, flush_bufs is not None),
              "rule": f"blocks of --steps steps repeated until {args.min_timed_s} s of timed work; "
                      "ms_per_step = the median block / steps"}
    peak, peak_kind = load_peaks()
    achieved = all_b / (ms_step / 1e3) / 1e9
    state_gbs = state_b / (ms_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "ms_per_step_median_single_step": median_ms,
        "timing": timing, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if args.state_dtype == "f32" else "f32 compute, bf16 state storage",
        "data": "synthetic", "config": workload_config(w, args),
        "state_gbs": state_gbs, "state_frac_of_peak": state_gbs / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": measured_traffic(w.name, args.state_dtype, args.v_split),
                     "kernel": step_kernel_name(w, args.state_dtype, args.v_split),
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s"},
        "e2e": {"value": whole_job_rate(world, w.rows, e2e_steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "overlap": "uploads and downloads on streams of their own, two buffer sets; blocks of "
                           f"{E2E_BLOCK} steps recorded as a CUDA graph"},
        "gpu_launches": args.steps * len(blocks),
        "clocks": sampler.summary(t_host0, t_host1),
    }
    if direct is not None:
        line["direct_launch"] = direct_record(direct, w, state_b, all_b, peak)
    if dist is not None:
        dist.destroy_process_group()
    if world == 1 and not args.no_per_workload:
        del dw, copies
        torch.cuda.empty_cache()
        line["per_workload"] = {name: measure_workload(I.WORKLOADS[name], device, args)
                                for name in PER_WORKLOAD if name != w.name}
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(si, state_dtype=args.state_dtype)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
