"""KDA decode / spec-verify core on GB300 (sm_103a): thin Python binding.

Every step of the path runs in the CUDA kernels of ``libkda.so`` (built
in-tree from ``csrc/kda_step.cu``); this module only marshals arguments
through the C ABI declared in ``include/kda.h``.  PyTorch supplies device
memory and the current stream.  There is no fallback: if the library is
missing or fails to load, every call raises.

Low-level functions carry the C names (:func:`kda_prepare`, :func:`kda_step`,
:func:`kda_check`, :func:`kda_destroy`, :func:`kda_strerror`,
:func:`kda_launch_info`, :func:`kda_set_gate_mode`, :func:`kda_set_v_split`, :func:`kda_plan_create`,
:func:`kda_plan_launch`, :func:`kda_plan_destroy`) and take raw device pointers.  :class:`PreparedKda`
mirrors the PreparedKda wrapper on the
"vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.prepared" page:
weights prepared once, then ``run(projected, out, caches=..., slots=...,
accepted=None)`` per step, with ``accepted[:R]`` and contiguous ``slots[:R]``
for verify steps; ``plan(...)`` records a step with fixed buffers as a CUDA
graph (:class:`KdaPlan`) that each later step launches in one call.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

from ._build import DEBUG_LIB_PATH, LIB_PATH, build

__all__ = [
    "KdaError", "build", "load_library", "kda_prepare", "kda_step", "kda_check", "kda_destroy",
    "kda_strerror", "kda_launch_info", "kda_set_gate_mode", "kda_plan_create", "kda_layer_plan_create", "kda_plan_launch",
    "kda_plan_destroy", "kda_set_state_dtype", "kda_set_v_split", "kda_linear", "kda_linear_check", "linear", "PreparedKda", "KdaPlan", "KDA_STATE_F32", "KDA_STATE_BF16", "KDA_PDL_STEP", "KDA_PDL_O_PROJ", "KDA_ERR_SLOT", "KDA_ERR_ACCEPTED",
    "KDA_ERR_TIMEOUT", "KDA_ERR_DUPLICATE", "KDA_MAX_TOKENS", "DEBUG_LIB_PATH", "KDA_GATE_SIGMOID", "KDA_GATE_SOFTPLUS", "HEAD_DIM",
]

HEAD_DIM = 128
KDA_OK, KDA_EINVAL, KDA_ECUDA = 0, -1, -2
KDA_ERR_SLOT, KDA_ERR_ACCEPTED, KDA_ERR_TIMEOUT, KDA_ERR_DUPLICATE = 1, 2, 4, 8
KDA_MAX_TOKENS = 8
KDA_GATE_SIGMOID, KDA_GATE_SOFTPLUS = 0, 1
KDA_STATE_F32, KDA_STATE_BF16 = 0, 1
KDA_PDL_STEP, KDA_PDL_O_PROJ = 1, 2

_lib: Optional[ctypes.CDLL] = None


class KdaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {kda_strerror(code)} ({code})")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with linear_attention_decode_03_gb300.build()")
    lib = ctypes.CDLL(path)
    vp, ll, i32, f32 = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_float
    lib.kda_prepare.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp, f32, f32, ctypes.POINTER(vp)]
    lib.kda_prepare.restype = i32
    lib.kda_step.argtypes = [vp, vp, ll, ll, vp, i32, vp, ll, vp, i32, vp, vp, vp]
    lib.kda_step.restype = i32
    lib.kda_check.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint)]
    lib.kda_check.restype = i32
    lib.kda_destroy.argtypes = [vp]
    lib.kda_destroy.restype = None
    lib.kda_strerror.argtypes = [i32]
    lib.kda_strerror.restype = ctypes.c_char_p
    lib.kda_launch_info.argtypes = [i32, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.kda_launch_info.restype = i32
    lib.kda_set_gate_mode.argtypes = [vp, i32]
    lib.kda_set_gate_mode.restype = i32
    lib.kda_plan_create.argtypes = [vp, vp, ll, ll, vp, i32, vp, ll, vp, i32, vp, vp, ctypes.POINTER(vp)]
    lib.kda_plan_create.restype = i32
    lib.kda_layer_plan_create.argtypes = [vp, vp, ll, ll, ll, vp, vp, ll, vp, i32, vp, ll, vp, i32, vp, vp, vp, vp,
                                          ll, i32, ctypes.POINTER(vp)]
    lib.kda_layer_plan_create.restype = i32
    lib.kda_plan_launch.argtypes = [vp, vp]
    lib.kda_plan_launch.restype = i32
    lib.kda_plan_destroy.argtypes = [vp]
    lib.kda_plan_destroy.restype = None
    lib.kda_set_state_dtype.argtypes = [vp, i32]
    lib.kda_set_state_dtype.restype = i32
    lib.kda_set_v_split.argtypes = [vp, i32]
    lib.kda_set_v_split.restype = i32
    lib.kda_linear.argtypes = [vp, ll, ll, vp, ll, ll, vp, ll, vp]
    lib.kda_linear.restype = i32
    lib.kda_linear_check.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
    lib.kda_linear_check.restype = i32
    _lib = lib
    return lib


def kda_strerror(code: int) -> str:
    return load_library().kda_strerror(int(code)).decode()


def kda_prepare(heads: int, conv_width: int, conv_w: int, bias: int, f_b: int, A_log: int, dt_bias: int,
                o_norm: int, gate_lower_bound: float, eps: float) -> int:
    """Device pointers in, an opaque handle (int) out."""
    h = ctypes.c_void_p()
    rc = load_library().kda_prepare(heads, conv_width, conv_w, bias or None, f_b, A_log, dt_bias, o_norm,
                                    gate_lower_bound, eps, ctypes.byref(h))
    if rc != KDA_OK:
        raise KdaError("kda_prepare", rc)
    return h.value


def kda_step(handle: int, projected: int, rows: int, pitch: int, conv_state: int, conv_dim_first: bool,
             state_pool: int, pool_slots: int, slots: int, L: int, accepted: Optional[int], out: int,
             stream: int) -> None:
    rc = load_library().kda_step(handle, projected, rows, pitch, conv_state, 1 if conv_dim_first else 0,
                                 state_pool, pool_slots, slots, L, accepted or None, out, stream or None)
    if rc != KDA_OK:
        raise KdaError("kda_step", rc)


def kda_plan_create(handle: int, projected: int, rows: int, pitch: int, conv_state: int, conv_dim_first: bool,
                    state_pool: int, pool_slots: int, slots: int, L: int, accepted: Optional[int], out: int) -> int:
    """Record one step (arguments as kda_step, no stream) as a CUDA graph; an opaque plan (int) out."""
    p = ctypes.c_void_p()
    rc = load_library().kda_plan_create(handle, projected, rows, pitch, conv_state, 1 if conv_dim_first else 0,
                                        state_pool, pool_slots, slots, L, accepted or None, out, ctypes.byref(p))
    if rc != KDA_OK:
        raise KdaError("kda_plan_create", rc)
    return p.value


def kda_layer_plan_create(handle: int, x: int, rows: int, ldx: int, hidden: int, w_in: int, projected: int,
                          pitch: int, conv_state: int, conv_dim_first: bool, state_pool: int, pool_slots: int,
                          slots: int, L: int, accepted: Optional[int], core_out: int, w_o: int, y: int, ldy: int,
                          pdl: int = 0) -> int:
    """Record in_proj -> kda_step -> o_proj on these buffers as one CUDA graph (see include/kda.h)."""
    p = ctypes.c_void_p()
    rc = load_library().kda_layer_plan_create(handle, x, rows, ldx, hidden, w_in, projected, pitch, conv_state,
                                              1 if conv_dim_first else 0, state_pool, pool_slots, slots, L,
                                              accepted or None, core_out, w_o, y, ldy, int(pdl),
                                              ctypes.byref(p))
    if rc != KDA_OK:
        raise KdaError("kda_layer_plan_create", rc)
    return p.value


def kda_plan_launch(plan: int, stream: int = 0) -> None:
    rc = load_library().kda_plan_launch(plan, stream or None)
    if rc != KDA_OK:
        raise KdaError("kda_plan_launch", rc)


def kda_plan_destroy(plan: int) -> None:
    load_library().kda_plan_destroy(plan)


def kda_linear(x: int, rows: int, ldx: int, w: int, N: int, K: int, y: int, ldy: int, stream: int = 0) -> None:
    """y[rows, N] = x[rows, K] . W[N, K]^T on device pointers (see include/kda.h)."""
    rc = load_library().kda_linear(x, rows, ldx, w, N, K, y, ldy, stream or None)
    if rc != KDA_OK:
        raise KdaError("kda_linear", rc)


def kda_linear_check(stream: int = 0) -> int:
    """Synchronise `stream`, return and clear the projections' device error bits."""
    flags = ctypes.c_uint(0)
    rc = load_library().kda_linear_check(stream or None, ctypes.byref(flags))
    if rc != KDA_OK:
        raise KdaError("kda_linear_check", rc)
    return flags.value


def linear(x, w, out=None, stream=None):
    """y = x @ w.T for CUDA bf16 tensors x [rows, K] (unit column stride) and
    w [N, K] (contiguous), through kda_linear; `out` [rows, N] bf16 or None."""
    import torch

    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16 or not (x.is_cuda and w.is_cuda):
        raise TypeError("linear takes CUDA bf16 tensors")
    if x.dim() != 2 or w.dim() != 2 or x.stride(1) != 1 or not w.is_contiguous() or x.shape[1] != w.shape[1]:
        raise ValueError("x [rows, K] with unit column stride and contiguous w [N, K] expected")
    rows, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((rows, N), dtype=torch.bfloat16, device=x.device)
    if out.dtype != torch.bfloat16 or out.dim() != 2 or out.stride(1) != 1 or tuple(out.shape) != (rows, N):
        raise ValueError("out must be bf16 [rows, N] with unit column stride")
    if stream is None:
        stream = _current_stream(x.device)
    kda_linear(x.data_ptr(), rows, x.stride(0), w.data_ptr(), N, K, out.data_ptr(), out.stride(0), stream)
    return out


def kda_set_state_dtype(handle: int, dtype: int) -> None:
    """KDA_STATE_F32 (default) or KDA_STATE_BF16: the state pool's storage type for later steps."""
    rc = load_library().kda_set_state_dtype(handle, int(dtype))
    if rc != KDA_OK:
        raise KdaError("kda_set_state_dtype", rc)


def kda_set_v_split(handle: int, v_split: int) -> None:
    """1 (default) or 2 CTAs a (request, head) for the handle's later steps (see include/kda.h)."""
    rc = load_library().kda_set_v_split(handle, int(v_split))
    if rc != KDA_OK:
        raise KdaError("kda_set_v_split", rc)


def kda_set_gate_mode(handle: int, mode: int) -> None:
    """KDA_GATE_SIGMOID (default) or KDA_GATE_SOFTPLUS for the handle's later steps."""
    rc = load_library().kda_set_gate_mode(handle, int(mode))
    if rc != KDA_OK:
        raise KdaError("kda_set_gate_mode", rc)


def kda_check(handle: int, stream: int = 0) -> int:
    flags = ctypes.c_uint(0)
    rc = load_library().kda_check(handle, stream or None, ctypes.byref(flags))
    if rc != KDA_OK:
        raise KdaError("kda_check", rc)
    return int(flags.value)


def kda_destroy(handle: int) -> None:
    if handle:
        load_library().kda_destroy(handle)


def kda_launch_info(L: int) -> Tuple[int, int, int]:
    """(threads per CTA, dynamic shared bytes, resident CTAs per SM) for L tokens."""
    t, s, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = load_library().kda_launch_info(L, ctypes.byref(t), ctypes.byref(s), ctypes.byref(c))
    if rc != KDA_OK:
        raise KdaError("kda_launch_info", rc)
    return t.value, s.value, c.value


def _current_stream(device) -> int:
    """The raw handle of the device's current stream (without building a
    torch Stream object on every call)."""
    import torch

    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None and device.index is not None:
        return raw(device.index)
    return torch.cuda.current_stream(device).cuda_stream


def _dev(t, dtype, name):
    import torch

    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


class PreparedKda:
    """Prepared KDA core for one layer (weights copied into the handle).

    ``conv_w`` [3D, 1, W] bf16, ``conv_bias`` [3D] bf16 or None, ``f_b`` [D, 128]
    bf16, ``A_log`` [H] f32, ``dt_bias`` [D] f32, ``o_norm`` [128] f32 (cast
    to fp32 as the page's __init__ does).  ``gate_mode`` picks the decay gate
    (``KDA_GATE_SIGMOID``, the default, or ``KDA_GATE_SOFTPLUS``; see
    ``include/kda.h``); ``state_dtype`` the state pool's storage type ("f32",
    the default, or "bf16": computed in fp32, each stored state rounded);
    ``v_split`` the CTAs a (request, head) (1, the default, or 2; see
    ``kda_set_v_split`` in ``include/kda.h``).
    """

    def __init__(self, conv_w, conv_bias, f_b, A_log, dt_bias, o_norm, *, gate_lower_bound: float = -5.0,
                 eps: float = 1e-6, conv_dim_first: bool = True, gate_mode: int = KDA_GATE_SIGMOID,
                 state_dtype: str = "f32", v_split: int = 1):
        import torch

        self.heads = int(A_log.numel())
        self.dim = self.heads * HEAD_DIM
        self.width = int(conv_w.shape[-1])
        self.conv_dim_first = conv_dim_first
        o_norm = o_norm.detach().float().contiguous()
        self._keep = [_dev(conv_w.detach().contiguous(), torch.bfloat16, "conv_w"),
                      _dev(f_b.detach().contiguous(), torch.bfloat16, "f_b"),
                      _dev(A_log.detach().contiguous(), torch.float32, "A_log"),
                      _dev(dt_bias.detach().contiguous(), torch.float32, "dt_bias"),
                      _dev(o_norm, torch.float32, "o_norm")]
        bias_ptr = 0
        if conv_bias is not None:
            b = _dev(conv_bias.detach().contiguous(), torch.bfloat16, "conv_bias")
            self._keep.append(b)
            bias_ptr = b.data_ptr()
        cw, fb, al, dt, on = self._keep[:5]
        self.device = cw.device
        with torch.cuda.device(self.device):
            self.handle = kda_prepare(self.heads, self.width, cw.data_ptr(), bias_ptr, fb.data_ptr(),
                                      al.data_ptr(), dt.data_ptr(), on.data_ptr(), float(gate_lower_bound),
                                      float(eps))
            if gate_mode != KDA_GATE_SIGMOID:
                kda_set_gate_mode(self.handle, gate_mode)
            if state_dtype not in ("f32", "bf16"):
                raise ValueError("state_dtype must be 'f32' or 'bf16'")
            self.state_dtype = state_dtype
            if state_dtype == "bf16":
                kda_set_state_dtype(self.handle, KDA_STATE_BF16)
            if v_split != 1:
                kda_set_v_split(self.handle, v_split)

    def _args(self, projected, out, caches, slots, accepted):
        """kda_step's arguments (pointers and sizes) for these tensors, and the
        tensors they point into (kept alive by a plan).  The step reads the
        first rows of ``slots`` / ``accepted`` only, so longer ones are passed
        as they are; a copy is made only where a layout needs one (strided
        verify slots, a non-contiguous ``accepted``)."""
        import torch

        conv, state = caches[:2]
        batch = projected.shape[0]
        L = 1
        if accepted is not None:
            L = int(slots.shape[1])
            rows = batch // L
            if accepted.shape[0] < rows or slots.shape[0] < rows:
                raise ValueError("slots and accepted need a row for each request of the batch")
            if not accepted.is_contiguous():
                accepted = accepted[:rows].contiguous()
            _dev(accepted, torch.int32, "accepted")
            if slots.stride() != (L, 1):
                slots = slots[:rows].contiguous()
        elif slots.shape[0] < batch:
            raise ValueError("slots needs an entry for each row of the batch")
        _dev(slots, torch.int32, "slots")
        if projected.dtype != torch.bfloat16 or not projected.is_cuda or projected.stride(1) != 1:
            raise TypeError("projected must be a CUDA bf16 tensor with unit column stride")
        if batch > 0 and projected.shape[1] < 4 * self.dim + HEAD_DIM + self.heads:
            raise ValueError("projected needs the q|k|v|gate|f_a|beta columns (4D + 128 + H)")
        _dev(out, torch.bfloat16, "out")
        _dev(conv, torch.bfloat16, "conv_state")
        _dev(state, torch.bfloat16 if self.state_dtype == "bf16" else torch.float32, "state_pool")
        pool = state.shape[0]
        if out.numel() < batch * self.dim:
            raise ValueError("out needs [rows, D] elements")
        if state.numel() != pool * self.heads * HEAD_DIM * HEAD_DIM:
            raise ValueError("state_pool must be [pool, H, 128, 128]")
        if conv.numel() < pool * 3 * self.dim * (self.width - 1):
            raise ValueError("conv_state needs a window for every slot of the state pool")
        args = (projected.data_ptr(), batch, projected.stride(0), conv.data_ptr(), self.conv_dim_first,
                state.data_ptr(), pool, slots.data_ptr(), L,
                None if accepted is None else accepted.data_ptr(), out.data_ptr())
        return args, (projected, out, conv, state, slots, accepted)

    def run(self, projected, out, *, caches, slots, accepted=None, stream=None):
        """One step.  ``caches`` = (conv_state, state_pool); decode when
        ``accepted`` is None (``slots`` [>= B]), verify otherwise (``slots``
        [>= R, L], ``accepted`` [>= R])."""
        import torch

        args, _ = self._args(projected, out, caches, slots, accepted)
        if stream is None:
            stream = _current_stream(self.device)
        kda_step(self.handle, *args, stream)
        return out

    def plan(self, projected, out, *, caches, slots, accepted=None) -> "KdaPlan":
        """Record a step on these buffers (arguments as ``run``) as a CUDA graph.
        Each ``launch()`` of the plan is one step on whatever the buffers then
        hold; the gate mode is the one set when the plan is made."""
        import torch

        args, keep = self._args(projected, out, caches, slots, accepted)
        with torch.cuda.device(self.device):
            p = kda_plan_create(self.handle, *args)
        return KdaPlan(p, keep + (self,), self.device)

    def layer_plan(self, x, w_in, projected, core_out, w_o, y, *, caches, slots, accepted=None,
                   pdl=0) -> "KdaPlan":
        """Record one step of the layer on these buffers as a CUDA graph:
        ``projected = x @ w_in.T`` (in_proj), the core step ``projected ->
        core_out`` (arguments as ``run``), ``y = core_out @ w_o.T`` (o_proj).
        x [rows, hidden] bf16 (unit column stride), w_in [pitch, hidden] and
        w_o [hidden, D] contiguous bf16, projected [rows, pitch], core_out
        [rows, D] and y [rows, hidden] bf16.  ``pdl``: a mask of the edges
        launched as programmatic dependents (KDA_PDL_STEP | KDA_PDL_O_PROJ;
        True = both, 0 = plain stream order)."""
        import torch

        args, keep = self._args(projected, core_out, caches, slots, accepted)
        for t, name in ((x, "x"), (w_in, "w_in"), (w_o, "w_o"), (y, "y")):
            if t.dtype != torch.bfloat16 or not t.is_cuda or t.stride(1) != 1:
                raise TypeError(f"{name} must be a CUDA bf16 tensor with unit column stride")
        if not (w_in.is_contiguous() and w_o.is_contiguous() and projected.is_contiguous() and core_out.is_contiguous()):
            raise ValueError("w_in, w_o, projected and core_out must be contiguous")
        rows, hidden = x.shape
        pitch = projected.shape[1]
        if (tuple(w_in.shape) != (pitch, hidden) or tuple(w_o.shape) != (hidden, core_out.shape[1])
                or projected.shape[0] != rows or tuple(y.shape) != (rows, hidden)):
            raise ValueError("layer_plan: inconsistent shapes")
        (_, batch, _, conv, dim_first, state, pool, slot_ptr, L, acc, out) = args
        with torch.cuda.device(self.device):
            mask = (KDA_PDL_STEP | KDA_PDL_O_PROJ) if pdl is True else int(pdl)
            p = kda_layer_plan_create(self.handle, x.data_ptr(), rows, x.stride(0), hidden, w_in.data_ptr(),
                                      projected.data_ptr(), pitch, conv, dim_first, state, pool, slot_ptr, L, acc,
                                      out, w_o.data_ptr(), y.data_ptr(), y.stride(0), mask)
        return KdaPlan(p, keep + (x, w_in, w_o, y, self), self.device)

    def check(self, stream=None) -> int:
        """Synchronise the stream; return and clear the device error bits (plan launches included)."""
        import torch

        if stream is None:
            stream = torch.cuda.current_stream(self.device).cuda_stream
        return kda_check(self.handle, stream)

    def close(self) -> None:
        if getattr(self, "handle", None):
            kda_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class KdaPlan:
    """One step of a PreparedKda recorded as a CUDA graph on fixed buffers
    (``PreparedKda.plan``).  Keeps the buffers and the prepared handle alive."""

    def __init__(self, plan: int, keep, device):
        self.plan, self._keep, self.device = plan, keep, device

    def launch(self, stream=None) -> None:
        import torch

        if stream is None:
            stream = _current_stream(self.device)
        kda_plan_launch(self.plan, stream)

    def close(self) -> None:
        if getattr(self, "plan", None):
            kda_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
