"""Grok-1 top-2-of-8 MoE feed-forward layer on B300 (sm_103a): Python binding.

A thin ctypes layer over the C ABI in ``include/moe_layer.h`` and
``include/attn_block.h`` (library ``libmoe_layer.so`` in this directory).  It only checks and marshals
arguments: every step of the layer runs in the library's CUDA kernels.  PyTorch
is used for device memory and streams.  There is no CPU fallback: when the
library is missing or the device is not an sm_103 part, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
LIB_PATH = os.path.join(_PKG, "libmoe_layer.so")
HEADER_PATH = os.path.join(_ROOT, "include", "moe_layer.h")
ATTN_HEADER_PATH = os.path.join(_ROOT, "include", "attn_block.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_OOM = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_DEVICE_CHECK, MOE_ERR_TIMEOUT = 4, 5, 6
MOE_WEIGHT_BF16, MOE_WEIGHT_INT8 = 0, 1
MOE_FLAG_DEVICE_CHECKS, MOE_FLAG_FORCE_TC, MOE_FLAG_FORCE_GEMV, MOE_FLAG_DECODE_TC = 0x1, 0x2, 0x4, 0x8
KERNEL_NAMES = ("router", "group", "up_geglu", "down", "combine")
ATTN_KERNEL_NAMES = ("prenorm", "qkv", "rope", "attn", "oproj", "post")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {_status_name(status)}: {detail}")


class Config(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ffn", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("eps", ctypes.c_float),
                ("weight_dtype", ctypes.c_int32), ("flags", ctypes.c_uint32), ("scale_experts", ctypes.c_int32),
                ("scale_groups", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gate", "gate_bias", "w", "wv", "w1", "w_scale", "wv_scale",
                                                "w1_scale", "pre_norm_scale", "post_norm_scale")]


class AttnConfig(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("eps", ctypes.c_float),
                ("rope_base", ctypes.c_float), ("logit_clamp", ctypes.c_float)]


class AttnWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("wq", "wk", "wv", "wo", "s_pre", "s_post")]


class WorkspaceView(ctypes.Structure):
    _fields_ = [("rnorm", ctypes.c_void_p), ("counts", ctypes.c_void_p), ("row_offset", ctypes.c_void_p),
                ("row_of_slot", ctypes.c_void_p), ("xn_perm", ctypes.c_void_p), ("act", ctypes.c_void_p),
                ("y_rows", ctypes.c_void_p), ("rows_cap", ctypes.c_int64)]


_lib_handle = None


def lib():
    """The loaded C library (raises if it was not built)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} not found: build it with `python -m mixture_experts_transformer_gemv_b300.build`"
                              " (there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.moe_layer_create.restype = i32
        L.moe_layer_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), ctypes.POINTER(vp)]
        L.moe_layer_forward.restype = i32
        L.moe_layer_forward.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp]
        L.moe_layer_forward_host.restype = i32
        L.moe_layer_forward_host.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp]
        L.moe_layer_forward_host_async.restype = i32
        L.moe_layer_forward_host_async.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp]
        L.moe_layer_host_wait.restype = i32
        L.moe_layer_host_wait.argtypes = [vp, vp]
        L.moe_layer_sync_status.restype = i32
        L.moe_layer_sync_status.argtypes = [vp, vp]
        L.moe_layer_destroy.restype = i32
        L.moe_layer_destroy.argtypes = [vp]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [i32]
        L.moe_last_error_message.restype = ctypes.c_char_p
        L.moe_last_error_message.argtypes = []
        L.moe_layer_set_profiling.restype = i32
        L.moe_layer_set_profiling.argtypes = [vp, i32]
        L.moe_layer_profile_read.restype = i32
        L.moe_layer_profile_read.argtypes = [vp, vp, vp, i32]
        L.moe_layer_router_stats.restype = i32
        L.moe_layer_router_stats.argtypes = [vp, vp, vp]
        L.moe_layer_gemm_grid.restype = i32
        L.moe_layer_gemm_grid.argtypes = [vp, vp]
        L.moe_layer_launch_count.restype = i64
        L.moe_layer_launch_count.argtypes = [vp]
        L.moe_layer_workspace.restype = i32
        L.moe_layer_workspace.argtypes = [vp, ctypes.POINTER(WorkspaceView)]
        L.moe_group_slots_noalloc.restype = i32
        L.moe_group_slots_noalloc.argtypes = [vp, vp, i32, vp, vp, vp]
        L.moe_selftest_bounded_wait.restype = i32
        L.moe_selftest_bounded_wait.argtypes = [i32, ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64)]
        L.moe_selftest_gelu.restype = i32
        L.moe_selftest_gelu.argtypes = [vp, vp, i64, vp]
        L.attn_block_create.restype = i32
        L.attn_block_create.argtypes = [ctypes.POINTER(AttnConfig), ctypes.POINTER(AttnWeights), ctypes.POINTER(vp)]
        L.attn_block_forward.restype = i32
        L.attn_block_forward.argtypes = [vp, vp, vp, i32, vp]
        L.attn_block_sync_status.restype = i32
        L.attn_block_sync_status.argtypes = [vp, vp]
        L.attn_block_set_profiling.restype = i32
        L.attn_block_set_profiling.argtypes = [vp, i32]
        L.attn_block_profile_read.restype = i32
        L.attn_block_profile_read.argtypes = [vp, vp, vp, i32]
        L.attn_block_launch_count.restype = i32
        L.attn_block_launch_count.argtypes = [vp]
        L.attn_block_destroy.restype = i32
        L.attn_block_destroy.argtypes = [vp]
        _lib_handle = L
    return _lib_handle


def _status_name(s: int) -> str:
    try:
        return lib().moe_status_string(s).decode()
    except Exception:
        return f"status {s}"


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where, lib().moe_last_error_message().decode())


def declared_functions():
    """Names of the functions include/moe_layer.h and include/attn_block.h declare."""
    text = open(HEADER_PATH).read() + open(ATTN_HEADER_PATH).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\*?\s+\*?((?:moe|attn)_[a-z_0-9]+)\s*\(", text,
                                 re.M)))


def selftest_bounded_wait(mode: int, limit_s: float) -> tuple:
    """moe_selftest_bounded_wait: (status, waited seconds).  The expected status is
    MOE_ERR_TIMEOUT (the wait gave up and latched the error word)."""
    el = ctypes.c_uint64(0)
    st = lib().moe_selftest_bounded_wait(int(mode), int(limit_s * 1e9), ctypes.byref(el))
    return st, el.value / 1e9


def selftest_gelu(x, stream=None):
    """moe_selftest_gelu: the device GELU of the GeGLU epilogues applied to a
    contiguous float32 CUDA tensor; returns a new tensor."""
    import torch
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    y = torch.empty_like(x)
    with torch.cuda.device(x.device):
        _check(lib().moe_selftest_gelu(x.data_ptr(), y.data_ptr(), x.numel(), _stream_handle(stream)),
               "moe_selftest_gelu")
    return y


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def group_slots_noalloc(topk_idx, topk_prob, expert_counts, row_of_slot, stream=None):
    """moe_group_slots_noalloc: per-expert counts and the slot -> row map of the
    layer's grouping step, with no memory allocated (scratch is a static device
    array; T <= 16384; calls must not overlap on the GPU).  All tensors CUDA,
    int32 / fp32, contiguous, on one device: topk_idx, topk_prob [T, 2] in;
    expert_counts [8], row_of_slot [T, 2] out.  Mis-shaped tensors raise
    ValueError before anything is enqueued."""
    import torch
    # shapes first: the kernel indexes [T, 2] and [8] arrays, so a short buffer
    # would be read or written past its end
    if topk_idx.dim() != 2 or topk_idx.shape[1] != 2:
        raise ValueError(f"group_slots_noalloc: topk_idx must be [T, 2] (got {tuple(topk_idx.shape)})")
    T = topk_idx.shape[0]
    for name, t in (("topk_prob", topk_prob), ("row_of_slot", row_of_slot)):
        if tuple(t.shape) != (T, 2):
            raise ValueError(f"group_slots_noalloc: {name} must be [{T}, 2] (got {tuple(t.shape)})")
    if expert_counts.dim() != 1 or expert_counts.numel() < 8:
        raise ValueError(f"group_slots_noalloc: expert_counts must be [8] (got {tuple(expert_counts.shape)})")
    for t, dt in ((topk_idx, torch.int32), (topk_prob, torch.float32), (expert_counts, torch.int32),
                  (row_of_slot, torch.int32)):
        if not (t.is_cuda and t.dtype == dt and t.is_contiguous()):
            raise ValueError("group_slots_noalloc: tensors must be contiguous CUDA int32 / fp32")
    if len({t.device for t in (topk_idx, topk_prob, expert_counts, row_of_slot)}) != 1:
        raise ValueError("group_slots_noalloc: all tensors must be on the same device")
    _check(lib().moe_group_slots_noalloc(topk_idx.data_ptr(), topk_prob.data_ptr(), T, expert_counts.data_ptr(),
                                         row_of_slot.data_ptr(), _stream_handle(stream)), "moe_group_slots_noalloc")


class MoeLayer:
    """One MoE layer bound to device tensors (borrowed: keep them alive).

    weights: dict of CUDA tensors, contiguous:
      gate [E, d] fp32, gate_bias [E] fp32 or None, w / wv [E, F, d] and
      w1 [E, d, F] (bf16, or int8 with w_scale / wv_scale [E_s, G, F] and
      w1_scale [E_s, G, d] bf16, scale_shape = (E_s, G)), pre_norm_scale /
      post_norm_scale [d] fp32.
    """

    def __init__(self, d_model: int, d_ffn: int, max_tokens: int, weights: dict, eps: float = 1e-5,
                 weight_dtype: str = "bf16", flags: int = 0, num_experts: int = 8, top_k: int = 2,
                 scale_shape=(8, 1)):
        import torch
        self.d, self.F, self.max_tokens = d_model, d_ffn, max_tokens
        self._weights = dict(weights)  # keep the borrowed tensors alive
        cfg = Config(d_model, d_ffn, num_experts, top_k, max_tokens, eps,
                     MOE_WEIGHT_INT8 if weight_dtype == "int8" else MOE_WEIGHT_BF16, flags,
                     int(scale_shape[0]), int(scale_shape[1]))
        w = Weights()
        for name, _ in Weights._fields_:
            t = weights.get(name)
            if t is not None:
                if not (t.is_cuda and t.is_contiguous()):
                    raise ValueError(f"weight {name} must be a contiguous CUDA tensor")
                setattr(w, name, t.data_ptr())
        handle = ctypes.c_void_p()
        self._dev = torch.cuda.current_device()
        _check(lib().moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(handle)), "moe_layer_create")
        self._h = handle

    # ------------------------------------------------------------------ calls
    def forward(self, hidden, out=None, stream=None, routing: bool = False):
        """hidden [T, d] bf16 CUDA -> out [T, d] bf16 (in place when out is hidden).
        With routing=True also returns (topk_idx [T,2] int32, topk_prob [T,2] fp32,
        expert_counts [8] int32)."""
        import torch
        T = hidden.shape[0]
        self._check_act(hidden, "hidden")
        if out is None:
            out = torch.empty_like(hidden)
        self._check_act(out, "out")
        idx = prob = counts = None
        if routing:
            idx = torch.empty((T, 2), dtype=torch.int32, device=hidden.device)
            prob = torch.empty((T, 2), dtype=torch.float32, device=hidden.device)
            counts = torch.zeros((8,), dtype=torch.int32, device=hidden.device)
        _check(lib().moe_layer_forward(self._h, hidden.data_ptr(), out.data_ptr(), T, _stream_handle(stream),
                                       _ptr(idx), _ptr(prob), _ptr(counts)), "moe_layer_forward")
        return (out, idx, prob, counts) if routing else out

    def forward_host(self, hidden_host, out_host=None, stream=None, routing: bool = False):
        """Same layer on HOST tensors (pinned for full copy speed); synchronous."""
        import torch
        T = hidden_host.shape[0]
        if hidden_host.is_cuda or hidden_host.dtype != torch.bfloat16 or not hidden_host.is_contiguous():
            raise ValueError("hidden_host must be a contiguous CPU bf16 tensor")
        if out_host is None:
            out_host = torch.empty_like(hidden_host)
        idx = prob = counts = None
        if routing:
            idx = torch.empty((T, 2), dtype=torch.int32)
            prob = torch.empty((T, 2), dtype=torch.float32)
            counts = torch.zeros((8,), dtype=torch.int32)
        _check(lib().moe_layer_forward_host(self._h, hidden_host.data_ptr(), out_host.data_ptr(), T,
                                            _stream_handle(stream), _ptr(idx), _ptr(prob), _ptr(counts)),
               "moe_layer_forward_host")
        return (out_host, idx, prob, counts) if routing else out_host

    def router_stats(self, stream=None):
        """Routing diagnostics of the last forward, as a CUDA fp32 tensor [10]:
        mean router probability of experts 0-7, routing entropy (nats), collapse
        index 1 - entropy / ln 8.  Enqueued on `stream` (default: current)."""
        import torch
        out = torch.empty(10, dtype=torch.float32, device=torch.device("cuda", self._dev))
        _check(lib().moe_layer_router_stats(self._h, out.data_ptr(), _stream_handle(stream)), "moe_layer_router_stats")
        return out

    def forward_host_async(self, hidden_host, out_host, stream=None):
        """moe_layer_forward_host_async: enqueue the layer on HOST tensors (pinned)
        and return at once; call host_wait() before touching the buffers."""
        import torch
        if hidden_host.is_cuda or hidden_host.dtype != torch.bfloat16 or not hidden_host.is_contiguous():
            raise ValueError("hidden_host must be a contiguous CPU bf16 tensor")
        if out_host.is_cuda or out_host.dtype != torch.bfloat16 or not out_host.is_contiguous():
            raise ValueError("out_host must be a contiguous CPU bf16 tensor")
        _check(lib().moe_layer_forward_host_async(self._h, hidden_host.data_ptr(), out_host.data_ptr(),
                                                  hidden_host.shape[0], _stream_handle(stream), None, None, None),
               "moe_layer_forward_host_async")

    def host_wait(self, stream=None):
        _check(lib().moe_layer_host_wait(self._h, _stream_handle(stream)), "moe_layer_host_wait")

    def sync_status(self, stream=None):
        _check(lib().moe_layer_sync_status(self._h, _stream_handle(stream)), "moe_layer_sync_status")

    def set_profiling(self, on: bool):
        _check(lib().moe_layer_set_profiling(self._h, 1 if on else 0), "moe_layer_set_profiling")

    def profile_read(self, reset: bool = False):
        """{kernel name: (total ms, launches)} of the profiled forwards."""
        ms = (ctypes.c_double * len(KERNEL_NAMES))()
        n = (ctypes.c_int64 * len(KERNEL_NAMES))()
        _check(lib().moe_layer_profile_read(self._h, ms, n, 1 if reset else 0), "moe_layer_profile_read")
        return {k: (ms[i], n[i]) for i, k in enumerate(KERNEL_NAMES)}

    def gemm_grid(self) -> dict:
        """CTAs per grouped-GEMM launch: {"up_bf16", "down_bf16", "up_int8", "down_int8"}."""
        g = (ctypes.c_int32 * 4)()
        _check(lib().moe_layer_gemm_grid(self._h, g), "moe_layer_gemm_grid")
        return dict(zip(("up_bf16", "down_bf16", "up_int8", "down_int8"), list(g)))

    def launch_count(self) -> int:
        return int(lib().moe_layer_launch_count(self._h))

    def workspace(self) -> WorkspaceView:
        v = WorkspaceView()
        _check(lib().moe_layer_workspace(self._h, ctypes.byref(v)), "moe_layer_workspace")
        return v

    def close(self):
        if getattr(self, "_h", None):
            _check(lib().moe_layer_destroy(self._h), "moe_layer_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check_act(self, t, name):
        import torch
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 2
                and t.shape[1] == self.d):
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor [T, {self.d}]")


class AttnBlock:
    """The attention half of a Grok-1 decoder layer bound to device tensors.

    weights: dict of contiguous CUDA tensors: wq [Hq 128, d], wk / wv [Hkv 128, d],
    wo [d, Hq 128] (bf16), s_pre / s_post [d] (fp32).  wq, wk, wv are copied
    into the handle; wo and the norm scales are borrowed (kept alive here)."""

    def __init__(self, d_model: int, n_q_heads: int, n_kv_heads: int, max_tokens: int, weights: dict,
                 eps: float = 1e-5, rope_base: float = 10000.0, logit_clamp: float = 30.0, head_dim: int = 128):
        import torch
        self.d, self.max_tokens = d_model, max_tokens
        self._weights = dict(weights)
        cfg = AttnConfig(d_model, n_q_heads, n_kv_heads, head_dim, max_tokens, eps, rope_base, logit_clamp)
        w = AttnWeights()
        for name, _ in AttnWeights._fields_:
            t = weights.get(name)
            if t is not None:
                if not (t.is_cuda and t.is_contiguous()):
                    raise ValueError(f"weight {name} must be a contiguous CUDA tensor")
                setattr(w, name, t.data_ptr())
        handle = ctypes.c_void_p()
        _check(lib().attn_block_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(handle)), "attn_block_create")
        self._h = handle

    def forward(self, x, out=None, stream=None):
        """x [T, d] bf16 CUDA (one causal sequence) -> y [T, d] bf16."""
        import torch
        for t, name in ((x, "x"), (out, "out")):
            if t is not None and not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 2
                                      and t.shape[1] == self.d):
                raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor [T, {self.d}]")
        if out is None:
            out = torch.empty_like(x)
        _check(lib().attn_block_forward(self._h, x.data_ptr(), out.data_ptr(), x.shape[0], _stream_handle(stream)),
               "attn_block_forward")
        return out

    def sync_status(self, stream=None):
        _check(lib().attn_block_sync_status(self._h, _stream_handle(stream)), "attn_block_sync_status")

    def launch_count(self) -> int:
        return int(lib().attn_block_launch_count(self._h))

    def set_profiling(self, on: bool):
        _check(lib().attn_block_set_profiling(self._h, int(bool(on))), "attn_block_set_profiling")

    def profile_read(self, reset: bool = False) -> dict:
        """{kernel: (total ms, timed launches)} since the last reset."""
        ms = (ctypes.c_double * len(ATTN_KERNEL_NAMES))()
        n = (ctypes.c_int64 * len(ATTN_KERNEL_NAMES))()
        _check(lib().attn_block_profile_read(self._h, ms, n, int(reset)), "attn_block_profile_read")
        return {k: (ms[i], n[i]) for i, k in enumerate(ATTN_KERNEL_NAMES)}

    def close(self):
        if getattr(self, "_h", None):
            _check(lib().attn_block_destroy(self._h), "attn_block_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
