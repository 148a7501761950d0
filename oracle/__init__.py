"""CPU oracle of the Grok-1 top-2-of-8 MoE feed-forward layer.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this package.  The product
path (the CUDA library and its binding) never imports it and shares no code with
it: the two meet only through the seeded arrays of ``synth``.

The arithmetic lives in ``moe_oracle.c`` (plain loops, fp64, OpenMP across rows
only; its header cites the page passages each step follows).  This module only
marshals numpy arrays into it.

Functions
---------
route(inp)                       -> Route (xn, p, idx, w) for all T tokens
routing_stats(p)                 -> mean probability per expert, routing entropy, collapse index
moe_tokens(inp, tokens)          -> Layer (y, m, idx, w, p) for a token subset
expert_ffn(inp, xn, e)           -> (h, v, a, o) of one expert on one vector
attn_tokens(inp, tokens)         -> (y, ctx) of the attention block for a token subset
rope(v, pos, base)               -> rotary embedding of one head vector
dequant(q, scale, scale_E, scale_G) -> fp32 [E, N, K] dequantised weights
gelu_tanh(u), rmsnorm(v, s, eps)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

W_BF16, W_INT8 = 0, 1


def build(force: bool = False) -> str:
    """Compile moe_oracle.c with gcc (-O2, OpenMP, IEEE semantics: no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        # A test may point the wrapper at a deliberately broken build of the
        # oracle (mutation checks of the pins); nothing else sets this.
        lib = ctypes.CDLL(os.environ.get("MOE_ORACLE_LIB_OVERRIDE") or build())
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
        lib.oracle_max_threads.restype = i32
        lib.oracle_max_threads.argtypes = []
        lib.oracle_gelu_tanh.restype = dbl
        lib.oracle_gelu_tanh.argtypes = [dbl]
        lib.oracle_rmsnorm.restype = None
        lib.oracle_rmsnorm.argtypes = [i64, vp, vp, dbl, vp]
        lib.oracle_dequant.restype = None
        lib.oracle_dequant.argtypes = [i32, vp, vp, i32, i32, i64, i64, i64, vp]
        lib.oracle_route.restype = None
        lib.oracle_route.argtypes = [i64, i64, i64, vp, vp, vp, vp, dbl, vp, vp, vp, vp]
        lib.oracle_expert_ffn.restype = None
        lib.oracle_expert_ffn.argtypes = [i64, i64, i64, vp, i32, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                          vp, vp, vp, vp]
        lib.oracle_routing_stats.restype = None
        lib.oracle_routing_stats.argtypes = [i64, i64, vp, vp]
        lib.oracle_moe_tokens.restype = None
        lib.oracle_moe_tokens.argtypes = [i64, vp, i64, i64, i64, vp, vp, vp, vp, vp, dbl, i32, vp, vp, vp,
                                          vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        lib.oracle_rope.restype = None
        lib.oracle_rope.argtypes = [i64, vp, i64, dbl]
        lib.oracle_attn_tokens.restype = None
        lib.oracle_attn_tokens.argtypes = [i64, vp, i64, i64, i64, i64, i64, vp, vp, vp, dbl, vp, vp, vp, vp,
                                           dbl, dbl, vp, vp]
        _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def max_threads() -> int:
    """Threads the oracle's OpenMP loops run on."""
    return int(_load().oracle_max_threads())


def gelu_tanh(u: float) -> float:
    return float(_load().oracle_gelu_tanh(float(u)))


def rmsnorm(v: np.ndarray, s: np.ndarray, eps: float) -> np.ndarray:
    v = np.ascontiguousarray(v, np.float64)
    s = np.ascontiguousarray(s, np.float64)
    out = np.empty_like(v)
    _load().oracle_rmsnorm(v.size, _p(v), _p(s), eps, _p(out))
    return out


def dequant(q: np.ndarray, scale: Optional[np.ndarray] = None, scale_E: int = 1, scale_G: int = 1) -> np.ndarray:
    """Dequantise a stacked weight q [E, N, K] (PyTorch [out, in] order).

    bf16 weights (uint16 bits) need no scale.  int8 weights take bf16 scale bits of
    logical shape (scale_E, scale_G, N), applied with the grouped rule
    w[e, n, k] = q[e, n, k] * s[e if scale_E > 1 else 0, k // (K / scale_G), n].
    """
    q = np.ascontiguousarray(q)
    E, N, K = q.shape
    out = np.empty((E, N, K), np.float32)
    if q.dtype == np.uint16:
        _load().oracle_dequant(W_BF16, _p(q), None, 1, 1, E, N, K, _p(out))
    else:
        assert q.dtype == np.int8 and scale is not None and K % scale_G == 0
        sc = np.ascontiguousarray(scale, np.uint16)
        assert sc.size == scale_E * scale_G * N
        _load().oracle_dequant(W_INT8, _p(q), _p(sc), scale_E, scale_G, E, N, K, _p(out))
    return out


@dataclass
class Route:
    xn: Optional[np.ndarray]  # [T, d] float64 (pre-MoE RMSNorm output)
    p: np.ndarray  # [T, E] float64 softmax probabilities
    idx: np.ndarray  # [T, 2] int32, rank order
    w: np.ndarray  # [T, 2] float64 combine weights (= p at idx)


def _weight_args(inp):
    if inp.weight_dtype == "bf16":
        return W_BF16, inp.w, inp.wv, inp.w1, None, None, None, 1, 1, 1
    # logical scale shape (E_s, G, N): G groups along each weight's input dimension
    return (W_INT8, inp.w, inp.wv, inp.w1, inp.w_scale, inp.wv_scale, inp.w1_scale, inp.scale_experts,
            inp.scale_groups, inp.scale_groups)


def route(inp, keep_xn: bool = False) -> Route:
    T, d, E = inp.T, inp.d, inp.E
    xn = np.empty((T, d), np.float64) if keep_xn else None
    p = np.empty((T, E), np.float64)
    idx = np.empty((T, 2), np.int32)
    w = np.empty((T, 2), np.float64)
    _load().oracle_route(T, d, E, _p(inp.x), _p(inp.gate), _p(inp.bias), _p(inp.s_pre), inp.eps, _p(xn), _p(p),
                         _p(idx), _p(w))
    return Route(xn, p, idx, w)


def routing_stats(p: np.ndarray) -> dict:
    """Routing diagnostics of router probabilities p [T, E] (float64): the mean
    probability of each expert, the routing entropy of that mean distribution in
    nats, and the collapse index 1 - entropy / ln E."""
    p = np.ascontiguousarray(p, np.float64)
    T, E = p.shape
    out = np.empty(E + 2, np.float64)
    _load().oracle_routing_stats(T, E, _p(p), _p(out))
    return {"mean_prob": out[:E].copy(), "entropy": float(out[E]), "collapse": float(out[E + 1])}


def expert_ffn(inp, xn: np.ndarray, e: int):
    """(h, v, a, o) of expert e on the pre-normed vector xn [d] (float64)."""
    d, F = inp.d, inp.F
    xn = np.ascontiguousarray(xn, np.float64)
    h = np.empty(F, np.float64)
    v = np.empty(F, np.float64)
    a = np.empty(F, np.float64)
    o = np.empty(d, np.float64)
    dt, w, wv, w1, sw, swv, sw1, sE, gu, gd = _weight_args(inp)
    _load().oracle_expert_ffn(d, F, e, _p(xn), dt, _p(w), _p(wv), _p(w1), _p(sw), _p(swv), _p(sw1), sE, gu, gd,
                              _p(h), _p(v), _p(a), _p(o))
    return h, v, a, o


@dataclass
class Layer:
    tokens: np.ndarray  # [n] int64 token ids
    y: np.ndarray  # [n, d] float64 layer output
    m: np.ndarray  # [n, d] float64 combined expert output (before post-norm)
    idx: np.ndarray  # [n, 2] int32
    w: np.ndarray  # [n, 2] float64
    p: np.ndarray  # [n, E] float64


def moe_tokens(inp, tokens: Optional[Sequence[int]] = None) -> Layer:
    """The whole layer on a subset of tokens (all tokens when None)."""
    tok = np.arange(inp.T, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, np.int64)
    n, d, F, E = tok.size, inp.d, inp.F, inp.E
    assert n == 0 or (tok.min() >= 0 and tok.max() < inp.T)
    y = np.empty((n, d), np.float64)
    m = np.empty((n, d), np.float64)
    idx = np.empty((n, 2), np.int32)
    w = np.empty((n, 2), np.float64)
    p = np.empty((n, E), np.float64)
    scratch = np.empty(2 * F + 3 * d, np.float64)
    dt, wt, wv, w1, sw, swv, sw1, sE, gu, gd = _weight_args(inp)
    _load().oracle_moe_tokens(n, _p(tok), d, F, E, _p(inp.x), _p(inp.gate), _p(inp.bias), _p(inp.s_pre),
                              _p(inp.s_post), inp.eps, dt, _p(wt), _p(wv), _p(w1), _p(sw), _p(swv), _p(sw1), sE, gu,
                              gd, _p(y), _p(m), _p(idx), _p(w), _p(p), _p(scratch))
    return Layer(tok, y, m, idx, w, p)


def near_tie_tokens(p: np.ndarray, band: float = 1e-6) -> np.ndarray:
    """Mask of tokens whose 2nd and 3rd largest probabilities differ by < band
    (their top-2 set is not decided by the arithmetic; such tokens are excluded
    from exact routing comparisons and counted)."""
    s = -np.sort(-p, axis=1)
    return (s[:, 1] - s[:, 2]) < band


def near_order_tie_tokens(p: np.ndarray, band: float = 1e-6) -> np.ndarray:
    """Mask of tokens whose 1st and 2nd probabilities differ by < band (their
    rank order is compared as a set only)."""
    s = -np.sort(-p, axis=1)
    return (s[:, 0] - s[:, 1]) < band


def rope(v: np.ndarray, pos: int, base: float = 10000.0) -> np.ndarray:
    """Rotary embedding of one head vector (pairs (2i, 2i + 1)) at position pos."""
    out = np.array(v, dtype=np.float64, copy=True, order="C")
    _load().oracle_rope(out.size, _p(out), int(pos), float(base))
    return out


def attn_tokens(inp, tokens: Optional[Sequence[int]] = None, want_ctx: bool = False):
    """Attention block y = x + RMSNorm_post(Wo attn(RMSNorm_pre(x))) of one causal
    sequence, for a subset of its tokens (all when None).  Returns (tok, y, ctx);
    ctx [n, Hq Dh] is the attention output before Wo (None unless asked for)."""
    tok = np.arange(inp.T, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, np.int64)
    n = tok.size
    assert n == 0 or (tok.min() >= 0 and tok.max() < inp.T)
    y = np.empty((n, inp.d), np.float64)
    ctx = np.empty((n, inp.Hq * inp.Dh), np.float64) if want_ctx else None
    if n:
        _load().oracle_attn_tokens(n, _p(tok), inp.T, inp.d, inp.Hq, inp.Hkv, inp.Dh, _p(inp.x), _p(inp.s_pre),
                                   _p(inp.s_post), inp.eps, _p(inp.wq), _p(inp.wk), _p(inp.wv), _p(inp.wo),
                                   inp.rope_base, inp.clamp, _p(y), _p(ctx))
    return tok, y, ctx
