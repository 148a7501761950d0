"""Seeded synthetic inputs for the Grok-1 MoE feed-forward layer.

Data only: this module draws the arrays both the CPU oracle and the GPU library
consume (hidden states, router gate, norm scales, expert weights) and holds none
of the layer's arithmetic.  Every array is fixed by (seed, tensor id, element
index) through the counter-based generator in ``synth.c``.

Shapes follow the Grok-1 checkpoint as the HF bf16 conversion lists it
(model card "TevunahAi/Grok-1-BF16", section "Weight Verification"):
``linear`` / ``linear_v`` are [F, d] and ``linear_1`` is [d, F] per expert, in
PyTorch [out, in] order; ``moe_block.gate`` is [8, d]; the norm scales are [d].

Workloads (d = 6144, F = 32768, E = 8, top-2 unless noted):

==========  ======  ===============================================================
name        T       values
==========  ======  ===============================================================
tiny        64      d=256, F=512; x N(0,1) bf16; gate N(0, 1/sqrt d) fp32;
                    W, Wv, W1 N(0, 0.02) bf16; norm scales 1
decode      8       x N(0,1) bf16; gate N(0, 1/sqrt d); norm scales U(0.5, 1.5)
                    rounded to bf16; W, Wv, W1 N(0, 0.02) bf16
prefill     8192    as decode (logits come out close to N(0, 1))
int8        2048    weights int8 uniform on [-127, 127]; bf16 scales U(1e-4, 3e-4)
                    of logical shape (8, 1, N), one per expert and output channel
skew        4096    as prefill plus router bias [3, 1, 0, 0, 0, 0, 0, -2]
==========  ======  ===============================================================

The seed of workload k in the list above is 1000 + k.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into synth/_build/libsynth.so with gcc (OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, dbl, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_int32
        vp = ctypes.c_void_p
        lib.synth_stream_key.restype = u64
        lib.synth_stream_key.argtypes = [u64, u64]
        for name in ("synth_normal_f32", "synth_normal_bf16", "synth_uniform_f32", "synth_uniform_bf16"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = [u64, i64, dbl, dbl, vp]
        lib.synth_uniform_int8.restype = None
        lib.synth_uniform_int8.argtypes = [u64, i64, i32, i32, vp]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def key(seed: int, tensor_id: int) -> int:
    return int(_load().synth_stream_key(seed, tensor_id))


def normal_f32(seed, tid, shape, std=1.0, mean=0.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().synth_normal_f32(key(seed, tid), out.size, mean, std, _ptr(out))
    return out


def normal_bf16(seed, tid, shape, std=1.0, mean=0.0, out: Optional[np.ndarray] = None) -> np.ndarray:
    """bf16 values as their uint16 bit patterns."""
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_bf16(key(seed, tid), out.size, mean, std, _ptr(out))
    return out


def uniform_bf16(seed, tid, shape, lo, hi, out: Optional[np.ndarray] = None) -> np.ndarray:
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    _load().synth_uniform_bf16(key(seed, tid), out.size, lo, hi, _ptr(out))
    return out


def uniform_int8(seed, tid, shape, lo, hi, out: Optional[np.ndarray] = None) -> np.ndarray:
    if out is None:
        out = np.empty(shape, dtype=np.int8)
    _load().synth_uniform_int8(key(seed, tid), out.size, lo, hi, _ptr(out))
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


# tensor ids of the streams (one stream per tensor and expert)
TID_X, TID_GATE, TID_SPRE, TID_SPOST = 1, 2, 3, 4
TID_W, TID_WV, TID_W1 = 100, 200, 300
TID_SW, TID_SWV, TID_SW1 = 400, 500, 600


@dataclass
class MoeInputs:
    """One MoE layer's inputs. bf16 arrays hold uint16 bit patterns."""

    name: str
    seed: int
    T: int
    d: int
    F: int
    E: int
    top_k: int
    eps: float
    weight_dtype: str  # "bf16" | "int8"
    x: np.ndarray  # [T, d] bf16 bits
    gate: np.ndarray  # [E, d] float32
    bias: Optional[np.ndarray]  # [E] float32 or None
    s_pre: np.ndarray  # [d] float32 (bf16-representable)
    s_post: np.ndarray  # [d] float32 (bf16-representable)
    w: np.ndarray  # [E, F, d] bf16 bits or int8
    wv: np.ndarray  # [E, F, d]
    w1: np.ndarray  # [E, d, F]
    w_scale: Optional[np.ndarray] = None  # [E_s, G, F] bf16 bits (int8 only)
    wv_scale: Optional[np.ndarray] = None  # [E_s, G, F]
    w1_scale: Optional[np.ndarray] = None  # [E_s, G, d]
    scale_experts: int = 8  # E_s: 8 = one scale set per expert, 1 = shared by all experts
    scale_groups: int = 1   # G: groups along each weight's input dimension
    notes: dict = field(default_factory=dict)


def make_inputs(
    T: int,
    d: int,
    F: int,
    seed: int,
    *,
    name: str = "custom",
    E: int = 8,
    weight_dtype: str = "bf16",
    w_std: float = 0.02,
    gate_std: Optional[float] = None,
    norm_scales: str = "uniform",  # "uniform": U(0.5,1.5) bf16-rounded; "ones"
    bias=None,
    eps: float = 1e-5,
    int8_scale_range=(1e-4, 3e-4),
    int8_scale_shape=(8, 1),
) -> MoeInputs:
    """int8_scale_shape = (E_s, G): the logical scale shape (E_s, G, N) of every
    int8 weight ("TevunahAi/Grok-1-BF16", "Conversion Details" lists (8,1,N),
    (8,8,N), (1,N) and (8,N), the last two read as (1,1,N) and (1,8,N)); scale set
    es is drawn from the stream of expert es, so (8, 1) gives the same values
    whatever else changes."""
    x = normal_bf16(seed, TID_X, (T, d))
    gstd = (1.0 / np.sqrt(d)) if gate_std is None else gate_std
    gate = normal_f32(seed, TID_GATE, (E, d), std=gstd)
    if norm_scales == "ones":
        s_pre = np.ones(d, np.float32)
        s_post = np.ones(d, np.float32)
    else:
        s_pre = bf16_bits_to_f32(uniform_bf16(seed, TID_SPRE, (d,), 0.5, 1.5))
        s_post = bf16_bits_to_f32(uniform_bf16(seed, TID_SPOST, (d,), 0.5, 1.5))
    b = None if bias is None else np.asarray(bias, dtype=np.float32).reshape(E)
    if weight_dtype == "bf16":
        w = np.empty((E, F, d), np.uint16)
        wv = np.empty((E, F, d), np.uint16)
        w1 = np.empty((E, d, F), np.uint16)
        for e in range(E):
            normal_bf16(seed, TID_W + e, None, std=w_std, out=w[e])
            normal_bf16(seed, TID_WV + e, None, std=w_std, out=wv[e])
            normal_bf16(seed, TID_W1 + e, None, std=w_std, out=w1[e])
        sw = swv = sw1 = None
    elif weight_dtype == "int8":
        w = np.empty((E, F, d), np.int8)
        wv = np.empty((E, F, d), np.int8)
        w1 = np.empty((E, d, F), np.int8)
        es_n, g_n = int8_scale_shape
        assert es_n in (1, E) and d % g_n == 0 and F % g_n == 0
        sw = np.empty((es_n, g_n, F), np.uint16)
        swv = np.empty((es_n, g_n, F), np.uint16)
        sw1 = np.empty((es_n, g_n, d), np.uint16)
        lo, hi = int8_scale_range
        for e in range(E):
            uniform_int8(seed, TID_W + e, None, -127, 127, out=w[e])
            uniform_int8(seed, TID_WV + e, None, -127, 127, out=wv[e])
            uniform_int8(seed, TID_W1 + e, None, -127, 127, out=w1[e])
        for es in range(es_n):
            uniform_bf16(seed, TID_SW + es, None, lo, hi, out=sw[es])
            uniform_bf16(seed, TID_SWV + es, None, lo, hi, out=swv[es])
            uniform_bf16(seed, TID_SW1 + es, None, lo, hi, out=sw1[es])
    else:
        raise ValueError(weight_dtype)
    return MoeInputs(name=name, seed=seed, T=T, d=d, F=F, E=E, top_k=2, eps=eps, weight_dtype=weight_dtype,
                     x=x, gate=gate, bias=b, s_pre=s_pre, s_post=s_post, w=w, wv=wv, w1=w1,
                     w_scale=sw, wv_scale=swv, w1_scale=sw1,
                     scale_experts=int8_scale_shape[0] if weight_dtype == "int8" else E,
                     scale_groups=int8_scale_shape[1] if weight_dtype == "int8" else 1)


GROK_D, GROK_F = 6144, 32768

# The five workloads, in order; their seeds are 1000 + position.
WORKLOADS = ("tiny", "decode", "prefill", "int8", "skew")
SKEW_BIAS = (3.0, 1.0, 0.0, 0.0, 0.0, 0.0, 0.0, -2.0)


def workload(name: str, T: Optional[int] = None) -> MoeInputs:
    """Inputs of a named workload. ``T`` overrides the token count (same seed:
    the first rows of x are the same whatever T is)."""
    k = WORKLOADS.index(name)
    seed = 1000 + k
    if name == "tiny":
        return make_inputs(T or 64, 256, 512, seed, name=name, norm_scales="ones")
    if name == "decode":
        return make_inputs(T or 8, GROK_D, GROK_F, seed, name=name)
    if name == "prefill":
        return make_inputs(T or 8192, GROK_D, GROK_F, seed, name=name)
    if name == "int8":
        return make_inputs(T or 2048, GROK_D, GROK_F, seed, name=name, weight_dtype="int8")
    if name == "skew":
        return make_inputs(T or 4096, GROK_D, GROK_F, seed, name=name, bias=SKEW_BIAS)
    raise KeyError(name)


# ----------------------------------------------------------------------------
# Attention half of the decoder layer (GQA with rotary embeddings, logit clamp).
# Shapes from "TevunahAi/Grok-1-BF16", "Weight Verification": q_proj [Hq Dh, d],
# k_proj and v_proj [Hkv Dh, d], o_proj [d, Hq Dh] in PyTorch [out, in] order,
# pre/post-attention norm scales [d]; 48 query and 8 key/value heads of 128 at
# d = 6144 ("Jah-yee/grok" README).

TID_WQ, TID_WK, TID_WVA, TID_WO, TID_SPRE_A, TID_SPOST_A = 700, 701, 702, 703, 704, 705


@dataclass
class AttnInputs:
    """One attention block's inputs for a causal sequence of T tokens at
    positions 0..T-1. bf16 arrays hold uint16 bit patterns."""

    name: str
    seed: int
    T: int
    d: int
    Hq: int
    Hkv: int
    Dh: int
    eps: float
    rope_base: float
    clamp: float
    x: np.ndarray  # [T, d] bf16 bits
    s_pre: np.ndarray  # [d] float32 (bf16-representable)
    s_post: np.ndarray  # [d] float32
    wq: np.ndarray  # [Hq Dh, d] bf16 bits
    wk: np.ndarray  # [Hkv Dh, d]
    wv: np.ndarray  # [Hkv Dh, d]
    wo: np.ndarray  # [d, Hq Dh]


def make_attn_inputs(T: int, d: int, Hq: int, Hkv: int, seed: int, *, name: str = "custom", Dh: int = 128,
                     qk_gain: float = 1.6, eps: float = 1e-5, rope_base: float = 10000.0,
                     clamp: float = 30.0) -> AttnInputs:
    """x ~ N(0, 1); Wq, Wk ~ N(0, qk_gain / sqrt(d)) (1.6 gives attention logits
    of standard deviation about 2.5, 5 pushes most of them past the clamp);
    Wv ~ N(0, 1 / sqrt(d)); Wo ~ N(0, 1 / sqrt(Hq Dh)); norm scales U(0.5, 1.5)
    rounded to bf16."""
    x = normal_bf16(seed, TID_X, (T, d))
    s_pre = bf16_bits_to_f32(uniform_bf16(seed, TID_SPRE_A, (d,), 0.5, 1.5))
    s_post = bf16_bits_to_f32(uniform_bf16(seed, TID_SPOST_A, (d,), 0.5, 1.5))
    wq = normal_bf16(seed, TID_WQ, (Hq * Dh, d), std=qk_gain / np.sqrt(d))
    wk = normal_bf16(seed, TID_WK, (Hkv * Dh, d), std=qk_gain / np.sqrt(d))
    wv = normal_bf16(seed, TID_WVA, (Hkv * Dh, d), std=1.0 / np.sqrt(d))
    wo = normal_bf16(seed, TID_WO, (d, Hq * Dh), std=1.0 / np.sqrt(Hq * Dh))
    return AttnInputs(name=name, seed=seed, T=T, d=d, Hq=Hq, Hkv=Hkv, Dh=Dh, eps=eps, rope_base=rope_base,
                      clamp=clamp, x=x, s_pre=s_pre, s_post=s_post, wq=wq, wk=wk, wv=wv, wo=wo)


# Attention workloads; their seeds are 2000 + position.
ATTN_WORKLOADS = ("attn_tiny", "attn_clamp", "attn_prefill")


def attn_workload(name: str, T: Optional[int] = None) -> AttnInputs:
    """attn_tiny: T=200, d=768, 6 query heads on 1 key/value head (the 6:1 ratio
    of 48:8); attn_clamp: the same with Wq, Wk gain 5 so the +-30 clamp binds;
    attn_prefill: T=8192 at d=6144, 48/8 heads.  ``T`` overrides the length
    (the first rows of x do not depend on it)."""
    seed = 2000 + ATTN_WORKLOADS.index(name)
    if name == "attn_tiny":
        return make_attn_inputs(T or 200, 768, 6, 1, seed, name=name)
    if name == "attn_clamp":
        return make_attn_inputs(T or 200, 768, 6, 1, seed, name=name, qk_gain=5.0)
    if name == "attn_prefill":
        return make_attn_inputs(T or 8192, GROK_D, 48, 8, seed, name=name)
    raise KeyError(name)
