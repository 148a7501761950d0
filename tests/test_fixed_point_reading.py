"""The arithmetic of the int8 GEMV kernels (int8 weights, T <= 16) restated in
numpy, against the oracle: the slot rows (the fp16 normed rows, then the fp16
GeGLU activations) are put in 16-bit fixed point per 128-element block,
sx = max |x| / 32767 and X = rint(x / sx), the int8 x int16 products are summed
exactly per block and each block sum is scaled by sx (the per-channel weight
scales multiply the result).  This checks the reading on the CPU: every element
moves by at most sx / 2 (and the fp32 rounding of sx), and the fixed point costs a small part of the layer's
tolerance |y - y_ref| <= 0.02 |y_ref| + 0.02 rms(y_ref) next to the same
arithmetic without it.  (The GPU tests compare the kernels themselves with the
oracle.)"""
import numpy as np
import pytest

import oracle
import synth

BLOCK = 128


def bf16_bits_to_f32(u16):
    return (np.asarray(u16, np.uint32) << 16).view(np.float32)


def round_bf16(a):
    """fp32 -> bf16 (round to nearest even) -> fp32."""
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def gelu_tanh(u):
    return 0.5 * u * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (u + 0.044715 * u ** 3)))


def quantise(x):
    """Per 128-element block: sx, X, and x as the kernels see it (sx X)."""
    xb = x.reshape(-1, BLOCK).astype(np.float64)
    m = np.max(np.abs(xb), axis=1)
    sx = (m / 32767.0).astype(np.float32).astype(np.float64)
    inv = np.where(m > 0, 32767.0 / np.where(m > 0, m, 1.0), 0.0).astype(np.float32)
    X = np.rint(xb * inv[:, None].astype(np.float64)).astype(np.int64)
    return sx, X


def block_dot(q, sx, X):
    """sum_kb sx[kb] * (q[:, kb] . X[kb]), the integer dot exact per block."""
    nkb = X.shape[0]
    qb = q.astype(np.int64).reshape(q.shape[0], nkb, BLOCK)
    ints = np.einsum("nbk,bk->nb", qb, X)  # exact (int64)
    return ints.astype(np.float64) @ sx


def layer_gemv_arithmetic(inp, fixed_point=True):
    r = oracle.route(inp, keep_xn=True)
    x = bf16_bits_to_f32(inp.x).astype(np.float64)
    sw, sv, s1 = (bf16_bits_to_f32(a).astype(np.float64) for a in (inp.w_scale, inp.wv_scale, inp.w1_scale))
    y = np.zeros_like(x)
    worst = 0.0
    for t in range(inp.T):
        xn16 = round_bf16(r.xn[t].astype(np.float32)).astype(np.float16).astype(np.float64)
        m = np.zeros(inp.d)
        for rank in range(2):
            e = int(r.idx[t, rank])
            es = e if inp.scale_experts > 1 else 0
            if fixed_point:
                sx, X = quantise(xn16)
                worst = max(worst, np.max(np.abs(xn16.reshape(-1, BLOCK) - sx[:, None] * X) / np.maximum(sx[:, None], 1e-300)))
                h = block_dot(inp.w[e], sx, X)
                v = block_dot(inp.wv[e], sx, X)
            else:
                h = inp.w[e].astype(np.float64) @ xn16
                v = inp.wv[e].astype(np.float64) @ xn16
            a = gelu_tanh(sw[es, 0] * h) * (sv[es, 0] * v)
            a16 = np.clip(a, -65504, 65504).astype(np.float16).astype(np.float64)
            if fixed_point:
                sa, A = quantise(a16)
                worst = max(worst, np.max(np.abs(a16.reshape(-1, BLOCK) - sa[:, None] * A) / np.maximum(sa[:, None], 1e-300)))
                o = s1[es, 0] * block_dot(inp.w1[e], sa, A)
            else:
                o = s1[es, 0] * (inp.w1[e].astype(np.float64) @ a16)
            m += float(r.w[t, rank]) * o
        z = m / np.sqrt(np.mean(m ** 2) + inp.eps) * inp.s_post
        y[t] = x[t] + z
    return y, worst


@pytest.mark.parametrize("T,d,F,seed", [(8, 512, 1024, 61), (16, 384, 640, 62)])
def test_fixed_point_slot_rows_cost_little_of_the_tolerance(T, d, F, seed):
    inp = synth.make_inputs(T, d, F, seed, name=f"fixed_point{T}", weight_dtype="int8")
    ref = oracle.moe_tokens(inp).y
    y_q, worst = layer_gemv_arithmetic(inp, fixed_point=True)
    y_f, _ = layer_gemv_arithmetic(inp, fixed_point=False)
    # |x - sx X| <= sx / 2 on every element, up to the fp32 rounding of 1 / sx and sx
    # (|x / sx| <= 32767, so 32767 * 2^-24 * 2 of sx at most)
    assert worst <= 0.5 + 2 * 32767 * 2.0 ** -24
    tol = 0.02 * np.abs(ref) + 0.02 * np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    assert np.max(np.abs(y_q - ref) / tol) <= 0.75         # the arithmetic as a whole, inside
    assert np.max(np.abs(y_q - y_f) / tol) <= 0.05         # the fixed point alone: under 5 % of it
