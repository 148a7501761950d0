"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something its own code does not produce:
values the pages print, closed forms, exact identities, special cases that reduce
to library routines (torch fp64 on CPU), brute force on tiny inputs, and an
independent numpy dequantisation.  Together they catch a dropped term, a wrong
sign or index, a swapped W / Wv, a transposed W1, a renormalised combine, a
missing residual or norm, and a wrong tie-break.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def _f64(bits):
    return torch.from_numpy(synth.bf16_bits_to_f32(bits).astype(np.float64))


def _weights_f64(inp):
    """Dense fp64 weights, dequantised by an independent numpy broadcast."""
    if inp.weight_dtype == "bf16":
        return _f64(inp.w), _f64(inp.wv), _f64(inp.w1)

    def full(scale, q):
        # scale [E_s, G, N] -> [E, N, K]: group g covers inputs [g K/G, (g+1) K/G)
        E, N, K = q.shape
        s = synth.bf16_bits_to_f32(scale)
        s = np.repeat(np.transpose(s, (0, 2, 1)), K // s.shape[1], axis=2)
        return np.broadcast_to(s, (E, N, K))

    return tuple(torch.from_numpy((q.astype(np.float32) * full(s, q)).astype(np.float64))
                 for q, s in ((inp.w, inp.w_scale), (inp.wv, inp.wv_scale), (inp.w1, inp.w1_scale)))


def _torch_layer_dense(inp):
    """Brute force with library routines: every expert on every token, then a
    top-2 mask.  torch.rms_norm / softmax / topk / gelu(tanh) / matmul, fp64."""
    x = _f64(inp.x)
    s_pre = torch.from_numpy(inp.s_pre.astype(np.float64))
    s_post = torch.from_numpy(inp.s_post.astype(np.float64))
    G = torch.from_numpy(inp.gate.astype(np.float64))
    xn = Fn.rms_norm(x, (inp.d,), weight=s_pre, eps=inp.eps)
    logits = xn @ G.T
    if inp.bias is not None:
        logits = logits + torch.from_numpy(inp.bias.astype(np.float64))
    p = torch.softmax(logits, dim=-1)
    topv, topi = torch.topk(p, 2, dim=-1)
    W, Wv, W1 = _weights_f64(inp)
    m = torch.zeros_like(x)
    for e in range(inp.E):
        o = (Fn.gelu(xn @ W[e].T, approximate="tanh") * (xn @ Wv[e].T)) @ W1[e].T
        wsel = (topi == e).to(torch.float64) * topv
        m = m + wsel.sum(dim=1, keepdim=True) * o
    y = x + Fn.rms_norm(m, (inp.d,), weight=s_post, eps=inp.eps)
    return y.numpy(), m.numpy(), topi.numpy(), topv.numpy(), p.numpy()


def _relerr(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------- elementwise

def test_gelu_tanh_identities_and_library():
    assert oracle.gelu_tanh(0.0) == 0.0
    us = np.linspace(-8, 8, 161)
    for u in us:
        # odd part of x*Phi-like gates: gelu(u) - gelu(-u) = u exactly in real arithmetic
        assert abs(oracle.gelu_tanh(u) - oracle.gelu_tanh(-u) - u) <= 1e-14 * max(1.0, abs(u))
    ref = Fn.gelu(torch.tensor(us, dtype=torch.float64), approximate="tanh").numpy()
    got = np.array([oracle.gelu_tanh(u) for u in us])
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-15)
    # the tanh form is not the erf form: they differ by ~1e-3 near u=-2
    erf_form = Fn.gelu(torch.tensor([-2.0], dtype=torch.float64)).item()
    assert abs(oracle.gelu_tanh(-2.0) - erf_form) > 1e-5


def test_rmsnorm_closed_form():
    d, eps = 64, 1e-5
    s = np.linspace(0.5, 1.5, d)
    for c in (3.0, -0.25, 1e-3):
        out = oracle.rmsnorm(np.full(d, c), s, eps)
        expect = math.copysign(1.0, c) * s / math.sqrt(1.0 + eps / (c * c))
        np.testing.assert_allclose(out, expect, rtol=1e-15)
    v = np.random.default_rng(0).standard_normal(d)
    out = oracle.rmsnorm(v, np.ones(d), eps)
    ms = np.mean(v * v)
    assert abs(math.sqrt(np.mean(out * out)) - 1.0 / math.sqrt(1.0 + eps / ms)) < 1e-15


# -------------------------------------------------------------------- router

def test_uniform_router_matches_page_demo():
    g = _golden("uniform_router.txt")
    inp = synth.make_inputs(16, 256, 512, 7, norm_scales="ones")
    inp.gate[:] = 0.0
    r = oracle.route(inp)
    assert np.all(r.p == 1.0 / 8.0)
    assert round(float(r.p[0, 0]), 3) == g["expert_weight"]
    ent = -float(np.sum(r.p[0] * np.log(r.p[0])))
    assert abs(ent - math.log(8)) < 1e-12
    assert round(ent, 3) == g["routing_entropy"] == g["routing_entropy_max"]
    # all-equal probabilities: the two lowest indices, in order
    assert np.all(r.idx == np.array([0, 1]))
    assert np.all(r.w == 0.125)


def test_routing_stats_uniform_router_matches_page_demo():
    """The README demo's untrained router: 0.125 per expert, entropy 2.079 of 2.079."""
    g = _golden("uniform_router.txt")
    inp = synth.make_inputs(24, 256, 512, 9, norm_scales="ones")
    inp.gate[:] = 0.0
    s = oracle.routing_stats(oracle.route(inp).p)
    assert np.all(np.round(s["mean_prob"], 3) == g["expert_weight"])
    assert round(s["entropy"], 3) == g["routing_entropy"] == round(math.log(g["num_experts"]), 3)
    assert abs(s["entropy"] - math.log(8)) < 1e-12 and abs(s["collapse"]) < 1e-12


@pytest.mark.parametrize("hot,entropy", [
    ((5,), 0.0),                  # one expert takes every token: entropy 0, collapse 1
    ((2, 6), math.log(2)),        # two experts share every token equally: ln 2
    ((0, 3, 7, 1), math.log(4)),  # four equal experts: ln 4
])
def test_routing_stats_closed_forms(hot, entropy):
    inp = synth.make_inputs(20, 256, 512, 10, norm_scales="ones")
    inp.gate[:] = 0.0
    b = np.full(8, -1e4, np.float32)
    b[list(hot)] = 0.0
    inp.bias = b
    s = oracle.routing_stats(oracle.route(inp).p)
    expect = np.zeros(8)
    expect[list(hot)] = 1.0 / len(hot)
    np.testing.assert_allclose(s["mean_prob"], expect, atol=1e-12)
    assert abs(s["entropy"] - entropy) < 1e-9
    assert abs(s["collapse"] - (1.0 - entropy / math.log(8))) < 1e-9


def test_routing_stats_invariants():
    inp = synth.make_inputs(300, 256, 512, 11, bias=synth.SKEW_BIAS)
    r = oracle.route(inp)
    s = oracle.routing_stats(r.p)
    assert abs(s["mean_prob"].sum() - 1.0) < 1e-12
    assert 0.0 < s["entropy"] < math.log(8)
    # the skew bias favours expert 0 and disfavours expert 7
    assert s["mean_prob"].argmax() == 0 and s["mean_prob"].argmin() == 7
    # token order does not matter
    perm = np.random.default_rng(3).permutation(inp.T)
    s2 = oracle.routing_stats(r.p[perm])
    np.testing.assert_allclose(s2["mean_prob"], s["mean_prob"], rtol=1e-13)


@pytest.mark.parametrize("bias,expect", [
    ([0, 0, 0, 5, 0, 5, 0, 0], (3, 5)),
    ([1, 2, 2, 0, 0, 0, 0, 0], (1, 2)),
    ([0, 0, 0, 0, 0, 0, 0, 1], (7, 0)),
    ([4, 0, 0, 0, 0, 0, 0, 4], (0, 7)),
    ([0, 0, 0, 0, 0, 0, 3, 0], (6, 0)),
])
def test_router_tie_break_lower_index(bias, expect):
    inp = synth.make_inputs(4, 256, 512, 8, norm_scales="ones", bias=bias)
    inp.gate[:] = 0.0
    r = oracle.route(inp)
    assert np.all(r.idx == np.array(expect))


def test_routing_invariants():
    inp = synth.workload("tiny")
    r = oracle.route(inp)
    assert np.all(r.idx[:, 0] != r.idx[:, 1])
    assert np.all((r.idx >= 0) & (r.idx < 8))
    counts = np.bincount(r.idx.ravel(), minlength=8)
    assert counts.sum() == 2 * inp.T
    np.testing.assert_allclose(r.p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(r.w, np.take_along_axis(r.p, r.idx, axis=1))
    # no renormalisation: the two weights sum to less than one
    assert np.all(r.w.sum(axis=1) < 1.0)
    # rank order: the first pick has the larger probability
    assert np.all(r.w[:, 0] >= r.w[:, 1])


# ------------------------------------------------------------- whole layer

@pytest.mark.parametrize("which", ["tiny", "mid", "tiny_int8", "int8_8x8", "int8_1x1", "int8_1x8", "tiny_bias"])
def test_layer_equals_dense_bruteforce(which):
    if which == "tiny":
        inp = synth.workload("tiny")
    elif which == "mid":
        inp = synth.make_inputs(24, 384, 640, 11)
    elif which == "tiny_int8":
        inp = synth.make_inputs(32, 256, 512, 12, weight_dtype="int8", int8_scale_range=(1e-3, 3e-3))
    elif which.startswith("int8_"):  # grouped / shared scale shapes (8,8,N), (1,N), (8,N)
        es, g = (int(v) for v in which[5:].split("x"))
        inp = synth.make_inputs(32, 256, 512, 14, weight_dtype="int8", int8_scale_range=(1e-3, 3e-3),
                                int8_scale_shape=(es, g))
    else:
        inp = synth.make_inputs(32, 256, 512, 13, bias=synth.SKEW_BIAS)
    y_ref, m_ref, idx_ref, w_ref, p_ref = _torch_layer_dense(inp)
    lay = oracle.moe_tokens(inp)
    assert not oracle.near_tie_tokens(p_ref).any()
    np.testing.assert_array_equal(lay.idx, idx_ref)
    np.testing.assert_allclose(lay.w, w_ref, rtol=1e-13)
    np.testing.assert_allclose(lay.p, p_ref, rtol=1e-12, atol=1e-15)
    assert _relerr(lay.m, m_ref) < 1e-10
    assert _relerr(lay.y, y_ref) < 1e-12


def test_one_hot_router_is_one_dense_mlp():
    """b_e = +1e4 makes p_e = 1 exactly: y = x + post_norm(FFN_e(pre_norm(x)))."""
    inp = synth.make_inputs(8, 256, 512, 21)
    e = 5
    bias = np.zeros(8, np.float32)
    bias[e] = 1e4
    inp.bias = bias
    lay = oracle.moe_tokens(inp)
    assert np.all(lay.idx[:, 0] == e) and np.all(lay.w[:, 0] == 1.0) and np.all(lay.w[:, 1] == 0.0)
    x = _f64(inp.x)
    W, Wv, W1 = _weights_f64(inp)
    xn = Fn.rms_norm(x, (inp.d,), weight=torch.from_numpy(inp.s_pre.astype(np.float64)), eps=inp.eps)
    o = Fn.linear(Fn.gelu(Fn.linear(xn, W[e]), approximate="tanh") * Fn.linear(xn, Wv[e]), W1[e])
    y = x + Fn.rms_norm(o, (inp.d,), weight=torch.from_numpy(inp.s_post.astype(np.float64)), eps=inp.eps)
    assert _relerr(lay.m, o.numpy()) < 1e-12
    assert _relerr(lay.y, y.numpy()) < 1e-12


def test_two_hot_router_combines_half_and_half():
    """gate = 0 and b = +1e4 on experts a, b: weights are exactly 1/2 each."""
    inp = synth.make_inputs(6, 256, 512, 22)
    inp.gate[:] = 0.0
    a, b = 2, 6
    bias = np.zeros(8, np.float32)
    bias[[a, b]] = 1e4
    inp.bias = bias
    lay = oracle.moe_tokens(inp)
    assert np.all(lay.idx == np.array([a, b])) and np.all(lay.w == 0.5)
    x = _f64(inp.x)
    W, Wv, W1 = _weights_f64(inp)
    xn = Fn.rms_norm(x, (inp.d,), weight=torch.from_numpy(inp.s_pre.astype(np.float64)), eps=inp.eps)
    o = [(Fn.gelu(xn @ W[k].T, approximate="tanh") * (xn @ Wv[k].T)) @ W1[k].T for k in (a, b)]
    m = 0.5 * o[0] + 0.5 * o[1]
    assert _relerr(lay.m, m.numpy()) < 1e-12


def test_expert_ffn_intermediates():
    """h = W xn and v = Wv xn (not swapped), a = gelu(h) v, o = W1 a."""
    inp = synth.make_inputs(4, 256, 512, 23)
    r = oracle.route(inp, keep_xn=True)
    xn = r.xn[1]
    h, v, a, o = oracle.expert_ffn(inp, xn, 3)
    W, Wv, W1 = _weights_f64(inp)
    xt = torch.from_numpy(xn)
    np.testing.assert_allclose(h, (W[3] @ xt).numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(v, (Wv[3] @ xt).numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(a, (Fn.gelu(torch.from_numpy(h), approximate="tanh") * torch.from_numpy(v)).numpy(),
                               rtol=1e-14)
    np.testing.assert_allclose(o, (W1[3] @ torch.from_numpy(a)).numpy(), rtol=1e-12, atol=1e-15)


def test_token_order_invariance_bitwise():
    inp = synth.make_inputs(20, 256, 512, 24, bias=[0.5, 0, 0, 0, 0, 0, 0, -0.5])
    lay = oracle.moe_tokens(inp)
    perm = np.random.default_rng(3).permutation(inp.T)
    inp2 = synth.make_inputs(20, 256, 512, 24, bias=[0.5, 0, 0, 0, 0, 0, 0, -0.5])
    inp2.x = np.ascontiguousarray(inp.x[perm])
    lay2 = oracle.moe_tokens(inp2)
    np.testing.assert_array_equal(lay2.y, lay.y[perm])
    np.testing.assert_array_equal(lay2.idx, lay.idx[perm])
    # subsets give the same rows as the full run (tokens are independent)
    sub = oracle.moe_tokens(inp, [19, 3, 7])
    np.testing.assert_array_equal(sub.y, lay.y[[19, 3, 7]])


def test_zero_post_norm_scale_leaves_residual():
    inp = synth.make_inputs(5, 256, 512, 25)
    inp.s_post = np.zeros(inp.d, np.float32)
    lay = oracle.moe_tokens(inp)
    np.testing.assert_array_equal(lay.y, synth.bf16_bits_to_f32(inp.x).astype(np.float64))


def test_layer_is_not_renormalised():
    """Doubling both combine weights (renormalising to sum 1 would) changes m;
    check the oracle's m equals w0 o0 + w1 o1 with w = p, not p / (p0 + p1)."""
    inp = synth.make_inputs(3, 256, 512, 26)
    r = oracle.route(inp, keep_xn=True)
    lay = oracle.moe_tokens(inp)
    for t in range(inp.T):
        o0 = oracle.expert_ffn(inp, r.xn[t], int(r.idx[t, 0]))[3]
        o1 = oracle.expert_ffn(inp, r.xn[t], int(r.idx[t, 1]))[3]
        np.testing.assert_allclose(lay.m[t], r.p[t, r.idx[t, 0]] * o0 + r.p[t, r.idx[t, 1]] * o1, rtol=1e-13)


# --------------------------------------------------------------- dequant

def _numpy_grouped_dequant(q, s, scale_E, scale_G):
    """Independent grouped broadcast: view q as JAX [E, K, N], repeat the scale
    groups along K, broadcast over experts, transpose back to [E, N, K]."""
    E, N, K = q.shape
    qj = np.transpose(q, (0, 2, 1)).astype(np.float32)  # [E, K, N]
    sf = synth.bf16_bits_to_f32(s).reshape(scale_E, scale_G, N)
    sk = np.repeat(sf, K // scale_G, axis=1)  # [E_s, K, N]
    wj = qj * sk  # broadcasts E_s = 1 across experts
    return np.ascontiguousarray(np.transpose(wj, (0, 2, 1)))


@pytest.mark.parametrize("shape", [(1, 32), (8, 32), (8, 1, 32), (8, 8, 32)])
def test_int8_dequant_scale_shapes(shape):
    E, N, K = 8, 32, 64
    q = synth.uniform_int8(5, 1, (E, N, K), -127, 127)
    s = synth.uniform_bf16(5, 2, shape, 1e-4, 3e-4)
    # left-pad the scale shape with ones to (E_s, G, N); a 2-D (8, N) is 8 K-groups
    padded = (1,) * (3 - len(shape)) + tuple(shape)
    scale_E, scale_G = padded[0], padded[1]
    got = oracle.dequant(q, s.ravel(), scale_E, scale_G)
    ref = _numpy_grouped_dequant(q, s.ravel(), scale_E, scale_G)
    np.testing.assert_array_equal(got, ref)
    # plain numpy broadcasting of the JAX-order weight agrees where it applies
    if len(shape) == 2 and shape[0] == 1 or shape == (8, 1, 32):
        qj = np.transpose(q, (0, 2, 1)).astype(np.float32)
        b = np.transpose(qj * synth.bf16_bits_to_f32(s), (0, 2, 1))
        np.testing.assert_array_equal(got, b)
    # the product is exact in fp32: equals the fp64 product
    exact = _numpy_grouped_dequant(q.astype(np.float64).astype(np.int8), s.ravel(), scale_E, scale_G)
    np.testing.assert_array_equal(got.astype(np.float64), exact.astype(np.float64))


def test_bf16_weights_pass_through():
    q = synth.normal_bf16(3, 3, (2, 16, 32), std=0.02)
    np.testing.assert_array_equal(oracle.dequant(q), synth.bf16_bits_to_f32(q))
