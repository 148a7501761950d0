"""Pins of the attention-block oracle to facts outside itself (CPU only).

The oracle computes, for a causal sequence, y = x + RMSNorm_post(Wo ctx) with
ctx the grouped-query attention of RoPE-rotated queries and keys whose scaled
logits are clamped to [-30, 30] ("TevunahAi/Grok-1-BF16", "Grok-1 Specific
Behaviors"; "Jah-yee/grok" README, architecture diagram; rotary embedding of
Su et al., "RoFormer").  The checks below rest on:

- the complex-number form of the rotary embedding (each pair (2i, 2i + 1) is the
  complex number v_2i + i v_2i+1 multiplied by exp(i pos theta_i)), its
  identity at position 0, its norm preservation and its relative-position
  property;
- an independent formulation of the whole block with torch library routines in
  fp64 (matmul, complex multiply, clamp, causal mask, softmax, repeat_interleave);
- closed forms: the first token attends only to itself; when every logit is
  clamped to the same bound the attention is a plain causal mean of V;
- causality: outputs of a prefix do not depend on later tokens.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def small(T=37, d=64, Hq=6, Hkv=2, Dh=16, gain=1.6, seed=7):
    return synth.make_attn_inputs(T, d, Hq, Hkv, seed, Dh=Dh, qk_gain=gain)


def torch_block(inp, clamp=True):
    """The block written with torch primitives (fp64), independent of the oracle's loops."""
    T, d, Hq, Hkv, Dh = inp.T, inp.d, inp.Hq, inp.Hkv, inp.Dh
    x = torch.from_numpy(f64(inp.x))
    xn = x / torch.sqrt((x * x).mean(dim=1, keepdim=True) + inp.eps) * torch.from_numpy(inp.s_pre.astype(np.float64))
    q = (xn @ torch.from_numpy(f64(inp.wq)).T).reshape(T, Hq, Dh)
    k = (xn @ torch.from_numpy(f64(inp.wk)).T).reshape(T, Hkv, Dh)
    v = (xn @ torch.from_numpy(f64(inp.wv)).T).reshape(T, Hkv, Dh)
    freq = inp.rope_base ** (-torch.arange(0, Dh, 2, dtype=torch.float64) / Dh)
    rot = torch.polar(torch.ones(T, Dh // 2, dtype=torch.float64),
                      torch.arange(T, dtype=torch.float64)[:, None] * freq[None, :])
    q = torch.view_as_real(torch.view_as_complex(q.reshape(T, Hq, Dh // 2, 2).contiguous()) * rot[:, None, :])
    k = torch.view_as_real(torch.view_as_complex(k.reshape(T, Hkv, Dh // 2, 2).contiguous()) * rot[:, None, :])
    q, k = q.reshape(T, Hq, Dh), k.reshape(T, Hkv, Dh)
    k = k.repeat_interleave(Hq // Hkv, dim=1)
    v = v.repeat_interleave(Hq // Hkv, dim=1)
    s = torch.einsum("thc,jhc->htj", q, k) / np.sqrt(Dh)
    if clamp:
        s = s.clamp(-inp.clamp, inp.clamp)
    s = s.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), diagonal=1), float("-inf"))
    a = torch.softmax(s, dim=-1)
    ctx = torch.einsum("htj,jhc->thc", a, v).reshape(T, Hq * Dh)
    o = ctx @ torch.from_numpy(f64(inp.wo)).T
    y = x + o / torch.sqrt((o * o).mean(dim=1, keepdim=True) + inp.eps) * torch.from_numpy(
        inp.s_post.astype(np.float64))
    return y.numpy(), ctx.numpy(), s


# ---------------------------------------------------------------- rotary embedding

@pytest.mark.parametrize("Dh", [2, 8, 128])
def test_rope_is_complex_rotation(Dh):
    rng = np.random.default_rng(Dh)
    for pos in (0, 1, 5, 777, 8191):
        v = rng.standard_normal(Dh)
        got = oracle.rope(v, pos, 10000.0)
        z = (v[0::2] + 1j * v[1::2]) * np.exp(1j * pos * 10000.0 ** (-np.arange(0, Dh, 2) / Dh))
        want = np.empty(Dh)
        want[0::2], want[1::2] = z.real, z.imag
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12 * max(1, pos))


def test_rope_identity_at_zero_and_norm_preserving():
    rng = np.random.default_rng(1)
    v = rng.standard_normal(128)
    assert np.array_equal(oracle.rope(v, 0), v)
    for pos in (1, 100, 4095):
        r = oracle.rope(v, pos)
        pairs_in = v[0::2] ** 2 + v[1::2] ** 2
        pairs_out = r[0::2] ** 2 + r[1::2] ** 2
        np.testing.assert_allclose(pairs_out, pairs_in, rtol=1e-12)


def test_rope_frequencies():
    """Pair 0 turns by exactly pos radians; pair i by pos * base^(-2i/Dh); the
    rotation is counter-clockwise ((1, 0) goes to (cos, +sin))."""
    Dh, base = 128, 10000.0
    e = np.zeros(Dh)
    e[0::2] = 1.0
    r = oracle.rope(e, 1, base)
    ang = np.arctan2(r[1::2], r[0::2])
    assert abs(ang[0] - 1.0) < 1e-14
    assert r[1] > 0
    np.testing.assert_allclose(ang[-1], base ** (-(Dh - 2) / Dh), rtol=1e-12)
    np.testing.assert_allclose(ang[1:] / ang[:-1], base ** (-2.0 / Dh), rtol=1e-10)


def test_rope_relative_position():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for m, n, s in ((5, 2, 11), (100, 0, 900), (3, 3, 4000)):
        a = oracle.rope(q, m) @ oracle.rope(k, n)
        b = oracle.rope(q, m + s) @ oracle.rope(k, n + s)
        assert abs(a - b) < 1e-9 * (1 + abs(a))


# ---------------------------------------------------------------- whole block

@pytest.mark.parametrize("gain", [1.6, 8.0])
def test_block_matches_torch_formulation(gain):
    inp = small(gain=gain)
    _, y, ctx = oracle.attn_tokens(inp, want_ctx=True)
    y_t, ctx_t, s = torch_block(inp)
    np.testing.assert_allclose(ctx, ctx_t, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(y, y_t, rtol=1e-9, atol=1e-11)
    finite = s[torch.isfinite(s)]
    clamped = (finite.abs() >= inp.clamp).double().mean().item()
    if gain > 5:
        assert 0.2 < clamped < 0.9, clamped  # the clamp binds on part of the logits
        # and it matters: without it the block comes out different
        y_nc, _, _ = torch_block(inp, clamp=False)
        assert np.abs(y_nc - y).max() > 1e-3
    else:
        assert clamped == 0.0


def test_block_token_subset_and_ragged_gqa():
    inp = small(T=23, d=96, Hq=8, Hkv=2, Dh=8)
    y_t, ctx_t, _ = torch_block(inp)
    tok = [22, 0, 13, 13, 5]
    _, y, ctx = oracle.attn_tokens(inp, tok, want_ctx=True)
    np.testing.assert_allclose(y, y_t[tok], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(ctx, ctx_t[tok], rtol=1e-9, atol=1e-11)


def test_first_token_attends_to_itself():
    """Token 0 has one key: ctx of head h is V of key/value head h // (Hq/Hkv)
    (no rotation, no clamp involved)."""
    inp = small(T=5, d=64, Hq=6, Hkv=2, Dh=16)
    x = f64(inp.x)[0]
    xn = x / np.sqrt(np.mean(x * x) + inp.eps) * inp.s_pre
    v = (f64(inp.wv) @ xn).reshape(2, 16)
    ctx = np.concatenate([v[h // 3] for h in range(6)])
    o = f64(inp.wo) @ ctx
    y = x + o / np.sqrt(np.mean(o * o) + inp.eps) * inp.s_post
    _, y_or, ctx_or = oracle.attn_tokens(inp, [0], want_ctx=True)
    np.testing.assert_allclose(ctx_or[0], ctx, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(y_or[0], y, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_saturated_logits_give_causal_mean(sign):
    """Queries and keys built so every logit is past +30 (sign +1) or -30
    (sign -1): all clamp to the same value and each query averages V over the
    keys at or before it."""
    T, d, Hq, Hkv, Dh = 30, 64, 6, 2, 4
    inp = small(T=T, d=d, Hq=Hq, Hkv=Hkv, Dh=Dh)
    x = f64(inp.x)
    x[:, 0] = 8.0  # a large constant column; every row's normalised entry 0 is positive
    inp.x = synth.f32_to_bf16_bits(x.astype(np.float32))
    x = f64(inp.x)
    wq = np.zeros((Hq * Dh, d))
    wk = np.zeros((Hkv * Dh, d))
    for h in range(Hq):
        wq[h * Dh + 2, 0] = 64.0 * sign  # only the slow pair (2, 3) is used
    for g in range(Hkv):
        wk[g * Dh + 2, 0] = 64.0
    inp.wq = synth.f32_to_bf16_bits(wq.astype(np.float32))
    inp.wk = synth.f32_to_bf16_bits(wk.astype(np.float32))
    xn = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + inp.eps) * inp.s_pre
    a = xn[:, 0] * 64.0
    # pair 1 turns by (t - j) * 10000^(-1/2) <= 0.29 rad over 30 tokens: cos > 0.95
    assert (a.min() ** 2 * 0.95 / np.sqrt(Dh)) > inp.clamp
    v = (xn @ f64(inp.wv).T).reshape(T, Hkv, Dh)
    cm = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None, None]
    want = np.concatenate([cm[:, h // (Hq // Hkv), :] for h in range(Hq)], axis=1)
    _, _, ctx = oracle.attn_tokens(inp, want_ctx=True)
    np.testing.assert_allclose(ctx, want, rtol=1e-12, atol=1e-13)


def test_prefix_outputs_do_not_see_later_tokens():
    inp = small(T=40)
    _, y_full, _ = oracle.attn_tokens(inp, range(25))
    short = synth.make_attn_inputs(25, inp.d, inp.Hq, inp.Hkv, 7, Dh=inp.Dh)
    assert np.array_equal(short.x, inp.x[:25])
    _, y_short, _ = oracle.attn_tokens(short)
    assert np.array_equal(y_full, y_short)
    x = inp.x.copy()
    x[25:] = synth.f32_to_bf16_bits(np.full((15, inp.d), 3.0, np.float32))
    inp.x = x
    _, y_pert, _ = oracle.attn_tokens(inp, range(40))
    assert np.array_equal(y_pert[:25], y_full)
    assert not np.array_equal(y_pert[25:], oracle.attn_tokens(small(T=40), range(25, 40))[1])


def test_workload_shapes():
    """Full-size shapes: 48 query and 8 key/value heads of 128 at d = 6144."""
    a = synth.make_attn_inputs(2, 6144, 48, 8, 1)
    assert a.wq.shape == (6144, 6144) and a.wk.shape == (1024, 6144)
    assert a.wv.shape == (1024, 6144) and a.wo.shape == (6144, 6144)
    assert a.clamp == 30.0 and a.Dh == 128


def test_multi_head_special_case():
    """Hkv = Hq (plain multi-head attention, no grouping) against the torch formulation."""
    inp = small(T=19, d=64, Hq=4, Hkv=4, Dh=8)
    y_t, ctx_t, _ = torch_block(inp)
    _, y, ctx = oracle.attn_tokens(inp, want_ctx=True)
    np.testing.assert_allclose(ctx, ctx_t, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(y, y_t, rtol=1e-9, atol=1e-11)


def test_attention_branch_is_scale_invariant():
    """The pre-norm makes the attention branch independent of the scale of x:
    y(a x) - a x equals y(x) - x (a = 4, exact in bf16; eps = 0 so the norm's
    epsilon does not break the invariance)."""
    inp = small(T=21)
    inp.eps = 0.0
    _, y1, _ = oracle.attn_tokens(inp)
    x1 = f64(inp.x)
    inp.x = synth.f32_to_bf16_bits((4.0 * x1).astype(np.float32))
    _, y4, _ = oracle.attn_tokens(inp)
    np.testing.assert_allclose(y4 - 4.0 * x1, y1 - x1, rtol=1e-9, atol=1e-9)
