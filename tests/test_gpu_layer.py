"""GPU parity of the whole layer against the CPU oracle, through the C ABI, at
sizes the oracle runs in seconds: several tiles along every dimension, ragged
row blocks, ragged d, the degenerate routers and the argument edge cases."""
import numpy as np
import pytest
import torch

import oracle
import synth
import mixture_experts_transformer_gemv_b300 as moe

from layer_helpers import (assert_routing, assert_values, bf16_tensor, device_weights, make_layer, read_device,
                           run, value_report)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mixture_experts_transformer_gemv_b300 import build
    build.build()
    assert torch.cuda.is_available()


def _full_check(inp, flags=0, max_tokens=None):
    layer = make_layer(inp, max_tokens=max_tokens, flags=flags)
    y, idx, prob, counts = run(layer, inp)
    ref = oracle.moe_tokens(inp)
    assert_routing(idx, prob, counts, ref, inp.name)
    rep = assert_values(y, ref.y, inp.name)
    layer.close()
    return rep


def test_tiny_workload_all_tokens():
    _full_check(synth.workload("tiny"))


@pytest.mark.parametrize("T,d,F,seed", [
    (300, 512, 1024, 31),    # 8 up-tiles x 2 down-tiles, one ragged row block per expert
    (1000, 256, 640, 32),    # two row blocks per expert, F/128 = 5
    (200, 384, 512, 33),     # d = 384: the last down-projection tile is half outside d
    (7, 256, 512, 34),       # fewer slots than a tile in every expert
    (1500, 256, 512, 36),    # router: 148 CTAs, 1184 warps, runs of 1-2 tokens
    (2400, 256, 512, 37),    # router: runs of 2-3 tokens per warp
    (1200, 7680, 256, 38),   # wide rows: the scaled gate (8 x d fp32) exceeds shared memory, read from L2
    (600, 14464, 256, 39),   # wider still, 57 chunks per lane (a ragged last step)
    (1300, 3072, 256, 40),   # the gate in shared memory, 12 chunks per lane
    (1200, 7040, 256, 41),   # near the widest gate shared memory holds (220 KB)
    (2400, 256, 16384, 42),  # F >= 16384, T >= 2048: two m-blocks per tile; ~600 rows per expert = a
                             # pair of full m-blocks and a half block alone
    (2047, 256, 16384, 45),  # one token below the pairing threshold: one m-block per tile
])
def test_mid_shapes(T, d, F, seed):
    _full_check(synth.make_inputs(T, d, F, seed, name=f"mid{T}x{d}x{F}"))


@pytest.mark.parametrize("T,d,seed", [(1184, 256, 43), (40, 7680, 44)])
def test_routing_does_not_depend_on_the_batch(T, d, seed):
    """Every token's router sums run in the same order whatever the batch (the
    warp that takes it, its position, T), with the gate in shared memory (d =
    256) or read from L2 (d = 7680): a token routes the same to the last bit
    (expert pair and probabilities) in the whole batch, in a prefix, in a suffix
    and alone (T = 1, the decode path's size); up to 16 tokens the router runs
    as one CTA per token (router_small_kernel, the 12-token run), beyond that
    as warps over runs of tokens."""
    inp = synth.make_inputs(T, d, 256, seed, name=f"router_batch{T}x{d}")
    layer = make_layer(inp)
    x = bf16_tensor(inp.x)
    _, idx_a, prob_a, _ = layer.forward(x, routing=True)
    idx_a, prob_a = idx_a.clone(), prob_a.clone()
    for lo, hi in ((0, T - 1), (T - 37, T), (T // 2, T // 2 + 1), (5, 17)):
        _, idx_b, prob_b, _ = layer.forward(x[lo:hi].contiguous(), routing=True)
        torch.cuda.synchronize()
        assert torch.equal(idx_a[lo:hi], idx_b), (lo, hi)
        assert torch.equal(prob_a[lo:hi], prob_b), (lo, hi)
    layer.sync_status()
    layer.close()


def test_skewed_bias_small():
    inp = synth.make_inputs(256, 256, 512, 35, bias=synth.SKEW_BIAS, name="skew_small")
    _full_check(inp)


def test_single_token_and_empty():
    inp = synth.make_inputs(1, 256, 512, 36, name="one")
    _full_check(inp, max_tokens=16)
    layer = make_layer(inp, max_tokens=16)
    x = bf16_tensor(inp.x)
    before = layer.launch_count()
    layer.forward(x[:0])
    assert layer.launch_count() == before  # T = 0 enqueues nothing
    layer.close()


def test_one_hot_router_single_expert():
    """All tokens to expert 5 with weight 1; the second pick has weight 0."""
    inp = synth.make_inputs(200, 256, 512, 37, name="onehot")
    b = np.zeros(8, np.float32)
    b[5] = 1e4
    inp.bias = b
    layer = make_layer(inp)
    y, idx, prob, counts = run(layer, inp)
    assert np.all(idx[:, 0] == 5) and np.all(idx[:, 1] == 0)
    assert np.all(prob[:, 0] == 1.0) and np.all(prob[:, 1] == 0.0)
    assert counts[5] == 200 and counts[0] == 200
    ref = oracle.moe_tokens(inp)
    assert_values(y, ref.y, "one-hot")


def test_uniform_router_picks_first_two():
    inp = synth.make_inputs(64, 256, 512, 38, name="uniform")
    inp.gate[:] = 0.0
    layer = make_layer(inp)
    y, idx, prob, counts = run(layer, inp)
    assert np.all(idx == np.array([0, 1]))
    assert np.all(prob == 0.125)
    assert list(counts) == [64, 64, 0, 0, 0, 0, 0, 0]
    assert_values(y, oracle.moe_tokens(inp).y, "uniform")


def test_in_place_and_host_entry_point():
    inp = synth.make_inputs(96, 256, 512, 39, name="inplace")
    layer = make_layer(inp)
    y_ref = oracle.moe_tokens(inp).y
    x = bf16_tensor(inp.x)
    out = layer.forward(x.clone())
    xi = x.clone()
    layer.forward(xi, out=xi)
    torch.cuda.synchronize()
    layer.sync_status()
    assert torch.equal(out, xi)
    assert_values(xi.float().cpu().numpy().astype(np.float64), y_ref, "in place")
    xh = bf16_tensor(inp.x, device=None).pin_memory()
    oh, idx, prob, counts = layer.forward_host(xh, routing=True)
    assert torch.equal(oh, out.cpu())
    assert counts.sum().item() == 2 * inp.T


def test_async_host_calls_match_device_calls():
    """Four moe_layer_forward_host_async calls in flight on alternating staging
    slots: each output equals a device-buffer forward of the same input."""
    inp = synth.make_inputs(96, 256, 512, 96, name="async")
    layer = make_layer(inp)
    x = bf16_tensor(inp.x)
    xs = [torch.roll(x, shifts=7 * i, dims=0).contiguous() for i in range(4)]
    xh = [t.cpu().pin_memory() for t in xs]
    oh = [torch.empty_like(h).pin_memory() for h in xh]
    for h, o in zip(xh, oh):
        layer.forward_host_async(h, o)
    layer.host_wait()
    for t, o in zip(xs, oh):
        direct = layer.forward(t)
        torch.cuda.synchronize()
        assert torch.equal(o, direct.cpu())
    layer.close()


def test_token_permutation():
    inp = synth.make_inputs(400, 256, 512, 40, name="perm")
    layer = make_layer(inp)
    y, idx, prob, counts = run(layer, inp)
    perm = np.random.default_rng(1).permutation(inp.T)
    x2 = bf16_tensor(np.ascontiguousarray(inp.x[perm]))
    y2, idx2, prob2, counts2 = run(layer, inp, x_dev=x2)
    np.testing.assert_array_equal(idx2, idx[perm])
    np.testing.assert_array_equal(prob2, prob[perm])
    np.testing.assert_array_equal(counts2, counts)
    r = value_report(y2, y[perm])
    assert r["violations"] == 0, r


def test_token_limits():
    inp = synth.make_inputs(32, 256, 512, 41, name="limits")
    layer = make_layer(inp, max_tokens=32)
    x = bf16_tensor(inp.x)
    layer.forward(x)  # T == max_tokens
    big = torch.zeros((33, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        layer.forward(big)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    layer.sync_status()


def test_device_checks_flag_clean_run():
    inp = synth.make_inputs(128, 256, 512, 42, name="checks")
    _full_check(inp, flags=moe.MOE_FLAG_DEVICE_CHECKS)


def test_intermediates_match_oracle():
    """Normed rows, expert grouping, GeGLU activations and scaled expert outputs."""
    inp = synth.workload("tiny")
    layer = make_layer(inp)
    run(layer, inp)
    ws = layer.workspace()
    R = ws.rows_cap
    T, d, F = inp.T, inp.d, inp.F
    rnorm = read_device(ws.rnorm, (inp.T,), torch.float32)
    xn_perm = read_device(ws.xn_perm, (R, d), torch.bfloat16)
    counts = read_device(ws.counts, (8,), torch.int32)
    off = read_device(ws.row_offset, (9,), torch.int32)
    ros = read_device(ws.row_of_slot, (T, 2), torch.int32)
    act = read_device(ws.act, (R, F), torch.bfloat16)
    yr = read_device(ws.y_rows, (R, d), torch.float32)
    r = oracle.route(inp, keep_xn=True)
    # the router's 1 / rms, and the normed rows the gather formed from it
    xs = synth.bf16_bits_to_f32(inp.x).astype(np.float64)
    np.testing.assert_allclose(rnorm, 1.0 / np.sqrt(np.mean(xs * xs, axis=1) + inp.eps), rtol=1e-5)
    for k in range(2):
        np.testing.assert_allclose(xn_perm[ros[:, k]], r.xn, rtol=2 ** -8, atol=1e-6)
    pad = np.setdiff1d(np.arange(int(off[8])), ros.ravel())
    assert pad.size == int(off[8]) - 2 * T and np.all(xn_perm[pad] == 0)
    np.testing.assert_array_equal(counts, np.bincount(r.idx.ravel(), minlength=8))
    # each expert's block is its slots padded to the next multiple of 128 rows
    assert off[0] == 0 and np.all(off % 128 == 0)
    np.testing.assert_array_equal(np.diff(off), (counts + 127) // 128 * 128)
    for t in (0, 17, T - 1):
        for rank in range(2):
            e = int(r.idx[t, rank])
            row = int(ros[t, rank])
            assert off[e] <= row < off[e] + counts[e]
            h, v, a, o = oracle.expert_ffn(inp, r.xn[t], e)
            ga = act[row]
            assert np.max(np.abs(ga - a)) <= 0.02 * np.max(np.abs(a)) + 1e-6, (t, rank)
            go = yr[row]
            wo = r.w[t, rank] * o
            assert np.max(np.abs(go - wo)) <= 0.02 * np.max(np.abs(wo)) + 1e-7, (t, rank)
    # rows of each expert are in token order (stable grouping)
    for e in range(8):
        toks = sorted(t for t in range(T) for k in range(2) if r.idx[t, k] == e)
        rows = [int(ros[t, k]) for t in toks for k in range(2) if r.idx[t, k] == e]
        assert rows == list(range(off[e], off[e] + counts[e]))


@pytest.mark.parametrize("T,d,F,seed", [
    (1, 256, 512, 61),
    (5, 384, 640, 62),     # ragged: d/128 = 3 row blocks, F/64 = 10 -> 2-way split
    (8, 512, 1024, 63),
    (16, 256, 512, 64),    # the largest T the decode path takes
])
@pytest.mark.parametrize("flags", [0, moe.MOE_FLAG_FORCE_TC])
def test_decode_path_and_forced_tensor_core_path(T, d, F, seed, flags):
    """T <= 16 runs the weight-streaming decode kernels unless the tensor-core
    grouped GEMM path is forced; both must match the oracle."""
    _full_check(synth.make_inputs(T, d, F, seed, name=f"dec{T}x{d}x{F}"), flags=flags)


def test_force_gemv_flag():
    inp = synth.make_inputs(40, 256, 512, 65, name="force_gemv")
    layer = make_layer(inp, flags=moe.MOE_FLAG_FORCE_GEMV)
    x = bf16_tensor(inp.x)
    with pytest.raises(moe.MoeError) as ei:
        layer.forward(x)  # 40 tokens: beyond the decode path's 16
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    sub = synth.make_inputs(12, 256, 512, 65, name="force_gemv12")
    y, idx, prob, counts = run(layer, sub, x_dev=x[:12].contiguous())
    ref = oracle.moe_tokens(sub)
    assert_routing(idx, prob, counts, ref, "force_gemv")
    assert_values(y, ref.y, "force_gemv")


def test_decode_and_tensor_core_paths_agree_on_one_expert_heavy_batch():
    """All 16 tokens to expert 3 (16 slots, the decode path's limit)."""
    inp = synth.make_inputs(16, 256, 512, 66, name="dec_onehot")
    b = np.zeros(8, np.float32)
    b[3] = 1e4
    inp.bias = b
    outs = []
    for flags in (0, moe.MOE_FLAG_FORCE_TC):
        layer = make_layer(inp, flags=flags)
        y, idx, prob, counts = run(layer, inp)
        assert counts[3] == 16
        outs.append(y)
        layer.close()
    ref = oracle.moe_tokens(inp)
    for y in outs:
        assert_values(y, ref.y, "dec_onehot")


# ------------------------------------------------------------- int8 weights
# int8 expert weights with bf16 scales, one per expert and output channel (the
# (8, 1, N) scale shape; "TevunahAi/Grok-1-BF16", "Conversion Details").  The
# kernels convert int8 -> bf16 in shared memory and apply the scale in the epilogue.

@pytest.mark.parametrize("T,d,F,seed", [
    (300, 512, 1024, 71),    # several up and down tiles, ragged row blocks
    (200, 384, 640, 72),     # ragged d (half a down tile) and F/128 = 5
])
def test_int8_weights(T, d, F, seed):
    inp = synth.make_inputs(T, d, F, seed, name=f"int8_{T}x{d}x{F}", weight_dtype="int8")
    _full_check(inp)


def test_int8_paired_mblocks_skewed():
    """F >= 16384 and T >= 2048: two m-blocks per tile.  The skewed router gives
    experts of 9.5, 4.5, 1.5 and 0.5 m-blocks: full pairs, a full block with a
    half one in one down tile (alone in the up projection), lone half blocks;
    ragged d (1.5 down n-blocks)."""
    inp = synth.make_inputs(2400, 384, 16384, 80, name="int8_pair_skew", weight_dtype="int8",
                            bias=synth.SKEW_BIAS)
    _full_check(inp, flags=moe.MOE_FLAG_DEVICE_CHECKS)


@pytest.mark.parametrize("T,d,F,seed", [
    (1, 256, 512, 76),
    (5, 384, 640, 77),      # ragged: d/128 = 3 weight blocks, F/64 = 10 -> 2-way split
    (9, 512, 1024, 73),
    (16, 256, 512, 78),     # the largest T the decode path takes
])
@pytest.mark.parametrize("flags", [0, moe.MOE_FLAG_FORCE_TC, moe.MOE_FLAG_DECODE_TC])
def test_int8_decode_path_and_forced_tensor_core_path(T, d, F, seed, flags):
    """int8 weights at T <= 16 run the int8 weight-streaming kernels unless the
    grouped GEMMs are forced: the CUDA-core GEMV kernels (integer dot products),
    or with MOE_FLAG_DECODE_TC the tensor-core kernels (weights converted into
    Tensor Memory).  T = 9 and 16 can put more than 8 slots on one expert (two
    slot groups in the GEMV)."""
    inp = synth.make_inputs(T, d, F, seed, name=f"int8dec{T}x{d}x{F}", weight_dtype="int8")
    _full_check(inp, flags=flags)


def test_int8_decode_one_expert_heavy_batch():
    """All 16 tokens to expert 6, int8 weights (two full slot groups of 8 in the
    GEMV kernels): GEMV, tensor-core decode and grouped-GEMM paths."""
    inp = synth.make_inputs(16, 384, 640, 79, name="int8dec_onehot", weight_dtype="int8")
    b = np.zeros(8, np.float32)
    b[6] = 1e4
    inp.bias = b
    ref = oracle.moe_tokens(inp)
    for flags in (0, moe.MOE_FLAG_FORCE_TC, moe.MOE_FLAG_FORCE_GEMV, moe.MOE_FLAG_DECODE_TC):
        layer = make_layer(inp, flags=flags)
        y, idx, prob, counts = run(layer, inp)
        assert counts[6] == 16
        assert_values(y, ref.y, f"int8dec_onehot flags={flags}")
        layer.close()


def test_int8_gemv_eight_slots_on_one_expert():
    """T = 8 with every token's first choice on expert 6: eight slot rows on one
    expert, one full slot group of the CUDA-core GEMV kernels; both int8 decode
    kernels."""
    inp = synth.make_inputs(8, 384, 640, 85, name="int8gemv_onehot", weight_dtype="int8")
    b = np.zeros(8, np.float32)
    b[6] = 1e4
    inp.bias = b
    ref = oracle.moe_tokens(inp)
    for flags in (0, moe.MOE_FLAG_DECODE_TC):
        layer = make_layer(inp, flags=flags)
        y, idx, prob, counts = run(layer, inp)
        assert counts[6] == 8
        assert_values(y, ref.y, f"int8gemv_onehot flags={flags}")
        layer.close()


def test_int8_skewed_and_checks():
    inp = synth.make_inputs(256, 256, 512, 74, name="int8_skew", weight_dtype="int8", bias=synth.SKEW_BIAS)
    _full_check(inp, flags=moe.MOE_FLAG_DEVICE_CHECKS)


@pytest.mark.parametrize("T", [64, 8])  # grouped tensor-core GEMM path; T <= 16 decode path
def test_int8_fp16_saturation_is_reported(T):
    """int8 layers carry their GeGLU activations in fp16, which saturates at
    +-65504.  With scales ~1000x the synthetic workload's, the activations pass
    that bound (checked on the oracle first).  Device checks off: the forward
    reports nothing.  Device checks on: moe_layer_sync_status reports
    MOE_ERR_DEVICE_CHECK naming the saturation, and the read clears it."""
    inp = synth.make_inputs(T, 256, 512, 90 + T, name="int8_sat", weight_dtype="int8", int8_scale_range=(0.2, 0.4))
    r = oracle.route(inp, keep_xn=True)
    _, _, a, _ = oracle.expert_ffn(inp, r.xn[0], int(r.idx[0, 0]))
    assert np.max(np.abs(a)) > 65504.0
    x = bf16_tensor(inp.x)
    layer = make_layer(inp)
    layer.forward(x)
    torch.cuda.synchronize()
    layer.sync_status()
    layer.close()
    layer = make_layer(inp, flags=moe.MOE_FLAG_DEVICE_CHECKS)
    layer.forward(x)
    with pytest.raises(moe.MoeError) as ei:
        layer.sync_status()
    assert ei.value.status == moe.MOE_ERR_DEVICE_CHECK and "65504" in str(ei.value)
    layer.sync_status()  # cleared by the read
    layer.close()


def test_device_gelu_matches_the_oracle():
    """The GeGLU epilogues' GELU (evaluated as u / (1 + 2^(-2 z log2 e)), z the
    tanh argument, on the ex2 and reciprocal instructions) against the oracle's
    fp64 tanh form: a dense sweep of [-16, 16], both tails out to the fp32 range,
    and +-0.  Bound: relative 2e-6 + 3e-7 |t|, t = 2 z log2 e the exponent (its
    rounding error grows with |t|, and 2^t is flushed past |t| ~ 126); plus the
    oracle's own cancellation in 1 + tanh z for u << 0 (2.3e-16 |u|) and 1e-37
    where the device result is flushed to zero."""
    import torch
    xs = np.concatenate([np.linspace(-16.0, 16.0, 100001), -np.logspace(-30, 38, 400), np.logspace(-30, 38, 400),
                         [0.0, -0.0]]).astype(np.float32)
    y = moe.selftest_gelu(torch.from_numpy(xs).cuda()).cpu().numpy().astype(np.float64)
    u = xs.astype(np.float64)
    ref = np.array([oracle.gelu_tanh(float(v)) for v in u])
    t = np.abs(2.0 * 0.7978845608028654 / np.log(2.0) * (u + 0.044715 * u ** 3))
    bound = (2e-6 + 3e-7 * np.minimum(t, 128.0)) * np.abs(ref) + 2.3e-16 * np.abs(u) + 1e-37
    err = np.abs(y - ref)
    worst = int(np.argmax(err / bound))
    assert np.all(err <= bound), f"u={u[worst]!r}: device {y[worst]!r} oracle {ref[worst]!r}"
    assert np.all(np.isfinite(y))
    assert y[-2] == 0.0 and y[-1] == 0.0
    # the ends: GELU(u) = u for u >> 0, -0 for u << 0
    assert y[np.argmax(u)] == u.max() and y[np.argmin(u)] == 0.0


def test_int8_intermediates_match_oracle():
    """GeGLU activations and scaled expert outputs of int8 experts."""
    inp = synth.make_inputs(64, 256, 512, 75, name="int8_inter", weight_dtype="int8")
    layer = make_layer(inp)
    run(layer, inp)
    ws = layer.workspace()
    act = read_device(ws.act, (ws.rows_cap, inp.F), torch.float16)  # int8 layers carry fp16 rows
    yr = read_device(ws.y_rows, (ws.rows_cap, inp.d), torch.float32)
    ros = read_device(ws.row_of_slot, (inp.T, 2), torch.int32)
    r = oracle.route(inp, keep_xn=True)
    for t in (0, 31, inp.T - 1):
        for rank in range(2):
            e = int(r.idx[t, rank])
            row = int(ros[t, rank])
            h, v, a, o = oracle.expert_ffn(inp, r.xn[t], e)
            assert np.max(np.abs(act[row] - a)) <= 0.02 * np.max(np.abs(a)) + 1e-6, (t, rank)
            wo = r.w[t, rank] * o
            assert np.max(np.abs(yr[row] - wo)) <= 0.02 * np.max(np.abs(wo)) + 1e-7, (t, rank)
    layer.close()


@pytest.mark.parametrize("T,weights,flags", [
    (8, "bf16", 0),                           # weight-streaming decode kernels
    (8, "int8", 0),                           # int8 weight-streaming decode kernels
    (200, "bf16", 0),                         # grouped GEMMs on CTA pairs
    (200, "int8", 0),                         # int8 grouped GEMMs
    (8, "int8", moe.MOE_FLAG_FORCE_TC),
    (8, "int8", moe.MOE_FLAG_DECODE_TC),
])
def test_back_to_back_forwards_are_deterministic(T, weights, flags):
    """Forty forwards queued back to back on one stream: no device wait may run
    out, and every output must equal the first bit for bit (every reduction in
    the layer has a fixed order).  Races between pipeline roles or between
    consecutive launches show up here as timeouts or changed bits."""
    inp = synth.make_inputs(T, 384, 1280, 80, name=f"repeat{T}{weights}", weight_dtype=weights)
    layer = make_layer(inp, flags=flags)
    x = bf16_tensor(inp.x)
    outs = [torch.empty_like(x) for _ in range(40)]
    for o in outs:
        layer.forward(x, out=o)
    torch.cuda.synchronize()
    layer.sync_status()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert_values(outs[0].float().cpu().numpy().astype(np.float64), oracle.moe_tokens(inp).y, inp.name)
    layer.close()



# ----------------------------------------------------------- routing diagnostics

def _stats_case(name):
    if name == "uniform":
        inp = synth.make_inputs(64, 256, 512, 81, norm_scales="ones", name=name)
        inp.gate[:] = 0.0
    elif name == "onehot":
        inp = synth.make_inputs(40, 256, 512, 82, name=name)
        b = np.zeros(8, np.float32)
        b[4] = 1e4
        inp.bias = b
    elif name == "skew":
        inp = synth.make_inputs(1001, 256, 512, 83, bias=synth.SKEW_BIAS, name=name)
    elif name == "decode":
        inp = synth.make_inputs(7, 384, 640, 84, name=name)
    else:
        inp = synth.workload("tiny")
    return inp


@pytest.mark.parametrize("name", ["tiny", "skew", "uniform", "onehot", "decode"])
def test_router_stats_match_oracle(name):
    """moe_layer_router_stats after a forward: mean probability per expert,
    routing entropy and collapse index against the oracle's (fp32 sums of T
    probabilities: 2e-6 absolute)."""
    inp = _stats_case(name)
    layer = make_layer(inp)
    run(layer, inp)
    s = layer.router_stats().cpu().numpy().astype(np.float64)
    torch.cuda.synchronize()
    ref = oracle.routing_stats(oracle.route(inp).p)
    np.testing.assert_allclose(s[:8], ref["mean_prob"], atol=2e-6)
    assert abs(s[8] - ref["entropy"]) < 2e-5 and abs(s[9] - ref["collapse"]) < 2e-5
    if name == "uniform":
        assert round(float(s[8]), 3) == 2.079 and np.all(np.round(s[:8], 3) == 0.125)
    layer.close()


def test_router_stats_needs_a_forward():
    inp = synth.workload("tiny")
    layer = make_layer(inp)
    with pytest.raises(moe.MoeError) as ei:
        layer.router_stats()
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    layer.close()



# ------------------------------------------------------- int8 scale shapes
# The model card lists scale shapes (8,1,N), (8,8,N), (1,N) and (8,N) ("Conversion
# Details"); read as (E_s, G, N) = (8,1), (8,8), (1,1), (1,8).  G > 1 scales vary
# along the reduction and are applied to the weights as they are converted (one
# bf16 or fp16 rounding); G == 1 scales multiply the fp32 result.

@pytest.mark.parametrize("shape", [(8, 8), (1, 1), (1, 8), (8, 2)])
@pytest.mark.parametrize("T,flags", [(200, 0), (8, 0), (8, moe.MOE_FLAG_FORCE_TC), (8, moe.MOE_FLAG_DECODE_TC)])
def test_int8_scale_shapes(shape, T, flags):
    inp = synth.make_inputs(T, 1024, 1024, 90 + shape[0] + shape[1], name=f"int8_scales_{shape}",
                            weight_dtype="int8", int8_scale_shape=shape)
    _full_check(inp, flags=flags)


def test_forward_captured_in_a_cuda_graph():
    """moe_layer_forward reads nothing back to the host, so it can be captured in
    a CUDA graph: replaying the graph on new inputs must give what direct calls give."""
    inp = synth.make_inputs(64, 256, 512, 95, name="graph")
    layer = make_layer(inp)
    x = bf16_tensor(inp.x)
    x_static = x.clone()
    out_static = torch.empty_like(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x_static, out=out_static, stream=s)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(x_static, out=out_static, stream=s)
    x2 = torch.roll(x, shifts=5, dims=0).contiguous()
    for xin in (x, x2):
        x_static.copy_(xin)
        g.replay()
        torch.cuda.synchronize()
        layer.sync_status()
        direct = layer.forward(xin)
        torch.cuda.synchronize()
        assert torch.equal(out_static, direct)
    layer.close()


@pytest.mark.parametrize("shape", [(8, 8), (8, 1)])
def test_int8_gemv_two_slot_groups(shape):
    """T = 13 with every first choice on expert 3: 13 slots on one expert, two
    slot groups (8 + 5) in the int8 GEMV kernels, with per-channel and grouped
    scales; both int8 decode kernels against the oracle."""
    inp = synth.make_inputs(13, 1024, 1024, 97 + shape[1], name=f"int8gemv_groups_{shape}", weight_dtype="int8",
                            int8_scale_shape=shape)
    b = np.zeros(8, np.float32)
    b[3] = 1e4
    inp.bias = b
    ref = oracle.moe_tokens(inp)
    for flags in (0, moe.MOE_FLAG_DECODE_TC):
        layer = make_layer(inp, flags=flags)
        y, idx, prob, counts = run(layer, inp)
        assert counts[3] == 13
        assert_values(y, ref.y, f"int8gemv_groups {shape} flags={flags}")
        layer.close()
