"""GPU parity of the attention block (pre-norm, GQA with RoPE and the +-30 logit
clamp, output projection, post-norm, residual) against the CPU oracle, through
the C ABI.

Tolerance, per element, as for the MoE layer:
    |y - y_ref| <= 0.02 |y_ref| + 0.02 rms(y_ref row)
The GPU path carries xn, Wq, Wk, Wv, q and k in fp16 (relative 2^-12 each:
the logits' error scales with |q||k|), the softmax weights, v and ctx in bf16
(2^-9) and sums in fp32; y itself is rounded to bf16 (2^-9 |y|).  A CPU
emulation of exactly these roundings puts the attention workloads at about half
the tolerance (rms error about 0.004 of the row rms); the tests also bound the
rms error.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import mixture_experts_transformer_gemv_b300 as moe
from layer_helpers import assert_values, bf16_tensor, value_report

pytestmark = pytest.mark.gpu


def device_attn_weights(inp):
    return {"wq": bf16_tensor(inp.wq), "wk": bf16_tensor(inp.wk), "wv": bf16_tensor(inp.wv),
            "wo": bf16_tensor(inp.wo), "s_pre": torch.from_numpy(inp.s_pre).cuda(),
            "s_post": torch.from_numpy(inp.s_post).cuda()}


def make_block(inp, max_tokens=None, weights=None):
    return moe.AttnBlock(inp.d, inp.Hq, inp.Hkv, max_tokens or inp.T,
                         device_attn_weights(inp) if weights is None else weights, eps=inp.eps,
                         rope_base=inp.rope_base, logit_clamp=inp.clamp)


def run(block, inp, x=None):
    x = bf16_tensor(inp.x) if x is None else x
    y = block.forward(x)
    torch.cuda.synchronize()
    block.sync_status()
    return y.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", ["attn_tiny", "attn_clamp"])
def test_small_workloads_all_tokens(name):
    inp = synth.attn_workload(name)
    blk = make_block(inp)
    y = run(blk, inp)
    _, y_ref, _ = oracle.attn_tokens(inp)
    r = assert_values(y, y_ref, name)
    assert r["rms_err"] < 0.01, r
    blk.close()


@pytest.mark.parametrize("T", [1, 2, 127, 128, 129, 255, 256, 257, 300, 520])
def test_lengths_span_tiles_and_ragged_tails(T):
    """Query tiles and key blocks of 128, GEMM row tiles of 256: lengths on and
    around each boundary; one handle sized for the largest."""
    inp = synth.attn_workload("attn_tiny", T=T)
    blk = make_block(inp, max_tokens=520)
    y = run(blk, inp)
    _, y_ref, _ = oracle.attn_tokens(inp)
    assert_values(y, y_ref, f"T={T}")
    blk.close()


def test_more_heads_and_groups():
    """12 query heads on 4 key/value heads (groups of 3) at d = 512."""
    inp = synth.make_attn_inputs(333, 512, 12, 4, 2100, name="attn_gqa3")
    blk = make_block(inp)
    y = run(blk, inp)
    _, y_ref, _ = oracle.attn_tokens(inp)
    assert_values(y, y_ref, "gqa3")
    blk.close()


def test_prefix_rows_match_and_repeat_bitwise():
    """Outputs of a prefix do not depend on later tokens (causality) and the same
    call twice gives the same bits."""
    inp = synth.attn_workload("attn_tiny", T=400)
    blk = make_block(inp, max_tokens=400)
    x = bf16_tensor(inp.x)
    y1 = blk.forward(x).clone()
    y2 = blk.forward(x).clone()
    y_pre = blk.forward(x[:150].contiguous()).clone()
    torch.cuda.synchronize()
    blk.sync_status()
    assert torch.equal(y1, y2)
    assert torch.equal(y1[:150], y_pre)
    blk.close()


def test_full_shape_mid_length_sampled():
    """48 / 8 heads at d = 6144, T = 1000: sampled tokens against the oracle."""
    inp = synth.attn_workload("attn_prefill", T=1000)
    blk = make_block(inp)
    y = run(blk, inp)
    tok = [0, 1, 2, 127, 128, 129, 511, 640, 998, 999]
    _, y_ref, _ = oracle.attn_tokens(inp, tok)
    assert_values(y[tok], y_ref, "T=1000 sampled")
    blk.close()


def test_full_prefill_workload_sampled():
    """The full workload (T = 8192, 48 / 8 heads, d = 6144) in the configuration
    the benchmark times: sampled tokens across the sequence, including the last
    query tile (the longest causal rows)."""
    inp = synth.attn_workload("attn_prefill")
    blk = make_block(inp)
    y = run(blk, inp)
    rng = np.random.default_rng(5)
    tok = sorted(set([0, 1, 127, 128, 4095, 4096, 8064, 8190, 8191] + list(rng.integers(0, 8192, 7))))
    _, y_ref, _ = oracle.attn_tokens(inp, tok)
    r = assert_values(y[tok], y_ref, "T=8192 sampled")
    assert r["rms_err"] < 0.01, r
    assert np.all(np.isfinite(y))
    blk.close()


def test_graph_capture():
    """The forward enqueues kernels only (no host sync): it captures into a CUDA graph."""
    inp = synth.attn_workload("attn_tiny")
    blk = make_block(inp)
    x = bf16_tensor(inp.x)
    out = torch.empty_like(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        blk.forward(x, out=out, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        blk.forward(x, out=out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    blk.sync_status()
    _, y_ref, _ = oracle.attn_tokens(inp)
    assert_values(out.float().cpu().numpy().astype(np.float64), y_ref, "graph replay")
    blk.close()


@pytest.mark.parametrize("base,clamp", [(1_000_000.0, 20.0), (500.0, 40.0)])
def test_other_rope_base_and_clamp(base, clamp):
    """The rotation table and the clamp follow the configuration: another base and
    clamp bound (40 is the largest the fixed-offset softmax accepts) against the
    oracle with the same settings, on the workload whose logits reach the clamp."""
    inp = synth.make_attn_inputs(260, 768, 6, 1, 2010, name="attn_cfg", qk_gain=5.0, rope_base=base, clamp=clamp)
    blk = make_block(inp)
    y = run(blk, inp)
    _, y_ref, _ = oracle.attn_tokens(inp)
    assert_values(y, y_ref, f"base={base} clamp={clamp}")
    blk.close()
