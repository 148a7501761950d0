"""The allocation-free grouping entry point (moe_group_slots_noalloc).

It exists for callers that cannot call cudaMalloc (a serving runtime that
reserved all free device memory for its own pool, or a plugin host that hands an
op only its input and output buffers).  Its scratch is a static device array
shared by every call, so this checks two calls in a row, with different inputs,
each against the grouping the layer's own forward computed (moe_layer_forward,
read back through the workspace view).  Integer outputs must match exactly.
The groupings are also checked against the rule written out in numpy (stable
slot order, blocks padded to 128 rows).  Collected last so a
stop-at-first-failure run has already run everything else.
"""
import numpy as np
import pytest
import torch

import synth
import mixture_experts_transformer_gemv_b300 as moe

from layer_helpers import bf16_tensor, make_layer, read_device

pytestmark = pytest.mark.gpu


def _forward_grouping(layer, inp):
    x = bf16_tensor(inp.x)
    _, idx, prob, counts = layer.forward(x, routing=True)
    torch.cuda.synchronize()
    layer.sync_status()
    ros = read_device(layer.workspace().row_of_slot, (inp.T, 2), torch.int32)
    return idx, prob, counts.cpu().numpy(), ros


def _numpy_grouping(idx):
    """The grouping rule written out: slots s = 2t + r in order, each expert's
    block padded to a multiple of 128 rows, experts in index order."""
    idx = idx.reshape(-1)
    counts = np.bincount(idx, minlength=8)
    off = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    ros = np.empty_like(idx)
    nxt = off[:8].copy()
    for s, e in enumerate(idx):
        ros[s] = nxt[e]
        nxt[e] += 1
    return counts, ros.reshape(-1, 2), off


def _check_noalloc(layer, inp):
    idx, prob, counts_ref, ros_ref = _forward_grouping(layer, inp)
    counts = torch.full((8,), -1, dtype=torch.int32, device="cuda")
    ros = torch.full((inp.T, 2), -1, dtype=torch.int32, device="cuda")
    moe.group_slots_noalloc(idx, prob, counts, ros)
    torch.cuda.synchronize()
    counts_np, ros_np = counts.cpu().numpy(), ros.cpu().numpy()
    np.testing.assert_array_equal(counts_np, counts_ref)
    np.testing.assert_array_equal(ros_np, ros_ref)
    c2, r2, off = _numpy_grouping(idx.cpu().numpy())
    np.testing.assert_array_equal(counts_np, c2)
    np.testing.assert_array_equal(ros_np, r2)
    # every expert's block starts at a multiple of 128 rows
    assert np.all(off % 128 == 0)
    return counts_np


def test_noalloc_grouping_matches_layer_forward_twice():
    from mixture_experts_transformer_gemv_b300 import build
    build.build()
    a = synth.make_inputs(300, 256, 512, 51, name="noalloc_a")
    b = synth.make_inputs(1000, 256, 512, 52, bias=synth.SKEW_BIAS, name="noalloc_b")
    layer_a = make_layer(a)
    layer_b = make_layer(b)
    for inp, layer in ((a, layer_a), (b, layer_b)):
        _check_noalloc(layer, inp)
    layer_a.close()
    layer_b.close()


def test_noalloc_at_its_token_limit_with_skewed_routing():
    """T = 16384, the largest the static array takes, with the skewed router
    (most slots on expert 0): the padded row count comes closest to the
    array's capacity here."""
    inp = synth.make_inputs(16384, 256, 512, 53, bias=synth.SKEW_BIAS, name="noalloc_limit")
    layer = make_layer(inp)
    counts = _check_noalloc(layer, inp)
    assert counts.sum() == 2 * 16384 and counts[0] > counts[1:].max()
    layer.close()


def test_noalloc_rejects_sizes_beyond_its_limit():
    T = 16385
    idx = torch.zeros((T, 2), dtype=torch.int32, device="cuda")
    prob = torch.zeros((T, 2), dtype=torch.float32, device="cuda")
    counts = torch.zeros((8,), dtype=torch.int32, device="cuda")
    ros = torch.zeros((T, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.group_slots_noalloc(idx, prob, counts, ros)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    assert "16384" in str(ei.value)
