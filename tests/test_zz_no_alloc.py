"""The allocation-free grouping entry point (moe_group_slots_noalloc).

It exists for callers that cannot call cudaMalloc (a serving runtime that
reserved all free device memory for its own pool, or a plugin host that hands an
op only its input and output buffers).  Its scratch is a static device array
shared by every call, so this checks two calls in a row, with different inputs,
each against the grouping the layer's own forward computed (moe_layer_forward,
read back through the workspace view).  Integer outputs must match exactly.
Collected last so a stop-at-first-failure run has already run everything else.
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


def test_noalloc_grouping_matches_layer_forward_twice():
    from mixture_experts_transformer_gemv_b300 import build
    build.build()
    a = synth.make_inputs(300, 256, 512, 51, name="noalloc_a")
    b = synth.make_inputs(1000, 256, 512, 52, bias=synth.SKEW_BIAS, name="noalloc_b")
    layer_a = make_layer(a)
    layer_b = make_layer(b)
    for inp, layer in ((a, layer_a), (b, layer_b)):
        idx, prob, counts_ref, ros_ref = _forward_grouping(layer, inp)
        counts = torch.full((8,), -1, dtype=torch.int32, device="cuda")
        ros = torch.full((inp.T, 2), -1, dtype=torch.int32, device="cuda")
        moe.group_slots_noalloc(idx, prob, counts, ros)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(counts.cpu().numpy(), counts_ref)
        np.testing.assert_array_equal(ros.cpu().numpy(), ros_ref)
    layer_a.close()
    layer_b.close()


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
