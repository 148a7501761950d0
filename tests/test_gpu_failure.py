"""Failure detection on the GPU without a fault: a kernel waits on an mbarrier
phase that nothing completes, with a short limit; the wait must give up, latch
the device error word (MOE_ERR_TIMEOUT to the host) and leave the context
usable for the next forward."""
import numpy as np
import pytest
import torch

import oracle
import synth
import mixture_experts_transformer_gemv_b300 as moe
from layer_helpers import assert_values, make_layer, run

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [0, 1])  # the spinning wait, the sleeping wait
def test_wait_on_a_phase_nobody_completes_gives_up(mode):
    st, waited = moe.selftest_bounded_wait(mode, 0.02)
    assert st == moe.MOE_ERR_TIMEOUT, moe.lib().moe_last_error_message()
    assert 0.02 <= waited < 0.5


def test_raised_abort_flag_ends_the_wait_at_once():
    st, waited = moe.selftest_bounded_wait(2, 2.0)
    assert st == moe.MOE_ERR_TIMEOUT
    assert waited < 0.05


def test_context_usable_after_the_timeouts():
    for mode in (0, 1, 2):
        assert moe.selftest_bounded_wait(mode, 0.005)[0] == moe.MOE_ERR_TIMEOUT
    inp = synth.workload("tiny")
    layer = make_layer(inp)
    y, idx, _, _ = run(layer, inp)
    ref = oracle.moe_tokens(inp)
    assert np.array_equal(idx, ref.idx)
    assert_values(y, ref.y, "forward after the timeouts")
    layer.close()
