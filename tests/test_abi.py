"""C-ABI library: loads, exports what include/moe_layer.h declares, validates
arguments on the host (no GPU needed: these paths return before any CUDA call)."""
import ctypes
import os

import pytest

import mixture_experts_transformer_gemv_b300 as moe
from mixture_experts_transformer_gemv_b300 import build as moe_build


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.lib()


def test_header_declares_the_boundary():
    names = moe.declared_functions()
    for n in ("moe_layer_create", "moe_layer_forward", "moe_layer_destroy", "moe_layer_forward_host",
              "moe_layer_sync_status", "moe_status_string", "moe_last_error_message"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = moe.declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe_layer.h but not exported"


def test_library_is_built_for_sm_103a():
    src = open(moe_build.__file__).read()
    assert "arch=compute_103a,code=sm_103a" in src
    assert os.path.exists(moe.LIB_PATH)


def test_header_flag_values_match_the_binding():
    import re
    text = open(moe.HEADER_PATH).read()
    found = {m.group(1): int(m.group(2), 16) for m in re.finditer(r"#define (MOE_FLAG_\w+) (0x[0-9a-f]+)u", text)}
    assert found == {k: getattr(moe, k) for k in found} and len(found) == 4


def test_status_strings(lib):
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(1) == b"MOE_ERR_INVALID_ARG"
    assert lib.moe_status_string(6) == b"MOE_ERR_TIMEOUT"
    assert lib.moe_status_string(99) == b"MOE_ERR_UNKNOWN"


def _cfg(**kw):
    c = dict(d_model=256, d_ffn=512, num_experts=8, top_k=2, max_tokens=64, eps=1e-5, weight_dtype=0, flags=0)
    c.update(kw)
    return moe.Config(**c)


def _fake_weights(align=0):
    w = moe.Weights()
    for i, (name, _) in enumerate(moe.Weights._fields_):
        if name in ("gate_bias", "w_scale", "wv_scale", "w1_scale"):
            continue
        setattr(w, name, 0x10000 * (i + 1) + align)
    return w


def _create(lib, cfg, w):
    h = ctypes.c_void_p()
    s = lib.moe_layer_create(ctypes.byref(cfg) if cfg is not None else None,
                             ctypes.byref(w) if w is not None else None, ctypes.byref(h))
    return s, h


@pytest.mark.parametrize("kw,status", [
    (dict(num_experts=4), moe.MOE_ERR_UNSUPPORTED),
    (dict(top_k=1), moe.MOE_ERR_UNSUPPORTED),
    (dict(d_model=200), moe.MOE_ERR_UNSUPPORTED),
    (dict(d_ffn=100), moe.MOE_ERR_UNSUPPORTED),
    (dict(d_model=0), moe.MOE_ERR_UNSUPPORTED),
    (dict(d_model=32768), moe.MOE_ERR_UNSUPPORTED),
    (dict(max_tokens=0), moe.MOE_ERR_INVALID_ARG),
    (dict(eps=0.0), moe.MOE_ERR_INVALID_ARG),
    (dict(weight_dtype=7), moe.MOE_ERR_INVALID_ARG),
    (dict(weight_dtype=1), moe.MOE_ERR_INVALID_ARG),  # int8 weights without their scales
    (dict(weight_dtype=1, flags=moe.MOE_FLAG_FORCE_GEMV), moe.MOE_ERR_INVALID_ARG),  # no scales
    (dict(flags=moe.MOE_FLAG_FORCE_GEMV | moe.MOE_FLAG_FORCE_TC), moe.MOE_ERR_INVALID_ARG),
    (dict(weight_dtype=1, scale_experts=3), moe.MOE_ERR_INVALID_ARG),
    (dict(weight_dtype=1, scale_groups=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(weight_dtype=1, scale_groups=4), moe.MOE_ERR_UNSUPPORTED),  # d = 256 is not a multiple of 128 x 4
])
def test_create_rejects_bad_config(lib, kw, status):
    s, h = _create(lib, _cfg(**kw), _fake_weights())
    assert s == status, lib.moe_last_error_message()
    assert not h.value
    assert lib.moe_last_error_message() != b""


def test_create_rejects_null_and_misaligned_pointers(lib):
    assert _create(lib, None, _fake_weights())[0] == moe.MOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(), None)[0] == moe.MOE_ERR_INVALID_ARG
    w = _fake_weights()
    w.w1 = None
    assert _create(lib, _cfg(), w)[0] == moe.MOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(), _fake_weights(align=8))[0] == moe.MOE_ERR_INVALID_ARG


def test_null_handle_calls(lib):
    assert lib.moe_layer_forward(None, None, None, 1, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_host(None, None, None, 1, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_sync_status(None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_destroy(None) == moe.MOE_OK
    assert lib.moe_layer_launch_count(None) == 0
    assert lib.moe_layer_set_profiling(None, 1) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_router_stats(None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_gemm_grid(None, None) == moe.MOE_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(moe, "_lib_handle", None)
    with pytest.raises(ImportError):
        moe.lib()


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.dirname(moe.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text and "moe_oracle" not in text


# ------------------------------------------------------------- attention block

def _attn_cfg(**kw):
    c = dict(d_model=6144, n_q_heads=48, n_kv_heads=8, head_dim=128, max_tokens=8192, eps=1e-5, rope_base=10000.0,
             logit_clamp=30.0)
    c.update(kw)
    return moe.AttnConfig(**c)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), 2),            # only heads of 128
    (dict(d_model=6000), 2),           # d a multiple of 256
    (dict(n_kv_heads=7), 1),           # Hkv must divide Hq
    (dict(max_tokens=0), 1),
    (dict(max_tokens=70000), 1),
    (dict(logit_clamp=50.0), 2),       # exp(-2c) must stay a normal float
    (dict(logit_clamp=0.0), 2),
    (dict(eps=0.0), 1),
])
def test_attn_create_rejects_bad_config(lib, kw, status):
    cfg = _attn_cfg(**kw)
    w = moe.AttnWeights(16, 16, 16, 16, 16, 16)  # never dereferenced: validation fails first
    h = ctypes.c_void_p(1)
    assert lib.attn_block_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == status
    assert h.value is None
    assert lib.moe_last_error_message()


def test_attn_null_arguments(lib):
    cfg = _attn_cfg()
    h = ctypes.c_void_p()
    assert lib.attn_block_create(None, None, ctypes.byref(h)) == 1
    w = moe.AttnWeights(0, 16, 16, 16, 16, 16)
    assert lib.attn_block_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == 1
    w = moe.AttnWeights(24, 16, 16, 16, 16, 16)  # misaligned
    assert lib.attn_block_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == 1
    assert lib.attn_block_forward(None, 16, 32, 4, None) == 1
    assert lib.attn_block_sync_status(None, None) == 1
    assert lib.attn_block_destroy(None) == 0
    assert lib.attn_block_launch_count(None) == 0


def test_selftest_rejects_bad_arguments(lib):
    el = ctypes.c_uint64(0)
    assert lib.moe_selftest_bounded_wait(3, 10_000_000, ctypes.byref(el)) == 1
    assert lib.moe_selftest_bounded_wait(0, 10, ctypes.byref(el)) == 1            # below 1 ms
    assert lib.moe_selftest_bounded_wait(1, 3_000_000_000, ctypes.byref(el)) == 1  # above 2 s


@pytest.mark.parametrize("what", ["idx_1d", "idx_3col", "prob_short", "ros_short", "counts_short"])
def test_noalloc_binding_rejects_misshaped_tensors(what):
    """group_slots_noalloc checks every shape before anything reaches the GPU:
    a [T, 2] array shorter than topk_idx, or fewer than 8 counts, would make the
    grouping kernel read or write past the caller's buffers.  CPU tensors are
    enough: the shape check comes before the device check."""
    import torch
    import mixture_experts_transformer_gemv_b300 as moe
    T = 10
    a = {"idx": torch.zeros((T, 2), dtype=torch.int32), "prob": torch.zeros((T, 2), dtype=torch.float32),
         "counts": torch.zeros((8,), dtype=torch.int32), "ros": torch.zeros((T, 2), dtype=torch.int32)}
    if what == "idx_1d":
        a["idx"] = torch.zeros((2 * T,), dtype=torch.int32)
    elif what == "idx_3col":
        a["idx"] = torch.zeros((T, 3), dtype=torch.int32)
    elif what == "prob_short":
        a["prob"] = torch.zeros((T - 1, 2), dtype=torch.float32)
    elif what == "ros_short":
        a["ros"] = torch.zeros((T, 1), dtype=torch.int32)
    else:
        a["counts"] = torch.zeros((7,), dtype=torch.int32)
    with pytest.raises(ValueError, match="must be"):
        moe.group_slots_noalloc(a["idx"], a["prob"], a["counts"], a["ros"])
