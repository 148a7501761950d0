"""Helpers shared by the GPU tests: move seeded inputs to the device, run the
layer through the C ABI, and compare with the oracle under the stated rules.

Value tolerance (per element, rms over the token's row of the oracle output):
    |y - y_ref| <= 0.02 * |y_ref| + 0.02 * rms(y_ref)
Routing: the expert pair must match exactly, except tokens whose 2nd and 3rd
oracle probabilities differ by < 1e-6 (excluded and counted); the rank order is
compared only where the 1st and 2nd differ by >= 1e-6.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import mixture_experts_transformer_gemv_b300 as moe

REL_TOL = 0.02
RMS_TOL = 0.02
TIE_BAND = 1e-6


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device else t


def device_weights(inp) -> dict:
    w = {
        "gate": torch.from_numpy(inp.gate).cuda(),
        "gate_bias": None if inp.bias is None else torch.from_numpy(inp.bias).cuda(),
        "pre_norm_scale": torch.from_numpy(inp.s_pre).cuda(),
        "post_norm_scale": torch.from_numpy(inp.s_post).cuda(),
    }
    if inp.weight_dtype == "bf16":
        for k in ("w", "wv", "w1"):
            w[k] = bf16_tensor(getattr(inp, k))
    else:
        for k in ("w", "wv", "w1"):
            w[k] = torch.from_numpy(getattr(inp, k)).cuda()
        w["w_scale"] = bf16_tensor(inp.w_scale)
        w["wv_scale"] = bf16_tensor(inp.wv_scale)
        w["w1_scale"] = bf16_tensor(inp.w1_scale)
    return w


def make_layer(inp, max_tokens=None, flags=0, weights=None):
    weights = device_weights(inp) if weights is None else weights
    return moe.MoeLayer(inp.d, inp.F, max_tokens or inp.T, weights, eps=inp.eps, weight_dtype=inp.weight_dtype,
                        flags=flags, scale_shape=(inp.scale_experts, inp.scale_groups))


def run(layer, inp, x_dev=None):
    x = bf16_tensor(inp.x) if x_dev is None else x_dev
    out, idx, prob, counts = layer.forward(x, routing=True)
    torch.cuda.synchronize()
    layer.sync_status()
    return (out.float().cpu().numpy().astype(np.float64), idx.cpu().numpy(), prob.cpu().numpy(),
            counts.cpu().numpy())


def value_report(y, y_ref):
    rms = np.sqrt(np.mean(y_ref * y_ref, axis=1, keepdims=True))
    bound = REL_TOL * np.abs(y_ref) + RMS_TOL * rms
    err = np.abs(y - y_ref)
    return {"max_ratio": float(np.max(err / bound)), "violations": int(np.sum(err > bound)),
            "max_abs": float(np.max(err)), "rms_err": float(np.sqrt(np.mean(err * err)))}


def assert_values(y, y_ref, what=""):
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    r = value_report(y, y_ref)
    assert r["violations"] == 0, f"{what}: {r}"
    return r


def routing_report(idx, prob, ref_p, ref_idx, ref_w):
    """Compare GPU routing with the oracle's.  Returns counts of excluded tokens."""
    excl = oracle.near_tie_tokens(ref_p, TIE_BAND)
    order_tie = oracle.near_order_tie_tokens(ref_p, TIE_BAND)
    keep = ~excl
    same_set = np.sort(idx, axis=1) == np.sort(ref_idx, axis=1)
    set_mismatch = int(np.sum(~np.all(same_set, axis=1) & keep))
    ordered = keep & ~order_tie
    order_mismatch = int(np.sum(~np.all(idx == ref_idx, axis=1) & ordered))
    ok_rows = keep & np.all(same_set, axis=1)
    # probabilities of the chosen experts (fp32 kernel vs fp64 oracle)
    pg = np.sort(prob[ok_rows], axis=1)
    pr = np.sort(ref_w[ok_rows], axis=1)
    prob_err = float(np.max(np.abs(pg - pr))) if pg.size else 0.0
    return {"excluded": int(excl.sum()), "set_mismatch": set_mismatch, "order_mismatch": order_mismatch,
            "prob_max_abs_err": prob_err}


def assert_routing(idx, prob, counts, ref, what=""):
    r = routing_report(idx, prob, ref.p, ref.idx, ref.w)
    assert r["set_mismatch"] == 0 and r["order_mismatch"] == 0, f"{what}: {r}"
    assert r["prob_max_abs_err"] < 1e-5, f"{what}: {r}"
    ref_counts = np.bincount(ref.idx.ravel(), minlength=8)
    if r["excluded"] == 0:
        np.testing.assert_array_equal(counts, ref_counts)
    else:
        assert np.all(np.abs(counts - ref_counts) <= r["excluded"]), (counts, ref_counts)
    assert counts.sum() == idx.shape[0] * 2
    return r


def stratified_tokens(ref_idx, T, per_expert=3, seed=0, extra=(0,)):
    """A few tokens per expert (first choice), plus the first and last token."""
    rng = np.random.default_rng(seed)
    pick = set(int(t) for t in extra if 0 <= t < T)
    pick.add(T - 1)
    for e in range(8):
        cand = np.nonzero(ref_idx[:, 0] == e)[0]
        if cand.size == 0:
            cand = np.nonzero(ref_idx[:, 1] == e)[0]
        if cand.size:
            pick.update(int(t) for t in rng.choice(cand, size=min(per_expert, cand.size), replace=False))
    return np.array(sorted(pick), dtype=np.int64)


_CUDART = None


def _cudart():
    """libcudart of the CUDA toolkit, for device-to-device copies of raw
    workspace pointers into torch tensors (test introspection only)."""
    global _CUDART
    if _CUDART is None:
        import ctypes
        import glob
        for cand in ("libcudart.so", *sorted(glob.glob("/usr/local/cuda/lib64/libcudart.so*"))):
            try:
                _CUDART = ctypes.CDLL(cand)
                break
            except OSError:
                continue
        _CUDART.cudaMemcpy.restype = ctypes.c_int
        _CUDART.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
    return _CUDART


def read_device(ptr, shape, dtype):
    """Copy a raw device buffer (e.g. a workspace pointer) to a numpy array:
    float64 for floating types, int32 as is."""
    n = int(np.prod(shape))
    buf = torch.empty(n, dtype=dtype, device="cuda")
    torch.cuda.synchronize()
    rc = _cudart().cudaMemcpy(buf.data_ptr(), ptr, n * buf.element_size(), 3)  # device to device
    assert rc == 0, f"cudaMemcpy failed ({rc})"
    torch.cuda.synchronize()
    if dtype == torch.int32:
        return buf.view(*shape).cpu().numpy()
    return buf.view(*shape).float().cpu().numpy().astype(np.float64)
