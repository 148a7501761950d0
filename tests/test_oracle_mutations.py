"""The pins must fail when a plausible mistake is planted in the oracle.

Each case copies moe_oracle.c, applies one textual mutation, compiles it into a
temporary library and runs the pin suite against it in a subprocess; the suite
must fail.  Mistakes are planted only in the oracle, on the CPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTANTS = {
    "h_uses_Wv": ("hn += weight_at(W, e, n, k)", "hn += weight_at(Wv, e, n, k)"),
    "gelu_on_linear_branch": ("a[n] = oracle_gelu_tanh(hn) * vn", "a[n] = oracle_gelu_tanh(vn) * hn"),
    "down_proj_wrong_operand": ("oj += weight_at(W1, e, j, n) * a[n]", "oj += weight_at(W, e, n, j) * a[n]"),
    "combine_weight_dropped": ("m[j] += wts[2 * i + r] * o[j]", "m[j] += o[j]"),
    "combine_renormalised": ("w2[1] = p[i1];", "w2[1] = p[i1]; { double s_ = w2[0] + w2[1]; w2[0] /= s_; w2[1] /= s_; }"),
    "residual_dropped": ("(double)bf16_bits_to_float(x_row[j]) + m[j] * rr", "m[j] * rr"),
    "softmax_sign": ("p[e] = exp(l[e] - mx)", "p[e] = exp(mx - l[e])"),
    "tie_to_higher_index": ("if ((float)p[e] > (float)p[i0]) i0", "if ((float)p[e] >= (float)p[i0]) i0"),
    "pre_norm_scale_dropped": ("* r * (double)s_pre[j]", "* r"),
    "post_norm_eps_dropped": ("\n    double rr = 1.0 / sqrt(ss / (double)d + eps)", "\n    double rr = 1.0 / sqrt(ss / (double)d)"),
    "gelu_constant": ("0.044715 * u * u * u", "0.0447 * u * u * u"),
    "int8_scale_not_per_expert": ("int64_t es = (W->scale_E > 1) ? e : 0;", "int64_t es = 0;"),
    "bias_sign": ("l[e] = acc + (bias ? (double)bias[e] : 0.0)", "l[e] = acc - (bias ? (double)bias[e] : 0.0)"),
    "entropy_in_bits": ("if (out[e] > 0.0) h -= out[e] * log(out[e]);", "if (out[e] > 0.0) h -= out[e] * log2(out[e]);"),
    "stats_sum_not_mean": ("out[e] = s / (double)T;", "out[e] = s;"),
}

# planted in the attention block; checked by its own pin file
ATTN_MUTANTS = {
    "rope_sign": ("v[2 * i] = x0 * c - x1 * s;", "v[2 * i] = x0 * c + x1 * s;"),
    "rope_frequency": ("pow(base, -2.0 * (double)i / (double)Dh)", "pow(base, -1.0 * (double)i / (double)Dh)"),
    "rope_half_split_pairs": ("const double x0 = v[2 * i], x1 = v[2 * i + 1];",
                              "const double x0 = v[i], x1 = v[i + Dh / 2];"),
    "keys_not_rotated": ("for (int64_t g = 0; g < Hkv; ++g) oracle_rope(", "for (int64_t g = 0; g < 0; ++g) oracle_rope("),
    "logit_scale_dropped": ("s /= sqrt((double)Dh);", ""),
    "clamp_dropped": ("if (s > clamp_c) s = clamp_c;", ""),
    "gqa_heads_interleaved": ("const int64_t g = h / group;", "const int64_t g = h % Hkv;"),
    "values_from_key_weights": ("matvec_bf16(kvw, d, wv, xn, V + t * kvw);", "matvec_bf16(kvw, d, wk, xn, V + t * kvw);"),
    "attn_residual_dropped": ("(double)bf16_bits_to_float(x[t * d + n]) + o[n] * rr", "o[n] * rr"),
    "attn_post_norm_scale_dropped": ("o[n] * rr * (double)s_post[n]", "o[n] * rr"),
    "attn_softmax_unnormalised": ("ctx[h * Dh + c] = acc / z;", "ctx[h * Dh + c] = acc;"),
}

PIN_FILE = {name: "test_oracle_pins.py" for name in MUTANTS}
PIN_FILE.update({name: "test_oracle_attn_pins.py" for name in ATTN_MUTANTS})
MUTANTS.update(ATTN_MUTANTS)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", str(lib), str(mut), "-lm"])
    env = dict(os.environ, MOE_ORACLE_LIB_OVERRIDE=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", PIN_FILE[name])],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
