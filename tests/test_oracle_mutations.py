"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a scratch copy of ``oracle/moe_oracle.c``
(never in the real file), rebuilds it there and runs the pin suite
(tests/test_oracle_pins.py) against the copy: the suite must fail.  The
mistakes are the slips a reader checking the oracle against the pages would
worry about: a transposed operand, a dropped scale, a wrong rounding rule, a
wrong tie-break, a wrong bucket order, a wrong reduction order.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("router_transposed", "acc += (double)xt[d] * (double)we[d];",
     "acc += (double)xt[d] * (double)W[((int64_t)d * E + e) % ((int64_t)E * D)];"),
    ("topk_ties_to_higher", "if (!taken[e] && (best < 0 || l[e] > l[best]))",
     "if (!taken[e] && (best < 0 || l[e] >= l[best]))"),
    ("norm_ignored", "w[t * k + s] = (float)(norm ? ps / psel : ps);", "w[t * k + s] = (float)(ps);"),
    ("norm_always", "w[t * k + s] = (float)(norm ? ps / psel : ps);", "w[t * k + s] = (float)(ps / psel);"),
    ("softmax_unshifted", "p[e] = exp((double)l[e] - m);", "p[e] = exp((double)l[e]);"),
    ("round_half_even", "int qi = (int)roundf(v);", "int qi = (int)rintf(v);"),
    ("quant_from_fp16_scale", "float id = (d != 0.0f) ? 1.0f / d : 0.0f;",
     "float id = (d != 0.0f) ? 1.0f / oracle_half_to_float(oracle_float_to_half(d)) : 0.0f;"),
    ("scale_perturbed", "d16[b] = oracle_float_to_half(d);", "d16[b] = oracle_float_to_half(d * 1.0001f);"),
    ("half_round_half_up", "float r = rintf(ldexpf(a, 10 - E));", "float r = floorf(ldexpf(a, 10 - E) + 0.5f);"),
    ("bucket_slot_major",
     "    for (int64_t t = 0; t < N; ++t)\n        for (int s = 0; s < k; ++s) {\n            int e = idx[t * k + s];\n            int64_t j = fill[e]++;",
     "    for (int s = 0; s < k; ++s)\n        for (int64_t t = 0; t < N; ++t) {\n            int e = idx[t * k + s];\n            int64_t j = fill[e]++;"),
    ("block_dot_short", "for (int i = 0; i < QK; ++i)\n        s += (int32_t)a[i] * (int32_t)b[i];",
     "for (int i = 0; i < QK - 1; ++i)\n        s += (int32_t)a[i] * (int32_t)b[i];"),
    ("dropped_activation_scale", "(double)oracle_half_to_float(ad16[b]) * (double)isum;", "(double)isum;"),
    ("gate_up_swapped", "h[r] = (float)((g / (1.0 + exp(-g))) * u);", "h[r] = (float)((u / (1.0 + exp(-u))) * g);"),
    ("silu_sign", "h[r] = (float)((g / (1.0 + exp(-g))) * u);", "h[r] = (float)((g / (1.0 + exp(g))) * u);"),
    ("partial_row_slot_major", "float *dst = partials + (t * k + s) * (int64_t)D;",
     "float *dst = partials + ((int64_t)s * (expStart[E] / k) + t) * (int64_t)D;"),
    ("shared_unscaled", "S[t * D + c] = (float)((double)s[t] * y[c]);", "S[t * D + c] = (float)(y[c]);"),
    ("sigmoid_sign", "s[t] = (float)(1.0 / (1.0 + exp(-(double)g[t])));",
     "s[t] = (float)(1.0 / (1.0 + exp((double)g[t])));"),
    ("combine_mul_add", "acc = fmaf(w[t * k + s], partials[(t * k + s) * (int64_t)D + c], acc);",
     "acc = acc + w[t * k + s] * partials[(t * k + s) * (int64_t)D + c];"),
    ("combine_reverse_order", "for (int s = 0; s < k; ++s)\n                acc = fmaf(w[t * k + s], partials[(t * k + s) * (int64_t)D + c], acc);",
     "for (int s = k - 1; s >= 0; --s)\n                acc = fmaf(w[t * k + s], partials[(t * k + s) * (int64_t)D + c], acc);"),
    ("q4k_min_sign", "(d * sc * (double)isum - dmin * m * (double)xsum)", "(d * sc * (double)isum + dmin * m * (double)xsum)"),
    ("q4k_min_uses_isum", "(d * sc * (double)isum - dmin * m * (double)xsum)", "(d * sc * (double)isum - dmin * m * (double)isum)"),
    ("q4k_nibble_order", "q[l] = (int8_t)((j & 1) ? (p[l] >> 4) : (p[l] & 15));",
     "q[l] = (int8_t)((j & 1) ? (p[l] & 15) : (p[l] >> 4));"),
    ("q4k_scale_high_bits", "*sc = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 4);", "*sc = (s12[j + 4] & 15);"),
    ("q3k_high_bit_sense", "return h ? l : l - 4;", "return h ? l - 4 : l;"),
    ("q3k_scale_offset", "return (lo | (hi << 4)) - 32;", "return (lo | (hi << 4)) - 31;"),
    ("q3k_low_bits_shift", "(2 * ((i % 128) / 32))) & 3;", "(2 * ((i % 64) / 16))) & 3;"),
    ("q3k_scale_high_bits_byte", "int hi = (s12[8 + j % 4] >> (2 * (j / 4))) & 3;",
     "int hi = (s12[8 + j / 4] >> (2 * (j % 4))) & 3;"),
    ("q3k_one_scale_per_block", "sisum += (int64_t)q3_k_scale(blk, j) * isum;",
     "sisum += (int64_t)q3_k_scale(blk, 2 * b) * isum;"),
    ("combine_residual_first",
     "            if (S)\n                acc = acc + S[t * D + c];\n            acc = acc + R[t * D + c];",
     "            acc = acc + R[t * D + c];\n            if (S)\n                acc = acc + S[t * D + c];"),
    ("combine_residual_dropped", "            acc = acc + R[t * D + c];\n", ""),
    ("combine_shared_first", "            float acc = 0.0f;\n            for (int s = 0; s < k; ++s)",
     "            float acc = S ? S[t * D + c] : 0.0f;\n            if (S) S = S + 0 * c;\n            for (int s = 0; s < k; ++s)"),
    ("rmsnorm_without_epsilon", "double r = 1.0 / sqrt(ss / (double)D + eps);", "double r = 1.0 / sqrt(ss / (double)D);"),
    ("rmsnorm_sum_not_mean", "double r = 1.0 / sqrt(ss / (double)D + eps);", "double r = 1.0 / sqrt(ss + eps);"),
    ("rmsnorm_gamma_by_row", "* r * (double)gamma[c]);", "* r * (double)gamma[t % D]);"),
    ("rmsnorm_scale_from_the_routed_sum", "            ss += (double)o[c] * (double)o[c];",
     "            ss += ((double)o[c] - R[t * D + c]) * ((double)o[c] - R[t * D + c]);"),
]


def _scratch_copy(tmp_path):
    dst = tmp_path / "repo"
    (dst / "tests").mkdir(parents=True)
    shutil.copytree(os.path.join(ROOT, "oracle"), dst / "oracle", ignore=shutil.ignore_patterns("_build", "__pycache__"))
    pkg = dst / "mixture_experts_ffn_top_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "mixture_experts_ffn_top_gb300", "workloads.py"), pkg / "workloads.py")
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), dst / "tests" / f)
    return dst


def _run_pins(dst):
    # the regression fixtures record this oracle's own results: they are left out, so a planted
    # mistake counts as caught only when an independent pin fails
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           "-k", "not recorded_fixture", "tests/test_oracle_pins.py"], cwd=dst, capture_output=True,
                          text=True, timeout=300)


def test_unmodified_copy_passes_every_pin(tmp_path):
    """Control: the scratch copy without a planted mistake passes, so a failure below is the mistake's."""
    r = _run_pins(_scratch_copy(tmp_path))
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    dst = _scratch_copy(tmp_path)
    src = dst / "oracle" / "moe_oracle.c"
    text = src.read_text()
    assert old in text, f"mutation site for {name} not found"
    if name == "combine_shared_first":  # shared added first, and not again at the end
        text = text.replace("            if (S)\n                acc = acc + S[t * D + c];\n", "")
    src.write_text(text.replace(old, new, 1))
    r = _run_pins(dst)
    assert r.returncode != 0, f"planted mistake {name} passed every pin:\n{r.stdout[-2000:]}"
