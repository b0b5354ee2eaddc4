"""Plant one plausible mistake at a time in a copy of the oracle; some pin must catch it.

The mistakes are made on the CPU, in a temporary copy of the C source; the
committed oracle is never touched.  Each mutant must fail at least one pin,
which shows the pins are strong enough to notice a dropped term, a wrong sign,
a wrong index or a swapped operand.
"""
import os
import shutil
import tempfile

import pytest

import oracle as oracle_pkg
from tests import oracle_pins

MUTANTS = {
    "offset_uses_division": ("int off = t % block_size;", "int off = t / block_size;"),
    "cache_layout_transposed": (
        "size_t base = (((size_t)blk * n_kv + g) * block_size + off) * head_dim;",
        "size_t base = (((size_t)blk * block_size + off) * n_kv + g) * head_dim;"),
    "no_causal_limit": ("const long pos = (long)ctx - q_len + i;\n                const int nvis",
                        "const long pos = (long)ctx - 1;\n                const int nvis"),
    "scale_dropped": ("s[t] = scale * dot;", "s[t] = dot;"),
    "exp_sign_flipped": ("double w = exp(s[t] - mx);", "double w = exp(mx - s[t]);"),
    "not_normalised": ("orow[e] = acc[e] / denom;", "orow[e] = acc[e];"),
    "strided_group_map": ("for (int h = g * G; h < (g + 1) * G; ++h) {",
                          "for (int h = g; h < n_q; h += n_kv) {"),
    "scores_use_V": ("dot += bf16_value(qrow[e]) * K[(size_t)t * head_dim + e];",
                     "dot += bf16_value(qrow[e]) * V[(size_t)t * head_dim + e];"),
    "values_use_K": ("acc[e] += w * V[(size_t)t * head_dim + e];",
                     "acc[e] += w * K[(size_t)t * head_dim + e];"),
    "bf16_widening_wrong": ("uint32_t u = ((uint32_t)bits) << 16;",
                            "uint32_t u = ((uint32_t)bits) << 15;"),
    "own_token_excluded": ("(int)(pos + 1 < ctx ? pos + 1 : ctx);", "(int)(pos < ctx ? pos : ctx);"),
    "append_skips_slot0": ("if (slot < 0 || slot >= (long)num_blocks * block_size)",
                           "if (slot <= 0 || slot >= (long)num_blocks * block_size)"),
    "append_k_into_v": ("memcpy(v_cache + dst, v_new + src", "memcpy(v_cache + dst, k_new + src"),
    "kv_bytes_no_factor2": ("return (int64_t)2 * layers", "return (int64_t)1 * layers"),
    "merge_no_rescale": ("double w = exp(m[(size_t)s * rows + r] - M);", "double w = 1.0;"),
    "merge_denominator_unweighted": ("denom += w * ls;", "denom += ls;"),
    "partial_max_not_reported": ("m[row] = mx;", "m[row] = 0.0;"),
    "e4m3_bias_off_by_one": ("ldexp(8.0 + m, e - 10)", "ldexp(8.0 + m, e - 11)"),
    "e4m3_subnormal_scale": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "e4m3_ties_away": ("(long)rint(ldexp(a, 3 - e))", "(long)floor(ldexp(a, 3 - e) + 0.5)"),
    "e4m3_saturates_late": ("    if (a >= 448.0) {", "    if (a >= 480.0) {"),
    "e4m3_overflow_to_nan": ("code = 0x7E; /* the largest finite code", "code = 0x7F; /* the largest finite code"),
    "fp8_k_scale_dropped": (": c->kv8      ? (double)c->k_scale[g] : 0.0;",
                            ": c->kv8      ? 1.0 : 0.0;"),
    "fp8_v_uses_k_scale": (": c->kv8      ? (double)c->v_scale[g] : 0.0;",
                           ": c->kv8      ? (double)c->k_scale[g] : 0.0;"),
    "fp8_v_rows_not_offset": ("size_t vbase8 = kbase8 + (size_t)block_size * head_dim;",
                              "size_t vbase8 = kbase8;"),
    "fp8_append_head0_scale": ("/ k_scale[g];", "/ k_scale[0];"),
    "fp8_append_multiplies": ("/ v_scale[g];", "* v_scale[g];"),
    "window_one_too_wide": ("const long first_l = window > 0 ? pos - window + 1 : 0;",
                            "const long first_l = window > 0 ? pos - window : 0;"),
    "window_one_too_narrow": ("const long first_l = window > 0 ? pos - window + 1 : 0;",
                              "const long first_l = window > 0 ? pos - window + 2 : 0;"),
    "window_ignored": ("const long first_l = window > 0 ? pos - window + 1 : 0;",
                       "const long first_l = 0;"),
    "fp8_block_no_requantise": ("if (s_new > s_old && s_old > 0.0f) {", "if (0) {"),
    "fp8_block_ignores_restart": ("const float s_old = o_min > 0 ? sc[which] : 0.0f;",
                                  "const float s_old = sc[which];"),
    "fp8_block_scale_too_small": ("while (ldexp(448.0, e) < a)", "while (ldexp(224.0, e) < a)"),
    "fp8_block_scale_too_large": ("const float s_req = (float)ldexp(1.0, e);",
                                  "const float s_req = (float)ldexp(1.0, e + 1);"),
    "fp8_block_attn_logical_scale": (
        "(double)c->blk_scales[((size_t)blk * n_kv + g) * 4 + 0]",
        "(double)c->blk_scales[((size_t)(t / block_size) * n_kv + g) * 4 + 0]"),
    "fp8_block_v_uses_k_scale": ("(double)c->blk_scales[((size_t)blk * n_kv + g) * 4 + 1]",
                                 "(double)c->blk_scales[((size_t)blk * n_kv + g) * 4 + 0]"),
    "fp8_block_requantise_all_rows": ("for (long r = 0; r < o_min; ++r)",
                                      "for (long r = 0; r < block_size; ++r)"),
    "fp8_block_amax_first_token_only": (
        "                for (int j = i; j >= 0; j = next[j])\n"
        "                    for (int e = 0; e < head_dim; ++e) {\n"
        "                        const double x",
        "                for (int j = i; j == i; j = next[j])\n"
        "                    for (int e = 0; e < head_dim; ++e) {\n"
        "                        const double x"),
    "copy_direction_swapped": ("memcpy(k_cache + (size_t)dst * per_block, k_cache + (size_t)src * per_block,",
                               "memcpy(k_cache + (size_t)src * per_block, k_cache + (size_t)dst * per_block,"),
}


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="pkv_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(workdir, name):
    old, new = MUTANTS[name]
    src = open(oracle_pkg.SOURCE).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    path = os.path.join(workdir, f"{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle_pkg.compile_oracle(path, os.path.join(workdir, f"lib_{name}.so"), openmp=False)
    orc = oracle_pkg.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
