"""Plant one plausible mistake at a time in a copy of the oracle's source
(on the CPU) and check that the pins catch every one of them.

One natural-looking mutation is deliberately absent: reading the high nibble
as element 2i for BOTH operands.  Two codes that share a byte always share a
16-element scale block, so swapping the order in A and B together permutes
the terms of every dot product and leaves C unchanged; it is an equivalent
mutant, not a mistake in what the oracle computes.  (It matters only for how
callers pack bytes, which the check_nibble_order pin documents.)

Likewise absent: the quantiser's scale quotient taken as amax * (1/6) in
single precision.  check_quant_scales_exhaustive shows that it gives the same
E4M3FN scale as amax / 6 for every finite FP16 and BF16 absmax (an exact tie
m = amax / 6 on a midpoint stays within half an ulp of m), so it too is
equivalent for these inputs.  The same slip in the element quotient,
x * (1/s), is not: it moves exact E2M1 ties and is planted below.
"""
import os

import pytest

import oracle_checks as oc
from oracle import oracle

MUTANTS = {
    "scale_per_32_elements": (
        "nvfp4_oracle_e4m3fn(sf_row[k / 16]);",
        "nvfp4_oracle_e4m3fn(sf_row[k / 32]);"),
    "last_k_dropped": (
        "for (int k = 0; k < K; ++k)\n                sum += arow[k] * brow[k];",
        "for (int k = 0; k < K - 1; ++k)\n                sum += arow[k] * brow[k];"),
    "e2m1_sign_dropped": (
        "        mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);\n    return s ? -mag : mag;",
        "        mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);\n    return mag;"),
    "e2m1_exponent_bias": (
        "mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);",
        "mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 2);"),
    "e4m3_bias_8": (
        "mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);",
        "mag = ldexp(1.0 + (double)m / 8.0, (int)e - 8);"),
    "e4m3_subnormal_scale": (
        "mag = ldexp((double)m / 8.0, -6);",
        "mag = ldexp((double)m / 8.0, -7);"),
    "e4m3_nan_missing": (
        "if (e == 15 && m == 7)\n        return NAN;",
        "if (e == 16 && m == 7)\n        return NAN;"),
    "fp16_ties_away": (
        "(diff == 0.5 && fmod(fl, 2.0) != 0.0)",
        "(diff == 0.5)"),
    "fp16_subnormal_quantum": (
        "if (qexp < -24)\n        qexp = -24;",
        "if (qexp < -23)\n        qexp = -23;"),
    "output_transposed": (
        "size_t idx = (size_t)m * j->N + n;",
        "size_t idx = (size_t)n * j->M + m;"),
    "b_scales_of_row_zero": (
        "dequant_row(j->X + (size_t)r * (j->K / 2), j->SFX + (size_t)r * (j->K / 16), j->K,",
        "dequant_row(j->X + (size_t)r * (j->K / 2), j->SFX, j->K,"),
    "float32_accumulator": (
        "            double sum = 0.0;\n            for (int k = 0; k < K; ++k)\n                sum += arow",
        "            float sum = 0.0f;\n            for (int k = 0; k < K; ++k)\n                sum += arow"),
    "elements_b_scale_dropped": (
        "nvfp4_oracle_e2m1(fp4_code(brow, k)) * nvfp4_oracle_e4m3fn(sb[k / 16]);",
        "nvfp4_oracle_e2m1(fp4_code(brow, k));"),
    "atom_inner_layout": (
        "(r % 32) * 16 + (r / 32) * 4 + j] = v;",
        "(r / 4) * 16 + (r % 4) * 4 + j] = v;"),
    "atom_order_k_major": (
        "((size_t)rb * kblocks + kb) * 512",
        "((size_t)kb * ((rows + 127) / 128) + rb) * 512"),
    "quant_scale_over_4": (
        "const float s32 = amax / 6.0f;",
        "const float s32 = amax / 4.0f;"),
    "quant_absmax_signed": (
        "const float a = fabsf(v[i]);",
        "const float a = v[i];"),
    "quant_nibbles_swapped": (
        "(uint8_t)(lo | (hi << 4));",
        "(uint8_t)(hi | (lo << 4));"),
    "quant_negative_zero": (
        "return (best != 0 && q < 0.0f) ? (best | 8u) : best;",
        "return (q < 0.0f) ? (best | 8u) : best;"),
    "quant_e2m1_ties_up": (
        "    for (unsigned c = 1; c < 8; ++c) {\n        const double d = fabs(a - nvfp4_oracle_e2m1(c));\n"
        "        if (d < best_d || (d == best_d && (c & 1u) == 0 && (best & 1u) == 1)) {",
        "    for (unsigned c = 1; c < 8; ++c) {\n        const double d = fabs(a - nvfp4_oracle_e2m1(c));\n"
        "        if (d <= best_d) {"),
    "quant_e4m3_truncates": (
        "        const double d = fabs(x - nvfp4_oracle_e4m3fn(c));\n"
        "        if (d < best_d || (d == best_d && (c & 1u) == 0 && (best & 1u) == 1)) {",
        "        const double d = fabs(x - nvfp4_oracle_e4m3fn(c));\n"
        "        if (nvfp4_oracle_e4m3fn(c) <= x) {"),
    "quant_reciprocal_multiply": (
        " / sdec)",
        " * (1.0f / sdec))"),
    "swiglu_gate_up_swapped": (
        "const double g = alpha * acc[(size_t)m * N + 256 * j + c];\n"
        "                const double u = alpha * acc[(size_t)m * N + 256 * j + 128 + c];",
        "const double g = alpha * acc[(size_t)m * N + 256 * j + 128 + c];\n"
        "                const double u = alpha * acc[(size_t)m * N + 256 * j + c];"),
    "swiglu_alpha_after_silu": (
        "v = nvfp4_oracle_silu(g) * u;",
        "v = nvfp4_oracle_silu(g / alpha) * alpha * u;"),
    "bf16_mantissa_9_bits": (
        "int qexp = ex - 8;\n    if (qexp < -133)",
        "int qexp = ex - 9;\n    if (qexp < -133)"),
    "silu_sign": (
        "return x / (1.0 + exp(-x));",
        "return x / (1.0 + exp(x));"),
    "fixed_point_shift": (
        "int shift = ea + eb - 2 + 20;",
        "int shift = ea + eb - 1 + 20;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(mutated)
    so = oracle.compile_oracle(path, os.path.join(tmp_path, f"libmutant_{name}.so"))
    o = oracle.Oracle(so)
    failed = []
    for check in oc.ALL_CHECKS:
        try:
            check(o)
        except (AssertionError, ValueError):
            failed.append(check.__name__)
            break                       # one failing pin is enough
    assert failed, f"no pin caught the planted mistake {name}"
