"""Planted mistakes in the oracle, on the CPU: every build of the oracle's C
source with one plausible mistake (a swapped index, a wrong rounding, a
dropped term, a flipped sign, a transposed operand) must fail at least one of
the oracle's pins, and the unchanged source must pass them all."""
import os
import subprocess

import numpy as np
import pytest

import tests.test_oracle as T
from oracle import oracle as O
from verify_matvec_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# name: (text of the oracle source, its replacement)
MUTANTS = {
    "nibble halves swapped": ("if (i < 16) return qs[i] & 0x0f;\n    return qs[i - 16] >> 4;",
                              "if (i < 16) return qs[i] >> 4;\n    return qs[i - 16] & 0x0f;"),
    "rounding half away from zero": ("float q = rintf(xb[i] / d);", "float q = roundf(xb[i] / d);"),
    "activation scale over 128": ("const float d = amax / 127.0f;", "const float d = amax / 128.0f;"),
    "activation scale dropped": ("acc += dw * (double)dxc[b] * s;", "acc += dw * s;"),
    "weight scale dropped": ("acc += dw * (double)dxc[b] * s;", "acc += (double)dxc[b] * s;"),
    "blocks of a row reversed": ("const uint8_t *blk = Wrow + b * ORACLE_BLOCK_BYTES;",
                                 "const uint8_t *blk = Wrow + (nb - 1 - b) * ORACLE_BLOCK_BYTES;"),
    "codebook level off by one": ("-127, -104, -83, -65, -49, -35, -22, -10,",
                                  "-127, -104, -83, -65, -49, -35, -22, -11,"),
    "silu sign flipped": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "gate and up rows swapped": (
        "const double g = row_dot(gu + r * nbH * ORACLE_BLOCK_BYTES, nbH, qh, dh);\n"
        "                const double u = row_dot(gu + (F + r) * nbH * ORACLE_BLOCK_BYTES, nbH, qh, dh);",
        "const double g = row_dot(gu + (F + r) * nbH * ORACLE_BLOCK_BYTES, nbH, qh, dh);\n"
        "                const double u = row_dot(gu + r * nbH * ORACLE_BLOCK_BYTES, nbH, qh, dh);"),
    "router weight of the slot index only": ("const double wj = (double)wts[p];", "const double wj = (double)wts[j];"),
    "shared expert weighted by slot 0's router weight": ("sh_wts[t] = 1.0f;", "sh_wts[t] = wts[t * k];"),
    "shared expert output dropped": ("y[i] += ys[i];", "y[i] += 0.0 * ys[i];"),
    "router ties to the higher index": ("l[e] > l[best]", "l[e] >= l[best]"),
    "router weights not normalised": ("for (int j = 0; j < k; ++j) wts[t * k + j] /= sum;", ""),
    "converter ties to the higher index": ("if (d < best_d) {", "if (d <= best_d) {"),
    "converter scale over -128": ("oracle_float_to_half(m / -127.0f)", "oracle_float_to_half(m / -128.0f)"),
    "converter scale sign flipped": ("oracle_float_to_half(m / -127.0f)", "oracle_float_to_half(m / 127.0f)"),
    "converter keeps the last largest weight": ("if (fabsf(w[i]) > fabsf(w[imax])) imax = i;",
                                                "if (fabsf(w[i]) >= fabsf(w[imax])) imax = i;"),
    "converter nibble halves swapped": ("if (i < 16) blk[2 + i] |= (uint8_t)best;\n        else blk[2 + i - 16] |= (uint8_t)(best << 4);",
                                        "if (i < 16) blk[2 + i] |= (uint8_t)(best << 4);\n        else blk[2 + i - 16] |= (uint8_t)best;"),
    "half rounding truncates": ("double q = nearbyint(ldexp(a, 11 - e));", "double q = floor(ldexp(a, 11 - e));"),
    "half subnormals flushed": ("const double q = nearbyint(ldexp(a, 24));", "const double q = 0.0;"),
    "sinkhorn without the exponential": ("P[i] = exp((double)c[i] - cmax);", "P[i] = (double)c[i] - cmax;"),
    "sinkhorn row step dropped": ("for (int j = 0; j < nhc; ++j) P[r * nhc + j] /= sum;", ""),
    "sinkhorn column step dropped": ("for (int r = 0; r < nhc; ++r) P[r * nhc + j] /= sum;", ""),
    "sinkhorn one round short": ("for (int t = 0; t < iters; ++t)", "for (int t = 1; t < iters; ++t)"),
    "sinkhorn transposed": ("const float *c = logits + m * nn;\n        double *P = out + m * nn;",
                            "const float *c = logits + m * nn;\n        double *P = out + m * nn;\n        float ct[64];\n"
                            "        for (int i = 0; i < nn; ++i) ct[(i % nhc) * nhc + i / nhc] = c[i];\n        c = ct;"),
}


def _tiny():
    return (synth.expert_blocks(T.E_, 2 * T.F_, T.H_, stream=31),
            synth.expert_blocks(T.E_, T.H_, T.F_, stream=32))


def _pins():
    tiny = _tiny()
    return [
        lambda: T.test_codebook_matches_fixture(GOLDEN),
        lambda: T.test_half_to_float_every_pattern(),
        lambda: T.test_quantize_golden_blocks(GOLDEN),
        lambda: T.test_quantize_exact_rational_properties(),
        lambda: T.test_quantize_sign_symmetry_and_power_of_two_scaling(),
        lambda: T.test_nibble_layout_one_hot(),
        lambda: T.test_block_dots_golden(GOLDEN),
        lambda: T.test_block_dots_brute_force_small(),
        lambda: T.test_matvec_equals_dequantize_then_dot(33, 320, 3),
        lambda: T.test_matvec_scale_linearity_exact(),
        lambda: T.test_silu_identities(),
        lambda: T.test_moe_k1_reduces_to_matvecs(tiny, 1),
        lambda: T.test_moe_gate_and_up_are_not_interchangeable(tiny),
        lambda: T.test_moe_router_weights_and_slots(tiny),
        lambda: T.test_moe_tokens_are_independent(tiny),
        lambda: T.test_moe_bad_ids_and_duplicates(tiny),
        lambda: T.test_moe_down_combine_matches_full(tiny),
        lambda: T.test_moe_shared_zero_scales_give_the_routed_layer(tiny),
        lambda: T.test_moe_shared_alone_is_one_dense_ffn(tiny, 1),
        lambda: T.test_moe_shared_is_one_more_slot_of_weight_one(tiny),
        lambda: T.test_moe_shared_equal_to_a_routed_expert(tiny),
        lambda: T.test_router_topk_golden(GOLDEN),
        lambda: T.test_router_topk_invariants(),
        lambda: T.test_float_to_half_matches_numpy(),
        lambda: T.test_convert_golden_blocks(GOLDEN),
        lambda: T.test_convert_grid_round_trip(),
        lambda: T.test_convert_brute_force_exact(),
        lambda: T.test_convert_error_bound_and_zero_blocks(),
        lambda: T.test_sinkhorn_zero_rounds_is_the_shifted_exponential(),
        lambda: T.test_sinkhorn_rank_one_is_uniform_after_one_round(4),
        lambda: T.test_sinkhorn_two_by_two_limit_closed_form(),
        lambda: T.test_sinkhorn_doubly_stochastic_input_is_a_fixed_point(),
        lambda: T.test_sinkhorn_sums_row_shift_and_permutations(),
    ]


def _build(tmp_path, name, source):
    src = tmp_path / f"{name}.c"
    src.write_text(source)
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", *O._CFLAGS, "-I", os.path.dirname(O._SRC), str(src), "-o", str(lib), "-lm"],
                   check=True)
    return str(lib)


def _failures(lib):
    failed = 0
    with O.using_library(lib):
        for pin in _pins():
            try:
                pin()
            except Exception:  # an assertion, or any other sign that the pin does not hold
                failed += 1
    return failed


def test_unchanged_source_passes_every_pin(tmp_path):
    with open(O._SRC) as f:
        source = f.read()
    assert _failures(_build(tmp_path, "unchanged", source)) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    with open(O._SRC) as f:
        source = f.read()
    assert old in source, "the mutation no longer matches the oracle source"
    mutant = source.replace(old, new, 1)
    lib = _build(tmp_path, "mutant", mutant)
    assert _failures(lib) >= 1, f"no pin fails when the oracle has: {name}"
