"""The pins must catch plausible mistakes in the oracle.

Each case below is a deliberately broken copy of the oracle's C source (a
dropped term, a wrong sign or order, a transposed operand, a wrong head map),
compiled into a temporary library on the CPU.  Every mutant must fail at least
one pin of tests/test_oracle_pins.py; the real oracle passes all of them.
"""

import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

_SRC = os.path.join(os.path.dirname(oracle.__file__), "gdr_oracle.c")

DECAY = "for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] *= alpha;"

MUTANTS = {
    # gate applied after the recall instead of before it
    "decay_after_recall": [
        (f"        /* S <- alpha S */\n        {DECAY}\n", ""),
        ("        /* S <- S + k_t ((v_t - u) beta_t)^T */\n",
         f"        /* S <- S + k_t ((v_t - u) beta_t)^T */\n        {DECAY}\n"),
    ],
    # beta dropped from the correction
    "no_beta": [("u[j] = (vt[j] - u[j]) * b;", "u[j] = (vt[j] - u[j]);")],
    # wrong sign of the recalled value
    "recall_sign": [("u[j] = (vt[j] - u[j]) * b;", "u[j] = (vt[j] + u[j]) * b;")],
    # recall skipped (plain gated linear attention)
    "no_recall": [("u[j] = (vt[j] - u[j]) * b;", "u[j] = vt[j] * b;")],
    # state transposed in the recall (S k instead of S^T k; dims must match)
    "recall_transposed": [("u[j] += row[j] * ki;", "u[j] += S[(size_t)j * dv + i] * ki + 0.0 * row[j];")],
    # gate read as exp(-g)
    "gate_sign": [("const double alpha = exp(J->g[", "const double alpha = exp(-J->g[")],
    # wrong QK head for a V head (interleaved instead of contiguous pairs)
    "head_map": [("const int hq = h / group;", "const int hq = h % J->h_qk;")],
    # scale ignored
    "no_scale": [("for (int j = 0; j < dv; ++j) ot[j] *= J->scale;", "")],
    # output read before the update (from the decayed S_{t-1})
    "readout_before_update": [
        ("        /* S <- S + k_t ((v_t - u) beta_t)^T */\n", "        goto readout; back:\n        /* S <- S + k_t ((v_t - u) beta_t)^T */\n"),
        ("        /* o_t <- scale S^T q_t */\n", "        continue;\n        readout: ;\n"),
        ("        for (int j = 0; j < dv; ++j) ot[j] *= J->scale;\n", "        for (int j = 0; j < dv; ++j) ot[j] *= J->scale;\n        goto back;\n"),
    ],
    # L2 norm: epsilon outside the square root
    "l2norm_eps_outside": [("const double inv = 1.0 / sqrt(ss + eps);", "const double inv = 1.0 / (sqrt(ss) + eps);")],
    # RMSNorm: sum of squares instead of their mean
    "rmsnorm_sum_not_mean": [("const double inv = 1.0 / sqrt(ss / d + eps);", "const double inv = 1.0 / sqrt(ss + eps);")],
    # gate: sigmoid(z) instead of silu(z)
    "gate_sigmoid_not_silu": [("const double silu = zz / (1.0 + exp(-zz));", "const double silu = 1.0 / (1.0 + exp(-zz));")],
    # norm weight dropped
    "rmsnorm_no_weight": [("yr[j] = w[j] * orow[j] * inv * silu;", "yr[j] = orow[j] * inv * silu;")],
    # beta logit with the wrong sign
    "sigmoid_sign": [("beta[i] = 1.0 / (1.0 + exp(-b[i]));", "beta[i] = 1.0 / (1.0 + exp(b[i]));")],
}

PIN_CASES = [
    pins.test_beta_zero_is_pure_geometric_decay,
    pins.test_alpha_one_beta_zero_freezes_state,
    pins.test_orthogonal_keys_give_cumulative_linear_attention,
    pins.test_orthonormal_keys_beta_one_overwrite_slots,
    pins.test_scalar_case_by_hand,
    pins.test_exact_rational_brute_force_matrix_products,
    pins.test_superposition_in_state_and_values,
    pins.test_scale_multiplies_output_only,
    pins.test_padding_rows_are_a_no_op,
    pins.test_qk_head_shared_by_contiguous_pair_of_v_heads,
    pins.test_contraction_bound_per_step,
    lambda: pins.test_chunk_forms_match_sequential(16, 40),
    pins.test_l2norm_rows_closed_forms,
    pins.test_sigmoid_closed_forms,
    pins.test_gated_rmsnorm_by_hand_and_invariants,
]


def _build_mutant(tmp_path, name, edits):
    src = open(_SRC).read()
    for old, new in edits:
        assert old in src, f"mutant {name}: pattern not found: {old[:60]!r}"
        src = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(src)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(c), "-lpthread", "-lm"])
    return str(so)


def _failures():
    failed = 0
    for case in PIN_CASES:
        try:
            case()
        except AssertionError:
            failed += 1
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_mutant_fails_some_pin(tmp_path, name):
    so = _build_mutant(tmp_path, name, MUTANTS[name])
    with oracle.using_library(so):
        assert _failures() > 0, f"mutant {name} passed every pin"


def test_real_oracle_passes_the_same_pins():
    assert _failures() == 0
