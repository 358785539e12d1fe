"""Plants plausible mistakes in copies of the oracle (CPU only) and checks the pins catch each one
(the forward's pins for mistakes in the forward, the reverse mode's for mistakes in the reverse mode).

Every mutant is compiled from a string-edited copy of ``oracle/dplr_oracle.c``
into a temporary directory, swapped in for the real library, and run through
the pin functions of ``test_oracle_pins``. A mutant that passes every pin
would mean the pins leave that part of the oracle unchecked.
"""

import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_backward as bpins
import test_oracle_gdp as gpins
import test_oracle_hla as hpins
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "dplr_oracle.c")

MUTANTS = {
    # generic mode
    "generic_sign_of_low_rank": ("s -= At[(size_t)i * dk + c] * w[i * nc + n];",
                                 "s += At[(size_t)i * dk + c] * w[i * nc + n];"),
    "generic_drops_decay": ("double s = d * S[c * nc + n];", "double s = S[c * nc + n];"),
    "generic_drops_write": ("for (int l = 0; l < p; ++l)\n", "for (int l = 0; l < 0; ++l)\n"),
    "generic_swaps_A_and_B": ("s += Bt[(size_t)i * dk + c] * S[c * nc + n];",
                              "s += At[(size_t)i * dk + c] * S[c * nc + n];"),
    # GDN mode
    "gdn_gate_on_write_too": ("S[c * nc + n] = gate * (S[c * nc + n] - bt * kt[c] * w[n])\n"
                              "                                        + bt * kt[c] * vt[c0 + n];",
                              "S[c * nc + n] = gate * (S[c * nc + n] - bt * kt[c] * w[n]\n"
                              "                                        + bt * kt[c] * vt[c0 + n]);"),
    "gdn_drops_erase": ("gate * (S[c * nc + n] - bt * kt[c] * w[n])", "gate * (S[c * nc + n])"),
    # HDLA mode
    "hdla_drops_first_erase": ("for (int n = 0; n < nc; ++n) S[c * nc + n] -= bt * kt[c] * w[n];\n"
                               "                /* 2:",
                               "for (int n = 0; n < nc; ++n) S[c * nc + n] -= 0.0 * w[n];\n"
                               "                /* 2:"),
    "hdla_write_sign": ("w[n] = s - vt[c0 + n];", "w[n] = s + vt[c0 + n];"),
    "hdla_decay_inverted": ("const double lam = exp(lt[c]);", "const double lam = exp(-lt[c]);"),
    # readout
    "readout_before_update_index": ("double* ot = a->o + (size_t)t * dv + c0;",
                                    "double* ot = a->o + (size_t)(t > 0 ? t - 1 : 0) * dv + c0;"),
    "readout_uses_k_not_q": ("for (int c = 0; c < dk; ++c) s += S[c * nc + n] * qt[c];",
                             "for (int c = 0; c < dk; ++c) s += S[c * nc + n] * (a->k ? a->k[(size_t)t * dk + c] : qt[c]);"),
    "initial_state_ignored": ("S[i * nc + n] = a->S0 ? a->S0[(size_t)i * dv + c0 + n] : 0.0;",
                              "S[i * nc + n] = 0.0;"),
    "initial_state_transposed": ("S[i * nc + n] = a->S0 ? a->S0[(size_t)i * dv + c0 + n] : 0.0;",
                                 "S[i * nc + n] = a->S0 ? a->S0[(size_t)(c0 + n) * dv + i % dv] : 0.0;"),
}

PIN_CALLS = [
    lambda: pins.test_hand_worked_examples("gdn_two_tokens"),
    lambda: pins.test_hand_worked_examples("hdla_two_tokens"),
    lambda: pins.test_hand_worked_examples("generic_one_token"),
    pins.test_no_decay_reduces_to_causal_linear_attention,
    pins.test_diagonal_decay_reduces_to_gla,
    pins.test_gdn_zero_beta_is_pure_gate,
    pins.test_gdn_delta_rule_closed_form_same_key,
    pins.test_hdla_reflection_without_forgetting_is_linear_attention,
    pins.test_hdla_transition_is_similar_to_its_diagonal,
    lambda: pins.test_explicit_transition_matrices("gdn"),
    lambda: pins.test_explicit_transition_matrices("hdla"),
    pins.test_generic_explicit_transition,
]


BWD_MARK = "/*\n * Reverse mode of the same serial recurrence"

# Mistakes planted in the reverse mode (after BWD_MARK), caught by the finite-difference and closed-form pins.
BWD_MUTANTS = {
    "bwd_readout_adjoint_dropped": ("for (int n = 0; n < dv; ++n) dS[(size_t)c * dv + n] += qt[c] * dot[n];",
                                    "for (int n = 0; n < dv; ++n) dS[(size_t)c * dv + n] += 0.0 * qt[c] * dot[n];"),
    "bwd_generic_decay_not_transposed": ("double s = exp(lt[c]) * dS[(size_t)c * dv + n];",
                                         "double s = dS[(size_t)c * dv + n];"),
    "bwd_gdn_gate_on_write_adjoint": ("for (size_t e = 0; e < SS; ++e) dT[e] = gate * dS[e];   /* dX */",
                                      "for (size_t e = 0; e < SS; ++e) dT[e] = dS[e];   /* dX */"),
    "bwd_erase_beta_sign": ("    *dbt -= db;", "    *dbt += db;"),
    "bwd_hdla_decay_grad_uses_wrong_state": ("for (int n = 0; n < dv; ++n) dd += dT[(size_t)c * dv + n] * S1[(size_t)c * dv + n];",
                                             "for (int n = 0; n < dv; ++n) dd += dT[(size_t)c * dv + n] * S2[(size_t)c * dv + n];"),
    "bwd_final_state_gradient_ignored": ("for (size_t e = 0; e < SS; ++e) dS[e] = a->dST ? a->dST[e] : 0.0;",
                                         "for (size_t e = 0; e < SS; ++e) dS[e] = 0.0;"),
}

BWD_PIN_CALLS = [
    bpins.test_gdn_backward_matches_finite_differences,
    bpins.test_hdla_backward_matches_finite_differences,
    lambda: bpins.test_generic_backward_matches_finite_differences(2, 1),
    bpins.test_linear_attention_closed_form,
    bpins.test_state_gradient_is_the_transposed_map,
]


HLA_MARK = "/*\n * HLA's query-conditioned composition"

# Mistakes planted in the HLA composition (after HLA_MARK), caught by its pins.
HLA_MUTANTS = {
    "hla_gate_drops_retention": ("X[(size_t)r * dv + n] = (1.0 - wij) * S[(size_t)r * dv + n] + wij * (s + Bj[(size_t)r * dv + n]);",
                                 "X[(size_t)r * dv + n] = wij * (s + Bj[(size_t)r * dv + n]);"),
    "hla_gate_on_write_only": ("X[(size_t)r * dv + n] = (1.0 - wij) * S[(size_t)r * dv + n] + wij * (s + Bj[(size_t)r * dv + n]);",
                               "X[(size_t)r * dv + n] = s + wij * Bj[(size_t)r * dv + n];"),
    "hla_skips_current_prefix": ("for (int t = c * L; t <= i; ++t)", "for (int t = c * L; t < i; ++t)"),
    "hla_threshold_inverted": ("if (wij < theta) wij = 0.0;", "if (wij > theta) wij = 0.0;"),
}

GDP_MARK = "/*\n * Gated DeltaProduct-style stacked Householders"

# Mistakes planted in the stacked-Householder oracle (after GDP_MARK), caught by its pins.
GDP_MUTANTS = {
    "gdp_gate_per_step": ("for (size_t e = 0; e < SS; ++e) S[e] *= gate;\n                for (int h = 0; h < nh; ++h) {",
                          "for (int h = 0; h < nh; ++h) {\n                for (size_t e = 0; e < SS; ++e) S[e] *= gate;"),
    "gdp_write_sign": ("w[n] = s - vt[n];", "w[n] = s + vt[n];"),
    "gdp_last_step_only": ("for (int h = 0; h < nh; ++h) {\n                    const double* kt", "for (int h = nh - 1; h < nh; ++h) {\n                    const double* kt"),
}

GDP_PIN_CALLS = [
    gpins.test_one_step_is_gated_deltanet,
    gpins.test_second_step_with_zero_beta_is_gated_deltanet,
    gpins.test_explicit_transition_and_write,
    gpins.test_rank_nh_transition_in_the_generic_form,
]

HLA_PIN_CALLS = [
    hpins.test_all_gates_one_is_the_gdn_recurrence,
    hpins.test_all_gates_zero_restarts_each_chunk,
    hpins.test_one_gate_selects_one_chunk_of_history,
    hpins.test_gates_below_the_threshold_are_zero,
    hpins.test_output_is_affine_in_each_gate,
]


def _build_mutant(tmp_path, name, old, new, backward=False, hla=False, gdp=False):
    text = open(SRC).read()
    cut, cut2, cut3 = text.index(BWD_MARK), text.index(HLA_MARK), text.index(GDP_MARK)
    parts = [text[:cut], text[cut:cut2], text[cut2:cut3], text[cut3:]]
    k = 3 if gdp else (2 if hla else (1 if backward else 0))
    assert parts[k].count(old) == 1, f"mutation anchor for {name} not unique/found"
    parts[k] = parts[k].replace(old, new)
    src = tmp_path / f"{name}.c"
    src.write_text("".join(parts))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(src), "-o", str(so), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_forward.restype = ctypes.c_int
    lib.oracle_forward.argtypes = [ctypes.c_int] * 8 + [dp] * 12 + [ctypes.c_int]
    lib.oracle_gdp.restype = ctypes.c_int
    lib.oracle_gdp.argtypes = [ctypes.c_int] * 6 + [dp] * 8 + [ctypes.c_int]
    lib.oracle_hla.restype = ctypes.c_int
    lib.oracle_hla.argtypes = [ctypes.c_int] * 6 + [ctypes.c_double] + [dp] * 7 + [ctypes.c_int]
    lib.oracle_backward.restype = ctypes.c_int
    lib.oracle_backward.argtypes = [ctypes.c_int] * 8 + [dp] * 22 + [ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    oracle._lib()                                  # make sure the real one is initialised first
    monkeypatch.setattr(oracle, "_handle", lib)
    caught = 0
    for call in PIN_CALLS:
        try:
            call()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin failed for mutant {name}"


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_backward_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    old, new = BWD_MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new, backward=True)
    oracle._lib()
    monkeypatch.setattr(oracle, "_handle", lib)
    caught = 0
    for call in BWD_PIN_CALLS:
        try:
            call()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin failed for mutant {name}"


@pytest.mark.parametrize("name", sorted(HLA_MUTANTS))
def test_hla_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    old, new = HLA_MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new, hla=True)
    oracle._lib()
    monkeypatch.setattr(oracle, "_handle", lib)
    caught = 0
    for call in HLA_PIN_CALLS:
        try:
            call()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin failed for mutant {name}"


@pytest.mark.parametrize("name", sorted(GDP_MUTANTS))
def test_gdp_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    old, new = GDP_MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new, gdp=True)
    oracle._lib()
    monkeypatch.setattr(oracle, "_handle", lib)
    caught = 0
    for call in GDP_PIN_CALLS:
        try:
            call()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin failed for mutant {name}"
