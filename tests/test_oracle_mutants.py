"""Mutation tests: plant a plausible mistake in a copy of the oracle (on the CPU) and
check that the pins catch it. Each mutant must make at least one pin fail."""
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_bwd_pins as bpins
from tests import test_oracle_dropout_pins as dpins
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "fa_oracle.cpp")

# (name, text to replace, replacement, pins to run)
MUTANTS = [
    ("causal mask off by one", "if (causal && (int64_t)j > i) { s[j] = NEG_INF; continue; }",
     "if (causal && (int64_t)j >= i && j > 0) { s[j] = NEG_INF; continue; }",
     ["causal_row0", "sdpa_causal", "zero_query_causal"]),
    ("scale dropped", "s[j] = scale * acc;", "s[j] = acc;", ["sdpa_full", "brute", "worked_row_final"]),
    ("logsumexp without the max", "*L = m + std::log(den);", "*L = std::log(den);",
     ["sdpa_full", "worked_row_final", "zero_query_full"]),
    ("scores against V instead of K", "const double* k = K + (int64_t)j * d;",
     "const double* k = V + (int64_t)j * d;", ["sdpa_full", "brute", "dominant"]),
    ("output weights not normalised", "for (int j = 0; j < Nk; ++j) s[j] = std::exp(s[j] - m) / den;",
     "for (int j = 0; j < Nk; ++j) s[j] = std::exp(s[j] - m);", ["sdpa_full", "probs", "hull"]),
    ("online softmax: old sum not re-based", "l = l * std::exp(m - m_new) + add;", "l = l + add;",
     ["worked_row_intermediates", "online_lse"]),
    ("merge: weight sign flipped", "const double wa = (m_a == NEG_INF) ? 0.0 : std::exp(m_a - m);",
     "const double wa = (m_a == NEG_INF) ? 0.0 : std::exp(m - m_a);", ["merge_closed", "merge_blocking"]),
    ("block state: causal mask ignored", "if (causal && (int64_t)j > i) v = NEG_INF;",
     "if (false) v = NEG_INF;", ["merge_blocking_causal"]),
    ("backward: D not subtracted", "const double ds = pij * (dprow[(size_t)j] - Di);",
     "const double ds = pij * dprow[(size_t)j];", ["bwd_torch", "bwd_closed"]),
    ("backward: dK without the scale", "gk[(int64_t)j * d + c] += scale * ds * q[i * d + c];",
     "gk[(int64_t)j * d + c] += ds * q[i * d + c];", ["bwd_torch", "bwd_fd"]),
    ("backward: dV from dS instead of P", "gv[(int64_t)j * d + c] += pz * go[i * d + c];",
     "gv[(int64_t)j * d + c] += ds * go[i * d + c];", ["bwd_torch", "bwd_closed"]),
    ("backward: dQ uses V instead of K", "gq[i * d + c] += scale * ds * k[(int64_t)j * d + c];",
     "gq[i * d + c] += scale * ds * v[(int64_t)j * d + c];", ["bwd_torch", "bwd_fd"]),
    ("philox: multipliers swapped", "const uint64_t p0 = (uint64_t)0xD2511F53u * c0;",
     "const uint64_t p0 = (uint64_t)0xCD9E8D57u * c0;", ["philox_kat"]),
    ("philox: second key word not bumped", "k1 += 0xBB67AE85u;", "k1 += 0u;", ["philox_kat"]),
    ("dropout: keep only above the threshold", "return x >= dr.t;", "return x > dr.t;",
     ["dropout_kat_bits"]),
    ("dropout: bytes of a word taken in natural order",
     "const int byte = (int)((j & 1) * 2 + ((j >> 1) & 1));", "const int byte = (int)(j & 3);",
     ["dropout_kat_bits"]),
    ("dropout: row and head swapped in the counter",
     "{(uint32_t)(j >> 4), (uint32_t)i, (uint32_t)bh, dr.offset}",
     "{(uint32_t)(j >> 4), (uint32_t)bh, (uint32_t)i, dr.offset}", ["dropout_layout"]),
    ("dropout: eight keys per generator call", "{(uint32_t)(j >> 4), (uint32_t)i,",
     "{(uint32_t)(j >> 3), (uint32_t)i,", ["dropout_layout"]),
    ("dropout: threshold truncated", "std::floor(p * 256.0 + 0.5)", "std::floor(p * 256.0)",
     ["dropout_threshold"]),
    ("dropout: kept entries not rescaled", "dr.z_keep = 256.0 / (256.0 - (double)t);",
     "dr.z_keep = 1.0;", ["dropout_unbiased", "dropout_onehot"]),
    ("dropout backward: dP without the mask", "dprow[(size_t)j] = acc * zrow[(size_t)j];",
     "dprow[(size_t)j] = acc;", ["dropout_torch", "dropout_fd"]),
    ("dropout backward: dV without the mask", "gv[(int64_t)j * d + c] += pz * go[i * d + c];",
     "gv[(int64_t)j * d + c] += pij * go[i * d + c];", ["dropout_torch", "dropout_fd"]),
]

PINS = {
    "causal_row0": lambda: pins.test_causal_row0_is_v0(oracle),
    "sdpa_causal": lambda: pins.test_attention_matches_torch_sdpa_float64(oracle, (1, 1, 100, 100, 32), True),
    "sdpa_full": lambda: pins.test_attention_matches_torch_sdpa_float64(oracle, (3, 2, 37, 53, 16), False),
    "zero_query_causal": lambda: pins.test_zero_query_is_uniform_average(oracle, True),
    "zero_query_full": lambda: pins.test_zero_query_is_uniform_average(oracle, False),
    "brute": lambda: pins.test_attention_brute_force_tiny(oracle),
    "worked_row_final": lambda: pins.test_worked_row_final_softmax_and_errata(oracle),
    "worked_row_intermediates": lambda: pins.test_worked_row_intermediates(oracle),
    "dominant": lambda: pins.test_dominant_key_selects_its_value(oracle),
    "probs": lambda: pins.test_probs_rows_sum_to_one_and_match_softmax(oracle),
    "hull": lambda: pins.test_output_in_convex_hull_and_permutation_invariance(oracle),
    "online_lse": lambda: pins.test_online_softmax_matches_logsumexp(oracle, 3),
    "merge_closed": lambda: pins.test_merge_two_singletons_closed_form(oracle),
    "merge_blocking": lambda: pins.test_merge_any_blocking_any_order_equals_definition(oracle, False),
    "merge_blocking_causal": lambda: pins.test_merge_any_blocking_any_order_equals_definition(oracle, True),
    "bwd_torch": lambda: bpins.test_bwd_matches_torch_autograd_float64(oracle, (2, 3, 37, 53, 16), False),
    "bwd_closed": lambda: bpins.test_bwd_closed_forms(oracle),
    "bwd_fd": lambda: bpins.test_bwd_central_differences(oracle),
    "philox_kat": lambda: dpins.test_philox_known_answer_vectors(oracle),
    "dropout_kat_bits": lambda: dpins.test_mask_bits_from_the_first_known_answer_vector(oracle),
    "dropout_layout": lambda: dpins.test_philox_matches_triton_and_mask_layout(oracle),
    "dropout_threshold": lambda: dpins.test_threshold_rounding_and_range(oracle),
    "dropout_unbiased": lambda: dpins.test_dropout_is_unbiased_over_seeds(oracle),
    "dropout_onehot": lambda: dpins.test_one_hot_values_read_the_mask_out_of_the_output(oracle),
    "dropout_torch": lambda: dpins.test_dropout_forward_and_backward_match_torch_autograd(oracle, True),
    "dropout_fd": lambda: dpins.test_dropout_backward_central_differences(oracle),
}


@pytest.mark.parametrize("mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(mut, oracle_mod, tmp_path):
    name, old, new, which = mut
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old}"
    mutant = tmp_path / "mutant.cpp"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-fPIC", "-shared", "-pthread", str(mutant), "-o", str(lib)],
                   check=True)
    failures = []
    with oracle.using_library(str(lib)):
        for pin in which:
            try:
                PINS[pin]()
            except AssertionError:
                failures.append(pin)
    assert failures, f"mutant '{name}' survived pins {which}"
    # and the intact oracle passes the same pins
    for pin in which:
        PINS[pin]()
