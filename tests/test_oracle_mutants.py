"""Each plausible slip planted in a copy of the oracle fails at least one pin.

The slips are planted on the CPU, in copies of the oracle's C source compiled
into a temporary directory; the oracle itself is never modified.
"""
import os

import pytest

import oracle
from tests import oracle_pins

# (name, text in wkv7_oracle.c, replacement)
MUTANTS = [
    ("delta_on_decayed_state",
     "acc += (double)kkt[i] * S[(size_t)i * N + j];",
     "acc += (double)kkt[i] * exp((double)wt[i]) * S[(size_t)i * N + j];"),
    ("delta_sign_flipped", "- c * z[j] +", "+ c * z[j] +"),
    ("decay_dropped", "const double decay = exp((double)wt[i]);", "const double decay = 1.0;"),
    ("decay_inverted", "const double decay = exp((double)wt[i]);", "const double decay = exp(-(double)wt[i]);"),
    ("decay_on_columns", "decay * S[(size_t)i * N + j]", "exp((double)wt[j]) * S[(size_t)i * N + j]"),
    ("k_used_for_kk_in_projection", "acc += (double)kkt[i] * S[(size_t)i * N + j];",
     "acc += (double)kt[i] * S[(size_t)i * N + j];"),
    ("a_dropped", "const double c = (double)kkt[i] * (double)at[i];", "const double c = (double)kkt[i];"),
    ("readout_transposed", "acc += (double)rt[i] * S[(size_t)i * N + j];",
     "acc += (double)rt[i] * S[(size_t)j * N + i];"),
    ("readout_before_kv_write", "acc += (double)rt[i] * S[(size_t)i * N + j];",
     "acc += (double)rt[i] * (S[(size_t)i * N + j] - (double)kt[i] * (double)vt[j]);"),
    ("k_and_v_swapped", "(double)kt[i] * (double)vt[j]", "(double)vt[i] * (double)kt[j]"),
    ("initial_state_ignored", "if (s0)\n", "if (0)\n"),
    ("wrong_head_offset", "((size_t)t * (size_t)H + (size_t)h) * (size_t)N",
     "((size_t)t * (size_t)H + (size_t)(H - 1 - h)) * (size_t)N"),
    ("last_token_dropped", "for (t = t_begin; t < t_end; ++t)", "for (t = t_begin; t + 1 < t_end; ++t)"),
    # the time-mix tail
    ("tail_unbiased_variance", "var /= (double)N;", "var /= (double)(N - 1);"),
    ("tail_eps_outside_sqrt", "inv = 1.0 / sqrt(var + eps);", "inv = 1.0 / (sqrt(var) + eps);"),
    ("tail_mean_not_subtracted", "(o[base + j] - mu) * inv", "o[base + j] * inv"),
    ("tail_second_moment_not_centred", "var += (o[base + j] - mu) * (o[base + j] - mu);",
     "var += o[base + j] * o[base + j];"),
    ("tail_gate_only_on_norm", "y[base + j] = (normed + bonus * (double)v[base + j]) * (double)g[base + j];",
     "y[base + j] = normed * (double)g[base + j] + bonus * (double)v[base + j];"),
    ("tail_bonus_without_rk", "bonus += (double)r[base + i] * (double)k[base + i] * (double)rk[pbase + i];",
     "bonus += (double)r[base + i] * (double)k[base + i];"),
    ("tail_bonus_times_wrong_v", "bonus * (double)v[base + j]", "bonus * (double)v[base + (N - 1 - j)]"),
    ("tail_parameters_of_head_zero", "const size_t pbase = (size_t)h * (size_t)N;", "const size_t pbase = 0;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    path = tmp_path / f"{name}.c"
    path.write_text(mutated)
    lib = oracle.load(oracle.compile_source(str(path), str(tmp_path / f"lib{name}.so")))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted slip {name}"
