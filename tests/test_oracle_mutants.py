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
    # the backward
    ("bwd_dr_from_old_state", "acc_r += S_new[(size_t)i * N + j] * dot[j];",
     "acc_r += S_old[(size_t)i * N + j] * dot[j];"),
    ("bwd_dw_without_decay_factor", "job->dw[base + i] = exp((double)job->w[base + i]) * acc_d;",
     "job->dw[base + i] = acc_d;"),
    ("bwd_dw_on_new_state", "acc_d += G[(size_t)i * N + j] * S_old[(size_t)i * N + j];",
     "acc_d += G[(size_t)i * N + j] * S_new[(size_t)i * N + j];"),
    ("bwd_u_with_kk_not_c", "acc_u += G[(size_t)i * N + j] * (double)job->kk[base + i] * (double)job->a[base + i];",
     "acc_u += G[(size_t)i * N + j] * (double)job->kk[base + i];"),
    ("bwd_dkk_without_c_chain", "job->dkk[base + i] = -acc + (double)job->a[base + i] * dc[i];",
     "job->dkk[base + i] = -acc;"),
    ("bwd_da_without_kk", "job->da[base + i] = (double)job->kk[base + i] * dc[i];", "job->da[base + i] = dc[i];"),
    ("bwd_dc_sign", "dc[i] = -acc_c;", "dc[i] = acc_c;"),
    ("bwd_removal_sign_in_adjoint", "decay * G[(size_t)i * N + j] - (double)job->kk[base + i] * u[j];",
     "decay * G[(size_t)i * N + j] + (double)job->kk[base + i] * u[j];"),
    ("bwd_adjoint_not_decayed", "decay * G[(size_t)i * N + j] - (double)job->kk[base + i] * u[j];",
     "G[(size_t)i * N + j] - (double)job->kk[base + i] * u[j];"),
    ("bwd_readout_outer_transposed", "G[(size_t)i * N + j] += (double)job->r[base + i] * dot[j];",
     "G[(size_t)i * N + j] += (double)job->r[base + j] * dot[i];"),
    ("bwd_dk_transposed", "acc_k += G[(size_t)i * N + j] * (double)job->v[base + j];",
     "acc_k += G[(size_t)j * N + i] * (double)job->v[base + j];"),
    ("bwd_dv_with_kk", "acc_v += G[(size_t)i * N + j] * (double)job->k[base + i];",
     "acc_v += G[(size_t)i * N + j] * (double)job->kk[base + i];"),
    ("bwd_final_state_gradient_ignored", "if (job->d_sf)\n        memcpy(G,", "if (0)\n        memcpy(G,"),
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
