"""The oracle's pins must be able to fail.

Each case plants one plausible slip in a private copy of oracle/fa_ref.c,
compiles it on the CPU, swaps it in for the real oracle and checks that at
least one pin of test_oracle_pins rejects it.  Nothing here touches a GPU.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

MUTANTS = {
    "dropped_D": ("ds[j] = p[j] * (dpij - Di);", "ds[j] = p[j] * dpij;"),
    "dq_sign": ("dq[c] += scale * ds[j] * k[c];", "dq[c] -= scale * ds[j] * k[c];"),
    "dv_wrong_operand": ("dv[c] += p[j] * g_o[c];", "dv[c] += p[j] * q[c];"),
    "dk_missing_scale": ("dk[c] += scale * ds[j] * q[c];", "dk[c] += ds[j] * q[c];"),
    "causal_off_by_one": ("return j <= p;", "return j < p;"),
    "causal_top_left": ("const long p = i + (long)(S_k - S_q);", "const long p = i;"),
    "window_off_by_one": ("p - j >= window ||", "p - j > window ||"),
    "window_one_sided": ("(p - j >= window || (!causal && j - p >= window))", "(p - j >= window)"),
    "group_interleaved": ("for (int h = hk * g; h < (hk + 1) * g; ++h)\n                for (int i = 0; i < S_q; ++i) {\n                    const double* q",
                          "for (int h = hk; h < H; h += H_kv)\n                for (int i = 0; i < S_q; ++i) {\n                    const double* q"),
    "lse_ignored": ("p[j] = exp(sij - lse);", "p[j] = exp(sij);"),
    "D_wrong_vector": ("const double Di = dot(g_o, o, d);", "const double Di = dot(g_o, g_o, d);"),
    "dq_rows_no_scale": ("for (int c = 0; c < d; ++c) dq[c] += scale * dsij * k[c];",
                         "for (int c = 0; c < d; ++c) dq[c] += dsij * k[c];"),
    "dkv_rows_wrong_group": ("for (int h = hk * g; h < (hk + 1) * g; ++h)\n            for (int i = 0; i < S_q; ++i) {\n                if (!allowed(i, j",
                             "for (int h = hk; h < hk + 1; ++h)\n            for (int i = 0; i < S_q; ++i) {\n                if (!allowed(i, j"),
    "preprocess_wrong": ("D[r] = dot(dO + (size_t)r * d, O + (size_t)r * d, d);",
                         "D[r] = dot(dO + (size_t)r * d, dO + (size_t)r * d, d);"),
}

PIN_CALLS = [
    lambda: [pins.test_bwd_matches_torch_autograd(s) for s in pins.SHAPES],
    lambda: [pins.test_fwd_matches_torch_sdpa(s) for s in pins.SHAPES],
    lambda: pins.test_bwd_matches_finite_differences((1, 4, 2, 5, 5, 8, False)),
    lambda: pins.test_bwd_matches_finite_differences((1, 2, 1, 3, 3, 4, True)),
    lambda: pins.test_preprocess_equals_sum_p_dp(),
    lambda: pins.test_gqa_is_sum_over_group(True),
    lambda: pins.test_sampled_rows_match_full_backward(True),
    lambda: pins.test_sampled_rows_match_full_backward(False),
    lambda: [pins.test_window_matches_torch_sdpa_band(s) for s in pins.WSHAPES],
    lambda: pins.test_window_single_query_is_trailing_slice(True),
    lambda: pins.test_window_noncausal_first_row_is_leading_slice(),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path, monkeypatch):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "fa_ref.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(path), "-o", str(so), "-lm"],
                   check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.open_library(str(so)))
    caught = 0
    for call in PIN_CALLS:
        try:
            call()
        except AssertionError:
            caught += 1
    assert caught >= 1, f"no pin rejects mutant {name}"
