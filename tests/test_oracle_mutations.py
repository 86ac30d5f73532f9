"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle's C source to a temporary directory, plants one
mistake by a textual replacement, compiles the copy, points the oracle wrapper
at it and runs the pins of ``test_oracle_pins``; at least one pin has to
fail.  The committed oracle is never modified.
"""
import ctypes
import os
import shutil
import subprocess

import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kla_oracle.c")

MUTATIONS = {
    "no_decay": ("for (int64_t i = 0; i < dk * dv; ++i) S[i] = a * S[i];",
                 "for (int64_t i = 0; i < dk * dv; ++i) S[i] = S[i];"),
    "norm_not_squared": ("kk += kt[i] * kt[i];", "kk += fabs(kt[i]);"),
    "eps_outside_denominator": ("J->eta[tok] / (kk + J->eps)", "J->eta[tok] / kk + J->eps"),
    "update_sign": ("S[i * dv + j] += bk * x[j];", "S[i * dv + j] -= bk * x[j];"),
    "residual_from_undecayed_state": ("x[j] = vt[j] - x[j];", "x[j] = vt[j] - x[j] / a;"),
    "readout_with_key": ("ot[j] += S[i * dv + j] * qt[i];", "ot[j] += S[i * dv + j] * kt[i];"),
    "eta_ignored": ("beta = J->eta[tok] / (kk + J->eps);",
                    "beta = 1.0 / (kk + J->eps);"),
    "direct_beta_normalised": ("if (!(J->flags & KLA_ORACLE_BETA_DIRECT)) {", "if (1) {"),
    "direct_beta_flag_inverted": ("if (!(J->flags & KLA_ORACLE_BETA_DIRECT)) {",
                                  "if (J->flags & KLA_ORACLE_BETA_DIRECT) {"),
}

PINS = [
    pins.test_golden_hand_two_tokens,
    lambda: pins.test_projection_constraint_each_step("decay_only"),
    pins.test_relaxation_residual,
    pins.test_beta_zero_closed_form,
    lambda: pins.test_no_erase_equals_masked_attention(True),
    lambda: pins.test_normalised_sgd_step(0.37),
    pins.test_direct_beta_hand_worked_two_tokens,
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    # the mistakes are planted in the forward loop only (the reverse mode, after
    # the marker, recomputes the forward with its own copy of these lines)
    cut = src.index("/* Reverse mode.")
    fwd, rest = src[:cut], src[cut:]
    assert fwd.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "kla_oracle_mut.c"
    mutated.write_text(fwd.replace(old, new) + rest)
    so = tmp_path / "libmut.so"
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-o", str(so), str(mutated), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    real = oracle._load()
    lib.kla_oracle_forward.argtypes = real.kla_oracle_forward.argtypes
    lib.kla_oracle_forward.restype = ctypes.c_int
    monkeypatch.setattr(oracle, "_lib", lib)
    failures = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {name!r}"
