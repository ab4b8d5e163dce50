"""The oracle's pins catch plausible mistakes: the oracle is rebuilt with one
planted error at a time (on the CPU) and at least one pin must fail."""
import os
import tempfile

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

MUTATIONS = {
    1: "decay on value rows instead of key columns",
    2: "output read before the rank-one write",
    3: "wrong sign of the gate",
    4: "epsilon outside the square root",
    5: "dk misses the residual's S'^T dr term",
    6: "adjoint not decayed between steps",
    7: "sigmoid derivative s instead of s(1-s)",
    8: "dA_log without the exp(A_log) factor",
    9: "L2-norm chain without the projection",
    10: "residual with a wrong (transposed) state term",
    11: "grouped value heads mapped to query/key heads round robin",
}

PIN_TESTS = [
    lambda: pins.test_backward_matches_central_differences((4,), 1),
    lambda: pins.test_core_backward_matches_central_differences(),
    pins.test_single_token_closed_form,
    pins.test_single_token_zero_state_gradients,
    pins.test_reduces_to_linear_attention,
    pins.test_beta_zero_is_pure_decay,
    pins.test_decay_acts_on_key_channels,
    pins.test_delta_rule_exact_association,
    pins.test_euler_identity_in_v_and_h0,
    pins.test_parameter_gradient_identities,
    pins.test_l2_norm_invariances,
    lambda: pins.test_chunk_form_equals_recurrence(16),
    pins.test_grouped_heads_equal_repeated_query_key_heads,
    pins.test_grouped_heads_central_differences,
]


def _caught():
    for t in PIN_TESTS:
        try:
            t()
        except (AssertionError, FloatingPointError):
            return True
    return False


@pytest.mark.parametrize("m", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(m):
    d = tempfile.mkdtemp(prefix="kda_oracle_mut")
    lib = oracle.build(mutation=m, out=os.path.join(d, f"libkda_oracle_m{m}.so"))
    oracle.use_library(lib)
    try:
        assert _caught(), f"no pin caught mutation {m}: {MUTATIONS[m]}"
    finally:
        oracle.use_library(None)


def test_unmutated_build_passes_all_pins():
    d = tempfile.mkdtemp(prefix="kda_oracle_mut")
    oracle.use_library(oracle.build(mutation=0, out=os.path.join(d, "libkda_oracle_m0.so")))
    try:
        assert not _caught()
    finally:
        oracle.use_library(None)
