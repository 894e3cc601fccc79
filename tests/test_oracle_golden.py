"""The vectorised oracle reproduces the stored loop-oracle values of two tiny
layers (tests/golden/, written by tests/golden/make_golden.py from oracle.brute)."""
import os

import numpy as np
import pytest

from hybrid_attention_ssm_fwd_b300 import synth
from oracle import hymba_ref as ref
from tests.golden.make_golden import CASES, golden_shape

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("name", sorted(CASES))
def test_vectorised_oracle_matches_golden(name):
    s = golden_shape(**CASES[name])
    p = synth.make_layer_inputs(s, 11)
    want = np.loadtxt(os.path.join(HERE, f"tiny_layer_{name}.txt"))
    got = ref.layer_fwd(p, p["Xt"], s)["Y"][0]
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)
