"""Property tests of the float64 oracle over random tiny layers.

The vectorised oracle (blocked attention over the visible keys, whole-batch
NumPy) and the loop-only oracle (explicit Python loops over rows, heads, keys,
channels and states) are written independently from the same definition
("Hymba: A Hybrid-head Architecture for Small Language Models", section 2.1
eq. (3), sections 2.2-2.3 for the mask, meta rows and KV sharing).  Here they
must agree on shapes drawn at random: meta lengths including none, windows
from one key to past the sequence, grouped and plain multi-head attention,
conv widths 2-4, with and without RoPE and the residual.  The row-sampled
oracle must reproduce the whole layer's rows.
"""
import numpy as np
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

from hybrid_attention_ssm_fwd_b300 import synth
from oracle import brute
from oracle import hymba_ref as ref


@st.composite
def tiny_layers(draw):
    B = draw(st.integers(1, 2))
    T = draw(st.integers(1, 9))
    M = draw(st.integers(0, 5))
    Hkv = draw(st.sampled_from([1, 2]))
    Hq = Hkv * draw(st.sampled_from([1, 2, 3]))
    dh = draw(st.sampled_from([2, 4, 8]))
    dv = draw(st.sampled_from([2, 4]))
    d = draw(st.sampled_from([8, 16, 24]))
    N = draw(st.integers(1, 4))
    k = draw(st.integers(2, 4))
    window = draw(st.integers(0, M + T + 2))
    rope = draw(st.sampled_from([0.0, 100.0]))
    residual = draw(st.booleans())
    seed = draw(st.integers(0, 2**16))
    s = synth.LayerShape(B=B, T=T, M=M, d=d, Hq=Hq, Hkv=Hkv, dh=dh, dv=dv, di=Hq * dv, N=N, k=k,
                         R=synth.dt_rank(d), window=window, residual=residual, rope_theta=rope, dtype="f32")
    return s, seed


@settings(max_examples=60, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(tiny_layers())
def test_vectorised_oracle_equals_loop_oracle(case):
    s, seed = case
    p = synth.make_layer_inputs(s, seed)
    y = ref.layer_fwd(p, p["Xt"], s)["Y"]
    yb = np.array(brute.layer_fwd(p, p["Xt"], s)["Y"])
    np.testing.assert_allclose(y, yb, rtol=1e-11, atol=1e-11 * max(1.0, np.abs(yb).max()))


@settings(max_examples=40, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(tiny_layers(), st.data())
def test_row_sampled_oracle_equals_whole_layer(case, data):
    s, seed = case
    p = synth.make_layer_inputs(s, seed)
    y = ref.layer_fwd(p, p["Xt"], s)["Y"]
    rows = np.array(sorted(data.draw(st.sets(st.integers(0, s.L - 1), min_size=1, max_size=s.L))))
    np.testing.assert_allclose(ref.layer_fwd_rows(p, p["Xt"], s, rows), y[:, rows], rtol=1e-12,
                               atol=1e-12 * max(1.0, np.abs(y).max()))
