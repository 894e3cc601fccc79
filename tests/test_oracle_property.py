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


@settings(max_examples=40, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(tiny_layers(), st.integers(1, 5), st.integers(0, 2))
def test_prefill_then_decode_equals_longer_prefill(case, n, extra_cap):
    """T0 prefilled tokens with their cache, then n decode steps, reproduce the
    last n rows of one prefill over T0 + n tokens, and leave the same SSM
    state and conv tail (ring capacity = window, or a little more; a global
    layer's cache holds every token)."""
    s, seed = case
    T0 = s.T
    sl = synth.with_(s, T=T0 + n)
    p = synth.make_layer_inputs(sl, seed)
    cap = s.window + extra_cap if s.window > 0 else T0 + n
    s0 = synth.with_(sl, T=T0)
    cache = ref.layer_fwd(p, p["Xt"][:, : s0.L], s0, cache_cap=cap)["cache"]
    sd = synth.with_(sl, T=1)
    ys = []
    for i in range(n):
        r = ref.layer_decode(p, p["Xt"][:, s0.L + i], cache, sd)
        ys.append(r["y"])
        cache = r["cache"]
    full = ref.layer_fwd(p, p["Xt"], sl, cache_cap=cap)
    scale = max(1.0, np.abs(full["Y"]).max())
    np.testing.assert_allclose(np.stack(ys, 1), full["Y"][:, s.M + T0:], rtol=1e-11, atol=1e-11 * scale)
    np.testing.assert_allclose(cache["ssm_state"], full["cache"]["ssm_state"], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(cache["conv_state"], full["cache"]["conv_state"], rtol=1e-13, atol=1e-15)
    assert np.all(cache["pos"] == T0 + n)
