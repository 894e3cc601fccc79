"""Pins of the residual-block oracle (oracle/block_ref.py) against library
routines, tabulated values, brute-force loops and the identities its
definition implies.  Source: "Griffin: Mixing Gated Linear Recurrences with
Local Attention for Efficient Language Models", section 2.1 (residual block:
x = x + Mix(RMSNorm(x)); x = x + MLP(RMSNorm(x))) and section 2.2 (gated MLP,
GeLU on one branch, expansion 3)."""
import math

import numpy as np
import scipy.integrate
import torch

from hybrid_attention_ssm_fwd_b300 import synth
from oracle import block_ref as br
from oracle import hymba_ref as ref

F = np.float64


def test_round_bf16_matches_torch_and_ties_to_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.uniform(-6, 6, 5000),
                        [0.0, -0.0, 1.0, 65504.0, 3.0e38, 1e-40]])
    ref_t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy().astype(F)
    np.testing.assert_array_equal(br.round_bf16(x), ref_t)
    # exactly halfway between two bf16 values: to the even mantissa
    assert br.round_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert br.round_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6


def test_rmsnorm_unit_rms_scale_invariance_and_weight():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 300)) * 3.0
    w = np.ones(300)
    y = br.rmsnorm(x, w, 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, -1)), 1.0, rtol=1e-12)
    np.testing.assert_allclose(br.rmsnorm(7.5 * x, w, 0.0), y, rtol=1e-12)
    w2 = rng.uniform(0.5, 2.0, 300)
    np.testing.assert_allclose(br.rmsnorm(x, w2, 0.0), y * w2, rtol=1e-12)
    # a constant row c maps to sign(c) * w; eps shrinks it by sqrt(c^2 / (c^2 + eps))
    c = np.full((1, 10), -2.0)
    np.testing.assert_allclose(br.rmsnorm(c, np.ones(10), 1e-6), -np.sqrt(4.0 / (4.0 + 1e-6)), rtol=1e-14)


def test_gelu_values_and_odd_part():
    # Phi(1) = 0.8413447460685429 (standard normal table); GeLU(1) = Phi(1)
    assert abs(br.gelu(np.array([1.0]))[0] - 0.8413447460685429) < 1e-15
    assert br.gelu(np.array([0.0]))[0] == 0.0
    x = np.linspace(-6, 6, 121)
    # Phi(x) + Phi(-x) = 1  =>  GeLU(x) - GeLU(-x) = x
    np.testing.assert_allclose(br.gelu(x) - br.gelu(-x), x, atol=1e-14)
    # against the CDF by numerical integration of the normal density
    for v in (-2.5, -0.3, 0.7, 3.1):
        phi, _ = scipy.integrate.quad(lambda t: math.exp(-t * t / 2) / math.sqrt(2 * math.pi), -np.inf, v)
        assert abs(br.gelu(np.array([v]))[0] - v * phi) < 1e-12


def test_gated_mlp_matches_loops():
    rng = np.random.default_rng(2)
    d, Fh, rows = 5, 7, 3
    x = rng.standard_normal((rows, d))
    Wg, Wu, Wd = rng.standard_normal((Fh, d)), rng.standard_normal((Fh, d)), rng.standard_normal((d, Fh))
    out = np.zeros((rows, d))
    for r in range(rows):
        hid = []
        for f in range(Fh):
            a = sum(x[r, i] * Wg[f, i] for i in range(d))
            b = sum(x[r, i] * Wu[f, i] for i in range(d))
            hid.append(a * 0.5 * (1.0 + math.erf(a / math.sqrt(2.0))) * b)
        for o in range(d):
            out[r, o] = sum(hid[f] * Wd[o, f] for f in range(Fh))
    np.testing.assert_allclose(br.gated_mlp(x, Wg, Wu, Wd), out, rtol=1e-12, atol=1e-12)
    # a zero gate switches the MLP off; scaling W_down scales its output
    assert np.all(br.gated_mlp(x, 0 * Wg, Wu, Wd) == 0)
    np.testing.assert_allclose(br.gated_mlp(x, Wg, Wu, 3 * Wd), 3 * br.gated_mlp(x, Wg, Wu, Wd), rtol=1e-12)


def _block_case(seed=3):
    s = synth.tiny_f32(B=2, T=40, M=8, window=16)
    tok, blocks = synth.make_block_inputs(s, 3 * s.d, seed)
    return s, tok, blocks[0]


def test_block_composition():
    s, tok, pb = _block_case()
    X = tok["Xt"].astype(F)
    out = br.block_fwd(pb, X, s)
    # the mixer sub-block is the layer on the normalised, bf16-stored stream
    xn = br.round_bf16(br.rmsnorm(X, pb["norm1"], s.eps))
    np.testing.assert_allclose(out["Y1"], X + ref.layer_fwd(pb, xn, s)["Y"], rtol=1e-13, atol=1e-13)
    # the MLP sub-block adds the gated MLP of the normalised Y1
    hn = br.round_bf16(br.rmsnorm(out["Y1"], pb["norm2"], s.eps))
    mlp = br.gated_mlp(hn, pb["W_gate"], pb["W_up"], pb["W_down"])
    np.testing.assert_allclose(out["Y"], out["Y1"] + mlp, rtol=1e-13, atol=1e-13)


def test_block_rows_matches_whole_block():
    """The row-sampled block oracle (for sequences too long for block_fwd)
    reproduces the whole block's rows: meta rows, the first real row, both
    sides of the window edge, the last row, and a prefix that stops early."""
    s, tok, pb = _block_case(6)
    X = tok["Xt"].astype(F)
    Y = br.block_fwd(pb, X, s)["Y"]
    for rows in ([0, s.M - 1, s.M, s.M + 15, s.M + 16, s.L - 1], [1, 2, 3], [s.L - 1]):
        rows = np.array(rows)
        np.testing.assert_allclose(br.block_fwd_rows(pb, X, s, rows), Y[:, rows], rtol=1e-12,
                                   atol=1e-12 * np.abs(Y).max())


def test_block_with_zeroed_sub_blocks():
    s, tok, pb = _block_case(4)
    X = tok["Xt"].astype(F)
    q = dict(pb)
    q["W_out"] = np.zeros_like(pb["W_out"])      # mixer contributes nothing
    q["W_gate"] = np.zeros_like(pb["W_gate"])    # GeLU(0) = 0: MLP contributes nothing
    out = br.block_fwd(q, X, s)
    np.testing.assert_array_equal(out["Y"], X)
    # each sub-block alone moves the stream by its own term only
    q = dict(pb)
    q["W_gate"] = np.zeros_like(pb["W_gate"])
    out = br.block_fwd(q, X, s)
    np.testing.assert_array_equal(out["Y"], out["Y1"])
    assert np.abs(out["Y1"] - X).max() > 1e-3


def test_blocks_stack_is_composition():
    s = synth.tiny_f32(B=1, T=24, M=8, window=8)
    tok, blocks = synth.make_block_inputs(s, 3 * s.d, 5, n_blocks=2)
    X = tok["Xt"].astype(F)
    Y2 = br.blocks_fwd(blocks, X, [s, s])
    np.testing.assert_allclose(Y2, br.block_fwd(blocks[1], br.block_fwd(blocks[0], X, s)["Y"], s)["Y"], rtol=1e-14)
