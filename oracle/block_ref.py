"""Float64 CPU oracle of the full residual block around the hybrid-head layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module; the product never
calls it and shares no code with it.

The Hymba pages describe the block only loosely (no FFN sizes, no norm
placement).  The plainest reading, taken from the residual pattern the pages
give for the hybrid models they compare against ("Griffin: Mixing Gated Linear
Recurrences with Local Attention for Efficient Language Models", section 2.1
Residual block and section 2.2 MLP block):

* section 2.1: two sub-blocks in order, each pre-normalised and added back to
  the stream:  x = x + Mix(RMSNorm(x));  x = x + MLP(RMSNorm(x)).
  Mix is the hybrid-head layer (no residual of its own).
* section 2.2: gated MLP -- two branches D -> F (F = 3 D, expansion 3), GeLU on
  one branch, elementwise product, and a linear layer back to D.

Further readings (also listed in the design notes):

1.  RMSNorm with a learned per-channel weight: x / sqrt(mean(x^2) + eps) * w,
    eps the layer's eps (1e-6).
2.  GeLU is the exact form x * Phi(x), Phi the standard normal CDF.
3.  The sub-blocks' inputs are stored in bf16 (round to nearest even), the
    type of the hybrid-head layer's input X~; the residual stream is fp32.
4.  The meta rows are part of the sequence like any other row (the stream
    X~ = [meta | tokens] enters the first block).
"""
from __future__ import annotations

from typing import Dict, List

import numpy as np
from scipy.special import erf

from oracle import hymba_ref as hr

F = np.float64


round_bf16 = hr.round_bf16


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of each row with a learned weight (Griffin page, section 2.1)."""
    x = np.asarray(x, F)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(w, F)


def gelu(v: np.ndarray) -> np.ndarray:
    """GeLU(v) = v * Phi(v), Phi(v) = (1 + erf(v / sqrt 2)) / 2 (Griffin page,
    section 2.2: the non-linearity on one branch of the gated MLP)."""
    v = np.asarray(v, F)
    return v * 0.5 * (1.0 + erf(v / np.sqrt(2.0)))


def gated_mlp(x: np.ndarray, W_gate: np.ndarray, W_up: np.ndarray, W_down: np.ndarray) -> np.ndarray:
    """Griffin page, section 2.2: GeLU(x W_gate^T) * (x W_up^T), then W_down."""
    x = np.asarray(x, F)
    return (gelu(x @ np.asarray(W_gate, F).T) * (x @ np.asarray(W_up, F).T)) @ np.asarray(W_down, F).T


def block_fwd(pb: Dict[str, np.ndarray], X: np.ndarray, s) -> Dict[str, np.ndarray]:
    """One residual block on the stream X [B, L, d] (Griffin page, section 2.1).

    ``pb`` holds the hybrid-head layer's parameters plus norm1, norm2 [d],
    W_gate, W_up [F, d] and W_down [d, F].  ``s`` is the layer's shape with
    residual off (the block adds the stream itself).  Returns the stream after
    the mixer sub-block (Y1) and after the MLP sub-block (Y).
    """
    assert not s.residual
    X = np.asarray(X, F)
    xn = round_bf16(rmsnorm(X, pb["norm1"], s.eps))
    Y1 = X + hr.layer_fwd(pb, xn, s)["Y"]
    hn = round_bf16(rmsnorm(Y1, pb["norm2"], s.eps))
    Y = Y1 + gated_mlp(hn, pb["W_gate"], pb["W_up"], pb["W_down"])
    return {"Y1": Y1, "Y": Y}


def block_fwd_rows(pb: Dict[str, np.ndarray], X: np.ndarray, s, rows) -> np.ndarray:
    """The block's output Y at the rows ``rows`` only, for sequences too long
    for block_fwd.  The MLP sub-block and both norms act row by row, so row r
    needs only the mixer's output at r, which in turn needs only the causal
    prefix up to r (hymba_ref.layer_fwd_rows).  Returns [B, len(rows), d]."""
    assert not s.residual
    X = np.asarray(X, F)
    rows = np.asarray(rows)
    n = int(rows.max()) + 1
    xn = round_bf16(rmsnorm(X[:, :n], pb["norm1"], s.eps))
    Y1 = X[:, rows] + hr.layer_fwd_rows(pb, xn, s, rows)
    hn = round_bf16(rmsnorm(Y1, pb["norm2"], s.eps))
    return Y1 + gated_mlp(hn, pb["W_gate"], pb["W_up"], pb["W_down"])


def blocks_fwd(blocks: List[Dict[str, np.ndarray]], X: np.ndarray, shapes) -> np.ndarray:
    """A stack of residual blocks; each block's input is the previous output."""
    Y = np.asarray(X, F)
    for pb, s in zip(blocks, shapes):
        Y = block_fwd(pb, Y, s)["Y"]
    return Y
