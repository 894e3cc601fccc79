"""Seeded synthetic inputs for the Hymba hybrid-head layer workloads.

This module only draws random numbers and rounds them to the storage type.  It
holds none of the layer's arithmetic, so both the float64 oracle (``oracle/``)
and the CUDA path can be fed from it without sharing any computation.

Recipe (one generator per workload, ``numpy.random.default_rng(seed)``, PCG64),
drawn in this fixed order:

    X [B,T,d], meta [M,d], then per layer: W_in, W_out, W_x, W_dt, conv_w,
    A_log, dt0; then (decode workloads only) the carried cache.

* X, meta, ring/meta K/V, ssm_state, conv_state ~ N(0, 1).
* Every projection matrix and conv_w ~ N(0, 0.02^2).
* A_log = ln U[1, 16]  (so A = -exp(A_log) lies in [-16, -1]).
* dt0 = exp(U[ln 1e-3, ln 1e-1]); dt_bias is its inverse softplus, so that
  softplus(dt_bias) = dt0 lies in [1e-3, 1e-1] when the projection is zero.
* conv_b = 0, D = 1, beta1 = beta2 = 1.

For bf16 workloads the matrices, X and meta are rounded to bf16
(round-to-nearest-even) here; fp32 vectors stay fp32.  The oracle receives the
same rounded values widened to float64, so both sides see identical inputs.

Hymba's meta tokens are learned, input-independent embeddings prepended to
every sequence ("Hymba: A Hybrid-head Architecture for Small Language Models",
section 2.3); the M meta rows are therefore drawn once and broadcast over the
batch to form X~ = [meta; X].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Dict, List, Optional

import numpy as np

# ---------------------------------------------------------------------------
# shapes
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class LayerShape:
    """Shape and flags of one hybrid-head layer call (symbols as in the paper)."""

    B: int          # batch
    T: int          # real tokens per sequence
    M: int          # meta tokens (prefix rows of X~)
    d: int          # d_model
    Hq: int         # query heads
    Hkv: int        # key/value heads (GQA groups)
    dh: int         # query/key head dim
    dv: int         # value head dim (Hq * dv == di so both branches are di wide)
    di: int         # SSM inner width
    N: int          # SSM state size
    k: int          # conv width
    R: int          # dt rank
    window: int     # sliding window in keys incl. self; 0 = global
    kv_shared: bool = False
    residual: bool = False
    rope_theta: float = 0.0   # 0 disables RoPE
    eps: float = 1e-6
    dtype: str = "bf16"       # "bf16" or "f32"
    fusion: str = "sum"       # "sum" (eq. 3) or "concat" (the ablation: W_out is [d, 2 di])

    @property
    def L(self) -> int:
        return self.M + self.T

    @property
    def P_in(self) -> int:
        kv = 0 if self.kv_shared else self.Hkv * (self.dh + self.dv)
        return self.Hq * self.dh + kv + 2 * self.di

    @property
    def xproj_out(self) -> int:
        return self.R + 2 * self.N


def dt_rank(d: int) -> int:
    return -(-d // 16)


def _shape(B, T, M, d, Hq, Hkv, dh, di, N, k, window, dtype, **kw) -> LayerShape:
    return LayerShape(B=B, T=T, M=M, d=d, Hq=Hq, Hkv=Hkv, dh=dh, dv=di // Hq, di=di,
                      N=N, k=k, R=dt_rank(d), window=window, dtype=dtype, **kw)


def tiny_f32(**kw) -> LayerShape:
    """Tiny single layer, fp32: batch 1, 64 tokens + 16 meta, d 64, 2/1 heads of 16."""
    base = dict(B=1, T=64, M=16, d=64, Hq=2, Hkv=1, dh=16, di=128, N=8, k=4,
                window=32, dtype="f32")
    base.update(kw)
    return _shape(**base)


def hymba15b_swa(**kw) -> LayerShape:
    """Hymba-1.5B-shaped SWA layer: batch 8, 8192 tokens + 128 meta, window 1024."""
    base = dict(B=8, T=8192, M=128, d=1600, Hq=25, Hkv=5, dh=64, di=3200, N=16, k=4,
                window=1024, dtype="bf16")
    base.update(kw)
    return _shape(**base)


def hymba15b_global(**kw) -> LayerShape:
    """Same shapes as the SWA layer but global attention, batch 2."""
    base = dict(B=2, T=8192, M=128, d=1600, Hq=25, Hkv=5, dh=64, di=3200, N=16, k=4,
                window=0, dtype="bf16")
    base.update(kw)
    return _shape(**base)


def ablation300m_stack(B=32, T=2048, M=128, **kw) -> List[LayerShape]:
    """300M-ablation-shaped 4-layer stack: layer 0 global, 1-3 window 1024,
    layer 2 reuses layer 1's K/V; residual stream X_{l+1} = X_l + Y_l."""
    out = []
    for layer in range(4):
        base = dict(B=B, T=T, M=M, d=1024, Hq=16, Hkv=4, dh=64, di=2048, N=16, k=4,
                    window=0 if layer == 0 else 1024, dtype="bf16",
                    kv_shared=(layer == 2), residual=True)
        base.update(kw)
        out.append(_shape(**base))
    return out


def hymba15b_decode(**kw) -> LayerShape:
    """Decode step on the 1.5B shapes: batch 128, one token, 8192 cached tokens."""
    base = dict(B=128, T=1, M=128, d=1600, Hq=25, Hkv=5, dh=64, di=3200, N=16, k=4,
                window=1024, dtype="bf16")
    base.update(kw)
    return _shape(**base)


# ---------------------------------------------------------------------------
# rounding
# ---------------------------------------------------------------------------


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    r = ((u + bias) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bf16-representable."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def store_round(a: np.ndarray, dtype: str) -> np.ndarray:
    a = np.asarray(a, dtype=np.float32)
    return bf16_round(a) if dtype == "bf16" else a


# ---------------------------------------------------------------------------
# draws
# ---------------------------------------------------------------------------


def _normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def draw_layer_params(rng: np.random.Generator, s: LayerShape) -> Dict[str, np.ndarray]:
    """One layer's parameters in the documented draw order.

    Matrices are rounded to the storage dtype; vectors are float32.
    W_in rows are ordered [Q (Hq*dh) | K (Hkv*dh) | V (Hkv*dv) | x (di) | z (di)];
    a KV-sharing layer has no K/V rows.
    """
    p: Dict[str, np.ndarray] = {}
    p["W_in"] = store_round(_normal(rng, (s.P_in, s.d), 0.02), s.dtype)
    p["W_out"] = store_round(_normal(rng, (s.d, s.di * (2 if s.fusion == "concat" else 1)), 0.02), s.dtype)
    p["W_x"] = store_round(_normal(rng, (s.xproj_out, s.di), 0.02), s.dtype)
    p["W_dt"] = store_round(_normal(rng, (s.di, s.R), 0.02), s.dtype)
    p["conv_w"] = _normal(rng, (s.di, s.k), 0.02)
    p["A_log"] = np.log(rng.uniform(1.0, 16.0, size=(s.di, s.N))).astype(np.float32)
    dt0 = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=(s.di,)))
    # inverse softplus of dt0 (float64 then stored as float32)
    p["dt_bias"] = (dt0 + np.log(-np.expm1(-dt0))).astype(np.float32)
    p["conv_b"] = np.zeros((s.di,), np.float32)
    p["D"] = np.ones((s.di,), np.float32)
    p["beta1"] = np.ones((s.di,), np.float32)
    p["beta2"] = np.ones((s.di,), np.float32)
    return p


def draw_block_params(rng: np.random.Generator, s: LayerShape, F: int) -> Dict[str, np.ndarray]:
    """One residual block: the hybrid-head layer's parameters, then norm1,
    norm2 [d] (1 + N(0, 0.1^2)), W_gate, W_up [F, d] ~ N(0, 1/d) and W_down
    [d, F] ~ N(0, 1/F), matrices rounded to the storage dtype."""
    p = draw_layer_params(rng, s)
    p["norm1"] = (1.0 + _normal(rng, (s.d,), 0.1)).astype(np.float32)
    p["norm2"] = (1.0 + _normal(rng, (s.d,), 0.1)).astype(np.float32)
    p["W_gate"] = store_round(_normal(rng, (F, s.d), 1.0 / math.sqrt(s.d)), s.dtype)
    p["W_up"] = store_round(_normal(rng, (F, s.d), 1.0 / math.sqrt(s.d)), s.dtype)
    p["W_down"] = store_round(_normal(rng, (s.d, F), 1.0 / math.sqrt(F)), s.dtype)
    return p


def make_block_inputs(s: LayerShape, F: int, seed: int, n_blocks: int = 1):
    """The stream X~ [B, L, d] and n_blocks blocks' parameters."""
    rng = np.random.default_rng(seed)
    tok = draw_tokens(rng, s)
    return tok, [draw_block_params(rng, s, F) for _ in range(n_blocks)]


def draw_tokens(rng: np.random.Generator, s: LayerShape) -> Dict[str, np.ndarray]:
    """X [B,T,d] and meta [M,d] (storage-rounded), plus X~ = [meta; X] [B,L,d]."""
    X = store_round(_normal(rng, (s.B, s.T, s.d)), s.dtype)
    meta = store_round(_normal(rng, (s.M, s.d)), s.dtype)
    Xt = np.empty((s.B, s.L, s.d), np.float32)
    Xt[:, : s.M] = meta[None]
    Xt[:, s.M:] = X
    return {"X": X, "meta": meta, "Xt": Xt}


def make_layer_inputs(s: LayerShape, seed: int) -> Dict[str, np.ndarray]:
    rng = np.random.default_rng(seed)
    out = draw_tokens(rng, s)
    out.update(draw_layer_params(rng, s))
    return out


def make_stack_inputs(shapes: List[LayerShape], seed: int):
    rng = np.random.default_rng(seed)
    tok = draw_tokens(rng, shapes[0])
    layers = [draw_layer_params(rng, s) for s in shapes]
    return tok, layers


def draw_decode_cache(rng: np.random.Generator, s: LayerShape, cap: int,
                      pos: int) -> Dict[str, np.ndarray]:
    """Random carried state for a decode step: ring K/V, meta K/V, SSM state,
    conv tail and per-sequence positions (all sequences at ``pos``)."""
    c: Dict[str, np.ndarray] = {}
    c["k_ring"] = store_round(_normal(rng, (s.B, cap, s.Hkv, s.dh)), s.dtype)
    c["v_ring"] = store_round(_normal(rng, (s.B, cap, s.Hkv, s.dv)), s.dtype)
    c["k_meta"] = store_round(_normal(rng, (s.M, s.Hkv, s.dh)), s.dtype)
    c["v_meta"] = store_round(_normal(rng, (s.M, s.Hkv, s.dv)), s.dtype)
    c["ssm_state"] = _normal(rng, (s.B, s.di, s.N))
    c["conv_state"] = _normal(rng, (s.B, s.di, s.k - 1))
    c["pos"] = np.full((s.B,), pos, np.int32)
    return c


def make_decode_inputs(s: LayerShape, seed: int, cap: Optional[int] = None,
                       pos: int = 8192) -> Dict[str, np.ndarray]:
    """x_new [B,d], layer parameters and a random cache, in the documented order."""
    assert s.T == 1
    rng = np.random.default_rng(seed)
    tok = draw_tokens(rng, s)
    out = {"x_new": tok["X"][:, 0, :].copy()}
    out.update(draw_layer_params(rng, s))
    cap = cap if cap is not None else (s.window if s.window > 0 else pos + 1)
    out.update(draw_decode_cache(rng, s, cap, pos))
    return out


def with_(s: LayerShape, **kw) -> LayerShape:
    return replace(s, **kw)
