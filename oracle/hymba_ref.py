"""Float64 CPU oracle of Hymba's fused hybrid-head layer (forward and decode step).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The product (the CUDA
library and its binding) never calls it, and it shares no code with it.

Source: "Hymba: A Hybrid-head Architecture for Small Language Models" (Dong et
al., 2024), as summarised on the web pages about it:

* section 2.1, eq. (3): one shared input projection yields the attention Q/K/V,
  the SSM input and the output gate; each branch is normalised and scaled by a
  learnable per-channel vector, then summed and projected:
      Y = W_out( beta1 * norm(M_attn X~) + beta2 * norm(M_ssm X~) ).
* section 2.2: sliding-window attention in most layers, global attention in
  the first/middle/last; consecutive layers can share K and V.
* section 2.3: 128 learned meta tokens are prepended to every sequence and act
  as a learned initial attention cache and SSM state.
* section 2.5 / Table 11: local window 1024, SSM state 16; RoPE base changed
  for context extension (the base itself is not given).

The pages give no SSM equations, norm type or tensor layout.  The readings
used here (each also listed in the design notes):

1.  norm = RMSNorm over the full di-wide row, eps 1e-6, with no weight of its
    own (beta1/beta2 are the per-channel scales).
2.  Both branches are di wide: V head dim dv = di / Hq, so the concatenated
    attention heads are di wide and one W_out follows the sum.
3.  SSM branch (Mamba-1 selective parametrisation): u = silu(causal depthwise
    conv1d(x) + b); [dtr | B | C] = u W_x^T; delta = softplus(dtr W_dt^T + b_dt);
    A = -exp(A_log);  h_t = exp(delta_t A) * h_{t-1} + delta_t B_t u_t;
    y_t = C_t . h_t + D * u_t;  g = y * silu(z).  Euler input term, no ZOH.
4.  Conv: width k, bias, zero left padding before row 0 (the first meta row).
5.  Attention: causal GQA, scale 1/sqrt(dh), query head h uses KV head
    floor(h * Hkv / Hq).  Visible keys of row i: j <= i and (window == 0 or
    i - j < window or j < M).  Meta keys are always visible to later rows,
    meta rows attend causally among themselves.
6.  RoPE (optional): rotate-half pairing, base theta, absolute positions
    0..L-1 counting the meta rows; K is cached after rotation.
7.  Fusion is the beta-weighted sum of eq. (3) (no 1/2 factor).
8.  Decode: the cache holds the last tokens' K/V in a ring of ``cap`` slots
    (slot = pos mod cap), meta K/V, the SSM state and the conv tail (the last
    k-1 pre-conv x rows).  The new token sits at absolute position M + pos.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Tuple

import numpy as np

F = np.float64


# ---------------------------------------------------------------------------
# elementwise pieces
# ---------------------------------------------------------------------------


def silu(v: np.ndarray) -> np.ndarray:
    """silu(v) = v * sigmoid(v), written without overflow for large |v|."""
    v = np.asarray(v, F)
    out = np.empty_like(v)
    pos = v >= 0
    out[pos] = v[pos] / (1.0 + np.exp(-v[pos]))
    e = np.exp(v[~pos])
    out[~pos] = v[~pos] * e / (1.0 + e)
    return out


def softplus(v: np.ndarray) -> np.ndarray:
    """softplus(v) = log(1 + e^v)."""
    return np.logaddexp(0.0, np.asarray(v, F))


def rms_norm(v: np.ndarray, eps: float) -> np.ndarray:
    """v / sqrt(mean(v^2) + eps) over the last axis (no weight: reading 1)."""
    v = np.asarray(v, F)
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps)


def rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE on the last axis (size dh) of x [..., P, H, dh].

    ``positions`` has the length of axis -3.  Pair (i, i + dh/2) is rotated by
    angle position * theta^(-2i/dh).
    """
    x = np.asarray(x, F)
    dh = x.shape[-1]
    half = dh // 2
    inv_freq = theta ** (-(np.arange(half, dtype=F) * 2.0) / dh)
    ang = np.asarray(positions, F)[:, None] * inv_freq[None, :]        # [P, half]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


# ---------------------------------------------------------------------------
# attention branch
# ---------------------------------------------------------------------------


def visible_mask(rows: np.ndarray, keys: np.ndarray, M: int, window: int) -> np.ndarray:
    """Boolean [len(rows), len(keys)]: key j visible to row i (reading 5)."""
    i = np.asarray(rows)[:, None]
    j = np.asarray(keys)[None, :]
    vis = j <= i
    if window > 0:
        vis &= (i - j < window) | (j < M)
    return vis


def attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, M: int, window: int,
              rows: Optional[np.ndarray] = None, block: int = 256) -> np.ndarray:
    """Causal GQA softmax attention with the meta-prefix / window mask.

    Q [B,L,Hq,dh], K [B,L,Hkv,dh], V [B,L,Hkv,dv] -> [B, R, Hq*dv] for the
    query rows ``rows`` (default: all L).  One query block at a time, over the
    keys that can be visible to that block; the max-subtracted softmax is
    mathematically the plain softmax.
    """
    Q, K, V = (np.asarray(a, F) for a in (Q, K, V))
    B, L, Hq, dh = Q.shape
    Hkv, dv = K.shape[2], V.shape[3]
    rows = np.arange(L) if rows is None else np.asarray(rows)
    out = np.zeros((B, len(rows), Hq * dv), F)
    scale = 1.0 / math.sqrt(dh)
    group = [(h * Hkv) // Hq for h in range(Hq)]
    for r0 in range(0, len(rows), block):
        rr = rows[r0:r0 + block]
        lo, hi = int(rr.min()), int(rr.max())
        keys = np.arange(0, hi + 1)
        if window > 0:
            keep = (keys < M) | (keys > lo - window)
            keys = keys[keep]
        mask = visible_mask(rr, keys, M, window)                       # [r, n]
        for h in range(Hq):
            g = group[h]
            q = Q[:, rr, h, :]                                         # [B, r, dh]
            k = K[:, keys, g, :]                                       # [B, n, dh]
            v = V[:, keys, g, :]
            s = np.einsum("brd,bnd->brn", q, k) * scale
            s = np.where(mask[None], s, -np.inf)
            s = s - s.max(axis=-1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(axis=-1, keepdims=True)
            out[:, r0:r0 + len(rr), h * dv:(h + 1) * dv] = np.einsum("brn,bnd->brd", p, v)
    return out


# ---------------------------------------------------------------------------
# SSM branch
# ---------------------------------------------------------------------------


def conv1d_silu(x: np.ndarray, w: np.ndarray, b: np.ndarray,
                tail: Optional[np.ndarray] = None) -> np.ndarray:
    """u_t = silu(sum_j w[c,j] x_{t-k+1+j} + b_c), zero left padding (reading 4).

    x [B,L,di], w [di,k], b [di].  ``tail`` [B,di,k-1] replaces the zero
    padding (oldest first), as a decode step uses it.
    """
    x = np.asarray(x, F)
    w = np.asarray(w, F)
    Bsz, L, di = x.shape
    k = w.shape[1]
    pad = np.zeros((Bsz, k - 1, di), F) if tail is None else np.transpose(np.asarray(tail, F), (0, 2, 1))
    xp = np.concatenate([pad, x], axis=1)                              # [B, L+k-1, di]
    acc = np.zeros((Bsz, L, di), F)
    for j in range(k):
        acc += w[None, None, :, j] * xp[:, j:j + L, :]
    return silu(acc + np.asarray(b, F))


def selective_scan(u: np.ndarray, delta: np.ndarray, A: np.ndarray, Bm: np.ndarray,
                   Cm: np.ndarray, D: np.ndarray, h0: Optional[np.ndarray] = None
                   ) -> Tuple[np.ndarray, np.ndarray]:
    """The recurrence run literally, one time step after another.

    u, delta [B,L,di]; A [di,N]; Bm, Cm [B,L,N]; D [di]; h0 [B,di,N] (zero if None).
        h_t = exp(delta_t * A) * h_{t-1} + (delta_t * u_t) * B_t
        y_t = C_t . h_t + D * u_t
    Returns y [B,L,di] and the final state h [B,di,N].
    """
    u, delta, A, Bm, Cm, D = (np.asarray(a, F) for a in (u, delta, A, Bm, Cm, D))
    Bsz, L, di = u.shape
    N = A.shape[1]
    h = np.zeros((Bsz, di, N), F) if h0 is None else np.array(h0, F)
    y = np.empty((Bsz, L, di), F)
    for t in range(L):
        dt = delta[:, t, :]                                            # [B, di]
        h = np.exp(dt[:, :, None] * A[None]) * h + (dt * u[:, t, :])[:, :, None] * Bm[:, t, None, :]
        y[:, t, :] = np.einsum("bcn,bn->bc", h, Cm[:, t, :]) + D[None] * u[:, t, :]
    return y, h


# ---------------------------------------------------------------------------
# the layer
# ---------------------------------------------------------------------------


def split_projection(proj: np.ndarray, s) -> Dict[str, np.ndarray]:
    """Split [.., P_in] into Q, K, V, x, z following the W_in row order."""
    o = 0
    out = {}
    lead = proj.shape[:-1]

    def take(n):
        nonlocal o
        a = proj[..., o:o + n]
        o += n
        return a

    out["Q"] = take(s.Hq * s.dh).reshape(*lead, s.Hq, s.dh)
    if not s.kv_shared:
        out["K"] = take(s.Hkv * s.dh).reshape(*lead, s.Hkv, s.dh)
        out["V"] = take(s.Hkv * s.dv).reshape(*lead, s.Hkv, s.dv)
    out["x"] = take(s.di)
    out["z"] = take(s.di)
    assert o == proj.shape[-1]
    return out


def ssm_branch(x: np.ndarray, z: np.ndarray, p: Dict[str, np.ndarray], s,
               tail: Optional[np.ndarray] = None, h0: Optional[np.ndarray] = None):
    """conv -> x_proj -> dt_proj/softplus -> selective scan -> gate.  Returns (g, h_final)."""
    u = conv1d_silu(x, p["conv_w"], p["conv_b"], tail)
    xdbl = u @ np.asarray(p["W_x"], F).T                                  # [B,L,R+2N]
    dtr = xdbl[..., : s.R]
    Bm = xdbl[..., s.R: s.R + s.N]
    Cm = xdbl[..., s.R + s.N:]
    delta = softplus(dtr @ np.asarray(p["W_dt"], F).T + np.asarray(p["dt_bias"], F))
    A = -np.exp(np.asarray(p["A_log"], F))
    y, h = selective_scan(u, delta, A, Bm, Cm, p["D"], h0)
    return y * silu(z), h


def fuse_and_project(att: np.ndarray, g: np.ndarray, p, s, X: Optional[np.ndarray],
                     residual: Optional[bool] = None) -> np.ndarray:
    """Eq. (3): Y = W_out(beta1 * norm(att) + beta2 * norm(g)) (+ X if residual).

    With ``s.fusion == "concat"`` the ablation of the Hymba page's appendix B
    (Table 10, concatenation instead of the averaging fusion): the two
    normalised, beta-scaled branches are concatenated and W_out is [d, 2 di]:
    Y = W_out [beta1 * norm(att) ; beta2 * norm(g)].
    """
    a = np.asarray(p["beta1"], F) * rms_norm(att, s.eps)
    b = np.asarray(p["beta2"], F) * rms_norm(g, s.eps)
    sm = np.concatenate([a, b], axis=-1) if getattr(s, "fusion", "sum") == "concat" else a + b
    Y = sm @ np.asarray(p["W_out"], F).T
    if s.residual if residual is None else residual:
        Y = Y + np.asarray(X, F)
    return Y


def layer_fwd(p: Dict[str, np.ndarray], Xt: np.ndarray, s,
              kv_in: Optional[Tuple[np.ndarray, np.ndarray]] = None,
              cache_cap: Optional[int] = None, want_branches: bool = False,
              residual: Optional[bool] = None) -> Dict[str, np.ndarray]:
    """Prefill forward of one hybrid-head layer on X~ [B, L, d] (meta rows first).

    Returns a dict with Y [B,L,d]; K/V (post-RoPE, [B,L,Hkv,dh|dv]) for a
    sharing consumer; and, when ``cache_cap`` is given, the decode cache.
    ``residual`` overrides the shape's residual flag when given.
    """
    Xt = np.asarray(Xt, F)
    B, L, d = Xt.shape
    assert L == s.L and d == s.d
    proj = Xt @ np.asarray(p["W_in"], F).T
    parts = split_projection(proj, s)
    Q = parts["Q"]
    positions = np.arange(L)
    if s.rope_theta > 0:
        Q = rope(Q, positions, s.rope_theta)
    if s.kv_shared:
        assert kv_in is not None
        K, V = (np.asarray(a, F) for a in kv_in)
    else:
        K, V = parts["K"], parts["V"]
        if s.rope_theta > 0:
            K = rope(K, positions, s.rope_theta)
    att = attention(Q, K, V, s.M, s.window)
    g, h = ssm_branch(parts["x"], parts["z"], p, s)
    Y = fuse_and_project(att, g, p, s, Xt, residual)
    out = {"Y": Y, "K": K, "V": V}
    if want_branches:
        out.update(att=att, g=g, x=parts["x"], z=parts["z"])
    if cache_cap is not None:
        out["cache"] = emit_cache(K, V, parts["x"], h, s, cache_cap)
    return out


def layer_fwd_rows(p: Dict[str, np.ndarray], Xt: np.ndarray, s, rows,
                   kv_in: Optional[Tuple[np.ndarray, np.ndarray]] = None) -> np.ndarray:
    """Y at the query rows ``rows`` only (indices into X~'s L rows), for
    sequences too long for the whole-layer oracle.

    The same steps as layer_fwd, eq. (3) of the Hymba page, cut to what these
    rows depend on: the layer is causal, so only the prefix up to the last
    requested row is projected and scanned, and attention runs for the
    requested query rows alone.  Returns [B, len(rows), d].
    """
    Xt = np.asarray(Xt, F)
    rows = np.asarray(rows)
    n = int(rows.max()) + 1
    Xp = Xt[:, :n]
    proj = Xp @ np.asarray(p["W_in"], F).T
    parts = split_projection(proj, s)
    positions = np.arange(n)
    Q = parts["Q"]
    if s.rope_theta > 0:
        Q = rope(Q, positions, s.rope_theta)
    if s.kv_shared:
        assert kv_in is not None
        K, V = (np.asarray(a, F)[:, :n] for a in kv_in)
    else:
        K, V = parts["K"], parts["V"]
        if s.rope_theta > 0:
            K = rope(K, positions, s.rope_theta)
    att = attention(Q, K, V, s.M, s.window, rows=rows)
    g, _ = ssm_branch(parts["x"], parts["z"], p, s)
    return fuse_and_project(att, g[:, rows], p, s, Xt[:, rows])


def emit_cache(K, V, x, h, s, cap: int) -> Dict[str, np.ndarray]:
    """Decode state after a prefill of T real tokens (reading 8)."""
    B = K.shape[0]
    k_ring = np.zeros((B, cap, s.Hkv, s.dh), F)
    v_ring = np.zeros((B, cap, s.Hkv, s.dv), F)
    n_keep = s.T if s.window == 0 else min(s.T, cap)
    assert n_keep <= cap
    for t in range(s.T - n_keep, s.T):
        k_ring[:, t % cap] = K[:, s.M + t]
        v_ring[:, t % cap] = V[:, s.M + t]
    km1 = s.k - 1
    tail = np.zeros((B, s.di, km1), F)
    L = s.L
    for j in range(km1):
        row = L - km1 + j
        if row >= 0:
            tail[:, :, j] = x[:, row, :]
    return {"k_ring": k_ring, "v_ring": v_ring,
            "k_meta": np.array(K[0, : s.M]), "v_meta": np.array(V[0, : s.M]),
            "ssm_state": np.array(h), "conv_state": tail,
            "pos": np.full((B,), s.T, np.int64)}


def decode_visible_slots(pos: int, window: int, cap: int) -> np.ndarray:
    """Ring slots holding the real keys visible to the token at real index pos."""
    n_vis = min(pos + 1, window) if window > 0 else pos + 1
    assert n_vis <= cap, "cache too small for the visible window"
    return np.array([(pos - i) % cap for i in range(n_vis)], dtype=np.int64)


def layer_decode(p: Dict[str, np.ndarray], x_new: np.ndarray, cache: Dict[str, np.ndarray], s,
                 shared_cache: Optional[Dict[str, np.ndarray]] = None) -> Dict[str, np.ndarray]:
    """One decode step for B sequences.  ``cache`` is not modified; the
    updated cache is returned.  A KV-sharing layer reads K/V from
    ``shared_cache`` (the producer's cache, already holding this token)."""
    x_new = np.asarray(x_new, F)
    B = x_new.shape[0]
    pos = np.asarray(cache["pos"]).astype(np.int64)
    proj = x_new @ np.asarray(p["W_in"], F).T                              # [B, P_in]
    parts = split_projection(proj, s)
    q = parts["Q"]                                                         # [B, Hq, dh]
    abs_pos = s.M + pos
    new = {k: np.array(v, copy=True) for k, v in cache.items()}
    if s.rope_theta > 0:
        q = rope(q, abs_pos, s.rope_theta)
    if s.kv_shared:
        kv_src = shared_cache
        assert kv_src is not None
    else:
        k = parts["K"]
        v = parts["V"]
        if s.rope_theta > 0:
            k = rope(k, abs_pos, s.rope_theta)
        kv_src = new
        cap = new["k_ring"].shape[1]
        for b in range(B):
            slot = pos[b] % cap if s.window > 0 else pos[b]
            assert slot < cap
            new["k_ring"][b, slot] = k[b]
            new["v_ring"][b, slot] = v[b]
    cap = kv_src["k_ring"].shape[1]
    att = np.zeros((B, s.Hq * s.dv), F)
    scale = 1.0 / math.sqrt(s.dh)
    for b in range(B):
        slots = decode_visible_slots(int(pos[b]), s.window, cap)
        Kb = np.concatenate([np.asarray(kv_src["k_meta"], F), np.asarray(kv_src["k_ring"], F)[b, slots]], 0)
        Vb = np.concatenate([np.asarray(kv_src["v_meta"], F), np.asarray(kv_src["v_ring"], F)[b, slots]], 0)
        for h in range(s.Hq):
            gidx = (h * s.Hkv) // s.Hq
            sc = Kb[:, gidx, :] @ q[b, h] * scale
            sc = sc - sc.max()
            pr = np.exp(sc)
            pr /= pr.sum()
            att[b, h * s.dv:(h + 1) * s.dv] = pr @ Vb[:, gidx, :]
    # SSM branch, one step from the carried state
    x = parts["x"][:, None, :]
    z = parts["z"][:, None, :]
    g, h = ssm_branch(x, z, p, s, tail=cache["conv_state"], h0=cache["ssm_state"])
    conv_state = np.concatenate([np.asarray(cache["conv_state"], F)[:, :, 1:], parts["x"][:, :, None]], axis=2)
    Y = fuse_and_project(att, g[:, 0, :], p, s, x_new)
    new["ssm_state"] = h
    new["conv_state"] = conv_state
    new["pos"] = pos + 1
    return {"y": Y, "cache": new, "att": att, "g": g[:, 0, :]}


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even), returned as float64:
    float32 bits + 0x7FFF + (bit 16), truncated to the top 16 bits."""
    f = np.ascontiguousarray(np.asarray(a, np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(F)


def stack_fwd(layers, Xt: np.ndarray, shapes) -> Dict[str, list]:
    """Residual stack X_{l+1} = X_l + Y_l(X_l) of hybrid-head layers (the
    Hymba pages describe no pre-norm or FFN for it); a kv_shared layer
    consumes the previous layer's post-RoPE K/V (section 2.2).

    Reading: the stream is carried at full precision and every layer reads
    it unrounded (no rounding step is part of the definition; a device keeps
    its own stream in fp32 and rounds only its matmul operands).  Every
    layer's own residual flag is ignored: the stack adds the stream.
    Returns the stream after each layer.
    """
    X = np.asarray(Xt, F)
    outs, prev = [], None
    for p, s in zip(layers, shapes):
        kv = (prev["K"], prev["V"]) if s.kv_shared else None
        o = layer_fwd(p, X, s, kv_in=kv, residual=False)
        X = X + o["Y"]
        outs.append(X)
        prev = o
    return {"Y": outs}
