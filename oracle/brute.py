"""Loop-only second oracle of the hybrid-head layer, for tiny shapes.

TEST INFRASTRUCTURE ONLY (same import rule as ``oracle.hymba_ref``).

Everything is written with explicit Python loops over scalars (``math`` only):
no BLAS, no vectorisation and no code shared with ``oracle.hymba_ref``, so that
the two oracles can only agree if both follow the same definition.  It follows
"Hymba: A Hybrid-head Architecture for Small Language Models", section 2.1
eq. (3), section 2.2 (window / KV sharing) and section 2.3 (meta tokens), with
the readings listed in ``oracle.hymba_ref``'s header.
"""
from __future__ import annotations

import math


def _mat(a):
    return [list(map(float, row)) for row in a]


def _silu(v):
    return v / (1.0 + math.exp(-v)) if v >= 0 else v * math.exp(v) / (1.0 + math.exp(v))


def _softplus(v):
    return v + math.log1p(math.exp(-v)) if v > 0 else math.log1p(math.exp(v))


def _matvec(W, x):
    """W [n][m] times x [m] -> [n]."""
    out = []
    for row in W:
        acc = 0.0
        for a, b in zip(row, x):
            acc += a * b
        out.append(acc)
    return out


def _rope_vec(v, position, theta):
    dh = len(v)
    half = dh // 2
    out = [0.0] * dh
    for i in range(half):
        ang = position * theta ** (-(2.0 * i) / dh)
        c, s = math.cos(ang), math.sin(ang)
        out[i] = v[i] * c - v[i + half] * s
        out[i + half] = v[i + half] * c + v[i] * s
    return out


def _rms(v, eps):
    ms = 0.0
    for a in v:
        ms += a * a
    ms /= len(v)
    r = 1.0 / math.sqrt(ms + eps)
    return [a * r for a in v]


def layer_fwd(p, Xt, s, kv_in=None):
    """Y [B][L][d] (nested lists) for one layer; optionally also K/V."""
    W_in = _mat(p["W_in"])
    W_out = _mat(p["W_out"])
    W_x = _mat(p["W_x"])
    W_dt = _mat(p["W_dt"])
    conv_w = _mat(p["conv_w"])
    conv_b = [float(a) for a in p["conv_b"]]
    dt_bias = [float(a) for a in p["dt_bias"]]
    A = [[-math.exp(float(a)) for a in row] for row in p["A_log"]]
    Dv = [float(a) for a in p["D"]]
    b1 = [float(a) for a in p["beta1"]]
    b2 = [float(a) for a in p["beta2"]]
    Bsz, L = len(Xt), len(Xt[0])
    M, W = s.M, s.window
    Hq, Hkv, dh, dv, di, N, k, R = s.Hq, s.Hkv, s.dh, s.dv, s.di, s.N, s.k, s.R
    Ys, Ks, Vs = [], [], []
    for b in range(Bsz):
        X = [[float(a) for a in row] for row in Xt[b]]
        q_all, k_all, v_all, x_all, z_all = [], [], [], [], []
        for t in range(L):
            pr = _matvec(W_in, X[t])
            o = 0
            q = [pr[o + h * dh: o + (h + 1) * dh] for h in range(Hq)]
            o += Hq * dh
            if not s.kv_shared:
                kk = [pr[o + g * dh: o + (g + 1) * dh] for g in range(Hkv)]
                o += Hkv * dh
                vv = [pr[o + g * dv: o + (g + 1) * dv] for g in range(Hkv)]
                o += Hkv * dv
            xx = pr[o: o + di]
            o += di
            zz = pr[o: o + di]
            if s.rope_theta > 0:
                q = [_rope_vec(a, t, s.rope_theta) for a in q]
                if not s.kv_shared:
                    kk = [_rope_vec(a, t, s.rope_theta) for a in kk]
            q_all.append(q)
            if not s.kv_shared:
                k_all.append(kk)
                v_all.append(vv)
            x_all.append(xx)
            z_all.append(zz)
        if s.kv_shared:
            k_all = [[list(map(float, kv_in[0][b][t][g])) for g in range(Hkv)] for t in range(L)]
            v_all = [[list(map(float, kv_in[1][b][t][g])) for g in range(Hkv)] for t in range(L)]
        # attention branch: explicit visible set per row
        att = []
        for i in range(L):
            row = []
            for h in range(Hq):
                g = (h * Hkv) // Hq
                keys = [j for j in range(i + 1) if W == 0 or i - j < W or j < M]
                sc = []
                for j in keys:
                    acc = 0.0
                    for e in range(dh):
                        acc += q_all[i][h][e] * k_all[j][g][e]
                    sc.append(acc / math.sqrt(dh))
                mx = max(sc)
                w = [math.exp(a - mx) for a in sc]
                tot = sum(w)
                for e in range(dv):
                    acc = 0.0
                    for wj, j in zip(w, keys):
                        acc += wj * v_all[j][g][e]
                    row.append(acc / tot)
            att.append(row)
        # SSM branch: conv, x_proj, dt_proj, scan, gate
        u = []
        for t in range(L):
            ut = []
            for c in range(di):
                acc = conv_b[c]
                for j in range(k):
                    src = t - (k - 1) + j
                    if src >= 0:
                        acc += conv_w[c][j] * x_all[src][c]
                ut.append(_silu(acc))
            u.append(ut)
        h = [[0.0] * N for _ in range(di)]
        gate = []
        for t in range(L):
            xd = _matvec(W_x, u[t])
            dtr, Bt, Ct = xd[:R], xd[R:R + N], xd[R + N:]
            pre = _matvec(W_dt, dtr)
            gt = []
            for c in range(di):
                delta = _softplus(pre[c] + dt_bias[c])
                y = 0.0
                for n in range(N):
                    h[c][n] = math.exp(delta * A[c][n]) * h[c][n] + delta * u[t][c] * Bt[n]
                    y += Ct[n] * h[c][n]
                y += Dv[c] * u[t][c]
                gt.append(y * _silu(z_all[t][c]))
            gate.append(gt)
        Yb = []
        for t in range(L):
            na = _rms(att[t], s.eps)
            ng = _rms(gate[t], s.eps)
            sm = [b1[c] * na[c] + b2[c] * ng[c] for c in range(di)]
            yt = _matvec(W_out, sm)
            if s.residual:
                yt = [a + bb for a, bb in zip(yt, X[t])]
            Yb.append(yt)
        Ys.append(Yb)
        Ks.append(k_all)
        Vs.append(v_all)
    return {"Y": Ys, "K": Ks, "V": Vs}


def selective_scan(u, delta, A, Bm, Cm, D, h0=None):
    """Scan for a single sequence with nested lists: u, delta [L][di],
    A [di][N], Bm, Cm [L][N], D [di].  Returns y [L][di], h [di][N]."""
    L, di, N = len(u), len(A), len(A[0])
    h = [[0.0] * N for _ in range(di)] if h0 is None else [list(map(float, r)) for r in h0]
    y = []
    for t in range(L):
        yt = []
        for c in range(di):
            acc = 0.0
            for n in range(N):
                h[c][n] = math.exp(delta[t][c] * A[c][n]) * h[c][n] + delta[t][c] * u[t][c] * Bm[t][n]
                acc += Cm[t][n] * h[c][n]
            yt.append(acc + D[c] * u[t][c])
        y.append(yt)
    return y, h
