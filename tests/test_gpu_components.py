"""Component parity on the GPU through the C ABI: the tcgen05 GEMM, the scan
(closed form, special cases, random vs oracle), the attention kernels (the
uniform-mean pin of the visible set, random vs oracle) and the bounded wait."""
import math

import numpy as np
import pytest
import torch

from hybrid_attention_ssm_fwd_b300 import binding as hb
from oracle import hymba_ref as ref

pytestmark = pytest.mark.gpu
F = np.float64


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 200, 100), (1000, 1600, 3200), (37, 8960, 1600),
                                   (4500, 144, 96), (128, 64, 8),
                                   (1115, 520, 200), (2100, 300, 64), (1921, 176, 72),
                                   # 4+ row blocks and tiles at most 128 wide run as CTA pairs (256-row
                                   # tiles on tcgen05.mma.cta_group::2); 5, 9 and 17 row blocks leave an
                                   # empty half in the last pair; N not a multiple of the tile
                                   (512, 128, 256), (600, 64, 1600), (1047, 384, 200), (2100, 120, 3200),
                                   (1921, 96, 72)])
@pytest.mark.parametrize("ab", [1, 2, 3])
def test_gemm_tc_matches_fp64(M, N, K, ab):
    """ab 1: bf16 x bf16; 2: fp16 x fp16; 3: fp16 A against a bf16 B that the
    kernel converts to fp16 in shared memory (exact for these magnitudes)."""
    g = torch.Generator().manual_seed(M * 7 + N + K)
    dt = torch.bfloat16 if ab == 1 else torch.float16
    dtb = torch.bfloat16 if ab in (1, 3) else torch.float16
    A = torch.randn(M, K, generator=g).to(dt)
    B = (0.05 * torch.randn(N, K, generator=g)).to(dtb)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # rows must start on 16 bytes: pad the row stride to a multiple of 8 and
    # fill the padding with NaN, which the K tail must never read
    Kp = (K + 7) // 8 * 8
    Ad = torch.full((M, Kp), float("nan"), dtype=dt, device="cuda")
    Bd = torch.full((N, Kp), float("nan"), dtype=dtb, device="cuda")
    Ad[:, :K] = A.cuda()
    Bd[:, :K] = B.cuda()
    rc = hb.hymba_test_gemm(Ad[:, :K], Bd[:, :K], C, ab, status=st)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    ref_c = A.double() @ B.double().T
    got = C.cpu().double()
    err = (got - ref_c).abs().max().item()
    assert err <= 1e-5 * max(1.0, ref_c.abs().max().item()) * math.sqrt(K / 64), err


@pytest.mark.parametrize("M,N,K,ldc", [(300, 37, 64, 40), (1047, 45, 200, 48), (520, 203, 96, 208),
                                       (129, 3, 64, 4), (2100, 61, 72, 64)])
def test_gemm_tc_ragged_columns_in_padded_rows(M, N, K, ldc):
    """fp32 results whose last 32-column piece holds a number of columns that
    is not a multiple of four, in rows padded to a 16-byte stride: the staged
    store writes whole 4-column pieces and the tail element by element, and
    never the padding (left NaN)."""
    g = torch.Generator().manual_seed(M + 31 * N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (0.05 * torch.randn(N, K, generator=g)).to(torch.bfloat16)
    Cp = torch.full((M, ldc), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Kp = (K + 7) // 8 * 8
    Ad = torch.zeros(M, Kp, dtype=torch.bfloat16, device="cuda")
    Bd = torch.zeros(N, Kp, dtype=torch.bfloat16, device="cuda")
    Ad[:, :K] = A.cuda()
    Bd[:, :K] = B.cuda()
    assert hb.hymba_test_gemm(Ad[:, :K], Bd[:, :K], Cp[:, :N], 1, status=st) == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    got = Cp.cpu().double()
    ref_c = A.double() @ B.double().T
    err = (got[:, :N] - ref_c).abs().max().item()
    assert err <= 1e-5 * max(1.0, ref_c.abs().max().item()) * math.sqrt(K / 64), err
    assert torch.isnan(got[:, N:]).all()


def _scan_inputs(B, L, di, N, seed, u0=None, d0=None, b0=None, c0=None):
    rng = np.random.default_rng(seed)
    u = rng.standard_normal((B, L, di)) if u0 is None else np.full((B, L, di), u0)
    z = rng.standard_normal((B, L, di)) * 2
    dl = rng.uniform(1e-3, 0.1, (B, L, di)) if d0 is None else np.full((B, L, di), d0)
    Bm = rng.standard_normal((B, L, N)) if b0 is None else np.full((B, L, N), b0)
    Cm = rng.standard_normal((B, L, N)) if c0 is None else np.full((B, L, N), c0)
    A_log = np.log(rng.uniform(1, 16, (di, N)))
    D = rng.standard_normal(di)
    # fp16-representable u, z so both sides see the same values
    u = u.astype(np.float16).astype(F)
    z = z.astype(np.float16).astype(F)
    return u, z, dl.astype(np.float32).astype(F), Bm.astype(np.float32).astype(F), Cm.astype(np.float32).astype(F), \
        A_log.astype(np.float32).astype(F), D.astype(np.float32).astype(F)


def _run_scan(u, z, dl, Bm, Cm, A_log, D, tpc=0, cpt=0):
    B, L, di = u.shape
    N = Bm.shape[-1]
    dev = "cuda"
    tu = torch.from_numpy(u).to(dev, torch.float16)
    tz = torch.from_numpy(z).to(dev, torch.float16)
    td = torch.from_numpy(dl).to(dev, torch.float32)
    bc = torch.from_numpy(np.concatenate([Bm, Cm], -1)).to(dev, torch.float32).contiguous()
    ta = torch.from_numpy(A_log).to(dev, torch.float32)
    tD = torch.from_numpy(D).to(dev, torch.float32)
    g = torch.empty(B, L, di, device=dev, dtype=torch.float16)
    h = torch.empty(B, di, N, device=dev, dtype=torch.float32)
    assert hb.hymba_test_scan(tu, tz, td, bc, ta, tD, g, h, threads_per_channel=tpc, channels_per_thread=cpt) == 0
    torch.cuda.synchronize()
    return g.float().cpu().numpy().astype(F), h.cpu().numpy().astype(F)


@pytest.mark.parametrize("tpc,cpt", [(1, 1), (2, 1), (2, 2), (4, 1), (4, 2)])
def test_scan_closed_form_on_gpu(tpc, cpt):
    """Constant u, Delta, B, C with D = 0: the state follows the geometric
    series exactly, so C.h dominates the output (the case the end-to-end
    tolerance cannot see).  Every split of the 16 states over 1, 2 or 4
    threads per channel, and two channels per thread at two or four threads
    per channel."""
    B, L, di, N = 2, 700, 64, 16
    u, z, dl, Bm, Cm, A_log, D = _scan_inputs(B, L, di, N, 1, u0=0.75, d0=0.05, b0=1.25, c0=-0.5)
    D[:] = 0
    g, h = _run_scan(u, z, dl, Bm, Cm, A_log, D, tpc, cpt)
    A = -np.exp(A_log)
    a = np.exp(0.05 * A)                                              # [di, N]
    t = np.arange(L)[:, None, None]
    ht = 0.05 * 1.25 * 0.75 * (1 - a[None] ** (t + 1)) / (1 - a[None])
    y = -0.5 * ht.sum(-1)                                             # [L, di]
    expect_g = y[None] * ref.silu(z)
    np.testing.assert_allclose(h, np.broadcast_to(ht[-1], h.shape), rtol=2e-5)
    np.testing.assert_allclose(g, expect_g, rtol=3e-3, atol=1e-3 * np.abs(expect_g).max())


def test_scan_special_cases_on_gpu():
    B, L, di, N = 1, 300, 128, 16
    u, z, dl, Bm, Cm, A_log, D = _scan_inputs(B, L, di, N, 2)
    g, h = _run_scan(u, z, dl, np.zeros_like(Bm), Cm, A_log, D)       # B = 0: y = D u
    np.testing.assert_allclose(g, D * u * ref.silu(z), rtol=2e-3, atol=1e-3)
    assert np.all(h == 0)


@pytest.mark.parametrize("tpc,cpt,L", [(1, 1, 517), (2, 1, 517), (2, 2, 517), (4, 1, 517), (4, 2, 517), (2, 1, 3),
                                       (2, 2, 3), (4, 1, 18), (4, 2, 18)])
def test_scan_random_matches_oracle(tpc, cpt, L):
    B, di, N = 3, 192, 16
    u, z, dl, Bm, Cm, A_log, D = _scan_inputs(B, L, di, N, 3)
    g, h = _run_scan(u, z, dl, Bm, Cm, A_log, D, tpc, cpt)
    y, hr = ref.selective_scan(u, dl, -np.exp(A_log), Bm, Cm, D)
    gr = y * ref.silu(z)
    np.testing.assert_allclose(h, hr, rtol=1e-4, atol=1e-5 * np.abs(hr).max())
    np.testing.assert_allclose(g, gr, rtol=2e-3, atol=2e-3 * np.abs(gr).max())


def _attn_inputs(B, L, Hq, Hkv, dh, dv, seed, zero_q=False, q_scale=1.0):
    rng = np.random.default_rng(seed)
    Q = np.zeros((B, L, Hq, dh)) if zero_q else rng.standard_normal((B, L, Hq, dh)) * q_scale
    K = rng.standard_normal((B, L, Hkv, dh))
    V = rng.standard_normal((B, L, Hkv, dv))
    return [a.astype(np.float16).astype(F) for a in (Q, K, V)]


def _run_attn(Q, K, V, M, window, use_tc):
    B, L, Hq, dh = Q.shape
    dv = V.shape[-1]
    t = [torch.from_numpy(a).to("cuda", torch.float16).contiguous() for a in (Q, K, V)]
    O = torch.full((B, L, Hq * dv), float("nan"), device="cuda", dtype=torch.float16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = hb.hymba_test_attention(*t, O, M, window, use_tc, status=st)
    if rc == hb.HYMBA_ERR_UNSUPPORTED:
        pytest.skip("tensor-core attention not available for this shape")
    assert rc == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    return O.float().cpu().numpy().astype(F)


@pytest.mark.parametrize("use_tc", [0, 1])
@pytest.mark.parametrize("M,window,L", [(128, 1024, 1500), (16, 32, 300), (128, 0, 700), (0, 1, 260),
                                        (5, 8, 200), (128, 200, 333)])
def test_attention_uniform_mean_pins_visible_set(use_tc, M, window, L):
    """Q = 0: every visible score is 0, so each output row is the plain mean
    of V over meta-union-window; this pins |vis(i)| for every row."""
    B, Hq, Hkv, dh, dv = 2, 4, 2, 64, 128
    Q, K, V = _attn_inputs(B, L, Hq, Hkv, dh, dv, 4, zero_q=True)
    got = _run_attn(Q, K, V, M, window, use_tc)
    exp = ref.attention(Q, K, V, M, window)
    np.testing.assert_allclose(got, exp, atol=2e-3, rtol=2e-3)


@pytest.mark.parametrize("use_tc", [0, 1])
@pytest.mark.parametrize("M,window,L,q_scale", [(128, 1024, 1400, 1.0), (128, 0, 600, 1.0), (16, 64, 301, 3.0),
                                                (3, 0, 129, 6.0)])
def test_attention_random_matches_oracle(use_tc, M, window, L, q_scale):
    """Random Q/K/V, including large scores that force the running-max
    rescale path."""
    B, Hq, Hkv, dh, dv = 2, 10, 2, 64, 128
    Q, K, V = _attn_inputs(B, L, Hq, Hkv, dh, dv, 5, q_scale=q_scale)
    got = _run_attn(Q, K, V, M, window, use_tc)
    exp = ref.attention(Q, K, V, M, window)
    np.testing.assert_allclose(got, exp, atol=4e-3 * max(1, np.abs(exp).max()), rtol=1e-2)


@pytest.mark.parametrize("Hq,Hkv,dv,M,window,L", [(3, 3, 64, 16, 64, 301), (6, 1, 64, 128, 256, 700),
                                                  (7, 7, 128, 0, 0, 130), (5, 1, 128, 128, 0, 400)])
def test_attention_head_pairing_matches_oracle(Hq, Hkv, dv, M, window, L):
    """The tensor-core kernel runs two query heads of one KV group per unit
    and a group's odd head alone: groups of 1, 3, 5 and 6 heads, both V
    widths."""
    B, dh = 2, 64
    Q, K, V = _attn_inputs(B, L, Hq, Hkv, dh, dv, 6, q_scale=2.0)
    got = _run_attn(Q, K, V, M, window, 1)
    exp = ref.attention(Q, K, V, M, window)
    np.testing.assert_allclose(got, exp, atol=4e-3 * max(1, np.abs(exp).max()), rtol=1e-2)


def test_bounded_wait_reports_timeout():
    """A wait on a barrier nothing arrives on gives up after its limit and the
    status word says so; the context stays usable."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hb.hymba_test_wait_timeout(20000, st) == 0
    torch.cuda.synchronize()
    assert st.item() == hb.HYMBA_ERR_TIMEOUT
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum().item()) == 8.0


def _run_scan_fused(u, z, dtr, W_dt, dt_bias, Bm, Cm, A_log, D, tpc=0, cpt=0):
    B, L, di = u.shape
    N = Bm.shape[-1]
    R = W_dt.shape[1]
    Rp = (R + 7) // 8 * 8
    dev = "cuda"
    tu = torch.from_numpy(u).to(dev, torch.float16)
    tz = torch.from_numpy(z).to(dev, torch.float16)
    tdt = torch.full((B, L, Rp), float("nan"), device=dev, dtype=torch.float16)   # padding never read
    tdt[..., :R] = torch.from_numpy(dtr).to(dev, torch.float16)
    tw = torch.from_numpy(W_dt).to(dev, torch.bfloat16)
    tb = torch.from_numpy(dt_bias).to(dev, torch.float32)
    bc = torch.from_numpy(np.concatenate([Bm, Cm], -1)).to(dev, torch.float32).contiguous()
    ta = torch.from_numpy(A_log).to(dev, torch.float32)
    tD = torch.from_numpy(D).to(dev, torch.float32)
    g = torch.empty(B, L, di, device=dev, dtype=torch.float16)
    h = torch.empty(B, di, N, device=dev, dtype=torch.float32)
    assert hb.hymba_test_scan_fused(tu, tz, tdt, tw, tb, bc, ta, tD, g, h, threads_per_channel=tpc,
                                    channels_per_thread=cpt) == 0
    torch.cuda.synchronize()
    return g.float().cpu().numpy().astype(F), h.cpu().numpy().astype(F)


def test_fused_scan_closed_form_on_gpu():
    """Fused dt projection with W_dt = 0: delta = softplus(bias) = 0.05 for every
    row, so the geometric-series closed form must hold through the fused path."""
    B, L, di, N, R = 2, 650, 64, 16, 100
    u, z, _, Bm, Cm, A_log, D = _scan_inputs(B, L, di, N, 6, u0=0.75, b0=1.25, c0=-0.5)
    D[:] = 0
    rng = np.random.default_rng(7)
    dtr = rng.standard_normal((B, L, R)).astype(np.float16).astype(F)
    W_dt = np.zeros((di, R))
    d0 = 0.05
    bias = np.full(di, d0 + np.log(-np.expm1(-d0))).astype(np.float32).astype(F)
    g, h = _run_scan_fused(u, z, dtr, W_dt, bias, Bm, Cm, A_log, D)
    dl = ref.softplus(bias)[0]
    A = -np.exp(A_log)
    a = np.exp(dl * A)
    t = np.arange(L)[:, None, None]
    ht = dl * 1.25 * 0.75 * (1 - a[None] ** (t + 1)) / (1 - a[None])
    expect_g = (-0.5 * ht.sum(-1))[None] * ref.silu(z)
    np.testing.assert_allclose(h, np.broadcast_to(ht[-1], h.shape), rtol=5e-5)
    np.testing.assert_allclose(g, expect_g, rtol=3e-3, atol=1e-3 * np.abs(expect_g).max())


@pytest.mark.parametrize("R,di,L,tpc,cpt", [(100, 192, 517, 0, 0), (100, 192, 517, 1, 1), (100, 192, 517, 2, 1),
                                            (100, 192, 517, 2, 2), (100, 192, 517, 4, 1), (64, 128, 130, 2, 1),
                                            (64, 128, 130, 2, 2), (8, 64, 33, 1, 1), (128, 48, 70, 4, 1),
                                            (17, 64, 1, 2, 1), (17, 64, 1, 2, 2), (100, 192, 517, 4, 2),
                                            (64, 128, 130, 4, 2)])
def test_fused_scan_random_matches_oracle(R, di, L, tpc, cpt):
    B, N = 2, 16
    u, z, _, Bm, Cm, A_log, D = _scan_inputs(B, L, di, N, 8)
    rng = np.random.default_rng(9)
    dtr = (rng.standard_normal((B, L, R)) * 0.5).astype(np.float16).astype(F)
    W_dt = synth_bf16(rng.standard_normal((di, R)) * 0.1)
    dt0 = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), di))
    bias = (dt0 + np.log(-np.expm1(-dt0))).astype(np.float32).astype(F)
    g, h = _run_scan_fused(u, z, dtr, W_dt, bias, Bm, Cm, A_log, D, tpc, cpt)
    dl = ref.softplus(dtr @ W_dt.T + bias)
    y, hr = ref.selective_scan(u, dl, -np.exp(A_log), Bm, Cm, D)
    gr = y * ref.silu(z)
    np.testing.assert_allclose(h, hr, rtol=2e-3, atol=2e-4 * np.abs(hr).max())
    np.testing.assert_allclose(g, gr, rtol=3e-3, atol=3e-3 * np.abs(gr).max())


def synth_bf16(a):
    from hybrid_attention_ssm_fwd_b300 import synth
    return synth.bf16_round(np.asarray(a, np.float32)).astype(F)


@pytest.mark.parametrize("B,L,di,k,ld_x", [(3, 200, 256, 4, 520), (2, 64, 3200, 4, 3200), (1, 1, 136, 3, 136),
                                          (4, 131, 24, 2, 40)])
def test_conv_matches_oracle(B, L, di, k, ld_x):
    """Causal conv + SiLU of the SSM branch: each sequence starts from zero
    history (never the previous sequence's rows), ragged row and channel
    tiles, strided input rows as in the projection buffer."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((B, L, ld_x)).astype(np.float16)
    w = (rng.standard_normal((di, k)) * 0.5).astype(np.float32)
    bias = (rng.standard_normal(di) * 0.1).astype(np.float32)
    tx = torch.from_numpy(x).cuda()
    u = torch.full((B, L, di), float("nan"), dtype=torch.float16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hb.hymba_test_conv(tx, u, torch.from_numpy(w).cuda(), torch.from_numpy(bias).cuda(), status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ur = ref.conv1d_silu(x[:, :, :di].astype(F), w.astype(F), bias.astype(F))
    got = u.float().cpu().numpy()
    # fp16 output: half an ulp of |u| plus fp32 accumulation
    np.testing.assert_allclose(got, ur, rtol=1e-3, atol=1e-3)
