"""The bench's roofline arithmetic on the host: the algorithmic work of each
stage (the denominators of every reported fraction) and the choice of the
dominant kernel.

FLOP counts are checked against closed forms written from the layer's shapes
(2 FLOP per multiply-add; attention counts only the visible (query, key)
pairs of the meta-prefix / sliding-window mask, counted here by brute force
over the mask's definition) and against the figures worked out by hand for
the Hymba-1.5B-shaped SWA layer at batch 8 x (8192 + 128).
"""
import numpy as np
import pytest

import bench
from hybrid_attention_ssm_fwd_b300 import synth


def _visible_pairs(L, M, W):
    """Sum over query rows of |{j <= i : W == 0 or i - j < W or j < M}|."""
    total = 0
    j = np.arange(L)
    for i0 in range(0, L, 1024):
        i = np.arange(i0, min(L, i0 + 1024))[:, None]
        vis = j[None, :] <= i
        if W > 0:
            vis &= (i - j[None, :] < W) | (j[None, :] < M)
        total += int(vis.sum())
    return total


SHAPES = [synth.hymba15b_swa(), synth.hymba15b_global()] + synth.ablation300m_stack()


@pytest.mark.parametrize("s", SHAPES, ids=["swa_1p5b", "global_1p5b", "stack_l0", "stack_l1", "stack_l2",
                                           "stack_l3"])
def test_layer_flops_closed_forms(s):
    fl = bench.layer_flops(s)
    rows = s.B * s.L
    kv = 0 if s.kv_shared else s.Hkv * (s.dh + s.dv)
    P_in = s.Hq * s.dh + kv + 2 * s.di
    assert fl["in_proj"] == pytest.approx(2 * rows * P_in * s.d, rel=1e-12)
    assert fl["x_proj"] == pytest.approx(2 * rows * (s.R + 2 * s.N) * s.di, rel=1e-12)
    assert fl["dt_proj"] == pytest.approx(2 * rows * s.R * s.di, rel=1e-12)
    assert fl["out_proj"] == pytest.approx(2 * rows * s.d * s.di, rel=1e-12)
    pairs = _visible_pairs(s.L, s.M, s.window)
    assert fl["attention"] == pytest.approx(2 * (s.dh + s.dv) * s.Hq * s.B * pairs, rel=1e-12)


def test_layer_flops_swa_1p5b_hand_figures():
    """Batch 8 x 8320 rows, P_in = 25*64 + 5*(64+128) + 2*3200 = 8960:
    in_proj 2*66560*8960*1600 = 1908.4 GFLOP; out_proj 2*66560*1600*3200 =
    681.6; x_proj (R = 100, 2N = 32) 2*66560*132*3200 = 56.2; dt_proj 42.6;
    attention 685.2 (about 1072 visible keys per row)."""
    fl = bench.layer_flops(synth.hymba15b_swa())
    got = {k: round(fl[k] / 1e9, 1) for k in ("in_proj", "out_proj", "x_proj", "dt_proj", "attention")}
    assert got == {"in_proj": 1908.4, "out_proj": 681.6, "x_proj": 56.2, "dt_proj": 42.6, "attention": 685.2}


def test_stage_rooflines_dominant_kernel_and_scan_bounds():
    s = synth.hymba15b_swa()
    stage_ms = {"convert": 0.02, "in_proj": 1.40, "kv_export": 0.002, "attention": 0.90, "conv": 0.18,
                "x_proj": 0.13, "dt_proj": 0.002, "scan": 1.44, "fuse_norm": 0.22, "out_proj": 0.56,
                "cache": 0.002}
    peaks = dict(bench.PEAKS_FALLBACK)
    kernels, dom = bench.stage_rooflines(s, stage_ms, peaks)
    assert dom == "scan"
    assert set(kernels) == {"in_proj", "attention", "x_proj", "out_proj", "conv", "fuse_norm", "scan", "scan_hbm",
                            "scan_fma"}
    rows = s.B * s.L
    t = 1.44e-3
    # one exponential per state and row, against 32 per clock per SM
    ex2_peak = 32 * 148 * 2.032e9
    assert kernels["scan"]["frac"] == pytest.approx(rows * s.di * s.N / t / ex2_peak, abs=1e-4)
    # four fp32 operations per state and row, against 128 lanes per SM: the same fraction
    assert kernels["scan_fma"]["frac"] == pytest.approx(kernels["scan"]["frac"], abs=1e-4)
    assert kernels["in_proj"]["frac"] == pytest.approx(1908.4e9 / 1.40e-3 / 1e12 / peaks["bf16_tflops"], rel=1e-3)
    # x_proj against HBM: u (fp16) in, dt (fp16, R padded to 8) and B|C (fp32) out, W_x once:
    # 66560 * (3200*2 + 104*2 + 32*4) + 132*3200*2 bytes
    xb = rows * (s.di * 2 + 104 * 2 + 32 * 4) + 132 * s.di * 2
    assert kernels["x_proj"]["bound"] == "hbm"
    assert kernels["x_proj"]["frac"] == pytest.approx(xb / 0.13e-3 / 1e9 / peaks["hbm_gbs"], rel=1e-3)
    # the longest stage wins even when it is not the scan
    stage_ms["in_proj"] = 2.0
    assert bench.stage_rooflines(s, stage_ms, peaks)[1] == "in_proj"


def test_cpu_baseline_line():
    """The oracle's timed CPU baseline (prefill sample and decode sample)
    carries the keys of the bench line."""
    from types import SimpleNamespace
    cb = bench.cpu_baseline(SimpleNamespace(cpu_sample_tokens=64))
    assert cb["kind"] == "oracle" and cb["unit"] == "tokens/s" and cb["value"] > 0 and cb["cores"] >= 1
    assert isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    assert "64 + 128 meta" in cb["sample"]
    assert cb["decode"]["unit"] == "tokens/s" and cb["decode"]["value"] > 0
