"""Meta-prefix precompute on the GPU through the C ABI.

The M meta tokens are the same learned rows at the head of every sequence
("Hymba: A Hybrid-head Architecture for Small Language Models", section 2.3),
so hymba_meta_prefill runs the layer once over them and hymba_layer_fwd_meta
runs the real tokens of a whole batch from that state.  Checked against the
float64 oracle on the full sequences [meta | tokens]: Y of the real rows,
Y / SSM state / conv tail of the meta rows, the decode cache a prefill leaves
(through decode steps that follow it), and a KV-sharing residual stack.
"""
import numpy as np
import pytest
import torch

from hybrid_attention_ssm_fwd_b300 import layer as hl
from hybrid_attention_ssm_fwd_b300 import synth
from oracle import hymba_ref as ref
from tests.gpu_util import assert_bf16_close, run_prefill

pytestmark = pytest.mark.gpu


def small_bf16(**kw):
    base = dict(B=2, T=200, M=64, d=128, Hq=4, Hkv=2, dh=64, di=256, N=16, k=4, window=64, dtype="bf16",
                rope_theta=10000.0)
    base.update(kw)
    return synth._shape(**base)


META_CASES = [
    dict(),
    dict(M=128, window=0),
    dict(M=128, T=333, window=128, rope_theta=0.0),
    dict(residual=True),
    dict(B=3, T=2),                                                      # fewer real rows than one tile
    dict(B=2, T=300, M=128, d=1600, Hq=25, Hkv=5, di=3200, window=256),  # 1.5B widths (dv = 128)
    dict(B=4, T=300),                                                    # 1200 real rows: cluster-pair GEMMs
    dict(fusion="concat"),
]


def _sync_ok(layer):
    torch.cuda.synchronize()
    assert layer.check_status() == 0, f"device status {layer.check_status()}"


@pytest.mark.parametrize("kw", META_CASES)
def test_meta_prefix_matches_oracle(kw):
    s = small_bf16(**kw)
    p = synth.make_layer_inputs(s, 11)
    layer = hl.HymbaLayer(s, hl.params_to_device(p, s))
    meta = layer.meta_prefill(hl.tokens_to_device(p["meta"], s))
    y = layer.forward_meta(meta, hl.tokens_to_device(p["X"], s))
    _sync_ok(layer)
    o = ref.layer_fwd(p, p["Xt"], s)
    assert_bf16_close(y.cpu().numpy(), o["Y"][:, s.M:], f"real rows {kw}")
    assert_bf16_close(meta["y"].cpu().numpy(), o["Y"][0, : s.M], f"meta rows {kw}")
    # the meta rows' own state: SSM state and conv tail after row M-1
    sm = synth.with_(s, B=1, T=0)
    om = ref.layer_fwd(p, p["Xt"][:1, : s.M], sm, cache_cap=1)["cache"]
    assert_bf16_close(meta["ssm_state"].cpu().numpy(), om["ssm_state"][0], "meta ssm_state")
    assert_bf16_close(meta["conv_tail"].cpu().numpy(), om["conv_state"][0], "meta conv tail")
    # and the same rows of the one-call prefill over [meta | tokens]
    yf, _, _ = run_prefill(s, p)
    assert_bf16_close(y.cpu().numpy(), yf[:, s.M:], "meta path vs one-call prefill")


@pytest.mark.parametrize("T0", [150, 2])
def test_meta_prefix_then_decode_equals_longer_prefill(T0):
    """The cache a meta-path prefill leaves (ring, meta K/V, SSM state, conv
    tail: with T0 < k-1 part of it comes from the meta rows) carries decode
    on exactly as the oracle's longer prefill does."""
    n = 12
    s = small_bf16(T=T0 + n)
    p = synth.make_layer_inputs(s, 12)
    cap = s.window
    s0 = synth.with_(s, T=T0)
    layer = hl.HymbaLayer(s0, hl.params_to_device(p, s0))
    meta = layer.meta_prefill(hl.tokens_to_device(p["meta"], s0))
    cache = hl.alloc_cache(s0, cap)
    y0 = layer.forward_meta(meta, hl.tokens_to_device(p["X"][:, :T0], s0), cache_out=cache, cap=cap)
    _sync_ok(layer)
    sd = synth.with_(s, T=1)
    dec = hl.HymbaLayer(sd, hl.params_to_device(p, sd), decode=True)
    ys = [dec.decode(hl.tokens_to_device(p["X"][:, T0 + i], sd), cache, cap).cpu().numpy() for i in range(n)]
    _sync_ok(dec)
    o = ref.layer_fwd(p, p["Xt"], s)
    assert_bf16_close(y0.cpu().numpy(), o["Y"][:, s.M: s.M + T0], "prefill rows")
    assert_bf16_close(np.stack(ys, 1), o["Y"][:, s.M + T0:], "decode after meta-path prefill")
    assert np.all(cache["pos"].cpu().numpy() == T0 + n)


def test_meta_prefix_kv_sharing_stack():
    """Global layer, window layer exporting K/V, window layer reusing them
    (kv_shared), on the fp32 residual stream (residual mode 2): the meta rows
    go through the stack once, the real rows of the batch once."""
    shapes = synth.ablation300m_stack(B=2, T=200, M=64, d=128, Hq=4, Hkv=2, di=256)[:3]
    shapes = [synth.with_(s, window=(0 if i == 0 else 64), rope_theta=10000.0) for i, s in enumerate(shapes)]
    tok, layers = synth.make_stack_inputs(shapes, seed=13)
    out = ref.stack_fwd(layers, tok["Xt"], shapes)
    M = shapes[0].M
    y_meta = torch.from_numpy(tok["meta"].astype(np.float32)).cuda()
    y = torch.from_numpy(tok["X"].astype(np.float32)).cuda()
    kv_meta = kv_real = None
    for i, (p, s) in enumerate(zip(layers, shapes)):
        layer = hl.HymbaLayer(s, hl.params_to_device(p, s), residual_mode=2)
        meta = layer.meta_prefill(y_meta.to(torch.bfloat16), y=y_meta, kv_in=kv_meta if s.kv_shared else None)
        kv_out = None
        if i == 1:
            kd = hl.kv_dtype(s)
            kv_out = (torch.empty(s.B, s.T, s.Hkv, s.dh, device="cuda", dtype=kd),
                      torch.empty(s.B, s.T, s.Hkv, s.dv, device="cuda", dtype=kd))
        layer.forward_meta(meta, y.to(torch.bfloat16), y=y, kv_in=kv_real if s.kv_shared else None, kv_out=kv_out)
        _sync_ok(layer)
        assert_bf16_close(y.cpu().numpy(), out["Y"][i][:, M:], f"stack layer {i} real rows")
        assert_bf16_close(y_meta.cpu().numpy(), out["Y"][i][0, :M], f"stack layer {i} meta rows")
        if i == 1:
            kv_meta, kv_real = (meta["k"], meta["v"]), kv_out


def test_meta_prefix_unsupported_shapes_raise():
    s = small_bf16(M=96)
    p = synth.make_layer_inputs(s, 14)
    layer = hl.HymbaLayer(s, hl.params_to_device(p, s))
    with pytest.raises(Exception):
        layer.meta_prefill(hl.tokens_to_device(p["meta"], s))
