"""Layer-level parity on the GPU through the C ABI against the float64
oracle: fp32 tiny workload (relative <= 1e-4), bf16 layers over several
tiles with ragged tails (max-abs <= 2e-2, relative Frobenius <= 1e-2), the
decode step, KV sharing and prefill/decode consistency."""
import numpy as np
import pytest
import torch

from hybrid_attention_ssm_fwd_b300 import layer as hl
from hybrid_attention_ssm_fwd_b300 import synth
from oracle import hymba_ref as ref
from tests.gpu_util import assert_bf16_close, assert_f32_close, cache_np, run_prefill

pytestmark = pytest.mark.gpu
F = np.float64


# --------------------------------------------------------------------------- fp32 path


@pytest.mark.parametrize("kw", [dict(), dict(window=0), dict(rope_theta=10000.0), dict(T=37, window=8),
                                dict(B=3, T=5, M=0, window=1), dict(residual=True, rope_theta=500.0),
                                dict(fusion="concat")])
def test_fp32_tiny_prefill(kw):
    s = synth.tiny_f32(**kw)
    p = synth.make_layer_inputs(s, 0)
    y, _, _ = run_prefill(s, p)
    yr = ref.layer_fwd(p, p["Xt"], s)["Y"]
    assert_f32_close(y, yr, f"fp32 {kw}")


def test_fp32_tiny_decode_chain_matches_longer_prefill():
    T0, n = 40, 30
    s = synth.tiny_f32(T=T0 + n, rope_theta=10000.0)
    p = synth.make_layer_inputs(s, 0)
    cap = s.window
    s0 = synth.with_(s, T=T0)
    y0, cache, _ = run_prefill(s0, p, cap=cap, Xt=p["Xt"][:, : s0.L])
    sd = synth.with_(s, T=1)
    layer = hl.HymbaLayer(sd, hl.params_to_device(p, sd), decode=True)
    ys = []
    for i in range(n):
        xn = hl.tokens_to_device(p["Xt"][:, s0.L + i], sd)
        ys.append(layer.decode(xn, cache, cap).cpu().numpy())
    yr = ref.layer_fwd(p, p["Xt"], s)["Y"][:, s0.L:]
    assert_f32_close(np.stack(ys, 1), yr, "fp32 decode chain")
    assert int(cache["pos"][0].item()) == T0 + n


# --------------------------------------------------------------------------- bf16 path


def small_bf16(**kw):
    base = dict(B=2, T=200, M=16, d=128, Hq=4, Hkv=2, dh=64, di=256, N=16, k=4, window=64, dtype="bf16",
                rope_theta=10000.0)
    base.update(kw)
    return synth._shape(**base)


BF16_CASES = [
    dict(),
    dict(window=0),
    dict(T=333, M=128, window=128, rope_theta=0.0),
    dict(B=1, T=300, M=128, d=1024, Hq=16, Hkv=4, di=2048, window=128),   # 300M-ablation widths
    dict(B=1, T=300, M=128, d=1600, Hq=25, Hkv=5, di=3200, window=256),   # 1.5B widths
    dict(B=3, T=1, M=0, window=1),
    dict(residual=True),
    dict(B=3, T=333),                     # 1047 rows: the projections run as cluster pairs, 9 row blocks
    dict(B=5, T=240, residual=True),      # 1280 rows, 10 row blocks
    dict(fusion="concat"),                # concatenated branches, W_out [d, 2 di]
    dict(B=3, T=333, fusion="concat", residual=True),
]


@pytest.mark.parametrize("kw", BF16_CASES)
def test_bf16_prefill_matches_oracle(kw):
    s = small_bf16(**kw)
    p = synth.make_layer_inputs(s, 1)
    y, _, _ = run_prefill(s, p)
    yr = ref.layer_fwd(p, p["Xt"], s)["Y"]
    assert_bf16_close(y, yr, f"bf16 {kw}")


def test_bf16_prefill_many_row_blocks():
    """1047 rows (nine 128-row GEMM blocks, a ragged last one) through the
    whole layer against the oracle."""
    s = small_bf16(B=3, T=333)
    p = synth.make_layer_inputs(s, 16)
    params = hl.params_to_device(p, s)
    X = hl.tokens_to_device(p["Xt"], s)
    layer = hl.HymbaLayer(s, params)
    y = layer.forward(X).cpu().numpy()
    torch.cuda.synchronize()
    assert layer.check_status() == 0
    yr = ref.layer_fwd(p, p["Xt"], s)["Y"]
    assert_bf16_close(y, yr, "1047 rows")


@pytest.mark.parametrize("n_layers", [4, 3, 1])
def test_bf16_stack_call_matches_oracle(n_layers):
    """hymba_stack_fwd (global layer, window layer exporting K/V, window
    layer reusing them, window layer) against the oracle's stack, which
    rounds each layer's input to bf16 and adds the unrounded stream."""
    shapes = synth.ablation300m_stack(B=2, T=200, M=16, d=128, Hq=4, Hkv=2, di=256)[:n_layers]
    shapes = [synth.with_(s, window=(0 if i == 0 else 64), rope_theta=10000.0) for i, s in enumerate(shapes)]
    tok, layers = synth.make_stack_inputs(shapes, seed=23)
    out = ref.stack_fwd(layers, tok["Xt"], shapes)
    st = hl.HymbaStack(shapes, [hl.params_to_device(p, s) for p, s in zip(layers, shapes)])
    x = hl.tokens_to_device(tok["Xt"], shapes[0])
    for rep in range(2):                  # the call leaves x intact: a second call gives the same stream
        y = st.forward(x)
        torch.cuda.synchronize()
        assert st.check_status() == 0
        assert_bf16_close(y.cpu().numpy(), out["Y"][-1], f"stack of {n_layers}, call {rep}")


def test_bf16_beta_isolation():
    """beta2 = 0 leaves only the attention branch, beta1 = 0 only the SSM one."""
    s = small_bf16()
    p = synth.make_layer_inputs(s, 2)
    for zero in ("beta1", "beta2"):
        q = dict(p)
        q[zero] = np.zeros_like(p[zero])
        y, _, _ = run_prefill(s, q)
        yr = ref.layer_fwd(q, p["Xt"], s)["Y"]
        assert_bf16_close(y, yr, f"{zero}=0")


def test_bf16_kv_sharing_stack():
    """Layer 1 exports K/V, layer 2 consumes them (kv_shared), residual stack."""
    shapes = synth.ablation300m_stack(B=2, T=200, M=16, d=128, Hq=4, Hkv=2, di=256)
    shapes = [synth.with_(s, window=(0 if i == 0 else 64), rope_theta=10000.0) for i, s in enumerate(shapes)]
    tok, layers = synth.make_stack_inputs(shapes, seed=3)
    out = ref.stack_fwd(layers, tok["Xt"], shapes)
    # fp32 residual stream carried in y (residual mode 2); each layer reads it
    # rounded to bf16 as its input X~
    y = torch.from_numpy(tok["Xt"].astype(np.float32)).cuda()
    kv = None
    for i, (p, s) in enumerate(zip(layers, shapes)):
        X = y.to(torch.bfloat16)
        layer = hl.HymbaLayer(s, hl.params_to_device(p, s), residual_mode=2)
        kv_out = None
        if i == 1:
            kd = hl.kv_dtype(s)
            kv_out = (torch.empty(s.B, s.L, s.Hkv, s.dh, device="cuda", dtype=kd),
                      torch.empty(s.B, s.L, s.Hkv, s.dv, device="cuda", dtype=kd))
        layer.forward(X, y=y, kv_in=kv if s.kv_shared else None, kv_out=kv_out)
        torch.cuda.synchronize()
        assert layer.check_status() == 0
        assert_bf16_close(y.cpu().numpy(), out["Y"][i], f"stack layer {i}")
        if kv_out is not None:
            kv = kv_out


def test_bf16_decode_matches_oracle_random_cache():
    s = small_bf16(B=6, T=1, window=64)
    rng_seed = 4
    inp = synth.make_decode_inputs(s, rng_seed, cap=64, pos=500)
    cache = hl.cache_to_device(inp, s)
    layer = hl.HymbaLayer(s, hl.params_to_device(inp, s), decode=True)
    y = layer.decode(hl.tokens_to_device(inp["x_new"], s), cache, 64).cpu().numpy()
    torch.cuda.synchronize()
    assert layer.check_status() == 0
    r = ref.layer_decode(inp, inp["x_new"], {k: inp[k] for k in ("k_ring", "v_ring", "k_meta", "v_meta",
                                                                  "ssm_state", "conv_state", "pos")}, s)
    assert_bf16_close(y, r["y"], "decode y")
    c = cache_np(cache)
    assert_bf16_close(c["ssm_state"], r["cache"]["ssm_state"], "decode ssm_state")
    assert np.all(c["pos"] == 501)
    slot = 500 % 64
    assert_bf16_close(c["k_ring"][:, slot], r["cache"]["k_ring"][:, slot], "decode k slot")


def test_bf16_prefill_then_decode_equals_longer_prefill():
    T0, n = 150, 20
    s = small_bf16(T=T0 + n)
    p = synth.make_layer_inputs(s, 5)
    cap = s.window
    s0 = synth.with_(s, T=T0)
    _, cache, _ = run_prefill(s0, p, cap=cap, Xt=p["Xt"][:, : s0.L])
    sd = synth.with_(s, T=1)
    layer = hl.HymbaLayer(sd, hl.params_to_device(p, sd), decode=True)
    ys = [layer.decode(hl.tokens_to_device(p["Xt"][:, s0.L + i], sd), cache, cap).cpu().numpy() for i in range(n)]
    yr = ref.layer_fwd(p, p["Xt"], s)["Y"][:, s0.L:]
    assert_bf16_close(np.stack(ys, 1), yr, "bf16 prefill->decode")


@pytest.mark.parametrize("kw,cap,pos", [
    # ring not yet full, exactly full, wrapped into two slot ranges; meta of 16 (a partial chunk)
    (dict(B=6, T=1, window=64), 64, [0, 5, 62, 63, 64, 500]),
    # window smaller than the ring, ranges that straddle the ring's end
    (dict(B=4, T=1, window=40, M=70), 100, [3, 39, 130, 199]),
    # global layer: the cache holds every token, no wrap
    (dict(B=3, T=1, window=0, M=0), 300, [0, 150, 299 - 1]),
    # 1.5B widths: G = 5 query heads per KV head, dv = 128, a 1024-slot ring
    (dict(B=3, T=1, M=128, d=1600, Hq=25, Hkv=5, di=3200, window=1024), 1024, [1, 1023, 8192]),
])
def test_bf16_decode_per_sequence_positions(kw, cap, pos):
    """Each sequence at its own position: the visible ring slots form one or
    two ranges of any length, next to a meta prefix that fills a partial
    chunk or none."""
    s = small_bf16(**kw)
    inp = synth.make_decode_inputs(s, 7, cap=cap, pos=0)
    inp["pos"] = np.asarray(pos, np.int32)
    cache = hl.cache_to_device(inp, s)
    layer = hl.HymbaLayer(s, hl.params_to_device(inp, s), decode=True)
    y = layer.decode(hl.tokens_to_device(inp["x_new"], s), cache, cap).cpu().numpy()
    torch.cuda.synchronize()
    assert layer.check_status() == 0
    keys = ("k_ring", "v_ring", "k_meta", "v_meta", "ssm_state", "conv_state", "pos")
    r = ref.layer_decode(inp, inp["x_new"], {k: inp[k] for k in keys}, s)
    assert_bf16_close(y, r["y"], f"decode y {pos}")
    c = cache_np(cache)
    assert np.all(c["pos"] == np.asarray(pos) + 1)
    assert_bf16_close(c["k_ring"], r["cache"]["k_ring"], "decode k_ring")


@pytest.mark.parametrize("kw", [dict(), dict(residual=True)])
def test_bf16_decode_concat_fusion(kw):
    """The concatenation variant through the decode step (norm writes both
    halves, out_proj reduces over 2 di)."""
    s = small_bf16(B=6, T=1, window=64, fusion="concat", **kw)
    inp = synth.make_decode_inputs(s, 9, cap=64, pos=300)
    assert inp["W_out"].shape == (s.d, 2 * s.di)
    cache = hl.cache_to_device(inp, s)
    layer = hl.HymbaLayer(s, hl.params_to_device(inp, s), decode=True)
    y = layer.decode(hl.tokens_to_device(inp["x_new"], s), cache, 64).cpu().numpy()
    torch.cuda.synchronize()
    assert layer.check_status() == 0
    keys = ("k_ring", "v_ring", "k_meta", "v_meta", "ssm_state", "conv_state", "pos")
    r = ref.layer_decode(inp, inp["x_new"], {k: inp[k] for k in keys}, s)
    assert_bf16_close(y, r["y"], f"decode concat {kw}")


def test_fp32_decode_concat_fusion_chain():
    T0, n = 30, 8
    s = synth.tiny_f32(T=T0 + n, rope_theta=10000.0, fusion="concat")
    p = synth.make_layer_inputs(s, 10)
    s0 = synth.with_(s, T=T0)
    _, cache, _ = run_prefill(s0, p, cap=s.window, Xt=p["Xt"][:, : s0.L])
    sd = synth.with_(s, T=1)
    layer = hl.HymbaLayer(sd, hl.params_to_device(p, sd), decode=True)
    ys = [layer.decode(hl.tokens_to_device(p["Xt"][:, s0.L + i], sd), cache, s.window).cpu().numpy()
          for i in range(n)]
    yr = ref.layer_fwd(p, p["Xt"], s)["Y"][:, s0.L:]
    assert_f32_close(np.stack(ys, 1), yr, "fp32 concat decode chain")
