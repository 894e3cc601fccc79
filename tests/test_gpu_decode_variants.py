"""Decode-step variants on the GPU through the C ABI against the float64
oracle ("Hymba: A Hybrid-head Architecture for Small Language Models",
section 2.2: a window-bounded cache per sequence, K/V shared by consecutive
layers):

* a KV-sharing consumer layer decoding from its producer's cache, against
  the oracle's shared decode and, chained, against the longer prefill;
* admitting a new sequence into row b of a running batch-128 cache (a batch-1
  prefill whose cache_out points at that row), then stepping the whole batch:
  the admitted row and the rows around it against the oracle, and the other
  rows' caches untouched by the admission.
bf16 tolerances: max-abs <= 2e-2 and relative Frobenius <= 1e-2."""
import numpy as np
import pytest
import torch

from hybrid_attention_ssm_fwd_b300 import layer as hl
from hybrid_attention_ssm_fwd_b300 import synth
from oracle import hymba_ref as ref
from tests.gpu_util import assert_bf16_close, cache_np, run_prefill

pytestmark = pytest.mark.gpu
F = np.float64
KEYS = ("k_ring", "v_ring", "k_meta", "v_meta", "ssm_state", "conv_state", "pos")


def small_bf16(**kw):
    base = dict(B=4, T=1, M=16, d=128, Hq=4, Hkv=2, dh=64, di=256, N=16, k=4, window=64, dtype="bf16",
                rope_theta=10000.0)
    base.update(kw)
    return synth._shape(**base)


def _consumer_params(s, seed):
    """Parameters of a KV-sharing consumer: its own draw with the K/V rows of
    W_in dropped (the shared layer has no K/V projection)."""
    p = synth.make_layer_inputs(s, seed)
    qn = s.Hq * s.dh
    kvn = s.Hkv * (s.dh + s.dv)
    q = dict(p)
    q["W_in"] = np.concatenate([p["W_in"][:qn], p["W_in"][qn + kvn:]], 0)
    return q


@pytest.mark.parametrize("kw,cap,pos", [
    (dict(), 64, [3, 63, 64, 500]),
    (dict(window=0, M=0, B=3), 300, [0, 150, 298]),
    (dict(B=6, M=128, d=1600, Hq=25, Hkv=5, di=3200, window=1024), 1024, [0, 700, 1023, 1024, 5000, 8192]),
])
def test_decode_kv_shared_consumer_matches_oracle(kw, cap, pos):
    """Producer step (writes this token's K/V into its cache), then the
    consumer step reading the producer's cache; the consumer's y and SSM
    state against the oracle's shared decode."""
    s = small_bf16(**kw)
    inp = synth.make_decode_inputs(s, 31, cap=cap, pos=0)
    inp["pos"] = np.asarray(pos, np.int32)
    sc = synth.with_(s, kv_shared=True)
    cons = _consumer_params(s, 32)
    own = {"ssm_state": synth.make_decode_inputs(s, 33, cap=cap, pos=0)["ssm_state"],
           "conv_state": inp["conv_state"][::-1].copy(), "pos": inp["pos"].copy()}

    pcache = hl.cache_to_device(inp, s)
    ccache = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in own.items()}
    ccache["ssm_state"] = ccache["ssm_state"].float()
    ccache["conv_state"] = ccache["conv_state"].float()
    prod = hl.HymbaLayer(s, hl.params_to_device(inp, s), decode=True)
    con = hl.HymbaLayer(sc, hl.params_to_device(cons, sc), decode=True)
    xn = hl.tokens_to_device(inp["x_new"], s)
    prod.decode(xn, pcache, cap)
    y = con.decode(xn, ccache, cap, shared_cache=pcache, shared_cap=cap).cpu().numpy()
    torch.cuda.synchronize()
    assert prod.check_status() == 0 and con.check_status() == 0

    rp = ref.layer_decode(inp, inp["x_new"], {k: inp[k] for k in KEYS}, s)
    rc = ref.layer_decode(cons, inp["x_new"], own, sc, shared_cache=rp["cache"])
    assert_bf16_close(y, rc["y"], f"shared decode y {pos}")
    c = cache_np(ccache)
    assert_bf16_close(c["ssm_state"], rc["cache"]["ssm_state"], "shared decode ssm_state")
    assert np.all(c["pos"] == np.asarray(pos) + 1)


@pytest.mark.parametrize("T0,n,window", [(150, 20, 64), (40, 12, 0)])
def test_decode_chain_kv_shared_consumer_equals_longer_prefill(T0, n, window):
    """Producer and consumer prefill T0 tokens (the consumer from the
    producer's exported K/V), then n decode steps, producer first; the
    consumer's outputs against the oracle's longer prefill."""
    s = small_bf16(B=2, T=T0 + n, window=window)
    cap = window if window > 0 else T0 + n
    pp = synth.make_layer_inputs(s, 41)
    sc = synth.with_(s, kv_shared=True)
    cons = _consumer_params(s, 42)
    s0, sc0 = synth.with_(s, T=T0), synth.with_(sc, T=T0)
    X0 = pp["Xt"][:, : s0.L]
    _, pcache, kv = run_prefill(s0, pp, cap=cap, want_kv=True, Xt=X0)
    _, ccache, _ = run_prefill(sc0, cons, cap=cap, kv_in=kv, Xt=X0)
    sd, scd = synth.with_(s, T=1), synth.with_(sc, T=1)
    prod = hl.HymbaLayer(sd, hl.params_to_device(pp, sd), decode=True)
    con = hl.HymbaLayer(scd, hl.params_to_device(cons, scd), decode=True)
    ys = []
    for i in range(n):
        xn = hl.tokens_to_device(pp["Xt"][:, s0.L + i], sd)
        prod.decode(xn, pcache, cap)
        ys.append(con.decode(xn, ccache, cap, shared_cache=pcache, shared_cap=cap).cpu().numpy())
    torch.cuda.synchronize()
    assert prod.check_status() == 0 and con.check_status() == 0
    pf = ref.layer_fwd(pp, pp["Xt"], s)
    cf = ref.layer_fwd(cons, pp["Xt"], sc, kv_in=(pf["K"], pf["V"]), cache_cap=cap)
    assert_bf16_close(np.stack(ys, 1), cf["Y"][:, s.M + T0:], "shared consumer decode chain")
    assert_bf16_close(cache_np(ccache)["ssm_state"], cf["cache"]["ssm_state"], "shared consumer final state")


def test_admit_sequence_into_row_of_batch128_cache():
    """Continuous batching at the 1.5B decode shapes: 127 sequences sit at
    position 8192 in a batch-128 cache; a new sequence of 300 tokens is
    prefilled alone into row b (cache_out = that row's pointers, the meta
    K/V shared), then one decode step runs the whole batch with per-sequence
    positions (8192 for the others, 300 for row b)."""
    s = synth.hymba15b_decode(rope_theta=10000.0)
    cap, b, T0 = s.window, 77, 300
    inp = synth.make_decode_inputs(s, 51, cap=cap, pos=8192)
    cache = hl.cache_to_device(inp, s)
    before = {k: cache[k][[b - 1, b + 1]].clone() for k in ("k_ring", "v_ring", "ssm_state", "conv_state")}

    sp = synth.with_(s, B=1, T=T0)
    newseq = synth.make_layer_inputs(sp, 52)
    pa = {k: inp[k] for k in inp if k not in KEYS and k != "x_new"}   # the layer's weights
    for k in ("X", "meta", "Xt"):
        pa[k] = newseq[k]
    y0, _, _ = run_prefill(sp, pa, cap=cap)                   # warm, unrelated buffers
    layer = hl.HymbaLayer(sp, hl.params_to_device(pa, sp))
    layer.forward(hl.tokens_to_device(pa["Xt"], sp), cache_out=hl.cache_row(cache, b), cap=cap)
    torch.cuda.synchronize()
    assert layer.check_status() == 0
    assert int(cache["pos"][b].item()) == T0
    for k, v in before.items():
        assert torch.equal(cache[k][[b - 1, b + 1]], v), f"admission touched {k} of other rows"

    dec = hl.HymbaLayer(s, hl.params_to_device(inp, s), decode=True)
    y = dec.decode(hl.tokens_to_device(inp["x_new"], s), cache, cap).cpu().numpy()
    torch.cuda.synchronize()
    assert dec.check_status() == 0
    c = cache_np(cache)
    assert c["pos"][b] == T0 + 1 and np.all(np.delete(c["pos"], b) == 8193)

    # row b: the oracle's prefill of the new sequence, then its decode step
    pre = ref.layer_fwd(pa, pa["Xt"], sp, cache_cap=cap)
    rb = ref.layer_decode(inp, inp["x_new"][b:b + 1], pre["cache"], synth.with_(s, B=1))
    assert_bf16_close(y[b:b + 1], rb["y"], "admitted row y")
    assert_bf16_close(c["ssm_state"][b:b + 1], rb["cache"]["ssm_state"], "admitted row ssm_state")
    # its neighbours: their own random history, with the meta K/V the
    # admission wrote (the meta rows are the same for every sequence)
    idx = [b - 1, b + 1]
    sub = {k: inp[k][idx] for k in ("k_ring", "v_ring", "ssm_state", "conv_state", "pos")}
    sub.update(k_meta=pre["cache"]["k_meta"], v_meta=pre["cache"]["v_meta"])
    rn = ref.layer_decode(inp, inp["x_new"][idx], sub, synth.with_(s, B=2))
    assert_bf16_close(y[idx], rn["y"], "neighbour rows y")
