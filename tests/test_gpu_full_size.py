"""Parity at the full workload sizes, in the launch configuration the
benchmark times (same shapes, seeds and calls), on outputs the float64 oracle
can compute at these sizes.

The layer is causal and its sequences are independent, so a sampled row of a
sampled sequence needs only that sequence's prefix: ``layer_fwd_rows`` projects
and scans the prefix and attends for the sampled query rows alone.  The rows
sampled are the meta rows' edge, the first real row, both sides of the
sliding-window edge (meta always visible; "Hymba: A Hybrid-head Architecture
for Small Language Models", sections 2.2 and 2.3), a middle row and the last
rows.  Sequence 0 is checked on its early rows, the batch's last sequence on
all of them, so both ends of the batch and of the sequence are covered.

* Hymba-1.5B-shaped SWA layer: batch 8 x (8192 + 128 meta), window 1024.
* The same shapes as a global-attention layer: batch 2 x (8192 + 128).
* Decode step, batch 128, 8192 tokens of history in a 1024-slot ring plus
  the meta K/V: y, the SSM state and the ring slot written for three
  sequences (first, middle, last); pos of all.
* 300M-ablation-shaped 4-layer stack (global, then three SWA layers; layers
  1 -> 2 share K/V), batch 32 x (2048 + 128), through hymba_stack_fwd as the
  benchmark runs it: every row of the last sequence after 1, 2, 3 and 4
  layers, chained through the fp32 residual stream.
* The full residual block around the SWA layer (gated MLP, F = 3 d), batch
  8 x (8192 + 128): sampled rows against the row-wise block oracle.
"""
import numpy as np
import pytest
import torch

from hybrid_attention_ssm_fwd_b300 import layer as hl
from hybrid_attention_ssm_fwd_b300 import synth
from oracle import hymba_ref as ref
from tests.gpu_util import assert_bf16_close, cache_np, run_prefill

pytestmark = pytest.mark.gpu


def _rows(s):
    M, W, L = s.M, s.window if s.window > 0 else 1024, s.L
    return np.array(sorted({0, M - 1, M, M + 1, M + W - 1, M + W, M + W + 1, L // 2 + 3, L - 2, L - 1}))


@pytest.mark.parametrize("make,seed,what", [
    (lambda: synth.hymba15b_swa(rope_theta=10000.0), 1, "SWA layer, batch 8 x 8K"),
    (lambda: synth.hymba15b_global(rope_theta=10000.0), 2, "global layer, batch 2 x 8K"),
])
def test_full_size_prefill_sampled_rows(make, seed, what):
    s = make()
    p = synth.make_layer_inputs(s, seed)
    y, _, _ = run_prefill(s, p)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    rows = _rows(s)
    early = rows[rows <= s.M + 1025]
    last = s.B - 1
    assert_bf16_close(y[0, early], ref.layer_fwd_rows(p, p["Xt"][:1], s, early)[0], f"{what}, sequence 0")
    assert_bf16_close(y[last, rows], ref.layer_fwd_rows(p, p["Xt"][last:], s, rows)[0], f"{what}, sequence {last}")


def test_full_size_decode_batch128_sampled_sequences():
    s = synth.hymba15b_decode(rope_theta=10000.0)
    cap = s.window
    inp = synth.make_decode_inputs(s, 4, cap=cap, pos=8192)
    cache = hl.cache_to_device(inp, s)
    layer = hl.HymbaLayer(s, hl.params_to_device(inp, s), decode=True)
    y = layer.decode(hl.tokens_to_device(inp["x_new"], s), cache, cap).cpu().numpy()
    torch.cuda.synchronize()
    assert layer.check_status() == 0
    assert np.all(np.isfinite(y))
    idx = [0, s.B // 2 - 1, s.B - 1]
    per_seq = ("k_ring", "v_ring", "ssm_state", "conv_state", "pos")
    sub = {k: inp[k][idx] for k in per_seq}
    sub.update(k_meta=inp["k_meta"], v_meta=inp["v_meta"])
    r = ref.layer_decode(inp, inp["x_new"][idx], sub, synth.with_(s, B=len(idx)))
    assert_bf16_close(y[idx], r["y"], "decode batch 128, y")
    c = cache_np(cache)
    assert_bf16_close(c["ssm_state"][idx], r["cache"]["ssm_state"], "decode batch 128, ssm_state")
    slot = 8192 % cap
    assert_bf16_close(c["k_ring"][idx, slot], r["cache"]["k_ring"][:, slot], "decode batch 128, k slot")
    assert_bf16_close(c["v_ring"][idx, slot], r["cache"]["v_ring"][:, slot], "decode batch 128, v slot")
    assert np.all(c["pos"] == 8193)


@pytest.mark.parametrize("n_layers", [1, 2, 3, 4])
def test_full_size_stack_call_last_sequence(n_layers):
    """The first n layers of the 4-layer stack through one hymba_stack_fwd
    call each, as the benchmark runs it (n = 4): the fp32 stream after layer
    n - 1, every row of the last sequence, chained with no reset, against the
    oracle's stack (the stream at full precision)."""
    shapes = [synth.with_(s, rope_theta=10000.0) for s in synth.ablation300m_stack()]
    tok, layers = synth.make_stack_inputs(shapes, seed=3)
    b = shapes[0].B - 1
    out = ref.stack_fwd(layers[:n_layers], tok["Xt"][b:b + 1], [synth.with_(s, B=1) for s in shapes[:n_layers]])
    st = hl.HymbaStack(shapes[:n_layers], [hl.params_to_device(p, s) for p, s in zip(layers, shapes[:n_layers])])
    y = st.forward(hl.tokens_to_device(tok["Xt"], shapes[0]))
    torch.cuda.synchronize()
    assert st.check_status() == 0
    assert_bf16_close(y[b].cpu().numpy(), out["Y"][-1][0],
                      f"stack call, batch 32 x 2K, after layer {n_layers - 1}, sequence {b}")
    del st, y


def test_full_size_block_sampled_rows():
    """hymba_block_fwd over batch 8 x (8192 + 128) at the 1.5B shapes with
    F = 3 d, as the benchmark runs it, against block_fwd_rows on sampled
    rows of the first and last sequences."""
    from oracle import block_ref as br
    s = synth.hymba15b_swa(rope_theta=10000.0)
    d_ff = 3 * s.d
    tok, blocks = synth.make_block_inputs(s, d_ff, 4)
    blk = hl.HymbaBlock(s, hl.block_params_to_device(blocks[0], s), d_ff)
    x = torch.from_numpy(tok["Xt"]).cuda()
    blk.forward(x)
    torch.cuda.synchronize()
    assert blk.check_status() == 0
    y = x.cpu().numpy()
    assert np.all(np.isfinite(y))
    del blk, x
    rows = _rows(s)
    early = rows[rows <= s.M + 1025]
    last = s.B - 1
    assert_bf16_close(y[0, early], br.block_fwd_rows(blocks[0], tok["Xt"][:1], s, early)[0], "block, sequence 0")
    assert_bf16_close(y[last, rows], br.block_fwd_rows(blocks[0], tok["Xt"][last:], s, rows)[0],
                      f"block, sequence {last}")
