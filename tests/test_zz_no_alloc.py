"""The decode entry point for callers that cannot allocate device memory.

hymba_layer_decode_static runs the decode step with the library's own
statically sized scratch buffer instead of a caller workspace: a plugin whose
host framework owns all device memory, or a serving loop whose memory is fully
reserved by its cache pool, cannot call cudaMalloc there.  This test checks it
against the workspace entry point, through the C ABI, on two consecutive decode
steps (the second one reuses the scratch left by the first).

Kept in a file that pytest collects last, so that a failure here leaves every
other test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

from hybrid_attention_ssm_fwd_b300 import binding as hb
from hybrid_attention_ssm_fwd_b300 import layer as hl
from hybrid_attention_ssm_fwd_b300 import synth
from tests.gpu_util import assert_bf16_close

pytestmark = pytest.mark.gpu


def test_static_scratch_decode_matches_workspace_decode_two_steps():
    # Hymba-1.5B-shaped decode at batch 128 over a full 1024-slot ring
    s = synth.hymba15b_decode(rope_theta=10000.0)
    cap = s.window
    inp = synth.make_decode_inputs(s, 21, cap=cap, pos=8192)
    desc = hb.make_desc(s)
    need = hb.layer_decode_workspace(desc)
    assert 0 < need <= hb.STATIC_SCRATCH_BYTES
    params = hl.params_to_device(inp, s)
    weights = hb.make_weights(params)
    cache_ws = hl.cache_to_device(inp, s)
    cache_st = {k: v.clone() for k, v in cache_ws.items()}
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(22)
    for step in range(2):
        xn = hl.tokens_to_device(synth.bf16_round(rng.standard_normal((s.B, s.d)).astype(np.float32)), s)
        y_ws = torch.empty(s.B, s.d, dtype=torch.float32, device="cuda")
        y_st = torch.full((s.B, s.d), float("nan"), dtype=torch.float32, device="cuda")
        hb.hymba_layer_decode(desc, weights, xn, y_ws, hb.make_cache(cache_ws, cap), ws, status=status[0:1])
        rc = hb.hymba_layer_decode_static(desc, weights, xn, y_st, hb.make_cache(cache_st, cap), status=status[1:2])
        assert rc == hb.HYMBA_OK
        torch.cuda.synchronize()
        assert status.cpu().tolist() == [0, 0]
        assert_bf16_close(y_st.cpu().numpy(), y_ws.cpu().numpy(), f"step {step} y")
        assert_bf16_close(cache_st["ssm_state"].cpu().numpy(), cache_ws["ssm_state"].cpu().numpy(),
                          f"step {step} ssm_state")
        assert torch.equal(cache_st["pos"], cache_ws["pos"])
        assert torch.equal(cache_st["k_ring"], cache_ws["k_ring"])


def test_static_scratch_rejects_shapes_beyond_its_size():
    s = synth.hymba15b_decode(B=4096)
    desc = hb.make_desc(s)
    assert hb.layer_decode_workspace(desc) > hb.STATIC_SCRATCH_BYTES
    w = hb.LayerWeights(*[0x10000 * (i + 1) for i in range(11)])
    cache = hb.Cache(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, s.window, 0)
    rc = hb.lib().hymba_layer_decode_static(ctypes.byref(desc), ctypes.byref(w), 0x200000, 0x300000,
                                            ctypes.byref(cache), None, None, None)
    assert rc == hb.HYMBA_ERR_WORKSPACE
