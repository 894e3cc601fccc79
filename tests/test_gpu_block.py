"""The full residual block (hymba_block_fwd) on the GPU through the C ABI
against the float64 block oracle: RMSNorm -> hybrid-head layer -> add, then
RMSNorm -> GeLU-gated MLP -> add ("Griffin: Mixing Gated Linear Recurrences
with Local Attention for Efficient Language Models", sections 2.1 and 2.2).
bf16 tolerances of the layer tests (max-abs <= 2e-2, relative Frobenius <=
1e-2) on the fp32 stream."""
import numpy as np
import pytest
import torch

from hybrid_attention_ssm_fwd_b300 import layer as hl
from hybrid_attention_ssm_fwd_b300 import synth
from oracle import block_ref as br
from tests.gpu_util import assert_bf16_close

pytestmark = pytest.mark.gpu


def small_bf16(**kw):
    base = dict(B=2, T=200, M=16, d=128, Hq=4, Hkv=2, dh=64, di=256, N=16, k=4, window=64, dtype="bf16",
                rope_theta=10000.0)
    base.update(kw)
    return synth._shape(**base)


BLOCK_CASES = [
    (dict(), 384),
    (dict(window=0, rope_theta=0.0), 384),
    (dict(B=3, T=333), 384),                                              # 1047 rows: cluster-pair GEMMs
    (dict(B=1, T=300, M=128, d=1600, Hq=25, Hkv=5, di=3200, window=256), 4800),  # 1.5B widths, F = 3d
    (dict(), 200),                                                        # F not a multiple of the tile
]


def _run_block(s, pb, Xt, d_ff):
    blk = hl.HymbaBlock(s, hl.block_params_to_device(pb, s), d_ff)
    x = torch.from_numpy(np.ascontiguousarray(Xt, dtype=np.float32)).cuda()
    blk.forward(x)
    torch.cuda.synchronize()
    assert blk.check_status() == 0, f"device status {blk.check_status()}"
    return x.cpu().numpy()


@pytest.mark.parametrize("kw,d_ff", BLOCK_CASES)
def test_block_matches_oracle(kw, d_ff):
    s = small_bf16(**kw)
    tok, blocks = synth.make_block_inputs(s, d_ff, 21)
    y = _run_block(s, blocks[0], tok["Xt"], d_ff)
    ref = br.block_fwd(blocks[0], tok["Xt"], s)
    assert_bf16_close(y, ref["Y"], f"block {kw} F={d_ff}")


def test_block_mlp_off_equals_layer_sub_block():
    """W_gate = 0 switches the MLP off (GeLU(0) = 0): the stream after the
    block is the mixer sub-block alone."""
    s = small_bf16()
    tok, blocks = synth.make_block_inputs(s, 384, 22)
    pb = dict(blocks[0])
    pb["W_gate"] = np.zeros_like(pb["W_gate"])
    y = _run_block(s, pb, tok["Xt"], 384)
    ref = br.block_fwd(pb, tok["Xt"], s)
    np.testing.assert_array_equal(ref["Y"], ref["Y1"])
    assert_bf16_close(y, ref["Y1"], "mixer sub-block")


def test_two_block_stack():
    s = small_bf16(B=2, T=150)
    tok, blocks = synth.make_block_inputs(s, 384, 23, n_blocks=2)
    x = torch.from_numpy(np.ascontiguousarray(tok["Xt"], dtype=np.float32)).cuda()
    for pb in blocks:
        blk = hl.HymbaBlock(s, hl.block_params_to_device(pb, s), 384)
        blk.forward(x)
        torch.cuda.synchronize()
        assert blk.check_status() == 0
    ref = br.blocks_fwd(blocks, tok["Xt"], [s, s])
    assert_bf16_close(x.cpu().numpy(), ref, "two blocks")
