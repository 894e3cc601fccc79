"""Host-side checks of the C-ABI library, no GPU needed: it loads, exports
every entry point include/hymba.h declares, and rejects bad arguments
synchronously before touching CUDA."""
import ctypes
import os
import re

import pytest

from hybrid_attention_ssm_fwd_b300 import binding as hb
from hybrid_attention_ssm_fwd_b300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "hymba.h")).read()
    return sorted(set(re.findall(r"HYMBA_API\s+[\w\s\*]+?\b(hymba_\w+)\s*\(", text)))


def test_library_loads_and_exports_every_declared_symbol():
    L = hb.lib()
    syms = declared_symbols()
    assert len(syms) >= 10
    for name in syms:
        assert hasattr(L, name), name
    assert L.hymba_abi_version() == 1


def test_status_strings():
    for code in range(7):
        assert hb.status_str(code).startswith("HYMBA_")
    assert "unknown" in hb.status_str(99)


def _fake_weights():
    # 256-aligned fake device addresses: never dereferenced because every
    # call below fails validation first
    return hb.LayerWeights(*[0x10000 * (i + 1) for i in range(11)])


def _desc(**kw):
    s = synth.hymba15b_swa(B=2, T=64)
    d = hb.make_desc(s)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_workspace_query():
    d = _desc()
    n = hb.layer_fwd_workspace(d)
    s = synth.hymba15b_swa(B=2, T=64)
    rows = s.B * s.L
    assert n >= rows * s.P_in * 2 + rows * s.di * (2 * 4 + 4)
    assert hb.layer_decode_workspace(hb.make_desc(synth.hymba15b_decode(B=4))) > 0
    assert hb.layer_fwd_workspace(_desc(n_q_heads=7)) == 0          # Hq % Hkv != 0
    assert hb.layer_decode_workspace(_desc()) == 0                  # decode needs n_tokens == 1


@pytest.mark.parametrize("field,value", [("batch", 0), ("n_tokens", 0), ("head_dim", 63), ("d_state", 65),
                                         ("d_conv", 9), ("window", -1), ("kv_shared", 2), ("dtype", 5),
                                         ("v_head_dim", 64), ("eps", -1.0)])
def test_invalid_desc_rejected_before_launch(field, value):
    d = _desc(**{field: value})
    w = _fake_weights()
    ws = ctypes.c_void_p(0x100000)
    rc = hb.lib().hymba_layer_fwd(ctypes.byref(d), ctypes.byref(w), 0x200000, 0x300000, None, None, None, ws,
                                  1 << 40, None, None)
    assert rc == hb.HYMBA_ERR_INVALID


def test_reserved_fields_must_be_zero():
    d = _desc()
    d.reserved = 3
    assert hb.layer_fwd_workspace(d) == 0


def test_reserved0_must_be_zero():
    """desc.reserved0 is a reserved word: any nonzero value is rejected."""
    d = _desc()
    assert hb.layer_fwd_workspace(d) > 0
    d.reserved0 = 1
    assert hb.layer_fwd_workspace(d) == 0


def test_null_and_misaligned_pointers_rejected():
    d = _desc()
    w = _fake_weights()
    L = hb.lib()
    big = 1 << 40
    assert L.hymba_layer_fwd(ctypes.byref(d), ctypes.byref(w), None, 0x300000, None, None, None, 0x100000, big,
                             None, None) == hb.HYMBA_ERR_INVALID
    assert L.hymba_layer_fwd(ctypes.byref(d), ctypes.byref(w), 0x200002, 0x300000, None, None, None, 0x100000, big,
                             None, None) == hb.HYMBA_ERR_INVALID
    assert L.hymba_layer_fwd(ctypes.byref(d), ctypes.byref(w), 0x200000, 0x300000, None, None, None, 0x100010, big,
                             None, None) == hb.HYMBA_ERR_INVALID
    w.W_in = None
    assert L.hymba_layer_fwd(ctypes.byref(d), ctypes.byref(w), 0x200000, 0x300000, None, None, None, 0x100000, big,
                             None, None) == hb.HYMBA_ERR_INVALID


def test_kv_sharing_pairing_enforced():
    w = _fake_weights()
    L = hb.lib()
    kv = hb.KV(0x400000, 0x500000)
    d = _desc()
    assert L.hymba_layer_fwd(ctypes.byref(d), ctypes.byref(w), 0x200000, 0x300000, None, ctypes.byref(kv), None,
                             0x100000, 1 << 40, None, None) == hb.HYMBA_ERR_INVALID
    d = _desc(kv_shared=1)
    assert L.hymba_layer_fwd(ctypes.byref(d), ctypes.byref(w), 0x200000, 0x300000, None, None, None, 0x100000,
                             1 << 40, None, None) == hb.HYMBA_ERR_INVALID


def test_workspace_too_small():
    d = _desc()
    w = _fake_weights()
    need = hb.layer_fwd_workspace(d)
    rc = hb.lib().hymba_layer_fwd(ctypes.byref(d), ctypes.byref(w), 0x200000, 0x300000, None, None, None,
                                  0x100000, need - 1, None, None)
    assert rc == hb.HYMBA_ERR_WORKSPACE


def test_decode_argument_checks():
    s = synth.hymba15b_decode(B=4)
    d = hb.make_desc(s)
    w = _fake_weights()
    L = hb.lib()
    cache = hb.Cache(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 512, 0)   # cap < window
    rc = L.hymba_layer_decode(ctypes.byref(d), ctypes.byref(w), 0x200000, 0x300000, ctypes.byref(cache), None,
                              0x100000, 1 << 40, None, None)
    assert rc == hb.HYMBA_ERR_INVALID
    cache.cap = 1024
    cache.pos = None
    rc = L.hymba_layer_decode(ctypes.byref(d), ctypes.byref(w), 0x200000, 0x300000, ctypes.byref(cache), None,
                              0x100000, 1 << 40, None, None)
    assert rc == hb.HYMBA_ERR_INVALID


def test_unaligned_bf16_shapes_unsupported():
    d = _desc(d_model=1604)
    assert hb.layer_fwd_workspace(d) == 0


def test_meta_prefix_workspace_and_support():
    # the meta-prefix calls: bf16, dh 64, M a positive multiple of 64
    d = _desc()
    assert hb.meta_prefill_workspace(d) > 0
    assert hb.layer_fwd_meta_workspace(_desc(n_tokens=256)) > hb.meta_prefill_workspace(d)  # B*T vs M rows
    assert hb.meta_prefill_workspace(_desc(n_meta=96)) == 0
    assert hb.layer_fwd_meta_workspace(_desc(n_meta=0)) == 0
    assert hb.layer_fwd_meta_workspace(_desc(dtype=hb.HYMBA_F32)) == 0


def test_meta_prefix_rejects_bad_arguments_before_launch():
    d = _desc()
    w = _fake_weights()
    ws = ctypes.c_void_p(0x100000)
    full = hb.Meta(k=0x400000, v=0x500000, ssm_state=0x600000, conv_tail=0x700000, y=0x800000)
    L = hb.lib()
    # no meta state
    rc = L.hymba_layer_fwd_meta(ctypes.byref(d), ctypes.byref(w), None, 0x200000, 0x300000, None, None, None, ws,
                                1 << 40, None, None)
    assert rc == hb.HYMBA_ERR_INVALID
    # missing meta K/V on a layer that owns its K/V
    part = hb.Meta(k=0, v=0, ssm_state=0x600000, conv_tail=0x700000, y=0x800000)
    rc = L.hymba_layer_fwd_meta(ctypes.byref(d), ctypes.byref(w), ctypes.byref(part), 0x200000, 0x300000, None, None,
                                None, ws, 1 << 40, None, None)
    assert rc == hb.HYMBA_ERR_INVALID
    rc = L.hymba_meta_prefill(ctypes.byref(d), ctypes.byref(w), 0x200000, ctypes.byref(part), None, ws, 1 << 40,
                              None, None)
    assert rc == hb.HYMBA_ERR_INVALID
    # kv_in given on a layer that owns its K/V
    kv = hb.KV(k=0x900000, v=0xa00000)
    rc = L.hymba_meta_prefill(ctypes.byref(d), ctypes.byref(w), 0x200000, ctypes.byref(full), ctypes.byref(kv), ws,
                              1 << 40, None, None)
    assert rc == hb.HYMBA_ERR_INVALID
    # workspace too small
    rc = L.hymba_meta_prefill(ctypes.byref(d), ctypes.byref(w), 0x200000, ctypes.byref(full), None, ws, 16, None,
                              None)
    assert rc == hb.HYMBA_ERR_WORKSPACE
    # unsupported meta count
    d96 = _desc(n_meta=96)
    rc = L.hymba_layer_fwd_meta(ctypes.byref(d96), ctypes.byref(w), ctypes.byref(full), 0x200000, 0x300000, None,
                                None, None, ws, 1 << 40, None, None)
    assert rc == hb.HYMBA_ERR_UNSUPPORTED


def test_block_workspace_and_argument_checks():
    d = _desc(residual=0)
    n = hb.block_fwd_workspace(d, 4800)
    assert n > hb.layer_fwd_workspace(d)
    assert hb.block_fwd_workspace(d, 4801) == 0                      # d_ff % 8 != 0
    assert hb.block_fwd_workspace(_desc(residual=1), 4800) == 0      # the block adds the stream itself
    assert hb.block_fwd_workspace(_desc(residual=0, dtype=hb.HYMBA_F32), 4800) == 0
    w = hb.BlockWeights(mix=_fake_weights(), norm1=0x400000, norm2=0x500000, W_gu=0x600000, W_down=0)
    rc = hb.lib().hymba_block_fwd(ctypes.byref(d), ctypes.byref(w), 4800, 0x200000, ctypes.c_void_p(0x100000),
                                  1 << 40, None, None)
    assert rc == hb.HYMBA_ERR_INVALID                                 # W_down missing
    w.W_down = 0x700000
    rc = hb.lib().hymba_block_fwd(ctypes.byref(d), ctypes.byref(w), 4800, 0x200000, ctypes.c_void_p(0x100000),
                                  16, None, None)
    assert rc == hb.HYMBA_ERR_WORKSPACE


def test_stack_workspace_and_argument_checks():
    """hymba_stack_fwd: descriptors validated before any launch (one batch
    shape, residual 0, no sharing into layer 0, bf16 only), the workspace
    covers the largest layer plus the bf16 stream and the shared K/V."""
    shapes = synth.ablation300m_stack(B=2, T=100, M=16)
    descs = [hb.make_desc(s, residual_mode=0) for s in shapes]
    da, wa = hb.make_stack(descs, [_fake_weights() for _ in shapes])
    n = hb.stack_fwd_workspace(da)
    assert n > max(hb.layer_fwd_workspace(d) for d in descs)
    L = hb.lib()
    assert L.hymba_stack_fwd_workspace(0, da) == 0
    bad = [hb.make_desc(s, residual_mode=0) for s in shapes]
    bad[0].residual = 2
    assert hb.stack_fwd_workspace(hb.make_stack(bad, [_fake_weights()] * 4)[0]) == 0
    bad = [hb.make_desc(s, residual_mode=0) for s in shapes]
    bad[1].batch = 3
    assert hb.stack_fwd_workspace(hb.make_stack(bad, [_fake_weights()] * 4)[0]) == 0
    bad = [hb.make_desc(s, residual_mode=0) for s in shapes[2:]]   # starts with the shared layer
    assert hb.stack_fwd_workspace(hb.make_stack(bad, [_fake_weights()] * 2)[0]) == 0
    bad = [hb.make_desc(synth.with_(s, dtype="f32"), residual_mode=0) for s in shapes]
    assert hb.stack_fwd_workspace(hb.make_stack(bad, [_fake_weights()] * 4)[0]) == 0
    x, y = 0x200000, 0x40000000
    assert L.hymba_stack_fwd(4, da, wa, x, y, ctypes.c_void_p(0x100000), 16, None, None) == hb.HYMBA_ERR_WORKSPACE
    assert L.hymba_stack_fwd(4, da, wa, x, x, ctypes.c_void_p(0x100000), 1 << 40, None, None) == hb.HYMBA_ERR_INVALID
    assert L.hymba_stack_fwd(4, da, None, x, y, ctypes.c_void_p(0x100000), 1 << 40, None, None) == \
        hb.HYMBA_ERR_INVALID


def test_fusion_flag_values():
    assert hb.layer_fwd_workspace(_desc(fusion=1)) > hb.layer_fwd_workspace(_desc(fusion=0))   # s rows 2 di wide
    assert hb.layer_fwd_workspace(_desc(fusion=2)) == 0
    d = _desc(fusion=2)
    w = _fake_weights()
    rc = hb.lib().hymba_layer_fwd(ctypes.byref(d), ctypes.byref(w), 0x200000, 0x300000, None, None, None,
                                  ctypes.c_void_p(0x100000), 1 << 40, None, None)
    assert rc == hb.HYMBA_ERR_INVALID


def test_block_weight_interleave_layout():
    """W_gu rows 2j / 2j+1 hold W_gate row j / W_up row j, as the header
    documents for hymba_block_weights (checked on the host, no GPU)."""
    import numpy as np
    import torch
    from hybrid_attention_ssm_fwd_b300 import layer as hl
    s = synth.tiny_f32(B=1, T=8, M=0)
    _, blocks = synth.make_block_inputs(s, 24, 0)
    pb = blocks[0]
    dev = hl.block_params_to_device(pb, s, device="cpu")
    gu = dev["W_gu"].numpy()
    assert gu.shape == (48, s.d)
    np.testing.assert_array_equal(gu[0::2], pb["W_gate"])
    np.testing.assert_array_equal(gu[1::2], pb["W_up"])
    assert dev["W_down"].shape == (s.d, 24) and dev["norm1"].dtype == torch.float32


def test_binding_checks_tensor_arguments_before_the_call():
    """The ctypes wrappers check what a bare pointer cannot carry (dtype,
    contiguity, size, device) and raise before anything reaches the
    library."""
    import torch
    s = synth.hymba15b_swa(B=2, T=64)
    desc = hb.make_desc(s)
    w = hb.LayerWeights(*[0x10000 * (i + 1) for i in range(11)])
    n = s.B * s.L * s.d
    x = torch.zeros(s.B, s.L, s.d, dtype=torch.bfloat16)
    y = torch.zeros(s.B, s.L, s.d, dtype=torch.float32)
    ws = torch.zeros(16, dtype=torch.uint8)
    cases = [
        (x.float(), y, "dtype"),                       # fp32 input to a bf16 layer
        (x.transpose(0, 1), y, "contiguous"),
        (x.reshape(-1)[: n - 1], y, "elements"),       # one element short
        (x, y, "CUDA"),                                # right in every way but on the host
    ]
    for xx, yy, word in cases:
        with pytest.raises(ValueError, match=word):
            hb.hymba_layer_fwd(desc, w, xx, yy, ws)
    # y is checked the same way (each tensor's own checks run before the next's)
    with pytest.raises(ValueError, match="dtype"):
        hb._arg(y.to(torch.bfloat16), "y", hb._io_dtypes(desc)[1], n)
    with pytest.raises(ValueError, match="required"):
        hb._arg(None, "y")
    sd = synth.with_(s, T=1)
    dd = hb.make_desc(sd)
    with pytest.raises(ValueError, match="elements"):
        hb.hymba_layer_decode(dd, w, torch.zeros(sd.B, sd.d - 8, dtype=torch.bfloat16),
                              torch.zeros(sd.B, sd.d), hb.Cache(), ws)
    with pytest.raises(ValueError, match="dtype"):
        hb.hymba_block_fwd(desc, hb.BlockWeights(), 4800, x, ws)
