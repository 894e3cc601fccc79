"""Helpers shared by the GPU parity tests (tolerances, uploads, oracle runs)."""
import numpy as np
import torch

from hybrid_attention_ssm_fwd_b300 import layer as hl

# Tolerances of the workload statement: bf16 path max-abs <= 2e-2 and relative
# Frobenius <= 1e-2; fp32 path relative <= 1e-4.
BF16_MAX_ABS = 2e-2
BF16_REL_FRO = 1e-2
F32_REL = 1e-4


def errs(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    e = got - ref
    return float(np.abs(e).max()), float(np.linalg.norm(e) / max(np.linalg.norm(ref), 1e-300))


def assert_bf16_close(got, ref, what=""):
    mx, rf = errs(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert mx <= BF16_MAX_ABS and rf <= BF16_REL_FRO, f"{what}: max_abs {mx:.3e} rel_fro {rf:.3e}"
    return mx, rf


def assert_f32_close(got, ref, what="", tol=F32_REL):
    mx, rf = errs(got, ref)
    scale = float(np.abs(np.asarray(ref)).max())
    assert rf <= tol and mx <= tol * scale, f"{what}: max_abs {mx:.3e} (scale {scale:.3e}) rel_fro {rf:.3e}"
    return mx, rf


def run_prefill(s, p, cap=None, kv_in=None, want_kv=False, Xt=None):
    """Upload, run hymba_layer_fwd, return numpy Y (and the cache / kv if asked)."""
    dev = "cuda"
    params = hl.params_to_device(p, s, dev)
    layer = hl.HymbaLayer(s, params)
    X = hl.tokens_to_device(p["Xt"] if Xt is None else Xt, s, dev)
    cache = hl.alloc_cache(s, cap, dev, with_kv=not s.kv_shared) if cap else None
    kv_out = None
    if want_kv:
        kd = hl.kv_dtype(s)
        kv_out = (torch.empty(s.B, s.L, s.Hkv, s.dh, device=dev, dtype=kd),
                  torch.empty(s.B, s.L, s.Hkv, s.dv, device=dev, dtype=kd))
    y = layer.forward(X, cache_out=cache, cap=cap or 0, kv_in=kv_in, kv_out=kv_out)
    torch.cuda.synchronize()
    assert layer.check_status() == 0, f"device status {layer.check_status()}"
    return y.cpu().numpy(), cache, kv_out


def cache_np(c):
    return {k: v.float().cpu().numpy() if v.dtype != torch.int32 else v.cpu().numpy() for k, v in c.items()}
