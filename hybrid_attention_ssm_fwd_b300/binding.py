"""Thin ctypes binding of libhymba.so (include/hymba.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  There is no
fallback: if the shared library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_size_t, c_uint32, c_void_p
from typing import Dict, Optional

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libhymba.so")

HYMBA_OK = 0
HYMBA_ERR_INVALID = 1
HYMBA_ERR_UNSUPPORTED = 2
HYMBA_ERR_WORKSPACE = 3
HYMBA_ERR_CUDA = 4
HYMBA_ERR_TIMEOUT = 5
HYMBA_ERR_RANGE = 6

HYMBA_F32 = 0
HYMBA_BF16 = 1


class LayerDesc(ctypes.Structure):
    _fields_ = [
        ("batch", c_int32), ("n_tokens", c_int32), ("n_meta", c_int32), ("d_model", c_int32),
        ("n_q_heads", c_int32), ("n_kv_heads", c_int32), ("head_dim", c_int32), ("v_head_dim", c_int32),
        ("d_inner", c_int32), ("d_state", c_int32), ("d_conv", c_int32), ("dt_rank", c_int32),
        ("window", c_int32), ("kv_shared", c_int32), ("residual", c_int32), ("dtype", c_int32),
        ("rope_theta", c_float), ("eps", c_float), ("wait_limit_us", c_uint32), ("fusion", c_int32),
        ("reserved0", c_int32), ("reserved", c_int32),
    ]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("W_in", "W_out", "W_x", "W_dt", "dt_bias", "A_log", "D", "conv_w",
                                        "conv_b", "beta1", "beta2")]


class KV(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p)]


class Cache(ctypes.Structure):
    _fields_ = [("k_ring", c_void_p), ("v_ring", c_void_p), ("k_meta", c_void_p), ("v_meta", c_void_p),
                ("ssm_state", c_void_p), ("conv_state", c_void_p), ("pos", c_void_p), ("cap", c_int32),
                ("reserved", c_int32)]


class BlockWeights(ctypes.Structure):
    _fields_ = [("mix", LayerWeights), ("norm1", c_void_p), ("norm2", c_void_p), ("W_gu", c_void_p),
                ("W_down", c_void_p)]


class Meta(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p), ("ssm_state", c_void_p), ("conv_tail", c_void_p),
                ("y", c_void_p)]


WEIGHT_NAMES = [f[0] for f in LayerWeights._fields_]
CACHE_NAMES = ["k_ring", "v_ring", "k_meta", "v_meta", "ssm_state", "conv_state", "pos"]

_lib = None


def lib() -> ctypes.CDLL:
    """Load libhymba.so once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m hybrid_attention_ssm_fwd_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    P = POINTER
    L.hymba_abi_version.restype = c_int32
    L.hymba_status_str.argtypes = [c_int32]
    L.hymba_status_str.restype = c_char_p
    L.hymba_layer_fwd_workspace.argtypes = [P(LayerDesc)]
    L.hymba_layer_fwd_workspace.restype = c_size_t
    L.hymba_layer_decode_workspace.argtypes = [P(LayerDesc)]
    L.hymba_layer_decode_workspace.restype = c_size_t
    L.hymba_layer_fwd.argtypes = [P(LayerDesc), P(LayerWeights), c_void_p, c_void_p, P(Cache), P(KV), P(KV),
                                  c_void_p, c_size_t, c_void_p, c_void_p]
    L.hymba_layer_fwd.restype = c_int32
    L.hymba_layer_fwd_events.argtypes = [P(LayerDesc), P(LayerWeights), c_void_p, c_void_p, P(Cache), P(KV),
                                         P(KV), c_void_p, c_size_t, c_void_p, c_void_p, c_int32, c_void_p]
    L.hymba_layer_fwd_events.restype = c_int32
    L.hymba_layer_decode.argtypes = [P(LayerDesc), P(LayerWeights), c_void_p, c_void_p, P(Cache), P(Cache),
                                     c_void_p, c_size_t, c_void_p, c_void_p]
    L.hymba_layer_decode.restype = c_int32
    L.hymba_layer_decode_events.argtypes = [P(LayerDesc), P(LayerWeights), c_void_p, c_void_p, P(Cache), P(Cache),
                                            c_void_p, c_size_t, c_void_p, c_void_p, c_int32, c_void_p]
    L.hymba_layer_decode_events.restype = c_int32
    L.hymba_layer_decode_static.argtypes = [P(LayerDesc), P(LayerWeights), c_void_p, c_void_p, P(Cache),
                                            P(Cache), c_void_p, c_void_p]
    L.hymba_layer_decode_static.restype = c_int32
    L.hymba_meta_prefill_workspace.argtypes = [P(LayerDesc)]
    L.hymba_meta_prefill_workspace.restype = c_size_t
    L.hymba_layer_fwd_meta_workspace.argtypes = [P(LayerDesc)]
    L.hymba_layer_fwd_meta_workspace.restype = c_size_t
    L.hymba_meta_prefill.argtypes = [P(LayerDesc), P(LayerWeights), c_void_p, P(Meta), P(KV), c_void_p, c_size_t,
                                     c_void_p, c_void_p]
    L.hymba_meta_prefill.restype = c_int32
    L.hymba_layer_fwd_meta.argtypes = [P(LayerDesc), P(LayerWeights), P(Meta), c_void_p, c_void_p, P(Cache), P(KV),
                                       P(KV), c_void_p, c_size_t, c_void_p, c_void_p]
    L.hymba_layer_fwd_meta.restype = c_int32
    L.hymba_block_fwd_workspace.argtypes = [P(LayerDesc), c_int32]
    L.hymba_block_fwd_workspace.restype = c_size_t
    L.hymba_block_fwd.argtypes = [P(LayerDesc), P(BlockWeights), c_int32, c_void_p, c_void_p, c_size_t, c_void_p,
                                  c_void_p]
    L.hymba_block_fwd.restype = c_int32
    L.hymba_stack_fwd_workspace.argtypes = [c_int32, P(LayerDesc)]
    L.hymba_stack_fwd_workspace.restype = c_size_t
    L.hymba_stack_fwd.argtypes = [c_int32, P(LayerDesc), P(LayerWeights), c_void_p, c_void_p, c_void_p, c_size_t,
                                  c_void_p, c_void_p]
    L.hymba_stack_fwd.restype = c_int32
    L.hymba_test_gemm.argtypes = [c_int32, c_int32, c_int32, c_int32, c_void_p, c_int32, c_void_p, c_int32,
                                  c_void_p, c_int32, c_void_p, c_void_p]
    L.hymba_test_gemm.restype = c_int32
    L.hymba_test_conv.argtypes = [c_int32] * 4 + [c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                                  c_void_p]
    L.hymba_test_conv.restype = c_int32
    L.hymba_test_scan.argtypes = [c_int32, c_int32, c_int32, c_int32, c_void_p, c_int32, c_void_p, c_int32,
                                  c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32,
                                  c_void_p]
    L.hymba_test_scan.restype = c_int32
    L.hymba_test_scan_fused.argtypes = [c_int32] * 5 + [c_void_p, c_int32, c_void_p, c_int32, c_void_p, c_int32] + \
        [c_void_p] * 7 + [c_int32, c_int32, c_void_p]
    L.hymba_test_scan_fused.restype = c_int32
    L.hymba_test_attention.argtypes = [c_int32] * 9 + [c_void_p] * 6
    L.hymba_test_attention.restype = c_int32
    L.hymba_test_wait_timeout.argtypes = [c_uint32, c_void_p, c_void_p]
    L.hymba_test_wait_timeout.restype = c_int32
    _lib = L
    return L


class HymbaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_str(code)} ({code})")
        self.code = code


def status_str(code: int) -> str:
    return lib().hymba_status_str(code).decode()


def _check(code: int, where: str) -> int:
    if code != HYMBA_OK:
        raise HymbaError(code, where)
    return code


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _arg(t, what: str, dtype=None, numel: int = 0) -> int:
    """Device address of a tensor argument, after the checks the C side cannot
    make on a bare pointer: present, of the expected dtype, contiguous, with
    at least ``numel`` elements, on a CUDA device."""
    if t is None:
        raise ValueError(f"{what}: a tensor is required")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{what}: {t.numel()} elements, needs at least {numel}")
    if t.device.type != "cuda":
        raise ValueError(f"{what}: must be on a CUDA device, not {t.device}")
    return t.data_ptr()


def _io_dtypes(desc):
    """(activation input dtype, output dtype) of a layer call: x in the
    descriptor's dtype (bf16 or fp32), y always fp32."""
    import torch
    return (torch.bfloat16 if desc.dtype == HYMBA_BF16 else torch.float32), torch.float32


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def make_desc(shape, wait_limit_us: int = 0, residual_mode: Optional[int] = None) -> LayerDesc:
    """LayerDesc from a synth.LayerShape-like object.  residual_mode overrides
    the shape's flag: 1 adds the layer input, 2 accumulates into y in place."""
    return LayerDesc(batch=shape.B, n_tokens=shape.T, n_meta=shape.M, d_model=shape.d, n_q_heads=shape.Hq,
                     n_kv_heads=shape.Hkv, head_dim=shape.dh, v_head_dim=shape.dv, d_inner=shape.di,
                     d_state=shape.N, d_conv=shape.k, dt_rank=shape.R, window=shape.window,
                     kv_shared=int(shape.kv_shared),
                     residual=int(shape.residual) if residual_mode is None else residual_mode,
                     dtype=HYMBA_BF16 if shape.dtype == "bf16" else HYMBA_F32, rope_theta=shape.rope_theta,
                     eps=shape.eps, wait_limit_us=wait_limit_us,
                     fusion=1 if getattr(shape, "fusion", "sum") == "concat" else 0)


def make_weights(w: Dict[str, "object"]) -> LayerWeights:
    return LayerWeights(**{n: _ptr(w[n]) for n in WEIGHT_NAMES})


def make_cache(c: Optional[Dict[str, "object"]], cap: int) -> Optional[Cache]:
    if c is None:
        return None
    return Cache(**{n: _ptr(c.get(n)) for n in CACHE_NAMES}, cap=cap, reserved=0)


def layer_fwd_workspace(desc: LayerDesc) -> int:
    return lib().hymba_layer_fwd_workspace(ctypes.byref(desc))


def layer_decode_workspace(desc: LayerDesc) -> int:
    return lib().hymba_layer_decode_workspace(ctypes.byref(desc))


def hymba_layer_fwd(desc: LayerDesc, weights: LayerWeights, x, y, ws, cache_out: Optional[Cache] = None,
                    kv_in: Optional[KV] = None, kv_out: Optional[KV] = None, status=None, stream=None,
                    check: bool = True) -> int:
    """Prefill forward through the C ABI (see include/hymba.h)."""
    xd, yd = _io_dtypes(desc)
    n = desc.batch * (desc.n_tokens + desc.n_meta) * desc.d_model
    px, py = _arg(x, "hymba_layer_fwd x", xd, n), _arg(y, "hymba_layer_fwd y", yd, n)
    rc = lib().hymba_layer_fwd(ctypes.byref(desc), ctypes.byref(weights), px, py,
                               ctypes.byref(cache_out) if cache_out is not None else None,
                               ctypes.byref(kv_in) if kv_in is not None else None,
                               ctypes.byref(kv_out) if kv_out is not None else None,
                               _arg(ws, "ws"), ws.numel() * ws.element_size(), _ptr(status), _stream(stream))
    return _check(rc, "hymba_layer_fwd") if check else rc


def hymba_layer_fwd_events(desc: LayerDesc, weights: LayerWeights, x, y, ws, events, n_events: int,
                           cache_out: Optional[Cache] = None, kv_in: Optional[KV] = None,
                           kv_out: Optional[KV] = None, status=None, stream=None, check: bool = True) -> int:
    """hymba_layer_fwd that records per-stage CUDA events (``events`` is a
    ctypes array of cudaEvent_t handles)."""
    xd, yd = _io_dtypes(desc)
    n = desc.batch * (desc.n_tokens + desc.n_meta) * desc.d_model
    px, py = _arg(x, "hymba_layer_fwd_events x", xd, n), _arg(y, "hymba_layer_fwd_events y", yd, n)
    rc = lib().hymba_layer_fwd_events(ctypes.byref(desc), ctypes.byref(weights), px, py,
                                      ctypes.byref(cache_out) if cache_out is not None else None,
                                      ctypes.byref(kv_in) if kv_in is not None else None,
                                      ctypes.byref(kv_out) if kv_out is not None else None,
                                      _arg(ws, "ws"), ws.numel() * ws.element_size(), _ptr(status), events, n_events,
                                      _stream(stream))
    return _check(rc, "hymba_layer_fwd_events") if check else rc


def make_block_weights(w: Dict[str, "object"]) -> BlockWeights:
    return BlockWeights(mix=make_weights(w), norm1=_ptr(w["norm1"]), norm2=_ptr(w["norm2"]), W_gu=_ptr(w["W_gu"]),
                        W_down=_ptr(w["W_down"]))


def block_fwd_workspace(desc: LayerDesc, d_ff: int) -> int:
    return lib().hymba_block_fwd_workspace(ctypes.byref(desc), d_ff)


def hymba_block_fwd(desc: LayerDesc, weights: BlockWeights, d_ff: int, x, ws, status=None, stream=None,
                    check: bool = True) -> int:
    """One residual block on the fp32 stream x, in place (see include/hymba.h)."""
    px = _arg(x, "hymba_block_fwd x", _io_dtypes(desc)[1], desc.batch * (desc.n_tokens + desc.n_meta) * desc.d_model)
    rc = lib().hymba_block_fwd(ctypes.byref(desc), ctypes.byref(weights), d_ff, px, _arg(ws, "hymba_block_fwd ws"),
                               ws.numel() * ws.element_size(), _ptr(status), _stream(stream))
    return _check(rc, "hymba_block_fwd") if check else rc


def make_stack(descs, weights):
    """ctypes arrays of layer descriptors and weight structs for hymba_stack_fwd."""
    n = len(descs)
    da = (LayerDesc * n)(*descs)
    wa = (LayerWeights * n)(*weights)
    return da, wa


def stack_fwd_workspace(descs) -> int:
    return lib().hymba_stack_fwd_workspace(len(descs), descs)


def hymba_stack_fwd(descs, weights, x, y, ws, status=None, stream=None, check: bool = True) -> int:
    """The residual stack over x (bf16 [B, L, d]) into y (fp32), see
    include/hymba.h; descs/weights are the arrays make_stack returns."""
    import torch
    d0 = descs[0]
    n = d0.batch * (d0.n_tokens + d0.n_meta) * d0.d_model
    px = _arg(x, "hymba_stack_fwd x", torch.bfloat16, n)
    py = _arg(y, "hymba_stack_fwd y", torch.float32, n)
    rc = lib().hymba_stack_fwd(len(descs), descs, weights, px, py, _arg(ws, "hymba_stack_fwd ws"),
                               ws.numel() * ws.element_size(), _ptr(status), _stream(stream))
    return _check(rc, "hymba_stack_fwd") if check else rc


def make_meta(m: Dict[str, "object"]) -> Meta:
    return Meta(**{n: _ptr(m.get(n)) for n in ("k", "v", "ssm_state", "conv_tail", "y")})


def meta_prefill_workspace(desc: LayerDesc) -> int:
    return lib().hymba_meta_prefill_workspace(ctypes.byref(desc))


def layer_fwd_meta_workspace(desc: LayerDesc) -> int:
    return lib().hymba_layer_fwd_meta_workspace(ctypes.byref(desc))


def hymba_meta_prefill(desc: LayerDesc, weights: LayerWeights, x_meta, meta: Meta, ws, kv_in: Optional[KV] = None,
                       status=None, stream=None, check: bool = True) -> int:
    """The layer over the meta rows alone, once for the batch (see include/hymba.h)."""
    px = _arg(x_meta, "hymba_meta_prefill x_meta", _io_dtypes(desc)[0], desc.n_meta * desc.d_model)
    rc = lib().hymba_meta_prefill(ctypes.byref(desc), ctypes.byref(weights), px, ctypes.byref(meta),
                                  ctypes.byref(kv_in) if kv_in is not None else None,
                                  _arg(ws, "ws"), ws.numel() * ws.element_size(), _ptr(status), _stream(stream))
    return _check(rc, "hymba_meta_prefill") if check else rc


def hymba_layer_fwd_meta(desc: LayerDesc, weights: LayerWeights, meta: Meta, x, y, ws,
                         cache_out: Optional[Cache] = None, kv_in: Optional[KV] = None, kv_out: Optional[KV] = None,
                         status=None, stream=None, check: bool = True) -> int:
    """Prefill of the real tokens from a meta-prefix state (see include/hymba.h)."""
    xd, yd = _io_dtypes(desc)
    n = desc.batch * desc.n_tokens * desc.d_model
    px, py = _arg(x, "hymba_layer_fwd_meta x", xd, n), _arg(y, "hymba_layer_fwd_meta y", yd, n)
    rc = lib().hymba_layer_fwd_meta(ctypes.byref(desc), ctypes.byref(weights), ctypes.byref(meta), px, py,
                                    ctypes.byref(cache_out) if cache_out is not None else None,
                                    ctypes.byref(kv_in) if kv_in is not None else None,
                                    ctypes.byref(kv_out) if kv_out is not None else None,
                                    _arg(ws, "ws"), ws.numel() * ws.element_size(), _ptr(status), _stream(stream))
    return _check(rc, "hymba_layer_fwd_meta") if check else rc


def hymba_layer_decode(desc: LayerDesc, weights: LayerWeights, x_new, y, cache: Cache, ws,
                       shared_cache: Optional[Cache] = None, status=None, stream=None, check: bool = True) -> int:
    """One decode step through the C ABI (see include/hymba.h)."""
    xd, yd = _io_dtypes(desc)
    n = desc.batch * desc.d_model
    px, py = _arg(x_new, "hymba_layer_decode x_new", xd, n), _arg(y, "hymba_layer_decode y", yd, n)
    rc = lib().hymba_layer_decode(ctypes.byref(desc), ctypes.byref(weights), px, py,
                                  ctypes.byref(cache),
                                  ctypes.byref(shared_cache) if shared_cache is not None else None,
                                  _arg(ws, "ws"), ws.numel() * ws.element_size(), _ptr(status), _stream(stream))
    return _check(rc, "hymba_layer_decode") if check else rc


def hymba_layer_decode_events(desc: LayerDesc, weights: LayerWeights, x_new, y, cache: Cache, ws, events,
                              n_events: int, shared_cache: Optional[Cache] = None, status=None, stream=None,
                              check: bool = True) -> int:
    """hymba_layer_decode that records per-stage CUDA events."""
    xd, yd = _io_dtypes(desc)
    n = desc.batch * desc.d_model
    px, py = _arg(x_new, "hymba_layer_decode_events x_new", xd, n), _arg(y, "hymba_layer_decode_events y", yd, n)
    rc = lib().hymba_layer_decode_events(ctypes.byref(desc), ctypes.byref(weights), px, py,
                                         ctypes.byref(cache),
                                         ctypes.byref(shared_cache) if shared_cache is not None else None,
                                         _arg(ws, "ws"), ws.numel() * ws.element_size(), _ptr(status), events, n_events,
                                         _stream(stream))
    return _check(rc, "hymba_layer_decode_events") if check else rc


STATIC_SCRATCH_BYTES = 32 * 1024 * 1024


def hymba_layer_decode_static(desc: LayerDesc, weights: LayerWeights, x_new, y, cache: Cache,
                              shared_cache: Optional[Cache] = None, status=None, stream=None,
                              check: bool = True) -> int:
    """hymba_layer_decode with the library's built-in scratch buffer instead of
    a workspace, for callers that cannot allocate device memory (see
    include/hymba.h).  Calls must not overlap on the GPU."""
    xd, yd = _io_dtypes(desc)
    n = desc.batch * desc.d_model
    px, py = _arg(x_new, "hymba_layer_decode_static x_new", xd, n), _arg(y, "hymba_layer_decode_static y", yd, n)
    rc = lib().hymba_layer_decode_static(ctypes.byref(desc), ctypes.byref(weights), px, py,
                                         ctypes.byref(cache),
                                         ctypes.byref(shared_cache) if shared_cache is not None else None,
                                         _ptr(status), _stream(stream))
    return _check(rc, "hymba_layer_decode_static") if check else rc


def hymba_test_gemm(A, B, C, ab_dtype: int, status=None, stream=None) -> int:
    M, K = A.shape
    N = B.shape[0]
    return lib().hymba_test_gemm(M, N, K, ab_dtype, _ptr(A), A.stride(0), _ptr(B), B.stride(0), _ptr(C),
                                 C.stride(0), _ptr(status), _stream(stream))


def hymba_test_conv(x, u, conv_w, conv_b, status=None, stream=None) -> int:
    """x: fp16 [B, L, ld_x] (the first di columns are used); u: fp16 [B, L, di]."""
    B, L, di = u.shape
    k = conv_w.shape[1]
    return lib().hymba_test_conv(B, L, di, k, _ptr(x), x.stride(1), _ptr(u), _ptr(conv_w), _ptr(conv_b),
                                 _ptr(status), _stream(stream))


def hymba_test_scan(u, z, delta, BC, A_log, D, g, h_out=None, threads_per_channel=0, channels_per_thread=0,
                    stream=None) -> int:
    B, L, di = delta.shape
    N = A_log.shape[1]
    return lib().hymba_test_scan(B, L, di, N, _ptr(u), u.stride(1), _ptr(z), z.stride(1), _ptr(delta),
                                 _ptr(BC), _ptr(A_log), _ptr(D), _ptr(g), _ptr(h_out), threads_per_channel,
                                 channels_per_thread, _stream(stream))


def hymba_test_scan_fused(u, z, dtr, W_dt, dt_bias, BC, A_log, D, g, h_out=None, threads_per_channel=0,
                          channels_per_thread=0, stream=None) -> int:
    B, L, di = u.shape
    N = A_log.shape[1]
    R = W_dt.shape[1]
    return lib().hymba_test_scan_fused(B, L, di, N, R, _ptr(u), u.stride(1), _ptr(z), z.stride(1), _ptr(dtr),
                                       dtr.stride(1), _ptr(W_dt), _ptr(dt_bias), _ptr(BC), _ptr(A_log), _ptr(D),
                                       _ptr(g), _ptr(h_out), threads_per_channel, channels_per_thread,
                                       _stream(stream))


def hymba_test_attention(Q, K, V, O, M: int, window: int, use_tc: bool, status=None, stream=None) -> int:
    B, L, Hq, dh = Q.shape
    Hkv, dv = K.shape[2], V.shape[3]
    return lib().hymba_test_attention(B, L, M, Hq, Hkv, dh, dv, window, int(use_tc), _ptr(Q), _ptr(K), _ptr(V),
                                      _ptr(O), _ptr(status), _stream(stream))


def hymba_test_wait_timeout(limit_us: int, status, stream=None) -> int:
    return lib().hymba_test_wait_timeout(limit_us, _ptr(status), _stream(stream))
