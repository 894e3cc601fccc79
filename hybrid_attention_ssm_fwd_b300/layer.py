"""PyTorch-facing convenience wrapper around the C ABI.

Holds a layer's device parameters, its descriptor and a workspace, and calls
hymba_layer_fwd / hymba_layer_decode on the current stream.  Marshalling
only: the arithmetic is in libhymba.so.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

from . import binding as hb

MATRICES = ("W_in", "W_out", "W_x", "W_dt")
VECTORS = ("dt_bias", "A_log", "D", "conv_w", "conv_b", "beta1", "beta2")


def storage_dtype(shape) -> torch.dtype:
    return torch.bfloat16 if shape.dtype == "bf16" else torch.float32


def kv_dtype(shape) -> torch.dtype:
    """Element type of exported/imported K/V (fp16 on the bf16 path)."""
    return torch.float16 if shape.dtype == "bf16" else torch.float32


def params_to_device(p: Dict[str, np.ndarray], shape, device="cuda") -> Dict[str, torch.Tensor]:
    """Matrices in the storage dtype, vectors in fp32 (values are already
    storage-rounded by the generator, so the conversion is exact)."""
    out = {}
    dt = storage_dtype(shape)
    for n in MATRICES:
        out[n] = torch.from_numpy(np.ascontiguousarray(p[n], dtype=np.float32)).to(device=device, dtype=dt)
    for n in VECTORS:
        out[n] = torch.from_numpy(np.ascontiguousarray(p[n], dtype=np.float32)).to(device)
    return out


def tokens_to_device(Xt: np.ndarray, shape, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(Xt, dtype=np.float32)).to(device=device, dtype=storage_dtype(shape))


def alloc_cache(shape, cap: int, device="cuda", with_kv: bool = True) -> Dict[str, torch.Tensor]:
    dt = storage_dtype(shape)
    c = {
        "ssm_state": torch.zeros(shape.B, shape.di, shape.N, device=device, dtype=torch.float32),
        "conv_state": torch.zeros(shape.B, shape.di, max(shape.k - 1, 1), device=device, dtype=torch.float32),
        "pos": torch.zeros(shape.B, device=device, dtype=torch.int32),
    }
    if with_kv:
        c["k_ring"] = torch.zeros(shape.B, cap, shape.Hkv, shape.dh, device=device, dtype=dt)
        c["v_ring"] = torch.zeros(shape.B, cap, shape.Hkv, shape.dv, device=device, dtype=dt)
        c["k_meta"] = torch.zeros(max(shape.M, 1), shape.Hkv, shape.dh, device=device, dtype=dt)
        c["v_meta"] = torch.zeros(max(shape.M, 1), shape.Hkv, shape.dv, device=device, dtype=dt)
    return c


def cache_row(cache: Dict[str, torch.Tensor], b: int) -> Dict[str, torch.Tensor]:
    """Views of row b of a batch cache, for a batch-1 call: the per-sequence
    tensors sliced at b (their data pointers offset by b rows), the meta K/V
    shared.  A batch-1 prefill with this as cache_out admits a new sequence
    into row b of a running batch."""
    out = {k: cache[k][b:b + 1] for k in ("ssm_state", "conv_state", "pos") if k in cache}
    for k in ("k_ring", "v_ring"):
        if k in cache:
            out[k] = cache[k][b:b + 1]
    for k in ("k_meta", "v_meta"):
        if k in cache:
            out[k] = cache[k]
    return out


def cache_to_device(c: Dict[str, np.ndarray], shape, device="cuda") -> Dict[str, torch.Tensor]:
    dt = storage_dtype(shape)
    out = {}
    for n in ("k_ring", "v_ring", "k_meta", "v_meta"):
        if n in c:
            out[n] = torch.from_numpy(np.ascontiguousarray(c[n], dtype=np.float32)).to(device=device, dtype=dt)
    out["ssm_state"] = torch.from_numpy(np.ascontiguousarray(c["ssm_state"], dtype=np.float32)).to(device)
    out["conv_state"] = torch.from_numpy(np.ascontiguousarray(c["conv_state"], dtype=np.float32)).to(device)
    out["pos"] = torch.from_numpy(np.ascontiguousarray(c["pos"], dtype=np.int32)).to(device)
    return out


class HymbaLayer:
    """One hybrid-head layer on one device."""

    def __init__(self, shape, params: Dict[str, torch.Tensor], wait_limit_us: int = 0, decode: bool = False,
                 residual_mode: Optional[int] = None):
        self.shape = shape
        self.params = params
        self.desc = hb.make_desc(shape, wait_limit_us, residual_mode)
        self.weights = hb.make_weights(params)
        dev = params["W_in"].device
        nbytes = hb.layer_decode_workspace(self.desc) if decode else hb.layer_fwd_workspace(self.desc)
        if nbytes == 0:
            raise hb.HymbaError(hb.HYMBA_ERR_INVALID, "workspace query")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def forward(self, x: torch.Tensor, y: Optional[torch.Tensor] = None, cache_out=None, cap: int = 0,
                kv_in=None, kv_out=None) -> torch.Tensor:
        s = self.shape
        if y is None:
            y = torch.empty(s.B, s.L, s.d, dtype=torch.float32, device=x.device)
        hb.hymba_layer_fwd(self.desc, self.weights, x, y, self.ws,
                           cache_out=hb.make_cache(cache_out, cap) if cache_out is not None else None,
                           kv_in=hb.KV(kv_in[0].data_ptr(), kv_in[1].data_ptr()) if kv_in is not None else None,
                           kv_out=hb.KV(kv_out[0].data_ptr(), kv_out[1].data_ptr()) if kv_out is not None else None,
                           status=self.status)
        return y

    def _scratch(self, nbytes: int) -> torch.Tensor:
        if nbytes == 0:
            raise hb.HymbaError(hb.HYMBA_ERR_UNSUPPORTED, "workspace query")
        if self.ws.numel() < nbytes:
            self.ws = torch.empty(nbytes, dtype=torch.uint8, device=self.ws.device)
        return self.ws

    def meta_prefill(self, x_meta: torch.Tensor, y: Optional[torch.Tensor] = None,
                     kv_in=None) -> Dict[str, torch.Tensor]:
        """The layer over the M meta rows alone ([M, d]), once for a whole
        batch.  Returns the state forward_meta starts the real tokens from:
        meta K/V (fp16; the producer's when kv_in is given), the SSM state
        [di, N], the conv tail [di, k-1] and Y of the meta rows [M, d] (``y``,
        when given, is that buffer: residual mode 2 adds into it)."""
        s = self.shape
        dev = x_meta.device
        kd = kv_dtype(s)
        meta = {
            "ssm_state": torch.empty(s.di, s.N, device=dev, dtype=torch.float32),
            "conv_tail": torch.empty(s.di, max(s.k - 1, 1), device=dev, dtype=torch.float32),
            "y": y if y is not None else torch.empty(s.M, s.d, device=dev, dtype=torch.float32),
        }
        if kv_in is None:
            meta["k"] = torch.empty(s.M, s.Hkv, s.dh, device=dev, dtype=kd)
            meta["v"] = torch.empty(s.M, s.Hkv, s.dv, device=dev, dtype=kd)
        else:
            meta["k"], meta["v"] = kv_in
        ws = self._scratch(hb.meta_prefill_workspace(self.desc))
        hb.hymba_meta_prefill(self.desc, self.weights, x_meta, hb.make_meta(meta), ws,
                              kv_in=hb.KV(kv_in[0].data_ptr(), kv_in[1].data_ptr()) if kv_in is not None else None,
                              status=self.status)
        return meta

    def forward_meta(self, meta: Dict[str, torch.Tensor], x: torch.Tensor, y: Optional[torch.Tensor] = None,
                     cache_out=None, cap: int = 0, kv_in=None, kv_out=None) -> torch.Tensor:
        """Prefill of the real tokens x [B, T, d] from a meta_prefill state;
        returns Y of the real rows [B, T, d].  kv_in / kv_out hold T rows."""
        s = self.shape
        if y is None:
            y = torch.empty(s.B, s.T, s.d, dtype=torch.float32, device=x.device)
        ws = self._scratch(hb.layer_fwd_meta_workspace(self.desc))
        hb.hymba_layer_fwd_meta(self.desc, self.weights, hb.make_meta(meta), x, y, ws,
                                cache_out=hb.make_cache(cache_out, cap) if cache_out is not None else None,
                                kv_in=hb.KV(kv_in[0].data_ptr(), kv_in[1].data_ptr()) if kv_in is not None else None,
                                kv_out=hb.KV(kv_out[0].data_ptr(), kv_out[1].data_ptr()) if kv_out is not None
                                else None, status=self.status)
        return y

    def decode(self, x_new: torch.Tensor, cache: Dict[str, torch.Tensor], cap: int,
               y: Optional[torch.Tensor] = None, shared_cache=None, shared_cap: int = 0) -> torch.Tensor:
        s = self.shape
        if y is None:
            y = torch.empty(s.B, s.d, dtype=torch.float32, device=x_new.device)
        hb.hymba_layer_decode(self.desc, self.weights, x_new, y, hb.make_cache(cache, cap), self.ws,
                              shared_cache=hb.make_cache(shared_cache, shared_cap) if shared_cache else None,
                              status=self.status)
        return y

    def check_status(self) -> int:
        return int(self.status.item())


def block_params_to_device(pb: Dict[str, np.ndarray], shape, device="cuda") -> Dict[str, torch.Tensor]:
    """A residual block's parameters: the layer's, the two RMSNorm weights
    (fp32), W_gate / W_up interleaved row by row into W_gu [2F, d] and W_down
    [d, F] (storage dtype)."""
    out = params_to_device(pb, shape, device)
    dt = storage_dtype(shape)
    for n in ("norm1", "norm2"):
        out[n] = torch.from_numpy(np.ascontiguousarray(pb[n], dtype=np.float32)).to(device)
    Fh, d = pb["W_gate"].shape
    gu = np.empty((2 * Fh, d), np.float32)
    gu[0::2] = pb["W_gate"]
    gu[1::2] = pb["W_up"]
    out["W_gu"] = torch.from_numpy(gu).to(device=device, dtype=dt)
    out["W_down"] = torch.from_numpy(np.ascontiguousarray(pb["W_down"], dtype=np.float32)).to(device=device, dtype=dt)
    return out


class HymbaBlock:
    """One residual block (RMSNorm -> hybrid-head layer -> add; RMSNorm ->
    gated MLP -> add) on one device, applied in place to an fp32 stream."""

    def __init__(self, shape, params: Dict[str, torch.Tensor], d_ff: int, wait_limit_us: int = 0):
        self.shape = shape
        self.params = params
        self.d_ff = d_ff
        self.desc = hb.make_desc(shape, wait_limit_us, residual_mode=0)
        self.weights = hb.make_block_weights(params)
        nbytes = hb.block_fwd_workspace(self.desc, d_ff)
        if nbytes == 0:
            raise hb.HymbaError(hb.HYMBA_ERR_UNSUPPORTED, "block workspace query")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=params["W_in"].device)
        self.status = torch.zeros(1, dtype=torch.int32, device=params["W_in"].device)

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        """x: [B, L, d] fp32 stream, updated in place and returned."""
        hb.hymba_block_fwd(self.desc, self.weights, self.d_ff, x, self.ws, status=self.status)
        return x

    def check_status(self) -> int:
        return int(self.status.item())


class HymbaStack:
    """A residual stack X_{l+1} = X_l + Y_l(bf16(X_l)) of hybrid-head layers
    on one device, run by one hymba_stack_fwd call (a kv_shared layer reads
    the previous layer's K/V)."""

    def __init__(self, shapes, params, wait_limit_us: int = 0):
        self.shapes = list(shapes)
        self.params = list(params)
        descs = [hb.make_desc(s, wait_limit_us, residual_mode=0) for s in self.shapes]
        self.descs, self.weights = hb.make_stack(descs, [hb.make_weights(p) for p in self.params])
        nbytes = hb.stack_fwd_workspace(self.descs)
        if nbytes == 0:
            raise hb.HymbaError(hb.HYMBA_ERR_INVALID, "stack workspace query")
        dev = self.params[0]["W_in"].device
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def forward(self, x: torch.Tensor, y: Optional[torch.Tensor] = None) -> torch.Tensor:
        """x: [B, L, d] bf16; returns the fp32 stream after the last layer."""
        s = self.shapes[0]
        if y is None:
            y = torch.empty(s.B, s.L, s.d, dtype=torch.float32, device=x.device)
        hb.hymba_stack_fwd(self.descs, self.weights, x, y, self.ws, status=self.status)
        return y

    def check_status(self) -> int:
        return int(self.status.item())
