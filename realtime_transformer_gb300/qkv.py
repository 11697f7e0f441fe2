"""QKVPlan: torch-facing wrapper of the attention-input sublayer's C ABI
(include/frt_qkv.h): residual + RMSNorm + E4M3 quantise, FP8 fused-QKV GEMM,
QKV split + RoPE.  PyTorch supplies device memory and streams; every step
runs in libfrt_ffn.so."""
from __future__ import annotations

import torch

from . import _native as N
from .ffn import _bf16, _ptr, _stream


class QKVPlan:
    """n_layers attention-input sublayers: width d, n_q / n_kv heads of head_dim."""

    def __init__(self, d: int, n_q_heads: int, n_kv_heads: int, head_dim: int, rope_base: float, M_max: int,
                 n_layers: int):
        self.d, self.nq, self.nkv, self.hd = d, n_q_heads, n_kv_heads, head_dim
        self.M_max, self.n_layers = M_max, n_layers
        self.handle = N.frt_qkv_plan_create(d, n_q_heads, n_kv_heads, head_dim, float(rope_base), M_max, n_layers)

    def close(self):
        if getattr(self, "handle", None):
            N.frt_qkv_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_weights(self, layer, w_norm, w_q, w_k, w_v, stream=None, fold_norm=False):
        """fold_norm: fold the RMSNorm weight into the fused QKV weight (the Pi0 layout)."""
        d, hd = self.d, self.hd
        N.frt_qkv_load_weights_ex(self.handle, layer, _bf16(w_norm, (d,), "w_norm"),
                                  _bf16(w_q, (self.nq * hd, d), "w_q"), _bf16(w_k, (self.nkv * hd, d), "w_k"),
                                  _bf16(w_v, (self.nkv * hd, d), "w_v"), N.FRT_LOAD_FOLD_NORM if fold_norm else 0,
                                  _stream(stream))

    def calibrate(self, layer, residuals, hiddens=None, stream=None):
        M = residuals[0].shape[0]
        rp = [_bf16(r, (M, self.d), "residual") for r in residuals]
        hp = [_bf16(h, (M, self.d), "hidden") if h is not None else None for h in hiddens] if hiddens else None
        N.frt_qkv_calibrate(self.handle, layer, rp, hp, M, _stream(stream))

    def scales(self):
        s_x, s_qkv = N.frt_qkv_get_scales(self.handle, self.n_layers)
        return {"s_x": s_x, "s_qkv": s_qkv}

    def set_scales(self, s_x):
        N.frt_qkv_set_scales(self.handle, list(map(float, s_x)))

    def _outs(self, M, dev):
        return {"q": torch.empty((self.nq, M, self.hd), dtype=torch.bfloat16, device=dev),
                "k": torch.empty((self.nkv, M, self.hd), dtype=torch.bfloat16, device=dev),
                "v": torch.empty((self.nkv, M, self.hd), dtype=torch.bfloat16, device=dev),
                "r_prime": torch.empty((M, self.d), dtype=torch.bfloat16, device=dev)}

    def forward(self, layer, residual, hidden, positions, out=None, stream=None):
        """Returns {"q" [Hq,M,hd], "k" [Hkv,M,hd], "v" [Hkv,M,hd], "r_prime" [M,d]}
        (BF16); positions: int32 [M] on the device."""
        M = residual.shape[0]
        o = out if out is not None else self._outs(M, residual.device)
        if positions.dtype != torch.int32 or tuple(positions.shape) != (M,):
            raise ValueError("positions must be int32 [M]")
        N.frt_qkv_forward(self.handle, layer, _bf16(residual, (M, self.d), "residual"),
                          _bf16(hidden, (M, self.d), "hidden") if hidden is not None else None, _ptr(positions),
                          _ptr(o["r_prime"]), _ptr(o["q"]), _ptr(o["k"]), _ptr(o["v"]), M, _stream(stream))
        return o

    def trace(self, layer, residual, hidden, positions, stream=None):
        """forward plus the intermediates q_x [M,d] (E4M3 bytes) and qkv [M,N] (BF16)."""
        M = residual.shape[0]
        dev = residual.device
        o = self._outs(M, dev)
        o["q_x"] = torch.empty((M, self.d), dtype=torch.uint8, device=dev)
        o["qkv"] = torch.empty((M, (self.nq + 2 * self.nkv) * self.hd), dtype=torch.bfloat16, device=dev)
        N.frt_qkv_debug_trace(self.handle, layer, _bf16(residual, (M, self.d), "residual"),
                              _bf16(hidden, (M, self.d), "hidden") if hidden is not None else None,
                              _ptr(positions), _ptr(o["r_prime"]), _ptr(o["q"]), _ptr(o["k"]), _ptr(o["v"]),
                              _ptr(o["q_x"]), _ptr(o["qkv"]), M, _stream(stream))
        return o

    def trace_from_qx(self, layer, q_x, positions, stream=None):
        """The GEMM and split + RoPE from caller-supplied E4M3 codes q_x
        (uint8 [M, d]) in place of the norm's output; returns q, k, v and the
        GEMM's BF16 output (diagnostics)."""
        M = q_x.shape[0]
        dev = q_x.device
        if q_x.dtype != torch.uint8 or tuple(q_x.shape) != (M, self.d) or not q_x.is_contiguous():
            raise ValueError("q_x must be a contiguous uint8 [M, d] tensor")
        o = self._outs(M, dev)
        o["qkv"] = torch.empty((M, (self.nq + 2 * self.nkv) * self.hd), dtype=torch.bfloat16, device=dev)
        N.frt_qkv_debug_trace_qx(self.handle, layer, _ptr(q_x), _ptr(positions), _ptr(o["q"]), _ptr(o["k"]),
                                 _ptr(o["v"]), _ptr(o["qkv"]), M, _stream(stream))
        return o

    def weights(self, layer, device="cuda", stream=None):
        """The plan's fused E4M3 weight [W_q; W_k; W_v] of one layer as
        stored, a uint8 [(Hq + 2 Hkv) hd, d] tensor (diagnostics)."""
        w = torch.empty(((self.nq + 2 * self.nkv) * self.hd, self.d), dtype=torch.uint8, device=device)
        N.frt_qkv_debug_weights(self.handle, layer, _ptr(w), _stream(stream))
        return w

    def device_status(self, stream=None):
        N.frt_qkv_device_status(self.handle, _stream(stream))
