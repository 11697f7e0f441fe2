"""FFNPlan: torch-facing wrapper of the C-ABI plan.

PyTorch supplies device memory and streams; every step runs in
libfrt_ffn.so.  Also holds the calibration cache of the "FlashRT
docs/architecture.md", 6 Calibration Framework: scales saved as JSON under
a key made of a hash of the weights and the token count ("{hash}_Se{M}.json").
"""
from __future__ import annotations

import hashlib
import json
import os

import torch

from . import _native as N

ACTS = {"geglu_tanh": N.FRT_ACT_GEGLU_TANH, "swiglu": N.FRT_ACT_SWIGLU}


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    return t.data_ptr()


def _bf16(t, shape, name):
    if t.dtype != torch.bfloat16 or tuple(t.shape) != tuple(shape):
        raise ValueError("%s must be bfloat16 %s, got %s %s" % (name, tuple(shape), t.dtype, tuple(t.shape)))
    return _ptr(t)


class FFNPlan:
    """A stack of n_layers FP8 FFN sublayers (d, ff, act) for up to M_max tokens."""

    def __init__(self, d: int, ff: int, act: str | int, M_max: int, n_layers: int):
        self.d, self.ff, self.M_max, self.n_layers = d, ff, M_max, n_layers
        self.act = ACTS[act] if isinstance(act, str) else int(act)
        self.handle = N.frt_ffn_plan_create(d, ff, self.act, M_max, n_layers)
        self._digest = [None] * n_layers

    def close(self):
        if getattr(self, "handle", None):
            N.frt_ffn_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- weights / scales --------------------------------------------------
    def load_weights(self, layer, w_norm, w_gate, w_up, w_down, stream=None):
        d, ff = self.d, self.ff
        N.frt_ffn_load_weights(self.handle, layer, _bf16(w_norm, (d,), "w_norm"),
                               _bf16(w_gate, (ff, d), "w_gate"), _bf16(w_up, (ff, d), "w_up"),
                               _bf16(w_down, (d, ff), "w_down"), _stream(stream))
        h = hashlib.sha256()
        for t in (w_norm, w_gate, w_up, w_down):
            h.update(t.reshape(-1)[:: max(1, t.numel() // 4096)].contiguous().view(torch.int16).cpu().numpy().tobytes())
        self._digest[layer] = h.hexdigest()

    def calibrate(self, residuals, hiddens=None, stream=None):
        M = residuals[0].shape[0]
        rp = [_bf16(r, (M, self.d), "residual") for r in residuals]
        hp = [_bf16(h, (M, self.d), "hidden") if h is not None else None for h in hiddens] if hiddens else None
        N.frt_ffn_calibrate(self.handle, rp, hp, M, _stream(stream))

    def scales(self):
        s_x, s_h, s_gu, s_d = N.frt_ffn_get_scales(self.handle, self.n_layers)
        return {"s_x": s_x, "s_h": s_h, "s_gu": s_gu, "s_down": s_d}

    def set_scales(self, s_x, s_h):
        N.frt_ffn_set_scales(self.handle, list(map(float, s_x)), list(map(float, s_h)))

    # -- calibration cache ---------------------------------------------------
    def cache_key(self, M: int) -> str:
        h = hashlib.sha256()
        h.update(json.dumps([self.d, self.ff, self.act, self.n_layers]).encode())
        for dg in self._digest:
            h.update((dg or "").encode())
        return "%s_Se%d" % (h.hexdigest()[:16], M)

    def save_scales(self, directory: str, M: int) -> str:
        os.makedirs(directory, exist_ok=True)
        path = os.path.join(directory, self.cache_key(M) + ".json")
        sc = self.scales()
        with open(path, "w") as f:
            json.dump({"s_x": sc["s_x"], "s_h": sc["s_h"], "extra": {"s_gu": sc["s_gu"], "s_down": sc["s_down"]}},
                      f)
        return path

    def load_scales(self, directory: str, M: int) -> bool:
        path = os.path.join(directory, self.cache_key(M) + ".json")
        if not os.path.exists(path):
            return False
        with open(path) as f:
            js = json.load(f)
        self.set_scales(js["s_x"], js["s_h"])
        return True

    # -- forward -------------------------------------------------------------
    def forward(self, residual, hidden=None, out=None, stream=None):
        M = residual.shape[0]
        if out is None:
            out = torch.empty_like(residual)
        N.frt_ffn_forward(self.handle, _bf16(residual, (M, self.d), "residual"),
                          _bf16(hidden, (M, self.d), "hidden") if hidden is not None else None,
                          _bf16(out, (M, self.d), "out"), M, _stream(stream))
        return out

    def graph_capture(self, residual, hidden, out, stream):
        M = residual.shape[0]
        N.frt_ffn_graph_capture(self.handle, _bf16(residual, (M, self.d), "residual"),
                                _bf16(hidden, (M, self.d), "hidden") if hidden is not None else None,
                                _bf16(out, (M, self.d), "out"), M, _stream(stream))

    def graph_replay(self, M: int, stream=None):
        N.frt_ffn_graph_replay(self.handle, M, _stream(stream))

    def device_status(self, stream=None):
        N.frt_ffn_device_status(self.handle, _stream(stream))

    def debug_stall(self, stream=None):
        """Failure-path test hook: raises FrtError(FRT_ERR_DEVICE_TIMEOUT)
        after a kernel gives up its bounded wait (about 2 s)."""
        N.frt_ffn_debug_stall(self.handle, _stream(stream))

    def trace_layer(self, layer, residual, hidden=None, stream=None):
        """Run one layer alone and return its intermediates (diagnostics)."""
        M, d, ff = residual.shape[0], self.d, self.ff
        dev = residual.device
        out = {
            "r_prime": torch.empty((M, d), dtype=torch.bfloat16, device=dev),
            "q_x": torch.empty((M, d), dtype=torch.uint8, device=dev),
            "gu": torch.empty((M, 2 * ff), dtype=torch.bfloat16, device=dev),
            "q_h": torch.empty((M, ff), dtype=torch.uint8, device=dev),
            "out": torch.empty((M, d), dtype=torch.bfloat16, device=dev),
        }
        N.frt_ffn_debug_trace(self.handle, layer, _bf16(residual, (M, d), "residual"),
                              _bf16(hidden, (M, d), "hidden") if hidden is not None else None, M,
                              _ptr(out["r_prime"]), _ptr(out["q_x"]), _ptr(out["gu"]), _ptr(out["q_h"]),
                              _ptr(out["out"]), _stream(stream))
        return out

    def gemm(self, A, B, alpha=1.0, path=0, splits=0, stream=None):
        """Diagnostics: C = alpha * A B^T on the plan's FP8 GEMM kernels (A [M,K], B [N,K] uint8 E4M3)."""
        M, K = A.shape
        Nn = B.shape[0]
        C = torch.empty((M, Nn), dtype=torch.float32, device=A.device)
        N.frt_fp8_gemm(self.handle, _ptr(A), _ptr(B), _ptr(C), M, Nn, K, float(alpha), path, splits,
                       _stream(stream))
        return C
