"""FP4Plan: torch-facing wrapper of the NVFP4 sublayer stack's C ABI
(include/frt_nvfp4.h; itsolotime FlashRT article, 7.2): norm + AWQ + NVFP4
quantise, the gate/up NVFP4 GEMM that forms G and U as NVFP4 and applies the
FP4 -> FP4 gated activation in its epilogue, NVFP4 down GEMM + residual.
PyTorch supplies device memory and streams; every step runs in
libfrt_ffn.so."""
from __future__ import annotations

import torch

from . import _native as N
from .ffn import ACTS, _bf16, _ptr, _stream


class FP4Plan:
    """A stack of n_layers NVFP4 FFN sublayers (d, ff, act) for up to M_max tokens."""

    def __init__(self, d: int, ff: int, act: str | int, M_max: int, n_layers: int):
        self.d, self.ff, self.M_max, self.n_layers = d, ff, M_max, n_layers
        self.act = ACTS[act] if isinstance(act, str) else int(act)
        self.handle = N.frt_fp4_plan_create(d, ff, self.act, M_max, n_layers)

    def close(self):
        if getattr(self, "handle", None):
            N.frt_fp4_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_weights(self, layer, w_norm, w_gate, w_up, w_down, awq=None, stream=None):
        """awq: fp32 [d] device tensor of AWQ scales (gate/up columns times c,
        the activation divided by c), or None."""
        d, ff = self.d, self.ff
        if awq is not None and (awq.dtype != torch.float32 or tuple(awq.shape) != (d,)):
            raise ValueError("awq must be float32 (%d,)" % d)
        N.frt_fp4_load_weights(self.handle, layer, _bf16(w_norm, (d,), "w_norm"), _bf16(w_gate, (ff, d), "w_gate"),
                               _bf16(w_up, (ff, d), "w_up"), _bf16(w_down, (d, ff), "w_down"), _ptr(awq),
                               _stream(stream))

    def calibrate(self, residuals, hiddens=None, stream=None):
        M = residuals[0].shape[0]
        rp = [_bf16(r, (M, self.d), "residual") for r in residuals]
        hp = [_bf16(h, (M, self.d), "hidden") for h in hiddens] if hiddens else None
        N.frt_fp4_calibrate(self.handle, rp, hp, M, _stream(stream))

    def scales(self):
        """{'act': [L][s_x, s_g, s_u, s_h], 'weight': [L][s_wg, s_wu, s_wd]}"""
        act, w = N.frt_fp4_get_scales(self.handle, self.n_layers)
        return {"act": [act[4 * l:4 * l + 4] for l in range(self.n_layers)],
                "weight": [w[3 * l:3 * l + 3] for l in range(self.n_layers)]}

    def set_scales(self, act):
        """act: per layer (s_x, s_g, s_u, s_h)."""
        N.frt_fp4_set_scales(self.handle, [float(v) for row in act for v in row])

    def forward(self, residual, hidden=None, out=None, stream=None):
        M = residual.shape[0]
        if out is None:
            out = torch.empty_like(residual)
        N.frt_fp4_forward(self.handle, _bf16(residual, (M, self.d), "residual"),
                          _bf16(hidden, (M, self.d), "hidden") if hidden is not None else None,
                          _bf16(out, (M, self.d), "out"), M, _stream(stream))
        return out

    def forward_profile(self, residual, hidden=None, out=None, n_replays=20, stream=None):
        """Per-launch shares (us) of the forward replayed as one graph: index
        3 l + s for layer l and step s (0 norm, 1 gate/up, 2 down); the
        median of n_replays.  Needs a stream other than the legacy default."""
        M = residual.shape[0]
        if out is None:
            out = torch.empty_like(residual)
        return N.frt_fp4_forward_profile(self.handle, _bf16(residual, (M, self.d), "residual"),
                                         _bf16(hidden, (M, self.d), "hidden") if hidden is not None else None,
                                         _bf16(out, (M, self.d), "out"), M, n_replays, 3 * self.n_layers,
                                         _stream(stream))

    def trace(self, layer, residual, hidden=None, stream=None):
        """One layer with its intermediates: codes are packed uint8 (two per
        byte), x_sf / h_sf in the TMEM-ready layout, g_sf / u_sf row-major."""
        M, d, ff = residual.shape[0], self.d, self.ff
        dev = residual.device
        mt = (M + 127) // 128 * 128
        u8 = lambda *s: torch.empty(s, dtype=torch.uint8, device=dev)
        t = {"out": torch.empty_like(residual), "r_prime": torch.empty_like(residual),
             "x_codes": u8(M, d // 2), "x_sf": u8(mt * d // 16), "g_codes": u8(M, ff // 2), "g_sf": u8(M, ff // 16),
             "u_codes": u8(M, ff // 2), "u_sf": u8(M, ff // 16), "h_codes": u8(M, ff // 2), "h_sf": u8(mt * ff // 16)}
        N.frt_fp4_debug_trace(self.handle, layer, _bf16(residual, (M, d), "residual"),
                              _bf16(hidden, (M, d), "hidden") if hidden is not None else None,
                              *[t[k].data_ptr() for k in ("out", "r_prime", "x_codes", "x_sf", "g_codes", "g_sf",
                                                          "u_codes", "u_sf", "h_codes", "h_sf")], M, _stream(stream))
        if hidden is None:
            del t["r_prime"]
        return t

    def trace_from(self, layer, residual, hidden=None, x=None, h=None, stream=None):
        """One layer step by step: x = (codes [M, d/2] uint8, TMEM-ready scales) replaces the norm's X for
        the gate/up GEMM, h = (codes [M, ff/2], TMEM-ready scales) the gate/up output A for the down GEMM
        (None: the kernels' own).  Returns g/u codes and row-major scales, h as the gate/up GEMM produced
        it, and the layer output."""
        M, d, ff = residual.shape[0], self.d, self.ff
        dev = residual.device
        mt = (M + 127) // 128 * 128
        u8 = lambda *s: torch.empty(s, dtype=torch.uint8, device=dev)
        t = {"out": torch.empty_like(residual), "g_codes": u8(M, ff // 2), "g_sf": u8(M, ff // 16),
             "u_codes": u8(M, ff // 2), "u_sf": u8(M, ff // 16), "h_codes": u8(M, ff // 2), "h_sf": u8(mt * ff // 16)}

        def pair(v, kk, what):
            if v is None:
                return None, None
            codes, sf = v
            if codes.dtype != torch.uint8 or sf.dtype != torch.uint8 or tuple(codes.shape) != (M, kk // 2) or \
                    sf.numel() != mt * kk // 16 or not codes.is_contiguous() or not sf.is_contiguous():
                raise ValueError("%s: uint8 codes (%d, %d) and %d scale bytes" % (what, M, kk // 2, mt * kk // 16))
            return codes.data_ptr(), sf.data_ptr()

        xc, xs = pair(x, d, "x")
        hc, hs = pair(h, ff, "h")
        N.frt_fp4_debug_trace_from(self.handle, layer, _bf16(residual, (M, d), "residual"),
                                   _bf16(hidden, (M, d), "hidden") if hidden is not None else None, xc, xs, hc, hs,
                                   *[t[k].data_ptr() for k in ("out", "g_codes", "g_sf", "u_codes", "u_sf",
                                                               "h_codes", "h_sf")], M, _stream(stream))
        return t

    def weights(self, layer, which, stream=None):
        """which: 'gate', 'up' or 'down' -> (codes row-major [rows, K/2], TMEM-ready scales)."""
        w = {"gate": 0, "up": 1, "down": 2}[which]
        rows, K = (self.ff, self.d) if w < 2 else (self.d, self.ff)
        dev = torch.device("cuda")
        codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
        sf = torch.empty(rows * K // 16, dtype=torch.uint8, device=dev)
        N.frt_fp4_debug_weights(self.handle, layer, w, codes.data_ptr(), sf.data_ptr(), _stream(stream))
        return codes, sf

    def device_status(self, stream=None):
        N.frt_fp4_device_status(self.handle, _stream(stream))

    def debug_stall(self, M, stream=None):
        """Test hook: a gate/up GEMM whose bounded wait gives up; raises FrtError(DEVICE_TIMEOUT)."""
        N.frt_fp4_debug_stall(self.handle, M, _stream(stream))


def nvfp4_gemm(a_codes, a_sf, b_codes, b_sf, M, N_, K, alpha=1.0, splits=1, stream=None):
    """Diagnostic block-scaled GEMM: fp32 [M, N] = alpha * A . B^T over NVFP4
    operands, split-K into at most `splits` partials summed in split order
    (fresh zeroed arrival counters each call)."""
    dev = a_codes.device
    out = torch.empty((M, N_), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    tiles = (N_ // 128) * ((M + 127) // 128)
    ws = torch.empty(tiles * splits * 128 * 128 if splits > 1 else 4, dtype=torch.float32, device=dev)
    counters = torch.zeros(max(tiles, 1), dtype=torch.int32, device=dev)
    N.frt_nvfp4_gemm(_ptr(a_codes), _ptr(a_sf), _ptr(b_codes), _ptr(b_sf), M, N_, K, float(alpha), out.data_ptr(),
                     int(splits), ws.data_ptr(), counters.data_ptr(), err.data_ptr(), _stream(stream))
    return out, err, counters
