"""FFNPlan: torch-facing wrapper of the C-ABI plan.

PyTorch supplies device memory and streams; every step runs in
libfrt_ffn.so.  Also holds the calibration cache of the "FlashRT
docs/architecture.md", 6 Calibration Framework: scales saved as JSON under
a key made of a hash of the weights and the token count ("{hash}_Se{M}.json").
"""
from __future__ import annotations


import torch

from . import _native as N
from . import calibration

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
    def load_weights(self, layer, w_norm, w_gate, w_up, w_down, stream=None, fold_norm=False, digest=True):
        """Quantise one layer's BF16 weights into the plan; fold_norm: fold
        the RMSNorm weight into the gate/up weights (the Pi0 layout).
        digest: hash every weight element for the calibration cache key
        (reads the weights back to the host); a plan loaded with
        digest=False has no cache key."""
        d, ff = self.d, self.ff
        N.frt_ffn_load_weights_ex(self.handle, layer, _bf16(w_norm, (d,), "w_norm"),
                                  _bf16(w_gate, (ff, d), "w_gate"), _bf16(w_up, (ff, d), "w_up"),
                                  _bf16(w_down, (d, ff), "w_down"), N.FRT_LOAD_FOLD_NORM if fold_norm else 0,
                                  _stream(stream))
        self._digest[layer] = (calibration.weights_digest(b"fold" if fold_norm else b"plain",
                                                          (w_norm, w_gate, w_up, w_down)) if digest else None)

    def calibrate(self, residuals, hiddens=None, stream=None):
        M = residuals[0].shape[0]
        rp = [_bf16(r, (M, self.d), "residual") for r in residuals]
        hp = [_bf16(h, (M, self.d), "hidden") if h is not None else None for h in hiddens] if hiddens else None
        N.frt_ffn_calibrate(self.handle, rp, hp, M, _stream(stream))

    def set_modulation(self, mods):
        """AdaRMSNorm: mods = one BF16 tensor [R, 3d] (scale | shift | gate)
        per layer, R = 1 (shared by all tokens) or M_max; None: plain norm.
        The plan reads the tensors at every forward and replay: keep them."""
        if mods is None:
            N.frt_ffn_set_modulation(self.handle, None, 0)
            self._mods = None
            return
        rows = mods[0].shape[0]
        ptrs = [_bf16(m, (rows, 3 * self.d), "modulation") for m in mods]
        N.frt_ffn_set_modulation(self.handle, ptrs, rows)
        self._mods = list(mods)

    def scales(self):
        s_x, s_h, s_gu, s_d = N.frt_ffn_get_scales(self.handle, self.n_layers)
        return {"s_x": s_x, "s_h": s_h, "s_gu": s_gu, "s_down": s_d}

    def set_scales(self, s_x, s_h):
        N.frt_ffn_set_scales(self.handle, list(map(float, s_x)), list(map(float, s_h)))

    # -- calibration cache ---------------------------------------------------
    def _shape(self):
        return {"d": self.d, "ff": self.ff, "act": self.act, "n_layers": self.n_layers}

    def cache_key(self, M: int) -> str:
        """"{hash}_Se{M}": hash of the shape and the loaded weights."""
        missing = [l for l, dg in enumerate(self._digest) if dg is None]
        if missing:
            raise ValueError("no weight digest for layers %s (not loaded, or loaded with digest=False)"
                             % missing[:8])
        return calibration.cache_key(calibration.checkpoint_hash(self._shape(), self._digest), M)

    def save_scales(self, directory: str | None, M: int, extra: dict | None = None) -> str:
        """Save the plan's scales for token count M; returns the file path."""
        rec = calibration.make_record(self._shape(), M, self.scales(), extra)
        return calibration.save(directory or calibration.default_dir(), self.cache_key(M), rec)

    def load_scales(self, directory: str | None, M: int) -> dict | None:
        """Set the scales cached for M, if a record matching this plan's
        shape and weight scales exists; returns the record (None: miss)."""
        sc = self.scales()
        rec = calibration.load(directory or calibration.default_dir(), self.cache_key(M), self._shape(), M,
                               {"s_gu": sc["s_gu"], "s_down": sc["s_down"]})
        if rec is not None:
            self.set_scales(rec["s_x"], rec["s_h"])
        return rec

    def calibrate_cached(self, residuals, hiddens=None, directory: str | None = None, extra: dict | None = None,
                         stream=None) -> bool:
        """Cache hit: load the scales.  Miss: calibrate on the batches and
        save them.  Returns True on a hit."""
        M = residuals[0].shape[0]
        if self.load_scales(directory, M) is not None:
            return True
        self.calibrate(residuals, hiddens, stream)
        self.save_scales(directory, M, extra)
        return False

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

    def graph_autotune(self, residual, hidden, out, stream, n_tries=4, n_replays=20):
        """Capture n_tries times cycling through the result-neutral schedules
        (_native.GRAPH_TACTICS), keep the fastest capture (median of n_replays
        timed replays each); returns (its replay time in us, its schedule)."""
        M = residual.shape[0]
        return N.frt_ffn_graph_autotune(self.handle, _bf16(residual, (M, self.d), "residual"),
                                        _bf16(hidden, (M, self.d), "hidden") if hidden is not None else None,
                                        _bf16(out, (M, self.d), "out"), M, n_tries, n_replays, _stream(stream))

    def graph_replay(self, M: int, stream=None):
        N.frt_ffn_graph_replay(self.handle, M, _stream(stream))

    def graph_profile(self, M: int, n_replays: int = 20, stream=None):
        """Per-launch shares in microseconds of a replay of the graph held for
        M: launch 3 l + s is layer l's step s (norm, gate/up, down)."""
        return N.frt_ffn_graph_profile(self.handle, M, n_replays, 3 * self.n_layers, _stream(stream))

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

    def trace_layer_from_qx(self, layer, r_prime, q_x, stream=None):
        """Steps A2..A4 of one layer from caller-supplied r' (BF16 [M, d]) and
        q_x (E4M3 codes, uint8 [M, d]); returns g/u, q_h and the output
        (diagnostics: lets another implementation's codes feed the GEMMs)."""
        M, d, ff = r_prime.shape[0], self.d, self.ff
        dev = r_prime.device
        if q_x.dtype != torch.uint8 or tuple(q_x.shape) != (M, d) or not q_x.is_contiguous() or q_x.device != dev:
            raise ValueError("q_x must be a contiguous uint8 [M, d] tensor on the device of r_prime")
        out = {
            "gu": torch.empty((M, 2 * ff), dtype=torch.bfloat16, device=dev),
            "q_h": torch.empty((M, ff), dtype=torch.uint8, device=dev),
            "out": torch.empty((M, d), dtype=torch.bfloat16, device=dev),
        }
        N.frt_ffn_debug_trace_qx(self.handle, layer, _bf16(r_prime, (M, d), "r_prime"), _ptr(q_x), M,
                                 _ptr(out["gu"]), _ptr(out["q_h"]), _ptr(out["out"]), _stream(stream))
        return out

    def uses_stack_kernel(self, M: int) -> bool:
        """Whether the forward for M tokens is the one persistent stack kernel."""
        return N.frt_ffn_uses_stack_kernel(self.handle, M)

    def stack_timeline(self, residual, hidden=None, stream=None):
        """The forward through the persistent stack kernel (the product
        instantiation) with its per-CTA, per-layer timeline: int64
        [CTAs, L, 16] %globaltimer nanoseconds (diagnostics)."""
        M, d, ff, L = residual.shape[0], self.d, self.ff, self.n_layers
        dev = residual.device
        out = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
        times = torch.zeros(((ff // 128) * (d // 256), L, 32), dtype=torch.int64, device=dev)
        N.frt_ffn_debug_stack(self.handle, _bf16(residual, (M, d), "residual"),
                              _bf16(hidden, (M, d), "hidden") if hidden is not None else None, _ptr(out), M,
                              None, None, None, None, None, None, _ptr(times), _stream(stream))
        return out, times

    def debug_stack(self, residual, hidden=None, q_x_in=None, res_in=None, stream=None):
        """The forward through the persistent stack kernel with every layer's
        intermediates dumped (diagnostics).  q_x_in (uint8 [L, M, d])
        replaces each layer's own E4M3 codes of step A1 as the GEMMs' input;
        res_in (BF16 [L, M, d]) replaces the input of every layer >= 1."""
        M, d, ff, L = residual.shape[0], self.d, self.ff, self.n_layers
        dev = residual.device
        o = {
            "out": torch.empty((M, d), dtype=torch.bfloat16, device=dev),
            "q_x": torch.empty((L, M, d), dtype=torch.uint8, device=dev),
            "gu": torch.empty((L, M, 2 * ff), dtype=torch.bfloat16, device=dev),
            "q_h": torch.empty((L, M, ff), dtype=torch.uint8, device=dev),
            "layer_out": torch.empty((L, M, d), dtype=torch.bfloat16, device=dev),
            "times": torch.zeros(((ff // 128) * (d // 256), L, 32), dtype=torch.int64, device=dev),
        }
        for name, t, dt in (("q_x_in", q_x_in, torch.uint8), ("res_in", res_in, torch.bfloat16)):
            if t is not None and (t.dtype != dt or tuple(t.shape) != (L, M, d) or not t.is_contiguous()):
                raise ValueError("%s must be a contiguous [L, M, d] tensor of %s" % (name, dt))
        N.frt_ffn_debug_stack(self.handle, _bf16(residual, (M, d), "residual"),
                              _bf16(hidden, (M, d), "hidden") if hidden is not None else None, _ptr(o["out"]), M,
                              _ptr(q_x_in) if q_x_in is not None else None,
                              _ptr(res_in) if res_in is not None else None, _ptr(o["q_x"]), _ptr(o["gu"]),
                              _ptr(o["q_h"]), _ptr(o["layer_out"]), _ptr(o["times"]), _stream(stream))
        return o

    def weights(self, layer, device="cuda", stream=None):
        """The plan's E4M3 weights of one layer as stored (diagnostics):
        w_gu [2ff, d] with gate and up rows interleaved in blocks of 64, and
        w_down [d, ff], as uint8 tensors."""
        d, ff = self.d, self.ff
        w_gu = torch.empty((2 * ff, d), dtype=torch.uint8, device=device)
        w_down = torch.empty((d, ff), dtype=torch.uint8, device=device)
        N.frt_ffn_debug_weights(self.handle, layer, _ptr(w_gu), _ptr(w_down), _stream(stream))
        return w_gu, w_down

    def gemm(self, A, B, alpha=1.0, path=0, splits=0, stream=None):
        """Diagnostics: C = alpha * A B^T on the plan's FP8 GEMM kernels (A [M,K], B [N,K] uint8 E4M3)."""
        M, K = A.shape
        Nn = B.shape[0]
        C = torch.empty((M, Nn), dtype=torch.float32, device=A.device)
        N.frt_fp8_gemm(self.handle, _ptr(A), _ptr(B), _ptr(C), M, Nn, K, float(alpha), path, splits,
                       _stream(stream))
        return C
