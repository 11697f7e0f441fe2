"""ctypes binding of libfrt_ffn.so (include/frt_ffn.h, include/frt_qkv.h, include/frt_nvfp4.h).

Argument marshalling only: every step of the FFN path runs in the CUDA
library.  The functions keep the C names; a non-OK status raises FrtError
with the library's message.  There is no fallback: if the library has not
been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfrt_ffn.so")

FRT_OK = 0
STATUS = {
    0: "FRT_OK", 1: "FRT_ERR_INVALID_ARG", 2: "FRT_ERR_UNSUPPORTED", 3: "FRT_ERR_OOM", 4: "FRT_ERR_NOT_READY",
    5: "FRT_ERR_SHAPE", 6: "FRT_ERR_CAPTURE", 7: "FRT_ERR_STALE_GRAPH", 8: "FRT_ERR_CUDA",
    9: "FRT_ERR_DEVICE_TIMEOUT",
}
FRT_ACT_GEGLU_TANH = 0
FRT_ACT_SWIGLU = 1

# every symbol include/frt_ffn.h declares, with (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_FP = ctypes.POINTER(ctypes.c_float)
SIGNATURES = {
    "frt_ffn_plan_create": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_P)]),
    "frt_ffn_plan_destroy": (_I, [_P]),
    "frt_ffn_load_weights": (_I, [_P, _I, _P, _P, _P, _P, _P]),
    "frt_ffn_load_weights_ex": (_I, [_P, _I, _P, _P, _P, _P, ctypes.c_uint, _P]),
    "frt_ffn_calibrate": (_I, [_P, ctypes.POINTER(_P), ctypes.POINTER(_P), _I, _I, _P]),
    "frt_ffn_get_scales": (_I, [_P, _FP, _FP, _FP, _FP]),
    "frt_ffn_set_modulation": (_I, [_P, ctypes.POINTER(_P), _I]),
    "frt_ffn_set_scales": (_I, [_P, _FP, _FP]),
    "frt_ffn_forward": (_I, [_P, _P, _P, _P, _I, _P]),
    "frt_ffn_graph_capture": (_I, [_P, _P, _P, _P, _I, _P]),
    "frt_ffn_graph_replay": (_I, [_P, _I, _P]),
    "frt_ffn_graph_profile": (_I, [_P, _I, _I, _FP, ctypes.POINTER(ctypes.c_int), _P]),
    "frt_ffn_graph_autotune": (_I, [_P, _P, _P, _P, _I, _I, _I, ctypes.POINTER(ctypes.c_float),
                                   ctypes.POINTER(ctypes.c_int), _P]),
    "frt_ffn_debug_trace": (_I, [_P, _I, _P, _P, _I, _P, _P, _P, _P, _P, _P]),
    "frt_ffn_debug_trace_qx": (_I, [_P, _I, _P, _P, _I, _P, _P, _P, _P]),
    "frt_ffn_debug_weights": (_I, [_P, _I, _P, _P, _P]),
    "frt_ffn_uses_stack_kernel": (_I, [_P, _I]),
    "frt_ffn_debug_stack": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "frt_debug_e4m3_encode_range": (_I, [ctypes.c_uint, ctypes.c_ulonglong, _P, _P]),
    "frt_ffn_device_status": (_I, [_P, _P]),
    "frt_ffn_debug_stall": (_I, [_P, _P]),
    "frt_ffn_debug_step": (_I, [_P, _I, _I, _I, _P]),
    "frt_fp8_gemm": (_I, [_P, _P, _P, _P, _I, _I, _I, _F, _I, _I, _P]),
    "frt_ffn_last_error": (ctypes.c_char_p, []),
    "frt_fp8_gemm_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _F, _P]),
    "frt_fp8_gemm_noalloc_last_error": (ctypes.c_char_p, []),
    "frt_fp8_gemm_noalloc_status": (_I, [_P]),
    "frt_fp8_gemm_noalloc_debug_stall": (_I, [_P]),
    # include/frt_qkv.h
    "frt_qkv_plan_create": (_I, [_I, _I, _I, _I, _F, _I, _I, ctypes.POINTER(_P)]),
    "frt_qkv_plan_destroy": (_I, [_P]),
    "frt_qkv_load_weights": (_I, [_P, _I, _P, _P, _P, _P, _P]),
    "frt_qkv_load_weights_ex": (_I, [_P, _I, _P, _P, _P, _P, ctypes.c_uint, _P]),
    "frt_qkv_calibrate": (_I, [_P, _I, ctypes.POINTER(_P), ctypes.POINTER(_P), _I, _I, _P]),
    "frt_qkv_get_scales": (_I, [_P, _FP, _FP]),
    "frt_qkv_set_scales": (_I, [_P, _FP]),
    "frt_qkv_forward": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P]),
    "frt_qkv_debug_trace": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P]),
    "frt_qkv_device_status": (_I, [_P, _P]),
    "frt_qkv_debug_weights": (_I, [_P, _I, _P, _P]),
    "frt_qkv_debug_trace_qx": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _I, _P]),
    # include/frt_nvfp4.h
    "frt_fp4_plan_create": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_P)]),
    "frt_fp4_plan_destroy": (_I, [_P]),
    "frt_fp4_load_weights": (_I, [_P, _I, _P, _P, _P, _P, _P, _P]),
    "frt_fp4_calibrate": (_I, [_P, ctypes.POINTER(_P), ctypes.POINTER(_P), _I, _I, _P]),
    "frt_fp4_get_scales": (_I, [_P, _FP, _FP]),
    "frt_fp4_set_scales": (_I, [_P, _FP]),
    "frt_fp4_forward": (_I, [_P, _P, _P, _P, _I, _P]),
    "frt_fp4_forward_profile": (_I, [_P, _P, _P, _P, _I, _I, _FP, ctypes.POINTER(ctypes.c_int), _P]),
    "frt_fp4_debug_trace": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P]),
    "frt_fp4_debug_weights": (_I, [_P, _I, _I, _P, _P, _P]),
    "frt_fp4_debug_trace_from": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P]),
    "frt_nvfp4_gemm": (_I, [_P, _P, _P, _P, _I, _I, _I, _F, _P, _I, _P, _P, _P, _P]),
    "frt_fp4_device_status": (_I, [_P, _P]),
    "frt_fp4_debug_stall": (_I, [_P, _I, _P]),
}


class FrtError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS.get(status, str(status)), message))
        self.status = status
        self.name = STATUS.get(status, str(status))


_lib = None


def lib() -> ctypes.CDLL:
    """Load libfrt_ffn.so (built by realtime_transformer_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libfrt_ffn.so is not built; run `python -m realtime_transformer_gb300.build` "
                              "(or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != FRT_OK:
        msg = lib().frt_ffn_last_error()
        raise FrtError(status, msg.decode() if msg else "")


def _ptrs(values):
    arr = (_P * len(values))(*[v if v else None for v in values])
    return arr


def frt_ffn_plan_create(d: int, ff: int, act: int, M_max: int, n_layers: int) -> int:
    out = _P()
    _check(lib().frt_ffn_plan_create(d, ff, act, M_max, n_layers, ctypes.byref(out)))
    return out.value


def frt_ffn_plan_destroy(plan: int) -> None:
    _check(lib().frt_ffn_plan_destroy(plan))


def frt_ffn_load_weights(plan, layer, w_norm, w_gate, w_up, w_down, stream) -> None:
    _check(lib().frt_ffn_load_weights(plan, layer, w_norm, w_gate, w_up, w_down, stream))


FRT_LOAD_FOLD_NORM = 1


def frt_ffn_load_weights_ex(plan, layer, w_norm, w_gate, w_up, w_down, flags, stream) -> None:
    _check(lib().frt_ffn_load_weights_ex(plan, layer, w_norm, w_gate, w_up, w_down, flags, stream))


def frt_ffn_calibrate(plan, residual_ptrs, hidden_ptrs, M, stream) -> None:
    n = len(residual_ptrs)
    r = _ptrs(residual_ptrs)
    h = _ptrs(hidden_ptrs) if hidden_ptrs is not None else None
    _check(lib().frt_ffn_calibrate(plan, ctypes.cast(r, ctypes.POINTER(_P)),
                                   ctypes.cast(h, ctypes.POINTER(_P)) if h is not None else None, n, M, stream))


def frt_ffn_set_modulation(plan, mod_ptrs, mod_rows) -> None:
    if mod_ptrs is None:
        _check(lib().frt_ffn_set_modulation(plan, None, 0))
        return
    arr = _ptrs(mod_ptrs)
    _check(lib().frt_ffn_set_modulation(plan, ctypes.cast(arr, ctypes.POINTER(_P)), mod_rows))


def frt_ffn_get_scales(plan, n_layers: int):
    arrs = [(ctypes.c_float * n_layers)() for _ in range(4)]
    _check(lib().frt_ffn_get_scales(plan, *[ctypes.cast(a, _FP) for a in arrs]))
    return [list(a) for a in arrs]


def frt_ffn_set_scales(plan, s_x, s_h) -> None:
    n = len(s_x)
    ax = (ctypes.c_float * n)(*s_x)
    ah = (ctypes.c_float * n)(*s_h)
    _check(lib().frt_ffn_set_scales(plan, ctypes.cast(ax, _FP), ctypes.cast(ah, _FP)))


def frt_ffn_forward(plan, residual_in, hidden_in, out, M, stream) -> None:
    _check(lib().frt_ffn_forward(plan, residual_in, hidden_in, out, M, stream))


def frt_ffn_graph_capture(plan, residual_in, hidden_in, out, M, stream) -> None:
    _check(lib().frt_ffn_graph_capture(plan, residual_in, hidden_in, out, M, stream))


def frt_ffn_graph_replay(plan, M, stream) -> None:
    _check(lib().frt_ffn_graph_replay(plan, M, stream))


GRAPH_TACTICS = ("defaults", "global split-K exchange", "single-CTA tiles", "no programmatic dependent launch")


def frt_ffn_graph_autotune(plan, residual_in, hidden_in, out, M, n_tries, n_replays, stream):
    """-> (median replay time of the kept graph in us, index into GRAPH_TACTICS)."""
    best = ctypes.c_float(0.0)
    tactic = ctypes.c_int(0)
    _check(lib().frt_ffn_graph_autotune(plan, residual_in, hidden_in, out, M, n_tries, n_replays,
                                        ctypes.byref(best), ctypes.byref(tactic), stream))
    return best.value, tactic.value


def frt_ffn_graph_profile(plan, M, n_replays, n_slots, stream) -> list[float]:
    """Per-launch shares (us) of a replay of the graph held for M (median of n_replays)."""
    buf = (ctypes.c_float * n_slots)()
    n = ctypes.c_int(0)
    _check(lib().frt_ffn_graph_profile(plan, M, n_replays, buf, ctypes.byref(n), stream))
    return [float(buf[i]) for i in range(n.value)]


def frt_ffn_debug_trace(plan, layer, residual_in, hidden_in, M, r_prime, q_x, gu, q_h, out, stream) -> None:
    _check(lib().frt_ffn_debug_trace(plan, layer, residual_in, hidden_in, M, r_prime, q_x, gu, q_h, out, stream))


def frt_ffn_debug_trace_qx(plan, layer, r_prime, q_x, M, gu, q_h, out, stream) -> None:
    _check(lib().frt_ffn_debug_trace_qx(plan, layer, r_prime, q_x, M, gu, q_h, out, stream))


def frt_ffn_uses_stack_kernel(plan, M) -> bool:
    return bool(lib().frt_ffn_uses_stack_kernel(plan, M))


def frt_ffn_debug_stack(plan, r, h, out, M, q_x_in, res_in, q_x, gu, q_h, layer_out, times, stream) -> None:
    _check(lib().frt_ffn_debug_stack(plan, r, h, out, M, q_x_in, res_in, q_x, gu, q_h, layer_out, times, stream))


def frt_ffn_debug_weights(plan, layer, w_gu, w_down, stream) -> None:
    _check(lib().frt_ffn_debug_weights(plan, layer, w_gu, w_down, stream))


def frt_debug_e4m3_encode_range(start, n, codes, stream) -> None:
    _check(lib().frt_debug_e4m3_encode_range(start, n, codes, stream))


def frt_ffn_debug_step(plan, layer, step, M, stream) -> None:
    _check(lib().frt_ffn_debug_step(plan, layer, step, M, stream))


def frt_ffn_device_status(plan, stream) -> None:
    _check(lib().frt_ffn_device_status(plan, stream))


def frt_ffn_debug_stall(plan, stream) -> None:
    _check(lib().frt_ffn_debug_stall(plan, stream))


def frt_fp8_gemm(plan, A, B, C, M, N, K, alpha, path, splits, stream) -> None:
    _check(lib().frt_fp8_gemm(plan, A, B, C, M, N, K, alpha, path, splits, stream))


def frt_fp8_gemm_noalloc(A, B, C, M, N, K, alpha, stream) -> None:
    """FP8 GEMM with no plan and no allocation (scratch in a fixed device array)."""
    _check_noalloc(lib().frt_fp8_gemm_noalloc(A, B, C, M, N, K, alpha, stream))


def _check_noalloc(st: int) -> None:
    if st != FRT_OK:
        msg = lib().frt_fp8_gemm_noalloc_last_error()
        raise FrtError(st, msg.decode() if msg else "")


def frt_fp8_gemm_noalloc_status(stream) -> None:
    """Synchronise `stream`; raise FRT_ERR_DEVICE_TIMEOUT if an allocation-free GEMM gave up a wait."""
    _check_noalloc(lib().frt_fp8_gemm_noalloc_status(stream))


def frt_fp8_gemm_noalloc_debug_stall(stream) -> None:
    _check_noalloc(lib().frt_fp8_gemm_noalloc_debug_stall(stream))


def frt_ffn_last_error() -> str:
    msg = lib().frt_ffn_last_error()
    return msg.decode() if msg else ""



# -- attention-input sublayer (include/frt_qkv.h) ----------------------------

def frt_qkv_plan_create(d, n_q_heads, n_kv_heads, head_dim, rope_base, M_max, n_layers) -> int:
    out = _P()
    _check(lib().frt_qkv_plan_create(d, n_q_heads, n_kv_heads, head_dim, rope_base, M_max, n_layers,
                                     ctypes.byref(out)))
    return out.value


def frt_qkv_plan_destroy(plan) -> None:
    _check(lib().frt_qkv_plan_destroy(plan))


def frt_qkv_load_weights(plan, layer, w_norm, w_q, w_k, w_v, stream) -> None:
    _check(lib().frt_qkv_load_weights(plan, layer, w_norm, w_q, w_k, w_v, stream))


def frt_qkv_load_weights_ex(plan, layer, w_norm, w_q, w_k, w_v, flags, stream) -> None:
    _check(lib().frt_qkv_load_weights_ex(plan, layer, w_norm, w_q, w_k, w_v, flags, stream))


def frt_qkv_calibrate(plan, layer, residual_ptrs, hidden_ptrs, M, stream) -> None:
    n = len(residual_ptrs)
    r = _ptrs(residual_ptrs)
    h = _ptrs(hidden_ptrs) if hidden_ptrs is not None else None
    _check(lib().frt_qkv_calibrate(plan, layer, ctypes.cast(r, ctypes.POINTER(_P)),
                                   ctypes.cast(h, ctypes.POINTER(_P)) if h is not None else None, n, M, stream))


def frt_qkv_get_scales(plan, n_layers: int):
    arrs = [(ctypes.c_float * n_layers)() for _ in range(2)]
    _check(lib().frt_qkv_get_scales(plan, *[ctypes.cast(a, _FP) for a in arrs]))
    return [list(a) for a in arrs]


def frt_qkv_set_scales(plan, s_x) -> None:
    arr = (ctypes.c_float * len(s_x))(*s_x)
    _check(lib().frt_qkv_set_scales(plan, ctypes.cast(arr, _FP)))


def frt_qkv_forward(plan, layer, residual_in, hidden_in, positions, r_prime, q, k, v, M, stream) -> None:
    _check(lib().frt_qkv_forward(plan, layer, residual_in, hidden_in, positions, r_prime, q, k, v, M, stream))


def frt_qkv_debug_trace(plan, layer, residual_in, hidden_in, positions, r_prime, q, k, v, q_x, qkv, M,
                        stream) -> None:
    _check(lib().frt_qkv_debug_trace(plan, layer, residual_in, hidden_in, positions, r_prime, q, k, v, q_x, qkv,
                                     M, stream))


def frt_qkv_debug_trace_qx(plan, layer, q_x, positions, q, k, v, qkv, M, stream) -> None:
    _check(lib().frt_qkv_debug_trace_qx(plan, layer, q_x, positions, q, k, v, qkv, M, stream))


def frt_qkv_debug_weights(plan, layer, w_qkv, stream) -> None:
    _check(lib().frt_qkv_debug_weights(plan, layer, w_qkv, stream))


def frt_qkv_device_status(plan, stream) -> None:
    _check(lib().frt_qkv_device_status(plan, stream))


# -- NVFP4 sublayer (include/frt_nvfp4.h) -----------------------------------

def frt_fp4_plan_create(d, ff, act, M_max, n_layers) -> int:
    out = _P()
    _check(lib().frt_fp4_plan_create(d, ff, act, M_max, n_layers, ctypes.byref(out)))
    return out.value


def frt_fp4_plan_destroy(plan) -> None:
    _check(lib().frt_fp4_plan_destroy(plan))


def frt_fp4_load_weights(plan, layer, w_norm, w_gate, w_up, w_down, awq, stream) -> None:
    _check(lib().frt_fp4_load_weights(plan, layer, w_norm, w_gate, w_up, w_down, awq, stream))


def frt_fp4_calibrate(plan, residual_ptrs, hidden_ptrs, M, stream) -> None:
    n = len(residual_ptrs)
    r = _ptrs(residual_ptrs)
    h = _ptrs(hidden_ptrs) if hidden_ptrs is not None else None
    _check(lib().frt_fp4_calibrate(plan, ctypes.cast(r, ctypes.POINTER(_P)),
                                   ctypes.cast(h, ctypes.POINTER(_P)) if h is not None else None, n, M, stream))


def frt_fp4_get_scales(plan, n_layers: int):
    act = (ctypes.c_float * (4 * n_layers))()
    w = (ctypes.c_float * (3 * n_layers))()
    _check(lib().frt_fp4_get_scales(plan, ctypes.cast(act, _FP), ctypes.cast(w, _FP)))
    return list(act), list(w)


def frt_fp4_set_scales(plan, act) -> None:
    arr = (ctypes.c_float * len(act))(*act)
    _check(lib().frt_fp4_set_scales(plan, ctypes.cast(arr, _FP)))


def frt_fp4_forward(plan, residual_in, hidden_in, out, M, stream) -> None:
    _check(lib().frt_fp4_forward(plan, residual_in, hidden_in, out, M, stream))


def frt_fp4_forward_profile(plan, residual_in, hidden_in, out, M, n_replays, n_slots, stream) -> list[float]:
    """Per-launch shares (us) of a replayed graph of the NVFP4 forward (median of n_replays)."""
    buf = (ctypes.c_float * n_slots)()
    n = ctypes.c_int(0)
    _check(lib().frt_fp4_forward_profile(plan, residual_in, hidden_in, out, M, n_replays, buf, ctypes.byref(n),
                                         stream))
    return [float(buf[i]) for i in range(n.value)]


def frt_fp4_debug_trace(plan, layer, residual_in, hidden_in, out, r_prime, x_codes, x_sf, g_codes, g_sf, u_codes,
                        u_sf, h_codes, h_sf, M, stream) -> None:
    _check(lib().frt_fp4_debug_trace(plan, layer, residual_in, hidden_in, out, r_prime, x_codes, x_sf, g_codes,
                                     g_sf, u_codes, u_sf, h_codes, h_sf, M, stream))


def frt_fp4_debug_trace_from(plan, layer, residual_in, hidden_in, x_codes_in, x_sf_in, h_codes_in, h_sf_in, out,
                             g_codes, g_sf, u_codes, u_sf, h_codes, h_sf, M, stream) -> None:
    _check(lib().frt_fp4_debug_trace_from(plan, layer, residual_in, hidden_in, x_codes_in, x_sf_in, h_codes_in,
                                          h_sf_in, out, g_codes, g_sf, u_codes, u_sf, h_codes, h_sf, M, stream))


def frt_fp4_debug_weights(plan, layer, which, codes, sf, stream) -> None:
    _check(lib().frt_fp4_debug_weights(plan, layer, which, codes, sf, stream))


def frt_nvfp4_gemm(a_codes, a_sf, b_codes, b_sf, M, N, K, alpha, out, splits, ws, counters, err, stream) -> None:
    _check(lib().frt_nvfp4_gemm(a_codes, a_sf, b_codes, b_sf, M, N, K, alpha, out, splits, ws, counters, err,
                                stream))


def frt_fp4_device_status(plan, stream) -> None:
    _check(lib().frt_fp4_device_status(plan, stream))


def frt_fp4_debug_stall(plan, M, stream) -> None:
    _check(lib().frt_fp4_debug_stall(plan, M, stream))
