"""Plain CPU oracle of the FP8 FFN sublayer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (``realtime_transformer_gb300``
and its CUDA library) never imports, links or calls it, and the two share no
code: this package wraps ``frt_oracle.c`` (plain fp32 C, bit-level E4M3/BF16)
through ctypes and loops over layers in Python.

Every function cites the passage it restates (page title, section):
  * agentlenshq "flashrt-project/FlashRT" summary, "Main ideas": fused
    residual-norm-quantise, FP8 per-tensor calibration, cosine > 0.999.
  * itsolotime FlashRT article, 5.2 (FusedGateUp + Quant), 7.1 (FP8 path),
    7.2 (per-layer FFN loop).
  * "FlashRT docs/architecture.md", 6 "Calibration Framework" and "What
    happens when you call model.predict".

Arrays are numpy: BF16 tensors travel as ``uint16`` bit patterns, E4M3 tensors
as ``uint8`` codes, scales as Python floats (fp32 values).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "frt_oracle.c")
_LIB = os.path.join(_HERE, "libfrt_oracle.so")

ACT_GEGLU_TANH = 0
ACT_SWIGLU = 1
EPS = 1e-6  # reading: the pages never state the RMSNorm epsilon


def build(force: bool = False) -> str:
    """Compile frt_oracle.c with gcc (fp contraction off, OpenMP on)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-fvisibility=hidden", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, f32, u8, u16 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_uint8, ctypes.c_uint16
        sig = {
            "orc_e4m3_decode": (f32, [u8]),
            "orc_e4m3_encode": (u8, [f32]),
            "orc_bf16_encode": (u16, [f32]),
            "orc_bf16_decode": (f32, [u16]),
            "orc_e4m3_encode_array": (None, [P, i64, P]),
            "orc_bf16_encode_array": (None, [P, i64, P]),
            "orc_scale_from_amax": (f32, [f32]),
            "orc_amax_bf16": (f32, [P, i64]),
            "orc_amax_f32": (f32, [P, i64]),
            "orc_quantize_bf16": (None, [P, i64, f32, P]),
            "orc_quantize_f32": (None, [P, i64, f32, P]),
            "orc_quantize_weight": (f32, [P, i64, P]),
            "orc_residual_rmsnorm": (None, [i32, i32, f32, P, P, P, P, P]),
            "orc_gemm_e4m3": (None, [i32, i32, i32, P, P, P]),
            "orc_gelu_tanh": (f32, [f32]),
            "orc_silu": (f32, [f32]),
            "orc_gated_act": (None, [i32, i32, i32, P, P]),
            "orc_gated_act_f32": (None, [i64, i32, P, P, P]),
            "orc_ffn_layer": (i32, [i32, i32, i32, i32, f32, P, P, P, P, P, f32, f32, f32, f32, P, P, P, P, P]),
            "orc_calibrate_layer": (i32, [i32, i32, i32, i32, f32, i32, P, P, P, P, P, f32, f32,
                                          ctypes.POINTER(f32), ctypes.POINTER(f32), P]),
            "orc_ref_layer_f32": (i32, [i32, i32, i32, i32, f32, P, P, P, P, P, P, P]),
            "orc_ref_layer_f32_ex": (i32, [i32, i32, i32, i32, f32, P, P, P, P, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint16)


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint8)


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """E4M3 codes -> fp32 values (OCP E4M3 'fn' definition)."""
    c = _u8(codes)
    table = np.array([lib().orc_e4m3_decode(i) for i in range(256)], dtype=np.float32)
    return table[c]


def e4m3_encode(x) -> np.ndarray:
    """fp32 -> E4M3 codes, round to nearest even, saturating to +-448."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


def bf16_encode(x) -> np.ndarray:
    """fp32 -> BF16 bit patterns, round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_bf16_encode_array(_p(x), x.size, _p(out))
    return out


def bf16_decode(b) -> np.ndarray:
    b = _u16(b)
    return (b.astype(np.uint32) << 16).view(np.float32)


def scale_from_amax(amax: float) -> float:
    return float(lib().orc_scale_from_amax(amax))


def recip(s: float) -> float:
    """fp32 reciprocal 1/s, the multiplier every quantisation uses."""
    return float(np.float32(1.0) / np.float32(s))


# --------------------------------------------------------------------------
# Steps
# --------------------------------------------------------------------------

def quantize_weight(w_bf16) -> tuple[np.ndarray, float]:
    """Step A0: per-tensor E4M3 weight quantisation -> (codes, scale)."""
    w = _u16(w_bf16)
    q = np.empty(w.shape, dtype=np.uint8)
    s = lib().orc_quantize_weight(_p(w), w.size, _p(q))
    return q, float(s)


def quantize_layer_weights(w_gate, w_up, w_down):
    """Step A0 for one layer: one scale over [W_gate; W_up], one for W_down."""
    w_gu = np.concatenate([_u16(w_gate), _u16(w_up)], axis=0)
    q_gu, s_gu = quantize_weight(w_gu)
    q_d, s_d = quantize_weight(w_down)
    return q_gu, s_gu, q_d, s_d


BF16_ONE = 0x3F80


def fold_norm_weight(w_gate, w_up, w_norm) -> np.ndarray:
    """The RMSNorm weight folded into the gate/up weights (itsolotime
    article, 5.2: the Pi0 spec's FusedGateUp(..., norm_fuse=...) ahead of
    Quant()): W'[j][k] = W[j][k] * w[k] over [W_gate; W_up], fp32.  The
    product of two BF16 values has at most 16 significant bits, so it is
    exact in fp32 (reading: the fold happens on the BF16 checkpoint tensors,
    before quantisation, with no rounding of its own)."""
    w_gu = bf16_decode(np.concatenate([_u16(w_gate), _u16(w_up)], axis=0))
    return (w_gu * bf16_decode(w_norm)[None, :]).astype(np.float32)


def quantize_layer_weights_folded(w_gate, w_up, w_down, w_norm):
    """Step A0 with the norm weight folded into [W_gate; W_up]: one scale
    over the folded fp32 matrix (amax / 448, the same rule as every weight),
    codes E4M3(W' * (1/s)); W_down as without the fold.  The layer's norm
    then multiplies by ones (the weight now lives in the GEMM)."""
    w_f = fold_norm_weight(w_gate, w_up, w_norm)
    s_gu = scale_from_amax(amax_f32(w_f))
    q_gu = quantize_f32(w_f, recip(s_gu))
    q_d, s_d = quantize_weight(w_down)
    return q_gu, s_gu, q_d, s_d


def residual_rmsnorm(r, h, w_norm, eps: float = EPS):
    """Step A1 before quantisation -> (r' BF16 bits, y fp32)."""
    r = _u16(r)
    M, d = r.shape
    hh = _u16(h) if h is not None else None
    w = _u16(w_norm)
    rp = np.empty((M, d), dtype=np.uint16)
    y = np.empty((M, d), dtype=np.float32)
    lib().orc_residual_rmsnorm(M, d, eps, _p(r), _p(hh), _p(w), _p(rp), _p(y))
    return rp, y


def quantize_f32(x, inv_s: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.empty(x.shape, dtype=np.uint8)
    lib().orc_quantize_f32(_p(x), x.size, inv_s, _p(q))
    return q


def amax_f32(x) -> float:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return float(lib().orc_amax_f32(_p(x), x.size))


def gemm_e4m3(A, B) -> np.ndarray:
    """acc = dec(A) dec(B)^T in fp32, k ascending; A [M,K], B [N,K] codes."""
    A = _u8(A)
    B = _u8(B)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    acc = np.empty((M, N), dtype=np.float32)
    lib().orc_gemm_e4m3(M, N, K, _p(A), _p(B), _p(acc))
    return acc


def gelu_tanh(g: float) -> float:
    return float(lib().orc_gelu_tanh(g))


def silu(g: float) -> float:
    return float(lib().orc_silu(g))


def gated_act(gu_bf16, act: int) -> np.ndarray:
    """Step A3 before quantisation: a = act(g) * u from the BF16 [M, 2ff] GEMM output."""
    gu = _u16(gu_bf16)
    M, two_ff = gu.shape
    ff = two_ff // 2
    a = np.empty((M, ff), dtype=np.float32)
    lib().orc_gated_act(M, ff, act, _p(gu), _p(a))
    return a


@dataclass
class LayerTrace:
    out: np.ndarray       # [M,d] BF16 bits
    r_prime: np.ndarray   # [M,d] BF16 bits
    q_x: np.ndarray       # [M,d] E4M3 codes
    gu: np.ndarray        # [M,2ff] BF16 bits
    q_h: np.ndarray       # [M,ff] E4M3 codes


def ffn_layer(r, h, w_norm, q_gu, q_down, s_x, s_h, s_gu, s_d, act: int, eps: float = EPS,
              trace: bool = False):
    """Steps A1..A4 of one layer with fixed scales -> out (or a LayerTrace)."""
    r = _u16(r)
    M, d = r.shape
    q_gu = _u8(q_gu)
    q_down = _u8(q_down)
    ff = q_down.shape[1]
    assert q_gu.shape == (2 * ff, d) and q_down.shape == (d, ff)
    hh = _u16(h) if h is not None else None
    out = np.empty((M, d), dtype=np.uint16)
    if trace:
        rp = np.empty((M, d), dtype=np.uint16)
        qx = np.empty((M, d), dtype=np.uint8)
        gu = np.empty((M, 2 * ff), dtype=np.uint16)
        qh = np.empty((M, ff), dtype=np.uint8)
    else:
        rp = qx = gu = qh = None
    rc = lib().orc_ffn_layer(M, d, ff, act, eps, _p(r), _p(hh), _p(_u16(w_norm)), _p(q_gu), _p(q_down),
                             s_x, s_h, s_gu, s_d, _p(out), _p(rp), _p(qx), _p(gu), _p(qh))
    if rc != 0:
        raise MemoryError("oracle layer allocation failed")
    if trace:
        return LayerTrace(out, rp, qx, gu, qh)
    return out


def calibrate_layer(r_batches, h_batches, w_norm, q_gu, q_down, s_gu, s_d, act: int, eps: float = EPS):
    """Step A6 for one layer: progressive amax over the calibration batches.

    Returns (s_x, s_h, next_residuals)."""
    rb = [_u16(r) for r in r_batches]
    M, d = rb[0].shape
    ff = _u8(q_down).shape[1]
    nb = len(rb)
    hb = [_u16(h) for h in h_batches] if h_batches is not None else None
    outs = [np.empty((M, d), dtype=np.uint16) for _ in range(nb)]
    P = ctypes.c_void_p
    r_arr = (P * nb)(*[_p(a) for a in rb])
    h_arr = (P * nb)(*[_p(a) for a in hb]) if hb is not None else None
    o_arr = (P * nb)(*[_p(a) for a in outs])
    sx = ctypes.c_float()
    sh = ctypes.c_float()
    rc = lib().orc_calibrate_layer(M, d, ff, act, eps, nb, ctypes.cast(r_arr, P),
                                   ctypes.cast(h_arr, P) if h_arr is not None else None,
                                   _p(_u16(w_norm)), _p(_u8(q_gu)), _p(_u8(q_down)), s_gu, s_d,
                                   ctypes.byref(sx), ctypes.byref(sh), ctypes.cast(o_arr, P))
    if rc != 0:
        raise MemoryError("oracle calibration allocation failed")
    return float(sx.value), float(sh.value), outs


def ref_layer_f32(r, h, w_norm, w_gate, w_up, w_down, act: int, eps: float = EPS) -> np.ndarray:
    """Unquantised fp32 layer (the baseline of the cosine > 0.999 claim)."""
    r = np.ascontiguousarray(r, dtype=np.float32)
    M, d = r.shape
    ff = _u16(w_gate).shape[0]
    hh = np.ascontiguousarray(h, dtype=np.float32) if h is not None else None
    out = np.empty((M, d), dtype=np.float32)
    rc = lib().orc_ref_layer_f32(M, d, ff, act, eps, _p(r), _p(hh), _p(_u16(w_norm)), _p(_u16(w_gate)),
                                 _p(_u16(w_up)), _p(_u16(w_down)), _p(out))
    if rc != 0:
        raise MemoryError("oracle reference allocation failed")
    return out


# --------------------------------------------------------------------------
# Stack (step A5 semantics: r_{l+1} = out_l, hidden added at layer 0 only)
# --------------------------------------------------------------------------

@dataclass
class QuantLayer:
    w_norm: np.ndarray
    q_gu: np.ndarray
    s_gu: float
    q_down: np.ndarray
    s_d: float


def quantize_stack(layers, fold_norm: bool = False) -> list[QuantLayer]:
    """Step A0 over a list of dicts with w_norm, w_gate, w_up, w_down (BF16
    bits); fold_norm: the norm weight folded into the gate/up weights."""
    out = []
    for lw in layers:
        if fold_norm:
            q_gu, s_gu, q_d, s_d = quantize_layer_weights_folded(lw["w_gate"], lw["w_up"], lw["w_down"],
                                                                 lw["w_norm"])
            w_norm = np.full(_u16(lw["w_norm"]).shape, BF16_ONE, dtype=np.uint16)
        else:
            q_gu, s_gu, q_d, s_d = quantize_layer_weights(lw["w_gate"], lw["w_up"], lw["w_down"])
            w_norm = _u16(lw["w_norm"])
        out.append(QuantLayer(w_norm, q_gu, s_gu, q_d, s_d))
    return out


def calibrate_stack(qlayers, r_batches, h_batches, act: int, eps: float = EPS):
    """Step A6 over the stack -> (s_x[L], s_h[L])."""
    s_x, s_h = [], []
    rb = list(r_batches)
    hb = list(h_batches) if h_batches is not None else None
    for l, ql in enumerate(qlayers):
        sx, sh, rb = calibrate_layer(rb, hb if l == 0 else None, ql.w_norm, ql.q_gu, ql.q_down,
                                     ql.s_gu, ql.s_d, act, eps)
        s_x.append(sx)
        s_h.append(sh)
    return s_x, s_h


def calibrate_stack_unquantized(layers, r_batches, h_batches, act: int, eps: float = EPS):
    """Step A6, the other reading of "run one forward, record the amax": the
    scales from the unquantised fp32 forward (BF16 master weights, fp32
    activations, no E4M3 rounding anywhere), so no layer sees an earlier
    layer's quantisation.  A flag of the oracle, not the contract (the
    progressive calibrate_stack is).  Returns (s_x[L], s_h[L])."""
    cur = [bf16_decode(b) for b in r_batches]
    hb = [bf16_decode(b) for b in h_batches] if h_batches is not None else None
    s_x, s_h = [], []
    for l, lw in enumerate(layers):
        my, ma = 0.0, 0.0
        nxt = []
        for b, x in enumerate(cur):
            x = np.ascontiguousarray(x, dtype=np.float32)
            M, d = x.shape
            ff = _u16(lw["w_gate"]).shape[0]
            hh = np.ascontiguousarray(hb[b], dtype=np.float32) if (hb is not None and l == 0) else None
            out = np.empty((M, d), dtype=np.float32)
            ry = np.empty(M, dtype=np.float32)
            ra = np.empty(M, dtype=np.float32)
            rc = lib().orc_ref_layer_f32_ex(M, d, ff, act, eps, _p(x), _p(hh), _p(_u16(lw["w_norm"])),
                                            _p(_u16(lw["w_gate"])), _p(_u16(lw["w_up"])), _p(_u16(lw["w_down"])),
                                            _p(out), _p(ry), _p(ra))
            if rc != 0:
                raise MemoryError("oracle reference allocation failed")
            my, ma = max(my, float(ry.max())), max(ma, float(ra.max()))
            nxt.append(out)
        s_x.append(scale_from_amax(my))
        s_h.append(scale_from_amax(ma))
        cur = nxt
    return s_x, s_h


def stack_forward(qlayers, r, h, s_x, s_h, act: int, eps: float = EPS, trace: bool = False):
    """Quantised forward through all layers -> final out (or per-layer traces)."""
    cur = _u16(r)
    traces = []
    for l, ql in enumerate(qlayers):
        res = ffn_layer(cur, h if l == 0 else None, ql.w_norm, ql.q_gu, ql.q_down, s_x[l], s_h[l],
                        ql.s_gu, ql.s_d, act, eps, trace=trace)
        if trace:
            traces.append(res)
            cur = res.out
        else:
            cur = res
    return traces if trace else cur


def ref_stack_f32(layers, r, h, act: int, eps: float = EPS) -> np.ndarray:
    """fp32 unquantised forward through all layers (BF16 master weights)."""
    cur = bf16_decode(r) if np.asarray(r).dtype == np.uint16 else np.asarray(r, dtype=np.float32)
    hf = None
    if h is not None:
        hf = bf16_decode(h) if np.asarray(h).dtype == np.uint16 else np.asarray(h, dtype=np.float32)
    for l, lw in enumerate(layers):
        cur = ref_layer_f32(cur, hf if l == 0 else None, lw["w_norm"], lw["w_gate"], lw["w_up"],
                            lw["w_down"], act, eps)
    return cur


# --------------------------------------------------------------------------
# Attention-side input projections: residual + RMSNorm + E4M3 quantise ->
# FP8 fused-QKV GEMM -> QKV split + RoPE (agentlenshq FlashRT summary,
# "What it is": residual-norm-quantise and RoPE kernels; itsolotime article,
# 5.2: FusedQKV(q, k, v) quantised as one tensor; "FlashRT
# docs/architecture.md", 8 Kernel Library: "qkv split + RoPE").
# --------------------------------------------------------------------------

def rope_inv_freq(head_dim: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i / head_dim), i < head_dim / 2, evaluated in fp64
    and rounded to fp32 (reading: the usual inverse-frequency vector)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return (float(base) ** (-2.0 * i / head_dim)).astype(np.float32)


def rope(x, pos, inv_freq) -> np.ndarray:
    """Rotary position embedding, rotate-half layout (reading): element i of
    the first half pairs with element i + hd/2.  angle = fp32(pos * theta_i)
    (fp32 product), cos and sin of that fp32 angle rounded to fp32, then in
    fp32: o_i = x_i cos - x_{i+hd/2} sin, o_{i+hd/2} = x_{i+hd/2} cos + x_i sin.
    x [..., M, H, hd] fp32 values, pos [M] integers; returns fp32."""
    x = np.asarray(x, dtype=np.float32)
    hd = x.shape[-1]
    half = hd // 2
    ang = (np.asarray(pos).astype(np.float32)[:, None] * np.asarray(inv_freq, np.float32)[None, :])
    c = np.cos(ang.astype(np.float64)).astype(np.float32)[:, None, :]
    s = np.sin(ang.astype(np.float64)).astype(np.float32)[:, None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    o1 = (x1 * c).astype(np.float32) - (x2 * s).astype(np.float32)
    o2 = (x2 * c).astype(np.float32) + (x1 * s).astype(np.float32)
    return np.concatenate([o1.astype(np.float32), o2.astype(np.float32)], axis=-1)


def quantize_qkv_weights(w_q, w_k, w_v):
    """Step A0 for the fused QKV weight: [W_q; W_k; W_v] as one tensor with
    one per-tensor scale -> (codes, scale)."""
    return quantize_weight(np.concatenate([_u16(w_q), _u16(w_k), _u16(w_v)], axis=0))


def quantize_qkv_weights_folded(w_q, w_k, w_v, w_norm):
    """The fused QKV weight with the RMSNorm weight folded in (itsolotime
    article, 5.2: the Pi0 spec's FusedQKV(..., norm_fuse=...)): W'[j][k] =
    W[j][k] * w[k] over [W_q; W_k; W_v] in fp32 (exact), one scale
    amax(W') / 448 -> (codes, scale); the sublayer's norm then multiplies by
    ones."""
    w = bf16_decode(np.concatenate([_u16(w_q), _u16(w_k), _u16(w_v)], axis=0))
    f = (w * bf16_decode(w_norm)[None, :]).astype(np.float32)
    s = scale_from_amax(amax_f32(f))
    return quantize_f32(f, recip(s)), s


@dataclass
class QKVTrace:
    r_prime: np.ndarray   # [M,d] BF16 bits
    q_x: np.ndarray       # [M,d] E4M3 codes
    qkv: np.ndarray       # [M,(Hq+2Hkv)hd] BF16 bits (GEMM output)
    q: np.ndarray         # [Hq,M,hd] BF16 bits (rotated)
    k: np.ndarray         # [Hkv,M,hd] BF16 bits (rotated)
    v: np.ndarray         # [Hkv,M,hd] BF16 bits


def qkv_layer(r, h, w_norm, q_qkv, s_x, s_qkv, n_q: int, n_kv: int, head_dim: int, pos, inv_freq,
              eps: float = EPS) -> QKVTrace:
    """One attention-input sublayer with fixed scales: r' = bf16(r + h),
    y = RMSNorm(r') w, q_x = E4M3(y / s_x) (step A1); qkv = bf16(acc * alpha),
    acc = q_x . W_qkv^T in fp32, alpha = s_x s_qkv (as step A2, plain BF16
    output); split into heads (the first Hq*hd columns are Q, then K, then V)
    and RoPE on Q and K, each rounded to BF16; outputs head-major [H, M, hd]
    (reading: the layout an attention kernel reads per head)."""
    r = _u16(r)
    M, d = r.shape
    rp, y = residual_rmsnorm(r, h, w_norm, eps)
    q_x = quantize_f32(y, recip(s_x))
    acc = gemm_e4m3(q_x, q_qkv)
    alpha = np.float32(np.float32(s_x) * np.float32(s_qkv))
    qkv = bf16_encode((acc * alpha).astype(np.float32))
    vals = bf16_decode(qkv)
    nq, nk = n_q * head_dim, n_kv * head_dim
    qh = vals[:, :nq].reshape(M, n_q, head_dim)
    kh = vals[:, nq:nq + nk].reshape(M, n_kv, head_dim)
    vh = qkv[:, nq + nk:nq + 2 * nk].reshape(M, n_kv, head_dim)
    q = bf16_encode(rope(qh, pos, inv_freq)).transpose(1, 0, 2)
    k = bf16_encode(rope(kh, pos, inv_freq)).transpose(1, 0, 2)
    v = vh.transpose(1, 0, 2)
    return QKVTrace(rp, q_x, qkv, np.ascontiguousarray(q), np.ascontiguousarray(k), np.ascontiguousarray(v))


def calibrate_qkv_layer(r_batches, h_batches, w_norm, eps: float = EPS) -> float:
    """Step A6 for the QKV sublayer: s_x = amax(y) / 448 over the batches."""
    amax = 0.0
    for i, r in enumerate(r_batches):
        _, y = residual_rmsnorm(r, h_batches[i] if h_batches is not None else None, w_norm, eps)
        amax = max(amax, amax_f32(y))
    return scale_from_amax(np.float32(amax))


# --------------------------------------------------------------------------
# AdaRMSNorm variant (itsolotime FlashRT article, 5.2: Pi0.5's decoder
# modulates "via AdaRMSNorm Dense layers" instead of a norm weight).  The
# pages give no formula; reading (the adaptive-norm form of diffusion
# transformers): a Dense layer of the conditioning gives per-token
# modulation vectors scale, shift and gate [M, d] (one row shared by all
# tokens when the conditioning is per sample); the norm output is
# y = (r' * inv) * (1 + scale) + shift (no norm weight), and the sublayer
# output is r' + gate * FFN(y).  Each operation in fp32, in that order.
# --------------------------------------------------------------------------

def split_modulation(mod, M: int, d: int):
    """mod [R, 3d] BF16 bits (scale | shift | gate), R = 1 (shared) or M ->
    (scale, shift, gate) fp32 [M, d]."""
    m = bf16_decode(mod).reshape(-1, 3 * d)
    assert m.shape[0] in (1, M)
    m = np.broadcast_to(m, (M, 3 * d))
    return (np.ascontiguousarray(m[:, :d]), np.ascontiguousarray(m[:, d:2 * d]),
            np.ascontiguousarray(m[:, 2 * d:]))


def ada_rmsnorm(r, h, mod, eps: float = EPS):
    """Step A1 with AdaRMSNorm before quantisation -> (r' BF16 bits, y fp32)."""
    r = _u16(r)
    M, d = r.shape
    rp, y0 = residual_rmsnorm(r, h, np.full(d, BF16_ONE, dtype=np.uint16), eps)  # y0 = r' * inv exactly
    scale, shift, _ = split_modulation(mod, M, d)
    one_plus = (np.float32(1.0) + scale).astype(np.float32)
    y = ((y0 * one_plus).astype(np.float32) + shift).astype(np.float32)
    return rp, y


def ffn_layer_ada(r, h, mod, q_gu, q_down, s_x, s_h, s_gu, s_d, act: int, eps: float = EPS,
                  trace: bool = False):
    """Steps A1..A4 of one AdaRMSNorm layer with fixed scales: A1 as
    ada_rmsnorm then q_x = E4M3(y / s_x); A2, A3 as ffn_layer (BF16 g/u,
    a = act(g) u, q_h = E4M3(a / s_h)); A4 out = bf16(r' + (acc * alpha_d) *
    gate)."""
    r = _u16(r)
    M, d = r.shape
    ff = _u8(q_down).shape[1]
    rp, y = ada_rmsnorm(r, h, mod, eps)
    q_x = quantize_f32(y, recip(s_x))
    gu = bf16_encode((gemm_e4m3(q_x, q_gu) * np.float32(np.float32(s_x) * np.float32(s_gu))).astype(np.float32))
    a = gated_act(gu, act)
    q_h = quantize_f32(a, recip(s_h))
    t = (gemm_e4m3(q_h, q_down) * np.float32(np.float32(s_h) * np.float32(s_d))).astype(np.float32)
    _, _, gate = split_modulation(mod, M, d)
    t = (t * gate).astype(np.float32)
    out = bf16_encode((bf16_decode(rp) + t).astype(np.float32))
    if trace:
        return LayerTrace(out, rp, q_x, gu, q_h)
    return out


def calibrate_stack_ada(qlayers, mods, r_batches, h_batches, act: int, eps: float = EPS):
    """Step A6 over an AdaRMSNorm stack (progressive, as calibrate_stack);
    mods[l] is layer l's modulation -> (s_x[L], s_h[L])."""
    s_x, s_h = [], []
    rb = [_u16(r) for r in r_batches]
    hb = [_u16(h) for h in h_batches] if h_batches is not None else None
    for l, ql in enumerate(qlayers):
        hl = hb if l == 0 else None
        ys = [ada_rmsnorm(r, hl[i] if hl is not None else None, mods[l], eps) for i, r in enumerate(rb)]
        sx = scale_from_amax(np.float32(max(amax_f32(y) for _, y in ys)))
        acts = []
        for _, y in ys:
            q_x = quantize_f32(y, recip(sx))
            gu = bf16_encode((gemm_e4m3(q_x, ql.q_gu) * np.float32(np.float32(sx) * np.float32(ql.s_gu)))
                             .astype(np.float32))
            acts.append(gated_act(gu, act))
        sh = scale_from_amax(np.float32(max(amax_f32(a) for a in acts)))
        rb = [ffn_layer_ada(r, hl[i] if hl is not None else None, mods[l], ql.q_gu, ql.q_down, sx, sh, ql.s_gu,
                            ql.s_d, act, eps) for i, r in enumerate(rb)]
        s_x.append(sx)
        s_h.append(sh)
    return s_x, s_h


def stack_forward_ada(qlayers, mods, r, h, s_x, s_h, act: int, eps: float = EPS):
    cur = _u16(r)
    for l, ql in enumerate(qlayers):
        cur = ffn_layer_ada(cur, h if l == 0 else None, mods[l], ql.q_gu, ql.q_down, s_x[l], s_h[l], ql.s_gu,
                            ql.s_d, act, eps)
    return cur


# --------------------------------------------------------------------------
# NVFP4 variant of the sublayer (itsolotime article, 7.2: gate and up as two
# NVFP4 GEMMs that emit packed FP4 plus scales, a fused GeGLU kernel that
# requantises FP4 to FP4, an NVFP4 down GEMM, the residual kept in 16 bits,
# AWQ pre-scaling of the normalised activation).  The pages do not define the
# format; reading: NVFP4 as published by NVIDIA -- E2M1 elements, one E4M3
# scale per 16 consecutive elements along K, one fp32 scale per tensor.
# --------------------------------------------------------------------------

FP4_BLOCK = 16
E2M1_MAX = 6.0
NVFP4_RANGE = 448.0 * 6.0  # amax -> per-tensor scale: the block scales then span E4M3
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)


def e2m1_decode(codes) -> np.ndarray:
    """4-bit E2M1 codes (bit 3 sign, bits 2..1 exponent, bit 0 mantissa) -> fp32."""
    c = _u8(codes)
    mag = _E2M1_MAG[c & 7]
    return np.where(c & 8, -mag, mag).astype(np.float32)


def e2m1_encode(x) -> np.ndarray:
    """fp32 -> E2M1 codes: nearest of the eight magnitudes, a tie to the even
    mantissa bit, saturating at 6; the sign kept (a negative that rounds to 0
    gives code 8, -0)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    a = np.abs(x)
    lo = np.clip(np.searchsorted(_E2M1_MAG, a, side="right") - 1, 0, 7)
    hi = np.minimum(lo + 1, 7)
    d_lo = a - _E2M1_MAG[lo]
    d_hi = _E2M1_MAG[hi] - a
    up = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(a >= np.float32(E2M1_MAX), 7, np.where(up, hi, lo))
    return (idx | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def nvfp4_scale_from_amax(amax: float) -> float:
    """Per-tensor scale amax / (448 * 6) in fp32 (1 for an all-zero tensor)."""
    a = np.float32(amax)
    return float(a / np.float32(NVFP4_RANGE)) if a > 0 else 1.0


def nvfp4_quantize(x, s: float):
    """fp32 [rows, K] with per-tensor scale s -> (E2M1 codes [rows, K], E4M3
    block-scale codes [rows, K / 16]).  Per block of 16 along K (fp32 ops):
    b = E4M3(amax_block * (1 / (6 s))); then every element
    q = E2M1(x * (1 / (dec(b) * s))), or code 0 where dec(b) is 0."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, K = x.shape
    assert K % FP4_BLOCK == 0
    blk = x.reshape(rows, K // FP4_BLOCK, FP4_BLOCK)
    amax_b = np.abs(blk).max(axis=2)
    inv6 = np.float32(recip(np.float32(6.0) * np.float32(s)))
    sb = e4m3_encode((amax_b * inv6).astype(np.float32))
    den = (e4m3_decode(sb) * np.float32(s)).astype(np.float32)
    safe = np.where(den > 0, den, np.float32(1.0))
    inv = np.where(den > 0, np.float32(1.0) / safe, np.float32(0.0)).astype(np.float32)
    q = e2m1_encode((blk * inv[:, :, None]).astype(np.float32))
    return q.reshape(rows, K), sb


def nvfp4_decode(q, sb, s: float) -> np.ndarray:
    """Codes + block scales + tensor scale -> fp32 values: (e2m1 * dec(b)) is
    exact in fp32; the product with s is rounded once."""
    q = _u8(q)
    rows, K = q.shape
    v = e2m1_decode(q).reshape(rows, K // FP4_BLOCK, FP4_BLOCK) * e4m3_decode(sb)[:, :, None]
    return (v.astype(np.float32) * np.float32(s)).astype(np.float32).reshape(rows, K)


def nvfp4_gemm(qa, sa, qb, sb) -> np.ndarray:
    """Block-scaled product without the tensor scales: acc[m][n] =
    sum_k e2m1(A[m][k]) dec(sa[m][k/16]) e2m1(B[n][k]) dec(sb[n][k/16]),
    A [M, K], B [N, K]; evaluated in fp64 (every product exact), rounded to fp32."""
    a = (e2m1_decode(qa).astype(np.float64).reshape(_u8(qa).shape[0], -1, FP4_BLOCK)
         * e4m3_decode(sa).astype(np.float64)[:, :, None]).reshape(_u8(qa).shape)
    b = (e2m1_decode(qb).astype(np.float64).reshape(_u8(qb).shape[0], -1, FP4_BLOCK)
         * e4m3_decode(sb).astype(np.float64)[:, :, None]).reshape(_u8(qb).shape)
    return (a @ b.T).astype(np.float32)


@dataclass
class NVFP4Weight:
    q: np.ndarray    # [rows, K] E2M1 codes
    sb: np.ndarray   # [rows, K / 16] E4M3 block-scale codes
    s: float         # fp32 tensor scale


def quantize_weight_nvfp4(w_bf16, col_scale=None) -> NVFP4Weight:
    """NVFP4 weight preparation: W'[j][k] = fp32(W[j][k] * c[k]) (c the AWQ
    scale of input channel k, or none), one tensor scale amax(W') / 2688."""
    w = bf16_decode(w_bf16)
    if col_scale is not None:
        w = (w * np.asarray(col_scale, np.float32)[None, :]).astype(np.float32)
    s = nvfp4_scale_from_amax(amax_f32(w))
    q, sb = nvfp4_quantize(w, s)
    return NVFP4Weight(q, sb, s)


def awq_scales(y_batches, alpha: float = 0.5) -> np.ndarray:
    """AWQ per-input-channel scales from calibration activations (the
    normalised y the gate/up GEMMs read): c_k = max(mean_t |y[t][k]|, 1e-5)^alpha
    in fp64, rounded to fp32 (reading: the pages name AWQ and an alpha, not
    the search; this is the activation-magnitude rule of the AWQ method)."""
    y = np.concatenate([np.asarray(b, np.float64) for b in y_batches], axis=0)
    return np.power(np.maximum(np.abs(y).mean(axis=0), 1e-5), alpha).astype(np.float32)


@dataclass
class NVFP4Layer:
    w_norm: np.ndarray       # [d] BF16 bits
    awq: np.ndarray | None   # [d] fp32 AWQ scales (None: no pre-scaling)
    gate: NVFP4Weight        # [ff, d]
    up: NVFP4Weight          # [ff, d]
    down: NVFP4Weight        # [d, ff]


def quantize_layer_nvfp4(w_norm, w_gate, w_up, w_down, awq=None) -> NVFP4Layer:
    """Weights of one NVFP4 layer: gate and up quantised separately (the split
    gate/up of the pages), each with the AWQ column scales; down without."""
    return NVFP4Layer(_u16(w_norm), None if awq is None else np.asarray(awq, np.float32),
                      quantize_weight_nvfp4(w_gate, awq), quantize_weight_nvfp4(w_up, awq),
                      quantize_weight_nvfp4(w_down))


@dataclass
class NVFP4Scales:
    s_x: float   # normalised (and AWQ-divided) activation
    s_g: float   # gate GEMM output
    s_u: float   # up GEMM output
    s_h: float   # gated activation


@dataclass
class NVFP4Trace:
    out: np.ndarray      # [M, d] BF16 bits
    r_prime: np.ndarray  # [M, d] BF16 bits
    x: tuple             # (codes [M, d], block scales [M, d/16])
    g: tuple             # (codes [M, ff], block scales [M, ff/16])
    u: tuple
    h: tuple
    y: np.ndarray        # [M, d] fp32, before quantisation
    g_f32: np.ndarray    # [M, ff] fp32 gate GEMM output before quantisation
    u_f32: np.ndarray
    a: np.ndarray        # [M, ff] fp32 gated activation before quantisation


def _nvfp4_awq_divide(y, awq):
    if awq is None:
        return y
    inv = (np.float32(1.0) / np.asarray(awq, np.float32)).astype(np.float32)
    return (y * inv[None, :]).astype(np.float32)


def nvfp4_gated_act(g4, u4, s_g, s_u, act):
    """The combine step of the NVFP4 encoder FFN (itsolotime FlashRT article,
    7.2): act(dec G) * dec U in fp32 from G and U as (E2M1 codes, row-major
    block-scale codes) with tensor scales s_g, s_u."""
    return _nvfp4_gated(g4, u4, s_g, s_u, act)


def _nvfp4_gated(g4, u4, s_g, s_u, act):
    gd = nvfp4_decode(g4[0], g4[1], s_g)
    ud = nvfp4_decode(u4[0], u4[1], s_u)
    a = np.empty(gd.shape, dtype=np.float32)
    lib().orc_gated_act_f32(gd.size, act, _p(np.ascontiguousarray(gd)), _p(np.ascontiguousarray(ud)), _p(a))
    return a


def ffn_layer_nvfp4(r, h, L: NVFP4Layer, sc: NVFP4Scales, act: int, eps: float = EPS, trace: bool = False):
    """One NVFP4 layer with fixed scales, in the pages' order: r' = bf16(r + h);
    y = RMSNorm(r') (fp32); y / c (AWQ); X = NVFP4(y, s_x);
    G = NVFP4(acc(X, W_g) * (s_x s_g'), s_g), U likewise (s_g', s_u' the weight
    scales); A = NVFP4(act(dec G) * dec U, s_h);
    out = bf16(r' + acc(A, W_d) * (s_h s_d'))."""
    rp, y = residual_rmsnorm(r, h, L.w_norm, eps)
    ys = _nvfp4_awq_divide(y, L.awq)
    x4 = nvfp4_quantize(ys, sc.s_x)
    alpha_g = np.float32(np.float32(sc.s_x) * np.float32(L.gate.s))
    alpha_u = np.float32(np.float32(sc.s_x) * np.float32(L.up.s))
    g = (nvfp4_gemm(x4[0], x4[1], L.gate.q, L.gate.sb) * alpha_g).astype(np.float32)
    u = (nvfp4_gemm(x4[0], x4[1], L.up.q, L.up.sb) * alpha_u).astype(np.float32)
    g4 = nvfp4_quantize(g, sc.s_g)
    u4 = nvfp4_quantize(u, sc.s_u)
    a = _nvfp4_gated(g4, u4, sc.s_g, sc.s_u, act)
    h4 = nvfp4_quantize(a, sc.s_h)
    alpha_d = np.float32(np.float32(sc.s_h) * np.float32(L.down.s))
    o = (nvfp4_gemm(h4[0], h4[1], L.down.q, L.down.sb) * alpha_d).astype(np.float32)
    out = bf16_encode((bf16_decode(rp) + o).astype(np.float32))
    if trace:
        return NVFP4Trace(out, rp, x4, g4, u4, h4, ys, g, u, a)
    return out


def calibrate_layer_nvfp4(r_batches, h_batches, L: NVFP4Layer, act: int, eps: float = EPS):
    """Progressive per-tensor calibration of one NVFP4 layer: each scale is
    amax / 2688 over the batches of the tensor it quantises, measured with
    the scales before it already applied.  Returns (NVFP4Scales, outs)."""
    nb = len(r_batches)
    hb = h_batches if h_batches is not None else [None] * nb
    pre = [residual_rmsnorm(r_batches[b], hb[b], L.w_norm, eps) for b in range(nb)]
    ys = [_nvfp4_awq_divide(y, L.awq) for _, y in pre]
    s_x = nvfp4_scale_from_amax(max(amax_f32(y) for y in ys))
    x4 = [nvfp4_quantize(y, s_x) for y in ys]
    alpha_g = np.float32(np.float32(s_x) * np.float32(L.gate.s))
    alpha_u = np.float32(np.float32(s_x) * np.float32(L.up.s))
    g = [(nvfp4_gemm(q, sb, L.gate.q, L.gate.sb) * alpha_g).astype(np.float32) for q, sb in x4]
    u = [(nvfp4_gemm(q, sb, L.up.q, L.up.sb) * alpha_u).astype(np.float32) for q, sb in x4]
    s_g = nvfp4_scale_from_amax(max(amax_f32(t) for t in g))
    s_u = nvfp4_scale_from_amax(max(amax_f32(t) for t in u))
    a = [_nvfp4_gated(nvfp4_quantize(g[b], s_g), nvfp4_quantize(u[b], s_u), s_g, s_u, act) for b in range(nb)]
    s_h = nvfp4_scale_from_amax(max(amax_f32(t) for t in a))
    sc = NVFP4Scales(s_x, s_g, s_u, s_h)
    outs = [ffn_layer_nvfp4(r_batches[b], hb[b], L, sc, act, eps) for b in range(nb)]
    return sc, outs


def calibrate_stack_nvfp4(layers, r_batches, h_batches, act: int, eps: float = EPS):
    """Calibration over the stack (hidden added at layer 0 only) -> [NVFP4Scales]."""
    out = []
    rb = list(r_batches)
    for l, L in enumerate(layers):
        sc, rb = calibrate_layer_nvfp4(rb, h_batches if l == 0 else None, L, act, eps)
        out.append(sc)
    return out


def stack_forward_nvfp4(layers, scales, r, h, act: int, eps: float = EPS):
    cur = _u16(r)
    for l, L in enumerate(layers):
        cur = ffn_layer_nvfp4(cur, h if l == 0 else None, L, scales[l], act, eps)
    return cur

