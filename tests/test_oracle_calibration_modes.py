"""The oracle's two readings of calibration ("FlashRT docs/architecture.md",
6 Calibration Framework: run one forward, record the amax of every FP8 GEMM
input): the progressive contract (each layer measured in the quantised
pipeline) and the unquantised-forward flag.  Pinned against fp64 numpy
evaluations of the unquantised layer and against each other where they must
agree."""
import numpy as np

import oracle
import synthetic


def _case(L=2, M=8):
    wl = synthetic.WORKLOADS["tiny"].with_(L=L, M=M)
    layers = [{k: synthetic.bf16_bits(v) for k, v in synthetic.layer_weights(wl, l).items()} for l in range(L)]
    cb = synthetic.calibration_batches(wl)
    return wl, layers, [synthetic.bf16_bits(a) for a, _ in cb], [synthetic.bf16_bits(b) for _, b in cb]


def _fp64_layer(x, lw, act, eps=oracle.EPS):
    """fp64 unquantised layer: (y, a, out)."""
    w = oracle.bf16_decode(lw["w_norm"]).astype(np.float64)
    y = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + eps) * w
    g = y @ oracle.bf16_decode(lw["w_gate"]).astype(np.float64).T
    u = y @ oracle.bf16_decode(lw["w_up"]).astype(np.float64).T
    if act == oracle.ACT_SWIGLU:
        ag = g / (1 + np.exp(-g))
    else:
        ag = 0.5 * g * (1 + np.tanh(np.sqrt(2 / np.pi) * (g + 0.044715 * g ** 3)))
    a = ag * u
    return y, a, x + a @ oracle.bf16_decode(lw["w_down"]).astype(np.float64).T


def test_unquantized_scales_follow_the_fp64_forward():
    wl, layers, rb, hb = _case()
    s_x, s_h = oracle.calibrate_stack_unquantized(layers, rb, hb, wl.act_id)
    cur = [oracle.bf16_decode(r).astype(np.float64) + oracle.bf16_decode(h).astype(np.float64)
           for r, h in zip(rb, hb)]
    for l, lw in enumerate(layers):
        res = [_fp64_layer(x, lw, wl.act_id) for x in cur]
        my = max(np.abs(y).max() for y, _, _ in res)
        ma = max(np.abs(a).max() for _, a, _ in res)
        assert abs(s_x[l] - my / 448) <= 1e-5 * my / 448, (l, s_x[l], my / 448)
        assert abs(s_h[l] - ma / 448) <= 1e-4 * ma / 448, (l, s_h[l], ma / 448)
        cur = [o for _, _, o in res]


def test_the_two_readings_agree_where_no_quantisation_precedes():
    """Without a hidden input, layer 0's normalised activation is the same
    computation in both readings, so its scale is the same bit for bit; the
    gated activation's scale differs only by the quantisation before it."""
    wl, layers, rb, _ = _case(L=1)
    q = oracle.quantize_stack(layers)
    p_x, p_h = oracle.calibrate_stack(q, rb, None, wl.act_id)
    u_x, u_h = oracle.calibrate_stack_unquantized(layers, rb, None, wl.act_id)
    assert p_x[0] == u_x[0]
    assert p_h[0] != u_h[0] and abs(p_h[0] - u_h[0]) < 0.1 * u_h[0]
