"""Pins of the oracle's AdaRMSNorm variant (itsolotime FlashRT article, 5.2:
Pi0.5 modulates through AdaRMSNorm Dense layers instead of a norm weight).
Reading: y = (r' inv)(1 + scale) + shift, out = r' + gate FFN(y), with the
modulation rows given per token or shared by all tokens."""
import numpy as np
import pytest

import synthetic

WL = synthetic.WORKLOADS["tiny"]


def setup(orc, seed=0):
    w = {k: synthetic.bf16_bits(v) for k, v in synthetic.layer_weights(WL, 0).items()}
    q = orc.quantize_stack([w])[0]
    r, h = [synthetic.bf16_bits(x) for x in synthetic.inputs(WL)]
    return w, q, r, h


def mod_rows(orc, scale, shift, gate):
    return orc.bf16_encode(np.concatenate([scale, shift, gate], axis=-1).astype(np.float32))


def test_identity_modulation_is_the_plain_layer_with_unit_norm_weight(orc):
    """scale 0, shift 0, gate 1: the plain layer with norm weight 1, bit for bit."""
    w, q, r, h = setup(orc)
    d = WL.d
    mod = mod_rows(orc, np.zeros((1, d)), np.zeros((1, d)), np.ones((1, d)))
    ones = np.full(d, orc.BF16_ONE, dtype=np.uint16)
    for act in (0, 1):
        a = orc.ffn_layer_ada(r, h, mod, q.q_gu, q.q_down, 0.0123, 0.0071, q.s_gu, q.s_d, act, trace=True)
        b = orc.ffn_layer(r, h, ones, q.q_gu, q.q_down, 0.0123, 0.0071, q.s_gu, q.s_d, act, trace=True)
        for k in ("r_prime", "q_x", "gu", "q_h", "out"):
            assert np.array_equal(getattr(a, k), getattr(b, k)), (act, k)


def test_zero_gate_passes_the_residual_through(orc):
    w, q, r, h = setup(orc)
    d = WL.d
    rng = np.random.default_rng(1)
    mod = mod_rows(orc, rng.normal(0, 0.1, (1, d)), rng.normal(0, 0.1, (1, d)), np.zeros((1, d)))
    t = orc.ffn_layer_ada(r, h, mod, q.q_gu, q.q_down, 0.0123, 0.0071, q.s_gu, q.s_d, 0, trace=True)
    assert np.array_equal(t.out, t.r_prime)


def test_scale_minus_one_leaves_the_shift(orc):
    """1 + scale = 0: y = shift exactly, so every q_x code is E4M3(shift / s_x)."""
    w, q, r, h = setup(orc)
    d = WL.d
    shift = np.linspace(-2.0, 2.0, d).astype(np.float32)[None, :]
    shift = orc.bf16_decode(orc.bf16_encode(shift))
    mod = mod_rows(orc, -np.ones((1, d)), shift, np.ones((1, d)))
    s_x = 0.01
    t = orc.ffn_layer_ada(r, h, mod, q.q_gu, q.q_down, s_x, 0.0071, q.s_gu, q.s_d, 0, trace=True)
    expect = orc.e4m3_encode((np.broadcast_to(shift, (WL.M, d)) * np.float32(orc.recip(s_x))).astype(np.float32))
    assert np.array_equal(t.q_x, expect)


def test_shared_row_equals_per_token_copies_and_rows_are_independent(orc):
    w, q, r, h = setup(orc)
    d, M = WL.d, WL.M
    rng = np.random.default_rng(2)
    one = mod_rows(orc, rng.normal(0, 0.1, (1, d)), rng.normal(0, 0.1, (1, d)), rng.normal(1, 0.1, (1, d)))
    per = np.repeat(one, M, axis=0)
    a = orc.ffn_layer_ada(r, h, one, q.q_gu, q.q_down, 0.0123, 0.0071, q.s_gu, q.s_d, 1)
    b = orc.ffn_layer_ada(r, h, per, q.q_gu, q.q_down, 0.0123, 0.0071, q.s_gu, q.s_d, 1)
    assert np.array_equal(a, b)
    # per-token rows: permuting tokens and their modulation rows together permutes the output
    mods = mod_rows(orc, rng.normal(0, 0.1, (M, d)), rng.normal(0, 0.1, (M, d)), rng.normal(1, 0.1, (M, d)))
    perm = rng.permutation(M)
    c = orc.ffn_layer_ada(r, h, mods, q.q_gu, q.q_down, 0.0123, 0.0071, q.s_gu, q.s_d, 1)
    e = orc.ffn_layer_ada(r[perm], h[perm], mods[perm], q.q_gu, q.q_down, 0.0123, 0.0071, q.s_gu, q.s_d, 1)
    assert np.array_equal(c[perm], e)


def test_ada_layer_keeps_the_cosine_claim(orc):
    """Against an unquantised fp64 evaluation of the same modulated layer
    (agentlenshq FlashRT summary, "Main ideas": cosine > 0.999)."""
    w, q, r, h = setup(orc)
    d, M = WL.d, WL.M
    rng = np.random.default_rng(3)
    mod = mod_rows(orc, rng.normal(0, 0.2, (M, d)), rng.normal(0, 0.2, (M, d)), rng.normal(1, 0.2, (M, d)))
    cb = synthetic.calibration_batches(WL)
    s_x, s_h = orc.calibrate_stack_ada([q], [mod], [synthetic.bf16_bits(a) for a, _ in cb],
                                       [synthetic.bf16_bits(b) for _, b in cb], WL.act_id)
    out = orc.bf16_decode(orc.stack_forward_ada([q], [mod], r, h, s_x, s_h, WL.act_id)).astype(np.float64)
    sc, sh, gt = [x.astype(np.float64) for x in orc.split_modulation(mod, M, d)]
    rp = orc.bf16_decode(r).astype(np.float64) + orc.bf16_decode(h).astype(np.float64)
    y = rp / np.sqrt((rp ** 2).mean(1, keepdims=True) + orc.EPS) * (1 + sc) + sh
    wg, wu, wd = [orc.bf16_decode(w[k]).astype(np.float64) for k in ("w_gate", "w_up", "w_down")]
    g, u = y @ wg.T, y @ wu.T
    a = 0.5 * g * (1 + np.tanh(np.sqrt(2 / np.pi) * (g + 0.044715 * g ** 3))) * u
    ref = rp + gt * (a @ wd.T)
    assert float(out.ravel() @ ref.ravel() / np.linalg.norm(out) / np.linalg.norm(ref)) > 0.999
