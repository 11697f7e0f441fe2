"""Pins of the oracle's norm-weight fold (itsolotime FlashRT article, 5.2:
Pi0 folds the RMSNorm weight into the fused gate/up weights before
quantisation; Pi0.5 does not).  Folded layer: W'[j][k] = W[j][k] w[k] over
[W_gate; W_up], one E4M3 scale over W', and the norm multiplies by ones."""
import numpy as np
import pytest

import synthetic

WL = synthetic.WORKLOADS["tiny"]


def weights(layer=0, wl=WL):
    return {k: synthetic.bf16_bits(v) for k, v in synthetic.layer_weights(wl, layer).items()}


def const_norm(orc, d, c):
    return orc.bf16_encode(np.full(d, c, dtype=np.float32))


def test_folded_products_are_exact(orc):
    w = weights()
    f = orc.fold_norm_weight(w["w_gate"], w["w_up"], w["w_norm"])
    gu = np.concatenate([orc.bf16_decode(w["w_gate"]), orc.bf16_decode(w["w_up"])], 0).astype(np.float64)
    exact = gu * orc.bf16_decode(w["w_norm"]).astype(np.float64)[None, :]
    assert f.dtype == np.float32 and np.array_equal(f.astype(np.float64), exact)
    # column k is scaled by w[k], not row j by w[j]
    k = int(np.argmax(np.abs(orc.bf16_decode(w["w_norm"]) - 1.0)))
    assert f[3, k] == np.float32(gu[3, k] * orc.bf16_decode(w["w_norm"])[k])


def test_fold_with_unit_norm_weight_is_the_plain_quantisation(orc):
    w = weights()
    ones = const_norm(orc, WL.d, 1.0)
    assert np.all(ones == orc.BF16_ONE)
    a = orc.quantize_layer_weights_folded(w["w_gate"], w["w_up"], w["w_down"], ones)
    b = orc.quantize_layer_weights(w["w_gate"], w["w_up"], w["w_down"])
    assert np.array_equal(a[0], b[0]) and a[1] == b[1]
    assert np.array_equal(a[2], b[2]) and a[3] == b[3]


@pytest.mark.parametrize("c", [0.5, 2.0, 8.0])
def test_fold_with_power_of_two_norm_weight_scales_exactly(orc, c):
    w = weights()
    a = orc.quantize_layer_weights_folded(w["w_gate"], w["w_up"], w["w_down"], const_norm(orc, WL.d, c))
    b = orc.quantize_layer_weights(w["w_gate"], w["w_up"], w["w_down"])
    assert np.array_equal(a[0], b[0])
    assert np.float32(a[1]) == np.float32(b[1]) * np.float32(c)


@pytest.mark.parametrize("act", [0, 1])
def test_folded_layer_equals_unfolded_for_a_constant_norm_weight(orc, act):
    """Norm weight c (a power of two): the unfolded layer with s_x and the
    folded one with s_x / c quantise the same values and use the same alpha,
    so every code and the output agree bit for bit."""
    c = 0.5
    w = weights()
    wn = const_norm(orc, WL.d, c)
    r, h = [synthetic.bf16_bits(x) for x in synthetic.inputs(WL)]
    qu = orc.quantize_stack([dict(w, w_norm=wn)])[0]
    qf = orc.quantize_stack([dict(w, w_norm=wn)], fold_norm=True)[0]
    assert np.all(qf.w_norm == orc.BF16_ONE)
    s_x, s_h = 0.0123, 0.0071
    u = orc.ffn_layer(r, h, qu.w_norm, qu.q_gu, qu.q_down, s_x, s_h, qu.s_gu, qu.s_d, act, trace=True)
    f = orc.ffn_layer(r, h, qf.w_norm, qf.q_gu, qf.q_down, float(np.float32(s_x) / np.float32(c)), s_h, qf.s_gu,
                      qf.s_d, act, trace=True)
    assert np.array_equal(u.q_x, f.q_x)
    assert np.array_equal(u.gu, f.gu)
    assert np.array_equal(u.q_h, f.q_h)
    assert np.array_equal(u.out, f.out)


def test_folded_fp8_layer_keeps_the_cosine_claim(orc):
    """Folded or not, the layer computes W (norm(r') * w) in real arithmetic:
    the folded FP8 layer stays within cosine > 0.999 of the unfolded fp32
    forward (agentlenshq FlashRT summary, "Main ideas")."""
    w = weights()
    r, h = [synthetic.bf16_bits(x) for x in synthetic.inputs(WL)]
    cb = synthetic.calibration_batches(WL)
    q = orc.quantize_stack([w], fold_norm=True)
    s_x, s_h = orc.calibrate_stack(q, [synthetic.bf16_bits(a) for a, _ in cb],
                                   [synthetic.bf16_bits(b) for _, b in cb], WL.act_id)
    out = orc.stack_forward(q, r, h, s_x, s_h, WL.act_id)
    ref = orc.ref_stack_f32([w], r, h, WL.act_id)
    a = orc.bf16_decode(out).astype(np.float64).ravel()
    b = ref.astype(np.float64).ravel()
    assert a @ b / np.linalg.norm(a) / np.linalg.norm(b) > 0.999
    # and the fold matters: the same codes read with the norm weight applied
    # twice (folded weights, unfolded norm) move the output
    wrong = orc.stack_forward([orc.QuantLayer(w["w_norm"], q[0].q_gu, q[0].s_gu, q[0].q_down, q[0].s_d)], r, h,
                              s_x, s_h, WL.act_id)
    assert not np.array_equal(wrong, out)
