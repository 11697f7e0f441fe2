"""Pins of the oracle's per-step arithmetic: residual add + RMSNorm (step A1),
gated activations (step A3), weight quantisation (step A0) and calibration
(step A6).

Passages: agentlenshq FlashRT summary, "Main ideas" (fused
residual-norm-quantise); itsolotime FlashRT article, 3.3 (rms_norm row),
5.2 (FusedGateUp + Quant), 7.2 (GEGLU/SiLU gate + requantise);
"FlashRT docs/architecture.md", 6 "Calibration Framework".
"""
import math

import numpy as np
import torch
import torch.nn.functional as F


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def ulp32(x):
    x = np.abs(np.asarray(x, np.float32))
    return np.spacing(np.maximum(x, np.float32(np.finfo(np.float32).tiny)))


# --------------------------------------------------------------------- A1 --

def test_residual_add_is_bf16_rounded_sum(orc):
    rng = np.random.default_rng(0)
    r = bf16(rng.standard_normal((4, 64)))
    h = bf16(rng.standard_normal((4, 64)) * 20)
    w = bf16(np.ones(64))
    rp, _ = orc.residual_rmsnorm(r, h, w)
    rt = torch.from_numpy(r.view(np.int16)).view(torch.bfloat16).float()
    ht = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float()
    expect = (rt + ht).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(rp, expect)
    rp2, _ = orc.residual_rmsnorm(r, None, w)
    assert np.array_equal(rp2, r)


def test_rmsnorm_constant_rows_closed_form(orc):
    """A row of constant c has mean square c^2, so y_i = w_i c / sqrt(c^2 + eps)."""
    d = 128
    rng = np.random.default_rng(1)
    w = bf16(1 + 0.1 * rng.standard_normal(d))
    wf = orc.bf16_decode(w).astype(np.float64)
    for c in (1.0, -3.0, 0.5, 20.0, 2.0 ** -8):
        r = bf16(np.full((1, d), c))
        _, y = orc.residual_rmsnorm(r, None, w)
        expect = wf * c / math.sqrt(c * c + 1e-6)
        assert np.all(np.abs(y[0] - expect) <= 4 * ulp32(expect)), c


def test_rmsnorm_matches_fp64_and_torch(orc):
    rng = np.random.default_rng(2)
    M, d = 16, 1024
    r = bf16(rng.standard_normal((M, d)))
    w = bf16(1 + 0.1 * rng.standard_normal(d))
    _, y = orc.residual_rmsnorm(r, None, w)
    rf = orc.bf16_decode(r).astype(np.float64)
    wf = orc.bf16_decode(w).astype(np.float64)
    y64 = rf / np.sqrt((rf ** 2).mean(axis=1, keepdims=True) + 1e-6) * wf
    assert np.max(np.abs(y - y64) / np.abs(y64).max()) < 1e-6
    yt = F.rms_norm(torch.from_numpy(rf), (d,), weight=torch.from_numpy(wf), eps=1e-6).numpy()
    assert np.allclose(y, yt, rtol=1e-5, atol=1e-6)


def test_rmsnorm_zero_row_and_eps(orc):
    d = 64
    w = bf16(np.ones(d))
    _, y = orc.residual_rmsnorm(bf16(np.zeros((1, d))), None, w)
    assert np.all(y == 0)


# --------------------------------------------------------------------- A3 --

def test_activation_special_values(orc):
    assert orc.gelu_tanh(0.0) == 0.0
    assert orc.silu(0.0) == 0.0
    assert orc.gelu_tanh(10.0) == 10.0          # tanh saturates to 1 in fp32
    assert abs(orc.gelu_tanh(-10.0)) < 1e-30
    assert orc.silu(40.0) == 40.0
    assert abs(orc.silu(-40.0)) < 1e-15
    assert abs(orc.gelu_tanh(1.0) - 0.8411919906) < 1e-6   # 0.5(1+tanh(sqrt(2/pi)*1.044715))


def test_activations_match_library_routines(orc):
    g = np.linspace(-12, 12, 4001).astype(np.float32)
    ours_gelu = np.array([orc.gelu_tanh(float(v)) for v in g], np.float32)
    ours_silu = np.array([orc.silu(float(v)) for v in g], np.float32)
    gt = torch.from_numpy(g.astype(np.float64))
    ref_gelu = F.gelu(gt, approximate="tanh").numpy()
    ref_silu = F.silu(gt).numpy()
    # fp32 evaluation of 0.5 g (1 + tanh(.)) cancels where tanh rounds to -1:
    # the absolute error there is about |g| * 2^-23.
    tol = 2e-6 * np.abs(ref_gelu) + np.abs(g) * 2.0 ** -22
    assert np.all(np.abs(ours_gelu - ref_gelu) <= tol)
    tol = 2e-6 * np.abs(ref_silu) + 1e-30
    assert np.all(np.abs(ours_silu - ref_silu) <= tol)


def test_gated_act_uses_gate_half_then_up_half(orc):
    """GU output rows are [g_0..g_{ff-1}, u_0..u_{ff-1}]; a_j = act(g_j) u_j."""
    ff = 8
    g = np.linspace(-2, 2, ff).astype(np.float32)
    u = np.linspace(0.5, 3, ff).astype(np.float32)
    gu = bf16(np.concatenate([g, u])[None, :])
    gb = orc.bf16_decode(gu[0, :ff]).astype(np.float64)
    ub = orc.bf16_decode(gu[0, ff:]).astype(np.float64)
    for act, fn in ((orc.ACT_GEGLU_TANH, lambda x: F.gelu(torch.from_numpy(x), approximate="tanh").numpy()),
                    (orc.ACT_SWIGLU, lambda x: F.silu(torch.from_numpy(x)).numpy())):
        a = orc.gated_act(gu, act)[0]
        expect = fn(gb) * ub
        assert np.allclose(a, expect, rtol=3e-6, atol=1e-7)
        swapped = fn(ub) * gb
        assert not np.allclose(a, swapped, rtol=1e-3)


# --------------------------------------------------------------------- A0 --

def test_weight_quantisation_lossless_on_grid(orc):
    """W = s * dec(c) with s a power of two and a +-448 code present: the
    scale comes out as s and the codes come back unchanged."""
    rng = np.random.default_rng(4)
    c = rng.integers(0, 0x7F, (64, 96)).astype(np.uint8) | (rng.integers(0, 2, (64, 96)).astype(np.uint8) << 7)
    c[c & 0x7F == 0x7F] = 0x7E
    c[3, 5] = 0x7E
    w = orc.e4m3_decode(c).astype(np.float64) * 2.0 ** -10
    wb = bf16(w)
    assert np.array_equal(orc.bf16_decode(wb).astype(np.float64), w)
    q, s = orc.quantize_weight(wb)
    assert s == 448.0 * 2.0 ** -10 / 448.0
    assert np.array_equal(q, c)


def test_fused_gate_up_has_one_scale(orc):
    rng = np.random.default_rng(5)
    wg = bf16(0.02 * rng.standard_normal((32, 16)))
    wu = bf16(0.5 * rng.standard_normal((32, 16)))
    wd = bf16(0.02 * rng.standard_normal((16, 32)))
    q_gu, s_gu, q_d, s_d = orc.quantize_layer_weights(wg, wu, wd)
    amax = max(np.abs(orc.bf16_decode(wg)).max(), np.abs(orc.bf16_decode(wu)).max())
    assert s_gu == float(np.float32(amax) / np.float32(448.0))
    assert q_gu.shape == (64, 16)
    assert s_d == float(np.float32(np.abs(orc.bf16_decode(wd)).max()) / np.float32(448.0))


# --------------------------------------------------------------------- A6 --

def _tiny_layer(orc, rng, d=64, ff=128):
    wg = bf16(0.02 * rng.standard_normal((ff, d)))
    wu = bf16(0.02 * rng.standard_normal((ff, d)))
    wd = bf16(0.02 * rng.standard_normal((d, ff)))
    wn = bf16(1 + 0.1 * rng.standard_normal(d))
    q_gu, s_gu, q_d, s_d = orc.quantize_layer_weights(wg, wu, wd)
    return wn, q_gu, s_gu, q_d, s_d


def test_calibration_constant_magnitude_gives_known_amax(orc):
    """Rows of +-c give |y_i| = |w_i| c / sqrt(c^2 + eps), so s_x is known."""
    rng = np.random.default_rng(6)
    d = 64
    wn, q_gu, s_gu, q_d, s_d = _tiny_layer(orc, rng, d=d)
    c = 2.0
    signs = np.where(rng.integers(0, 2, (8, d)) == 1, 1.0, -1.0)
    r = bf16(c * signs)
    s_x, s_h, _ = orc.calibrate_layer([r], None, wn, q_gu, q_d, s_gu, s_d, orc.ACT_GEGLU_TANH)
    wf = np.abs(orc.bf16_decode(wn)).astype(np.float64)
    amax = wf.max() * c / math.sqrt(c * c + 1e-6)
    assert abs(s_x - amax / 448.0) <= 4 * float(ulp32(amax / 448.0))
    assert s_h > 0


def test_calibration_invariant_to_row_permutation_and_batch_split(orc):
    rng = np.random.default_rng(7)
    wn, q_gu, s_gu, q_d, s_d = _tiny_layer(orc, rng)
    r = bf16(rng.standard_normal((12, 64)))
    h = bf16(rng.standard_normal((12, 64)))
    sx, sh, out = orc.calibrate_layer([r], [h], wn, q_gu, q_d, s_gu, s_d, orc.ACT_SWIGLU)
    perm = rng.permutation(12)
    sx2, sh2, out2 = orc.calibrate_layer([r[perm]], [h[perm]], wn, q_gu, q_d, s_gu, s_d, orc.ACT_SWIGLU)
    assert (sx, sh) == (sx2, sh2)
    assert np.array_equal(out[0][perm], out2[0])
    # two batches of 6 rows: scales are the max over both halves
    sx3, sh3, _ = orc.calibrate_layer([r[:6], r[6:]], [h[:6], h[6:]], wn, q_gu, q_d, s_gu, s_d, orc.ACT_SWIGLU)
    assert (sx3, sh3) == (sx, sh)


def test_calibrated_scales_bound_the_layer_inputs(orc):
    """After calibration no activation quantised with the calibrated scales
    saturates on the calibration data: max |y| / s_x == 448 exactly at amax."""
    rng = np.random.default_rng(8)
    wn, q_gu, s_gu, q_d, s_d = _tiny_layer(orc, rng)
    r = bf16(rng.standard_normal((10, 64)))
    sx, sh, _ = orc.calibrate_layer([r], None, wn, q_gu, q_d, s_gu, s_d, orc.ACT_GEGLU_TANH)
    tr = orc.ffn_layer(r, None, wn, q_gu, q_d, sx, sh, s_gu, s_d, orc.ACT_GEGLU_TANH, trace=True)
    assert (tr.q_x & 0x7F).max() == 0x7E
    assert (tr.q_h & 0x7F).max() == 0x7E
