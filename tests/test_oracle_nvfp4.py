"""Pins of the oracle's NVFP4 variant (itsolotime FlashRT article, 7.2: split
gate/up NVFP4 GEMMs emitting packed FP4 and scales, a fused GeGLU FP4-to-FP4
requantise, NVFP4 down GEMM, AWQ pre-scaling).  Pinned against the E2M1 format
definition, brute-force nearest rounding, exact rational sums, exact
power-of-two invariances and the unquantised fp32 layer."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic
from parity import cosine

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def e2m1_from_bits(c: int) -> float:
    """The format: sign bit 3, two exponent bits (bias 1), one mantissa bit;
    exponent 0 is subnormal (m * 0.5)."""
    s, e, m = c >> 3, (c >> 1) & 3, c & 1
    v = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -v if s else v


def test_e2m1_decode_matches_the_format_definition():
    got = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    want = np.array([e2m1_from_bits(c) for c in range(16)], np.float32)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.arange(16) >= 8)


def test_e2m1_encode_is_nearest_with_ties_to_even_and_saturates():
    vals = np.array([e2m1_from_bits(c) for c in range(16)], np.float64)
    rng = np.random.default_rng(3)
    grid = np.arange(-8 * 64, 8 * 64 + 1) / 64.0  # every midpoint is on this grid
    x = np.concatenate([grid, rng.uniform(-7, 7, 4000), [1e-30, -1e-30, 1e30, -1e30]]).astype(np.float32)
    got = oracle.e2m1_encode(x)
    for xi, ci in zip(x.astype(np.float64), got):
        if abs(xi) >= 6:
            want = 7
        else:
            dist = np.abs(vals[:8] - abs(xi))
            best = np.nonzero(dist == dist.min())[0]
            want = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
        want |= 8 if np.signbit(xi) else 0
        assert ci == want, (xi, ci, want)


def test_round_trip_of_every_value():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(oracle.e2m1_encode(oracle.e2m1_decode(codes)), codes)


def _representable_blocks(rows, nblk, s, rng):
    """Blocks built from E2M1 values times an E4M3 block scale times s, each
    block holding a +-6 so that its scale is the one quantisation picks."""
    v = oracle.e2m1_decode(rng.integers(0, 16, (rows, nblk, 16)).astype(np.uint8))
    v[:, :, rng.integers(0, 16)] = 6.0 * rng.choice([-1, 1], (rows, nblk))
    sb = rng.integers(0x20, 0x68, (rows, nblk)).astype(np.uint8)  # normal E4M3 scales
    x = v * oracle.e4m3_decode(sb)[:, :, None] * np.float32(s)
    return x.reshape(rows, nblk * 16).astype(np.float32), v.reshape(rows, nblk * 16), sb


@pytest.mark.parametrize("s", [1.0, 2.0 ** -7, 2.0 ** 5])
def test_representable_blocks_quantise_exactly(s):
    rng = np.random.default_rng(11)
    x, v, sb = _representable_blocks(5, 6, s, rng)
    q, got_sb = oracle.nvfp4_quantize(x, s)
    assert np.array_equal(got_sb, sb)
    assert np.array_equal(oracle.e2m1_decode(q), v.astype(np.float32))
    assert np.array_equal(oracle.nvfp4_decode(q, got_sb, s), x)


def test_block_scale_is_the_e4m3_rounding_of_the_block_amax_over_six():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((16, 128)) * np.exp(rng.uniform(-3, 3, (16, 1)))).astype(np.float32)
    s = oracle.nvfp4_scale_from_amax(np.abs(x).max())
    assert s == np.float32(np.abs(x).max()) / np.float32(2688.0)
    q, sb = oracle.nvfp4_quantize(x, s)
    blk = np.abs(x.astype(np.float64)).reshape(16, 8, 16)
    ideal = blk.max(axis=2) / (6.0 * s)
    d = oracle.e4m3_decode(sb).astype(np.float64)
    # the nearest E4M3 value: within half of its spacing (2^(e-3) for normals)
    spacing = 2.0 ** (np.floor(np.log2(np.maximum(d, 2.0 ** -6))) - 3)
    assert np.all(np.abs(d - ideal) <= spacing / 2 * (1 + 1e-6))
    # the block's largest magnitude always lands on +-6
    mag = oracle.e2m1_decode(q).reshape(16, 8, 16)
    imax = blk.argmax(axis=2)
    top = np.take_along_axis(np.abs(mag), imax[:, :, None], axis=2)[:, :, 0]
    assert np.all(top == 6.0)
    # every element within half an E2M1 step of its scaled value
    scaled = x.reshape(16, 8, 16).astype(np.float64) / (d * s)[:, :, None]
    err = np.abs(scaled - mag)
    half = np.where(np.abs(scaled) < 2, 0.25, np.where(np.abs(scaled) < 4, 0.5, 1.0))
    assert np.all(err <= half * (1 + 1e-5) + 1e-6)


def test_zero_blocks_and_tensor():
    x = np.zeros((2, 32), np.float32)
    x[1, 16:] = np.linspace(-1, 1, 16)
    assert oracle.nvfp4_scale_from_amax(0.0) == 1.0
    q, sb = oracle.nvfp4_quantize(x, oracle.nvfp4_scale_from_amax(1.0))
    assert sb[0, 0] == 0 and sb[0, 1] == 0 and sb[1, 0] == 0 and sb[1, 1] != 0
    assert np.all(oracle.e2m1_decode(q[0]) == 0) and np.all(oracle.e2m1_decode(q[1, :16]) == 0)


def test_scaled_gemm_equals_the_exact_rational_sum():
    rng = np.random.default_rng(2)
    M, N, K = 3, 4, 48
    qa = rng.integers(0, 16, (M, K)).astype(np.uint8)
    qb = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sa = rng.integers(0x08, 0x70, (M, K // 16)).astype(np.uint8)
    sb = rng.integers(0x08, 0x70, (N, K // 16)).astype(np.uint8)
    got = oracle.nvfp4_gemm(qa, sa, qb, sb)
    dec = oracle.e4m3_decode(np.arange(0x70, dtype=np.uint8))
    fa = {c: Fraction(float(dec[c])) for c in range(0x08, 0x70)}
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(e2m1_from_bits(int(qa[m, k]))) * fa[sa[m, k // 16]]
                        * Fraction(e2m1_from_bits(int(qb[n, k]))) * fa[sb[n, k // 16]] for k in range(K))
            assert got[m, n] == np.float32(float(exact)), (m, n)


def _layer(name="tiny", awq=None):
    wl = synthetic.WORKLOADS[name]
    lw = {k: synthetic.bf16_bits(v) for k, v in synthetic.layer_weights(wl, 0).items()}
    r, h = synthetic.inputs(wl)
    cb = synthetic.calibration_batches(wl)
    rb = [synthetic.bf16_bits(a) for a, _ in cb]
    hb = [synthetic.bf16_bits(b) for _, b in cb]
    act = oracle.ACT_GEGLU_TANH if wl.act == "geglu_tanh" else oracle.ACT_SWIGLU
    return wl, lw, synthetic.bf16_bits(r), synthetic.bf16_bits(h), rb, hb, act


def test_uniform_power_of_two_awq_leaves_the_layer_bit_exact():
    """y / c with W c (c a power of two) moves only the tensor scales; dividing
    the weights or multiplying the activation instead would scale the output."""
    wl, lw, r, h, rb, hb, act = _layer()
    outs = []
    for awq in (None, np.full(wl.d, 4.0, np.float32)):
        L = oracle.quantize_layer_nvfp4(lw["w_norm"], lw["w_gate"], lw["w_up"], lw["w_down"], awq)
        sc, _ = oracle.calibrate_layer_nvfp4(rb, hb, L, act)
        outs.append((oracle.ffn_layer_nvfp4(r, h, L, sc, act, trace=True), sc, L))
    (a, sa, La), (b, sbb, Lb) = outs
    assert sbb.s_x == sa.s_x / 4 and Lb.gate.s == La.gate.s * 4 and Lb.up.s == La.up.s * 4
    for k in ("x", "g", "u", "h"):
        assert np.array_equal(getattr(a, k)[0], getattr(b, k)[0]), k
        assert np.array_equal(getattr(a, k)[1], getattr(b, k)[1]), k
    assert np.array_equal(a.out, b.out)


def test_awq_scales_closed_form():
    rng = np.random.default_rng(4)
    mag = np.exp(rng.uniform(-2, 2, 64))
    sign = rng.choice([-1.0, 1.0], (10, 64))
    c = oracle.awq_scales([sign[:6] * mag, sign[6:] * mag], alpha=0.5)
    assert np.allclose(c, np.sqrt(mag), rtol=1e-6)
    assert np.array_equal(oracle.awq_scales([np.zeros((2, 4))], alpha=1.0), np.full(4, 1e-5, np.float32))


def test_calibrated_scales_of_constant_magnitude_rows():
    d, ff = 64, 128
    r = oracle.bf16_encode(np.where(np.arange(d) % 3 == 0, -2.0, 2.0)[None, :].repeat(4, 0).astype(np.float32))
    ones = np.full(d, oracle.BF16_ONE, np.uint16)
    rng = np.random.default_rng(0)
    w = lambda a, b: oracle.bf16_encode((rng.standard_normal((a, b)) * 0.05).astype(np.float32))
    L = oracle.quantize_layer_nvfp4(ones, w(ff, d), w(ff, d), w(d, ff))
    sc, _ = oracle.calibrate_layer_nvfp4([r], None, L, oracle.ACT_SWIGLU)
    # y = +-1 / sqrt(1 + eps / 4) rounded to fp32: amax just below 1
    y = oracle.residual_rmsnorm(r, None, ones)[1]
    assert sc.s_x == np.float32(np.abs(y).max()) / np.float32(2688.0)
    assert abs(np.abs(y).max() - 1.0) < 1e-6


@pytest.mark.parametrize("name", ["tiny", "vla_action_expert"])
def test_nvfp4_layer_tracks_the_fp32_layer(name):
    wl, lw, r, h, rb, hb, act = _layer(name)
    L = oracle.quantize_layer_nvfp4(lw["w_norm"], lw["w_gate"], lw["w_up"], lw["w_down"])
    sc, outs = oracle.calibrate_layer_nvfp4(rb, hb, L, act)
    tr = oracle.ffn_layer_nvfp4(r, h, L, sc, act, trace=True)
    ref = oracle.ref_layer_f32(oracle.bf16_decode(r), oracle.bf16_decode(h), lw["w_norm"], lw["w_gate"],
                               lw["w_up"], lw["w_down"], act)
    rp = oracle.bf16_decode(tr.r_prime)
    assert np.array_equal(tr.r_prime, oracle.bf16_encode(oracle.bf16_decode(r) + oracle.bf16_decode(h)))
    # the FFN's own contribution (four FP4 roundings on its way) and the layer output
    assert cosine(oracle.bf16_decode(tr.out) - rp, ref - rp) > 0.93
    assert cosine(oracle.bf16_decode(tr.out), ref) > 0.998
    # calibration's own forward reproduces the fixed-scale forward
    assert np.array_equal(oracle.ffn_layer_nvfp4(rb[0], hb[0], L, sc, act), outs[0])
    # the per-tensor scales put each calibrated tensor's amax at 448 * 6
    assert sc.s_x == np.float32(max(np.abs(oracle._nvfp4_awq_divide(oracle.residual_rmsnorm(a, b, lw["w_norm"])[1],
                                                                   None)).max() for a, b in zip(rb, hb))) \
        / np.float32(2688.0)


def test_nvfp4_stack_tracks_the_fp32_stack():
    wl = synthetic.WORKLOADS["tiny"].with_(L=3)
    layers = [{k: synthetic.bf16_bits(v) for k, v in synthetic.layer_weights(wl, l).items()} for l in range(3)]
    r, h = synthetic.inputs(wl)
    cb = synthetic.calibration_batches(wl)
    rb = [synthetic.bf16_bits(a) for a, _ in cb]
    hb = [synthetic.bf16_bits(b) for _, b in cb]
    Ls = [oracle.quantize_layer_nvfp4(lw["w_norm"], lw["w_gate"], lw["w_up"], lw["w_down"]) for lw in layers]
    scs = oracle.calibrate_stack_nvfp4(Ls, rb, hb, oracle.ACT_GEGLU_TANH)
    out = oracle.stack_forward_nvfp4(Ls, scs, synthetic.bf16_bits(r), synthetic.bf16_bits(h), oracle.ACT_GEGLU_TANH)
    ref = oracle.ref_stack_f32(layers, synthetic.bf16_bits(r), synthetic.bf16_bits(h), oracle.ACT_GEGLU_TANH)
    assert cosine(oracle.bf16_decode(out), ref) > 0.999


def test_values_beyond_the_calibrated_range_saturate():
    """A block whose amax exceeds the tensor scale's range (an activation
    larger than any seen in calibration) gets the largest E4M3 scale, 448, and
    its largest elements the largest E2M1 code, 6."""
    s = 1.0 / 2688.0  # calibrated for amax 1
    x = np.zeros((1, 32), np.float32)
    x[0, :16] = np.linspace(-50.0, 50.0, 16)  # 50x the calibrated amax
    x[0, 16:] = np.linspace(-0.5, 0.5, 16)
    q, sb = oracle.nvfp4_quantize(x, s)
    assert oracle.e4m3_decode(sb)[0, 0] == 448.0
    assert oracle.e2m1_decode(q[0, [0, 15]]).tolist() == [-6.0, 6.0]
    # the in-range block is unaffected by its neighbour
    assert oracle.e4m3_decode(sb)[0, 1] < 448.0
    assert oracle.e2m1_decode(q[0, [16, 31]]).tolist() == [-6.0, 6.0]
