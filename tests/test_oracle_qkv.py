"""Pins of the oracle's attention-input sublayer: residual + RMSNorm + E4M3
quantise -> FP8 fused-QKV GEMM -> QKV split + RoPE (agentlenshq FlashRT
summary, "What it is"; itsolotime FlashRT article, 5.2 FusedQKV; "FlashRT
docs/architecture.md", 8 Kernel Library: "qkv split + RoPE").

RoPE is pinned against complex multiplication (numpy complex128), closed
forms of the frequencies, one-hot inputs and the relative-position property;
the sublayer against a composition from torch routines (float8 casts,
rms_norm, fp64 matmul, complex rotation)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synthetic


def test_inverse_frequencies_closed_form(orc):
    f = orc.rope_inv_freq(8, 10000.0)
    assert f.dtype == np.float32
    assert list(f) == [np.float32(1.0), np.float32(0.1), np.float32(0.01), np.float32(0.001)]
    g = orc.rope_inv_freq(128, 1.0e6)
    assert g[0] == 1.0 and g[64 - 1] == np.float32(1.0e6 ** (-126.0 / 128.0))
    assert np.all(np.diff(g) < 0)


def test_rope_at_position_zero_is_identity(orc):
    x = np.random.default_rng(1).standard_normal((4, 3, 64)).astype(np.float32)
    assert np.array_equal(orc.rope(x, np.zeros(4, np.int64), orc.rope_inv_freq(64, 10000.0)), x)


def test_rope_is_complex_rotation_of_half_pairs(orc):
    """(x_i + i x_{i+hd/2}) * exp(i pos theta_i), angle rounded to fp32 first."""
    rng = np.random.default_rng(2)
    hd = 32
    x = rng.standard_normal((5, 2, hd)).astype(np.float32)
    pos = np.array([0, 1, 7, 300, 4097])
    f = orc.rope_inv_freq(hd, 10000.0)
    got = orc.rope(x, pos, f).astype(np.float64)
    ang = (pos.astype(np.float32)[:, None] * f[None, :]).astype(np.float64)
    z = (x[..., :hd // 2].astype(np.float64) + 1j * x[..., hd // 2:].astype(np.float64)) * np.exp(1j * ang)[:, None, :]
    ref = np.concatenate([z.real, z.imag], axis=-1)
    bound = 4 * 2.0 ** -24 * (np.abs(x[..., :hd // 2]) + np.abs(x[..., hd // 2:])).astype(np.float64)
    assert np.all(np.abs(got - ref) <= np.concatenate([bound, bound], -1))


def test_rope_one_hot_pairs_element_i_with_i_plus_half(orc):
    hd = 16
    f = orc.rope_inv_freq(hd, 10000.0)
    for j in (0, 3, 7):
        x = np.zeros((1, 1, hd), np.float32)
        x[0, 0, j] = 1.0
        out = orc.rope(x, [5], f)[0, 0]
        a = np.float64(np.float32(np.float32(5.0) * f[j]))
        expect = np.zeros(hd, np.float32)
        expect[j] = np.float32(np.cos(a))
        expect[j + hd // 2] = np.float32(np.sin(a))
        assert np.array_equal(out, expect), j


def test_rope_scores_depend_on_relative_position(orc):
    rng = np.random.default_rng(3)
    hd = 64
    f = orc.rope_inv_freq(hd, 10000.0)
    q = rng.standard_normal((1, 1, hd)).astype(np.float32)
    k = rng.standard_normal((1, 1, hd)).astype(np.float32)
    s = lambda m, n: float(orc.rope(q, [m], f).astype(np.float64).ravel() @ orc.rope(k, [n], f).astype(np.float64).ravel())
    assert s(9, 4) == pytest.approx(s(14, 9), rel=1e-5, abs=1e-5)
    assert s(9, 4) == pytest.approx(s(5, 0), rel=1e-5, abs=1e-5)
    assert s(9, 4) != pytest.approx(s(4, 9), rel=1e-3)


def t_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)


def to_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("nq,nkv,hd,base", [(4, 1, 64, 10000.0), (4, 2, 32, 1.0e6)])
def test_qkv_layer_agrees_with_library_composition(orc, nq, nkv, hd, base):
    """Given the oracle's q_x codes (the norm and quantiser are pinned
    elsewhere), torch's float8 decode, an fp64 matmul, BF16 casts and a
    complex rotation reproduce the split, the head order and the RoPE."""
    wl = synthetic.WORKLOADS["tiny"]
    M, d = 8, wl.d
    g = torch.Generator().manual_seed(5)
    wq = (torch.randn(nq * hd, d, generator=g) * 0.02).to(torch.bfloat16)
    wk = (torch.randn(nkv * hd, d, generator=g) * 0.02).to(torch.bfloat16)
    wv = (torch.randn(nkv * hd, d, generator=g) * 0.02).to(torch.bfloat16)
    wn = (1 + 0.1 * torch.randn(d, generator=g)).to(torch.bfloat16)
    r, h = [synthetic.bf16_bits(x) for x in synthetic.inputs(wl, M=M)]
    codes, s_qkv = orc.quantize_qkv_weights(to_bits(wq), to_bits(wk), to_bits(wv))
    s_x = orc.calibrate_qkv_layer([r], [h], to_bits(wn))
    pos = np.arange(M) * 37 + 3
    f = orc.rope_inv_freq(hd, base)
    tr = orc.qkv_layer(r, h, to_bits(wn), codes, s_x, s_qkv, nq, nkv, hd, pos, f)
    # torch side
    dec = lambda c: torch.from_numpy(np.ascontiguousarray(c, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64)
    acc = dec(tr.q_x) @ dec(codes).T
    qkv = (acc * float(np.float32(np.float32(s_x) * np.float32(s_qkv)))).to(torch.float32).to(torch.bfloat16)
    assert np.abs(to_bits(qkv).astype(np.int32) - tr.qkv.astype(np.int32)).max() <= 1  # fp32 vs fp64 sums
    x = qkv.to(torch.float64).reshape(M, nq + 2 * nkv, hd)
    ang = torch.from_numpy((pos.astype(np.float32)[:, None] * f[None, :]).astype(np.float64))
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]
    def rope_t(t):
        z = torch.complex(t[..., :hd // 2], t[..., hd // 2:]) * rot
        return torch.cat([z.real, z.imag], -1).to(torch.bfloat16)
    q = rope_t(x[:, :nq]).transpose(0, 1)
    k = rope_t(x[:, nq:nq + nkv]).transpose(0, 1)
    v = x[:, nq + nkv:].to(torch.bfloat16).transpose(0, 1)
    for name, ours, ref in (("q", tr.q, q), ("k", tr.k, k), ("v", tr.v, v)):
        a = orc.bf16_decode(ours).astype(np.float64)
        b = orc.bf16_decode(to_bits(ref)).astype(np.float64)
        assert a.shape == b.shape, name
        c = float((a * b).sum() / np.sqrt((a * a).sum() * (b * b).sum()))
        assert c >= 0.9999, (name, c)
        assert np.abs(a - b).max() <= 2e-2 * np.sqrt((b * b).mean()), name


def test_qkv_calibration_constant_rows(orc):
    """Rows of constant magnitude normalise to +-w: s_x = max|w| / 448."""
    d = 256
    wn = orc.bf16_encode(np.linspace(0.5, 1.5, d).astype(np.float32))
    r = orc.bf16_encode(np.where(np.arange(4 * d).reshape(4, d) % 3, 2.0, -2.0).astype(np.float32))
    s = orc.calibrate_qkv_layer([r], None, wn, eps=0.0)
    assert np.float32(s) == np.float32(np.float32(orc.bf16_decode(wn).max()) / np.float32(448.0))


def test_qkv_fold_unit_and_power_of_two_norm_weights(orc):
    """Fold with w = 1 is the plain quantisation; with w = c (a power of two)
    the codes stay and the scale is multiplied by c exactly; the folded
    sublayer with s_x / c then equals the unfolded one with w = c bit for bit."""
    rng = np.random.default_rng(9)
    d, nq, nkv, hd = 256, 4, 1, 64
    wq, wk, wv = [orc.bf16_encode(rng.normal(0, 0.02, (n * hd, d)).astype(np.float32)) for n in (nq, nkv, nkv)]
    ones = np.full(d, orc.BF16_ONE, dtype=np.uint16)
    a = orc.quantize_qkv_weights_folded(wq, wk, wv, ones)
    b = orc.quantize_qkv_weights(wq, wk, wv)
    assert np.array_equal(a[0], b[0]) and a[1] == b[1]
    c = 0.5
    wc = orc.bf16_encode(np.full(d, c, np.float32))
    f = orc.quantize_qkv_weights_folded(wq, wk, wv, wc)
    assert np.array_equal(f[0], b[0]) and np.float32(f[1]) == np.float32(b[1]) * np.float32(c)
    r = orc.bf16_encode(rng.standard_normal((6, d)).astype(np.float32))
    pos = np.arange(6) * 5
    inv = orc.rope_inv_freq(hd, 1.0e4)
    s_x = 0.0113
    u = orc.qkv_layer(r, None, wc, b[0], s_x, b[1], nq, nkv, hd, pos, inv)
    g = orc.qkv_layer(r, None, ones, f[0], float(np.float32(s_x) / np.float32(c)), f[1], nq, nkv, hd, pos, inv)
    for k in ("q_x", "qkv", "q", "k", "v"):
        assert np.array_equal(getattr(u, k), getattr(g, k)), k
    # and a real norm weight changes the folded codes (columns scaled by w[k])
    wr = orc.bf16_encode((1 + 0.1 * rng.standard_normal(d)).astype(np.float32))
    assert not np.array_equal(orc.quantize_qkv_weights_folded(wq, wk, wv, wr)[0], b[0])
