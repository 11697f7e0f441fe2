"""Pins of the oracle's number formats against definitions and library casts.

E4M3 (OCP FP8 "fn" variant) and BF16 are the formats of the FP8 path
(agentlenshq FlashRT summary, "Main ideas": FP8 weights and activations;
itsolotime FlashRT article, 7.1 "FP8 path": E4M3).
"""
import numpy as np
import pytest
import torch


def closed_form_e4m3(c: int) -> float:
    """Value of an E4M3 code written from the format definition."""
    s = -1.0 if c & 0x80 else 1.0
    e = (c >> 3) & 0xF
    m = c & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_decode_matches_definition_all_codes(orc):
    for c in range(256):
        v = orc.lib().orc_e4m3_decode(c)
        ref = closed_form_e4m3(c)
        if np.isnan(ref):
            assert np.isnan(v), hex(c)
        else:
            assert v == ref, (hex(c), v, ref)


def test_closed_form_landmarks(orc):
    dec = orc.lib().orc_e4m3_decode
    assert dec(0x7E) == 448.0
    assert dec(0xFE) == -448.0
    assert dec(0x08) == 2.0 ** -6
    assert dec(0x01) == 2.0 ** -9
    assert dec(0x07) == 7 * 2.0 ** -9
    assert dec(0x38) == 1.0
    assert dec(0x3F) == 1.875
    assert dec(0x77) == 240.0
    assert np.isnan(dec(0x7F)) and np.isnan(dec(0xFF))


def test_round_trip_all_codes(orc):
    L = orc.lib()
    for c in range(256):
        if c & 0x7F == 0x7F:
            assert L.orc_e4m3_encode(L.orc_e4m3_decode(c)) == 0x7F
            continue
        assert L.orc_e4m3_encode(L.orc_e4m3_decode(c)) == c, hex(c)


def _next_up(x):
    return float(np.nextafter(np.float32(x), np.float32(np.inf)))


def _next_down(x):
    return float(np.nextafter(np.float32(x), np.float32(-np.inf)))


def test_midpoints_round_to_even_and_neighbours_to_nearest(orc):
    L = orc.lib()
    for sign in (0x00, 0x80):
        for c in range(0, 0x7E):
            lo, hi = sign | c, sign | (c + 1)
            vlo, vhi = closed_form_e4m3(lo), closed_form_e4m3(hi)
            mid = np.float32((vlo + vhi) / 2.0)
            assert float(mid) == (vlo + vhi) / 2.0  # midpoints are exact in fp32
            even = lo if (c & 1) == 0 else hi
            assert L.orc_e4m3_encode(float(mid)) == even, (hex(lo), float(mid))
            toward_lo = _next_down(mid) if sign == 0 else _next_up(mid)
            toward_hi = _next_up(mid) if sign == 0 else _next_down(mid)
            assert L.orc_e4m3_encode(toward_lo) == lo
            assert L.orc_e4m3_encode(toward_hi) == hi


def test_saturation_nan_and_signed_zero(orc):
    L = orc.lib()
    for v in (448.0, 448.5, 464.0, 480.0, 1e6, 3.0e38, float("inf")):
        assert L.orc_e4m3_encode(v) == 0x7E
        assert L.orc_e4m3_encode(-v) == 0xFE
    assert L.orc_e4m3_encode(float("nan")) == 0x7F
    assert L.orc_e4m3_encode(0.0) == 0x00
    assert L.orc_e4m3_encode(-0.0) == 0x80
    # half of the smallest subnormal is a tie between 0 and 2^-9: even -> 0
    assert L.orc_e4m3_encode(2.0 ** -10) == 0x00
    assert L.orc_e4m3_encode(_next_up(2.0 ** -10)) == 0x01
    assert L.orc_e4m3_encode(1e-30) == 0x00


def test_agrees_with_torch_float8_cast_over_all_binades(orc):
    """Every fp32 magnitude in [2^-12, 448] (all mantissas), both signs on a
    subset: oracle encode == torch float8_e4m3fn cast (RNE).  Saturation is
    not compared; torch does not saturate."""
    lo = np.float32(2.0 ** -12).view(np.uint32)
    hi = np.float32(448.0).view(np.uint32)
    step = 1 << 24
    for start in range(int(lo), int(hi) + 1, step):
        bits = np.arange(start, min(start + step, int(hi) + 1), dtype=np.uint32)
        x = bits.view(np.float32)
        ours = orc.e4m3_encode(x)
        theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        bad = np.nonzero(ours != theirs)[0]
        assert bad.size == 0, (x[bad[:5]], ours[bad[:5]], theirs[bad[:5]])
    rng = np.random.default_rng(7)
    x = -(rng.uniform(0, 448, 1 << 20).astype(np.float32))
    ours = orc.e4m3_encode(x)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_encode_is_monotone(orc):
    rng = np.random.default_rng(3)
    x = np.sort(rng.uniform(-500, 500, 200000).astype(np.float32))
    v = orc.e4m3_decode(orc.e4m3_encode(x))
    assert np.all(np.diff(v) >= 0)


def test_bf16_encode_matches_torch(orc):
    """All 2^16 upper halves x a set of lower halves that covers every
    rounding case (ties, just-below/above ties, zero, all ones, random)."""
    lows = np.array([0x0000, 0x0001, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xBFFF, 0xFFFF, 0x4000, 0xC000],
                    dtype=np.uint32)
    rng = np.random.default_rng(11)
    lows = np.concatenate([lows, rng.integers(0, 1 << 16, 22, dtype=np.uint32)])
    highs = np.arange(1 << 16, dtype=np.uint32)
    bits = (highs[:, None] << 16 | lows[None, :]).reshape(-1)
    x = bits.view(np.float32)
    ours = orc.bf16_encode(x)
    theirs = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], theirs[~nan])
    assert np.all(np.isnan(orc.bf16_decode(ours[nan])))


def test_bf16_decode_is_exact_widening(orc):
    b = np.arange(1 << 16, dtype=np.uint16)
    ours = orc.bf16_decode(b)
    theirs = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    same = (ours == theirs) | (np.isnan(ours) & np.isnan(theirs))
    assert same.all()


def test_scale_rule(orc):
    assert orc.scale_from_amax(0.0) == 1.0
    assert orc.scale_from_amax(448.0) == 1.0
    assert orc.scale_from_amax(3.5) == 2.0 ** -7
    v = orc.scale_from_amax(1.2345)
    assert v == float(np.float32(1.2345) / np.float32(448.0))
