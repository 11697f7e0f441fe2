"""Calibration cache ("FlashRT docs/architecture.md", 6 Calibration
Framework): key "{hash}_Se{M}", JSON records that keep fp32 scales exactly,
stale records (other shape, M or weight scales) not used.  Host logic only."""
import json
import os

import numpy as np
import pytest

from realtime_transformer_gb300 import calibration as C

SHAPE = {"d": 1024, "ff": 4096, "act": 0, "n_layers": 3}


def f32_list(xs):
    return [float(np.float32(x)) for x in xs]


SCALES = {
    "s_x": f32_list([0.1, 1e-40, 448.0 / 3.0]),  # 1e-40 is an fp32 subnormal
    "s_h": f32_list([np.nextafter(np.float32(1.0), np.float32(2.0)), 2.0 ** -20, 7.0]),
    "s_gu": f32_list([3.1e-4, 2.9e-4, 3.3e-4]),
    "s_down": f32_list([3.0e-4, 3.2e-4, 2.8e-4]),
}
WS = {"s_gu": SCALES["s_gu"], "s_down": SCALES["s_down"]}


def test_key_format_and_hash_inputs():
    h = C.checkpoint_hash(SHAPE, ["a", "b", "c"])
    assert len(h) == 16 and int(h, 16) >= 0
    assert C.cache_key(h, 50) == h + "_Se50"
    assert C.checkpoint_hash(SHAPE, ["a", "b", "x"]) != h
    assert C.checkpoint_hash(SHAPE, ["a", "b", None]) != h
    assert C.checkpoint_hash(dict(SHAPE, ff=2048), ["a", "b", "c"]) != h
    # concatenation of digests is not ambiguous
    assert C.checkpoint_hash(SHAPE, ["ab", "c", "d"]) != C.checkpoint_hash(SHAPE, ["a", "bc", "d"])
    with pytest.raises(ValueError):
        C.cache_key(h, 0)


def test_record_round_trip_is_bit_exact(tmp_path):
    rec = C.make_record(SHAPE, 50, SCALES, extra={"note": "calibrated on 1 batch", "n": 4})
    path = C.save(str(tmp_path), "k_Se50", rec)
    assert os.path.basename(path) == "k_Se50.json"
    assert os.listdir(tmp_path) == ["k_Se50.json"]  # no temporary left behind
    got = C.load(str(tmp_path), "k_Se50", SHAPE, 50, WS)
    assert got is not None
    for k in ("s_x", "s_h"):
        a = np.array(got[k], dtype=np.float32).view(np.uint32)
        b = np.array(SCALES[k], dtype=np.float32).view(np.uint32)
        assert np.array_equal(a, b), k
    assert got["extra"] == {"note": "calibrated on 1 batch", "n": 4}


@pytest.mark.parametrize("change", ["missing", "corrupt", "format", "M", "ff", "n_layers", "s_gu_ulp", "s_x_zero",
                                    "s_h_nan", "s_x_short"])
def test_stale_or_damaged_records_are_not_used(tmp_path, change):
    d = str(tmp_path)
    C.save(d, "k_Se50", C.make_record(SHAPE, 50, SCALES))
    path = os.path.join(d, "k_Se50.json")
    rec = json.load(open(path))
    shape, M, ws = SHAPE, 50, WS
    if change == "missing":
        os.remove(path)
    elif change == "corrupt":
        open(path, "w").write("{not json")
    elif change == "format":
        rec["format"] = "something/else"
    elif change == "M":
        M = 49
    elif change == "ff":
        shape = dict(SHAPE, ff=2048)
    elif change == "n_layers":
        shape = dict(SHAPE, n_layers=2)
    elif change == "s_gu_ulp":
        g = list(WS["s_gu"])
        g[1] = float(np.nextafter(np.float32(g[1]), np.float32(1.0)))
        ws = {"s_gu": g, "s_down": WS["s_down"]}
    elif change == "s_x_zero":
        rec["s_x"][0] = 0.0
    elif change == "s_h_nan":
        rec["s_h"][2] = float("nan")
    elif change == "s_x_short":
        rec["s_x"] = rec["s_x"][:2]
    if change not in ("missing", "corrupt"):
        json.dump(rec, open(path, "w"))
    assert C.load(d, "k_Se50", shape, M, ws) is None


def test_make_record_checks_layer_counts():
    bad = dict(SCALES, s_h=SCALES["s_h"][:2])
    with pytest.raises(ValueError):
        C.make_record(SHAPE, 50, bad)


def test_default_dir_follows_the_environment(monkeypatch, tmp_path):
    monkeypatch.setenv("FRT_FFN_CALIB_DIR", str(tmp_path))
    assert C.default_dir() == str(tmp_path)
    monkeypatch.delenv("FRT_FFN_CALIB_DIR")
    assert C.default_dir().endswith(os.path.join(".cache", "frt_ffn", "calibration"))


def test_weight_digest_covers_every_element():
    """The cache key's weight digest reads every element: two weight sets
    that differ in one element anywhere (here one that a strided sample of
    4096 elements would skip) get different digests, as do other tags and
    other tensor boundaries."""
    import torch
    g = torch.Generator().manual_seed(3)
    w = [(torch.randn(n, generator=g) * 0.02).to(torch.bfloat16) for n in (1024, 4096 * 1024, 1024 * 4096)]
    base = C.weights_digest(b"plain", w)
    assert base == C.weights_digest(b"plain", [t.clone() for t in w])
    stride = w[1].numel() // 4096
    for t_i, idx in ((1, 1), (1, stride + 1), (2, w[2].numel() - 1), (0, 17)):
        v = [t.clone() for t in w]
        flat = v[t_i].view(-1)
        flat[idx] = flat[idx] + torch.tensor(1.0, dtype=torch.bfloat16)
        assert C.weights_digest(b"plain", v) != base, (t_i, idx)
    assert C.weights_digest(b"fold", w) != base
    # moving an element across a tensor boundary changes the digest
    a = torch.cat([w[0], w[1][:1]])
    assert C.weights_digest(b"plain", [a, w[1][1:], w[2]]) != base
    # chunked reading gives the same digest as one read
    assert C.weights_digest(b"plain", w, chunk_elems=1000) == base
