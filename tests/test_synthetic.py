"""The seeded input recipe: shapes, determinism, outlier channels."""
import math

import numpy as np

import torch

import synthetic


def test_shapes_and_dtypes():
    wl = synthetic.WORKLOADS["tiny"]
    w = synthetic.layer_weights(wl, 0)
    assert w["w_norm"].shape == (256,) and w["w_gate"].shape == (1024, 256)
    assert w["w_up"].shape == (1024, 256) and w["w_down"].shape == (256, 1024)
    assert all(v.dtype == torch.bfloat16 for v in w.values())
    r, h = synthetic.inputs(wl)
    assert r.shape == (8, 256) and h.shape == (8, 256) and r.dtype == torch.bfloat16
    assert len(synthetic.calibration_batches(wl)) == 4


def test_deterministic_and_layers_independent():
    wl = synthetic.WORKLOADS["tiny"].with_(L=3)
    a = synthetic.layer_weights(wl, 1)
    b = synthetic.layer_weights(wl, 1)
    c = synthetic.layer_weights(wl, 2)
    assert torch.equal(a["w_gate"], b["w_gate"])
    assert not torch.equal(a["w_gate"], c["w_gate"])
    assert not torch.equal(a["w_gate"], a["w_up"])


def test_outlier_channels():
    for name, wl in synthetic.WORKLOADS.items():
        ch = synthetic.outlier_channels(wl)
        if not wl.outliers:
            assert ch == []
            continue
        assert len(ch) == math.ceil(0.001 * wl.d)
        r, h = synthetic.inputs(wl, M=64)
        rms = r.float().pow(2).mean(0).sqrt()
        mask = torch.zeros(wl.d, dtype=torch.bool)
        mask[ch] = True
        assert rms[mask].min() > 10 and rms[~mask].max() < 2
        (rc, hc), = synthetic.calibration_batches(wl, M=64)
        assert rc.float().pow(2).mean(0).sqrt()[mask].min() > 10


def test_distribution():
    wl = synthetic.WORKLOADS["vla_action_expert"]
    w = synthetic.layer_weights(wl, 0)
    assert abs(w["w_gate"].float().std().item() - 0.02) < 1e-3
    assert abs(w["w_norm"].float().mean().item() - 1.0) < 0.02
    assert abs(w["w_norm"].float().std().item() - 0.1) < 0.01


def test_attention_shapes_cover_every_workload():
    for name, wl in synthetic.WORKLOADS.items():
        nq, nkv, hd, base = synthetic.ATTENTION[name]
        assert nq % nkv == 0 and hd % 64 == 0 and base > 1
        assert ((nq + 2 * nkv) * hd) % 128 == 0
    wl = synthetic.WORKLOADS["tiny"]
    w = synthetic.qkv_weights(wl, 0)
    nq, nkv, hd, _ = synthetic.ATTENTION["tiny"]
    assert tuple(w["w_q"].shape) == (nq * hd, wl.d) and tuple(w["w_k"].shape) == (nkv * hd, wl.d)
    assert tuple(w["w_v"].shape) == (nkv * hd, wl.d) and tuple(w["w_norm"].shape) == (wl.d,)
    assert all(v.dtype == torch.bfloat16 for v in w.values())
    # seeded: the same layer twice is the same tensor, another layer is not
    assert torch.equal(synthetic.qkv_weights(wl, 0)["w_q"], w["w_q"])
    assert not torch.equal(synthetic.qkv_weights(wl, 1)["w_q"], w["w_q"])


def test_positions():
    assert list(synthetic.positions(synthetic.WORKLOADS["tiny"])) == list(range(8))
    p = synthetic.positions(synthetic.WORKLOADS["llm_decode"])
    assert p.dtype == np.int32 and list(p) == [synthetic.DECODE_CONTEXT]


def test_modulation_is_seeded_and_shaped():
    wl = synthetic.WORKLOADS["tiny"]
    a = synthetic.modulation(wl, 0, 8)
    b = synthetic.modulation(wl, 0, 8)
    c = synthetic.modulation(wl, 1, 8)
    assert a.shape == (8, 3 * wl.d) and a.dtype == torch.bfloat16
    assert torch.equal(a, b) and not torch.equal(a, c)
    gate = a[:, 2 * wl.d:].float()
    assert abs(gate.mean().item() - 1.0) < 0.05 and abs(a[:, :wl.d].float().mean().item()) < 0.05

