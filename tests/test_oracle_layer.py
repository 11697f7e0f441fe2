"""Pins of the oracle's whole layer and stack.

1. An independent composition of the layer from library routines (torch's
   BF16 and float8_e4m3fn casts, F.rms_norm, fp64 matmul, F.gelu / F.silu)
   must agree with the oracle under the same contract the GPU path is held to.
2. The FP8 path keeps cosine > 0.999 against the unquantised fp32 forward
   (agentlenshq FlashRT summary, "Main ideas").  Reading: the claim is applied
   per sublayer (teacher-forced: both paths see the same input).  It holds as
   stated where the residual stream carries most of the output energy (tiny,
   VLA action expert, VLA prefix).  On the decode and long-prefill shapes,
   N(0, 0.02) weights at d=5120, ff=17408 make the sublayer's update carry
   about 85% of the output energy, and the update's own cosine is set by E4M3
   resolution: RNE onto a 3-bit mantissa has a relative RMS error of about
   2.9% per rounding, and the update passes four roundings (x, W_gu, a,
   W_down), so 1 - cos(update) is about 4 * 0.029^2 / 2 = 1.7e-3.  Every
   workload is therefore held to 1 - cos(out) <= 3e-3 * E + 1e-4, where E is
   the update's share of the output energy.  Over a free-running stack the
   error adds up layer by layer: 1 - cos <= 2 * sum_l (1 - cos_l).
3. A degenerate case where every quantisation step up to the gate/up GEMM is
   lossless reproduces the unquantised math exactly.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synthetic


def t_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)


def to_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def cos(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / np.sqrt((a @ a) * (b @ b)))


def code_ordinal(c):
    """Position of an E4M3 code on the monotone value line (+-0 equal)."""
    c = np.asarray(c, np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def torch_layer(r, h, w, s_x, s_h, act):
    """The layer built from library routines, with its own weight quantisation."""
    d = r.shape[1]
    ff = w["w_gate"].shape[0]
    rb = t_bf16(r)
    rp = (rb.float() + t_bf16(h).float()).to(torch.bfloat16) if h is not None else rb
    y = F.rms_norm(rp.float(), (d,), weight=t_bf16(w["w_norm"]).float(), eps=1e-6)
    f8 = torch.float8_e4m3fn

    def wq(t):
        tf = t.float()
        s = (tf.abs().max() / 448.0).item()
        return (tf * (1.0 / torch.tensor(s, dtype=torch.float32))).to(f8), s

    wgu = torch.cat([t_bf16(w["w_gate"]), t_bf16(w["w_up"])], dim=0)
    q_gu, s_gu = wq(wgu)
    q_d, s_d = wq(t_bf16(w["w_down"]))
    inv_sx = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(s_x, dtype=torch.float32)
    inv_sh = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(s_h, dtype=torch.float32)
    q_x = (y * inv_sx).to(f8)
    acc = (q_x.double() @ q_gu.double().T).float()
    a_gu = torch.tensor(s_x, dtype=torch.float32) * torch.tensor(s_gu, dtype=torch.float32)
    gu = (acc * a_gu).to(torch.bfloat16).float()
    g, u = gu[:, :ff], gu[:, ff:]
    ag = F.gelu(g, approximate="tanh") if act == 0 else F.silu(g)
    a = ag * u
    q_h = (a * inv_sh).to(f8)
    acc_d = (q_h.double() @ q_d.double().T).float()
    a_d = torch.tensor(s_h, dtype=torch.float32) * torch.tensor(s_d, dtype=torch.float32)
    out = (rp.float() + acc_d * a_d).to(torch.bfloat16)
    return dict(out=to_bits(out), q_x=q_x.view(torch.uint8).numpy(), q_h=q_h.view(torch.uint8).numpy(),
                s_gu=s_gu, s_d=s_d)


def assert_contract(orc, ours_out, ref_out, ours_codes=(), ref_codes=()):
    for a, b in zip(ours_codes, ref_codes):
        same = np.mean(a == b)
        assert same >= 0.999, same
        assert np.abs(code_ordinal(a) - code_ordinal(b)).max() <= 1
    o = orc.bf16_decode(ours_out).astype(np.float64)
    r = orc.bf16_decode(ref_out).astype(np.float64)
    assert cos(o, r) >= 0.9999
    assert np.abs(o - r).max() <= 2e-2 * np.sqrt((r ** 2).mean())


@pytest.mark.parametrize("name", ["tiny", "vla_action_expert"])
def test_layer_agrees_with_library_composition(orc, name):
    wl = synthetic.WORKLOADS[name]
    M = min(wl.M, 16)
    w = {k: synthetic.bf16_bits(v) for k, v in synthetic.layer_weights(wl, 0).items()}
    r, h = [synthetic.bf16_bits(x) for x in synthetic.inputs(wl, M=M)]
    (ql,) = orc.quantize_stack([w])
    s_x, s_h = orc.calibrate_stack([ql], [r], [h], wl.act_id)
    tr = orc.ffn_layer(r, h, ql.w_norm, ql.q_gu, ql.q_down, s_x[0], s_h[0], ql.s_gu, ql.s_d, wl.act_id,
                       trace=True)
    ref = torch_layer(r, h, w, s_x[0], s_h[0], wl.act_id)
    assert ref["s_gu"] == pytest.approx(ql.s_gu, rel=1e-6) and ref["s_d"] == pytest.approx(ql.s_d, rel=1e-6)
    assert_contract(orc, tr.out, ref["out"], (tr.q_x, tr.q_h), (ref["q_x"], ref["q_h"]))


def test_lossless_degenerate_layer_matches_plain_math(orc):
    """eps = 0, rows of +-1, norm weight and all weights on scaled E4M3 grids
    with power-of-two scales: q_x, the weight codes and the gate/up GEMM are
    exact, so g and u equal the fp64 product of the unquantised operands up
    to the BF16 rounding of the GEMM output."""
    rng = np.random.default_rng(9)
    M, d, ff = 6, 64, 96

    def grid(shape, scale):
        c = rng.integers(0x20, 0x60, shape).astype(np.uint8) | (rng.integers(0, 2, shape).astype(np.uint8) << 7)
        c.flat[0] = 0x7E
        return orc.e4m3_decode(c).astype(np.float64) * scale

    wn = grid((d,), 2.0 ** -7)          # amax 3.5 -> s_x = 2^-7 on rows of +-1
    wg = grid((ff, d), 2.0 ** -12)
    wu = grid((ff, d), 2.0 ** -12)
    wd = grid((d, ff), 2.0 ** -12)
    to = lambda x: to_bits(torch.from_numpy(x).float().to(torch.bfloat16))
    r = to(np.where(rng.integers(0, 2, (M, d)) == 1, 1.0, -1.0))
    w = dict(w_norm=to(wn), w_gate=to(wg), w_up=to(wu), w_down=to(wd))
    (ql,) = orc.quantize_stack([w])
    s_x = 3.5 / 448.0
    tr = orc.ffn_layer(r, None, ql.w_norm, ql.q_gu, ql.q_down, s_x, 1.0, ql.s_gu, ql.s_d,
                       orc.ACT_GEGLU_TANH, eps=0.0, trace=True)
    y = orc.bf16_decode(r).astype(np.float64) * wn
    assert np.array_equal(orc.e4m3_decode(tr.q_x).astype(np.float64) * s_x, y)
    g = y @ wg.T
    u = y @ wu.T
    gu = orc.bf16_decode(tr.gu).astype(np.float64)
    expect = orc.bf16_decode(to_bits(torch.from_numpy(np.concatenate([g, u], 1)).float().to(torch.bfloat16)))
    assert np.array_equal(gu, expect.astype(np.float64))


def _teacher_forced_cosines(orc, wl, M, layers):
    r, h = [synthetic.bf16_bits(x) for x in synthetic.inputs(wl, M=M)]
    cb = synthetic.calibration_batches(wl, M=M)
    ws = [{k: synthetic.bf16_bits(v) for k, v in synthetic.layer_weights(wl, l).items()} for l in range(layers)]
    q = orc.quantize_stack(ws)
    s_x, s_h = orc.calibrate_stack(q, [synthetic.bf16_bits(a) for a, _ in cb],
                                   [synthetic.bf16_bits(b) for _, b in cb], wl.act_id)
    cur = orc.bf16_decode(r)
    hf = orc.bf16_decode(h)
    cur_q = r
    tf, energy, free = [], [], []
    for l in range(layers):
        hl = h if l == 0 else None
        rin = cur.astype(np.float64) + (hf.astype(np.float64) if l == 0 else 0.0)
        ref = orc.ref_layer_f32(cur, hf if l == 0 else None, ws[l]["w_norm"], ws[l]["w_gate"], ws[l]["w_up"],
                                ws[l]["w_down"], wl.act_id)
        out = orc.ffn_layer(orc.bf16_encode(cur), hl, q[l].w_norm, q[l].q_gu, q[l].q_down, s_x[l], s_h[l],
                            q[l].s_gu, q[l].s_d, wl.act_id)
        tf.append(cos(orc.bf16_decode(out), ref))
        ref64 = ref.astype(np.float64)
        energy.append(float(((ref64 - rin) ** 2).sum() / (ref64 ** 2).sum()))
        cur_q = orc.ffn_layer(cur_q, hl, q[l].w_norm, q[l].q_gu, q[l].q_down, s_x[l], s_h[l],
                              q[l].s_gu, q[l].s_d, wl.act_id)
        free.append(cos(orc.bf16_decode(cur_q), ref))
        cur = ref
    return tf, energy, free


@pytest.mark.parametrize("name,M,layers", [("tiny", 8, 1), ("vla_action_expert", 50, 18),
                                           ("vla_prefix", 4, 1), ("llm_decode", 1, 1),
                                           ("long_prefill", 4, 1)])
def test_fp8_path_cosine_against_fp32_forward(orc, name, M, layers):
    wl = synthetic.WORKLOADS[name]
    tf, energy, free = _teacher_forced_cosines(orc, wl, M, layers)
    if name in ("tiny", "vla_action_expert", "vla_prefix"):
        assert min(tf) > 0.999, tf
    for c, e in zip(tf, energy):
        assert 1.0 - c <= 3e-3 * e + 1e-4, (c, e)
    assert free[-1] >= 1.0 - 2.0 * sum(1.0 - c for c in tf), (tf, free)


def test_stack_hidden_enters_layer_zero_only(orc):
    wl = synthetic.WORKLOADS["tiny"].with_(L=2, d=64, ff=128, M=4)
    ws = [{k: synthetic.bf16_bits(v) for k, v in synthetic.layer_weights(wl, l).items()} for l in range(2)]
    q = orc.quantize_stack(ws)
    r, h = [synthetic.bf16_bits(x) for x in synthetic.inputs(wl)]
    s = [0.01, 0.01]
    out = orc.stack_forward(q, r, h, s, s, wl.act_id)
    l0 = orc.ffn_layer(r, h, q[0].w_norm, q[0].q_gu, q[0].q_down, 0.01, 0.01, q[0].s_gu, q[0].s_d, wl.act_id)
    l1 = orc.ffn_layer(l0, None, q[1].w_norm, q[1].q_gu, q[1].q_down, 0.01, 0.01, q[1].s_gu, q[1].s_d, wl.act_id)
    assert np.array_equal(out, l1)
