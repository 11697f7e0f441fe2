"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (full M, all layers, one captured graph per stack).

The oracle cannot run every row of the large shapes, but rows are
independent once the scales are fixed, so the checks run on sampled rows
(spread over the token tiles, the first and last row included) while the GPU
runs every row with the same kernels and tiling as the timed forward:

  * free-running: the whole graph-replayed stack on the workload's input
    against the oracle's quantised stack and the unquantised fp32 forward on
    the sampled rows: as close to fp32 as the oracle itself (within 1e-3),
    and within twice the oracle's own distance from fp32 of the oracle
    (cosine >= 0.999 where that is tighter; agentlenshq summary, "Main
    ideas", read per sublayer, and its extension to free-running stacks);
  * teacher-forced: three layers (first, middle, last) on a seeded input,
    every sampled row under the full contract (tests/parity.check_layer);
  * step A0: the stored E4M3 weight codes of those layers byte for byte.

The layers are generated, loaded and run through the oracle one at a time, so
host memory holds one layer's master weights at once.  Scales are the
oracle's progressive calibration ("FlashRT docs/architecture.md", 6) on a
seeded calibration batch of at most 64 rows."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import bits, check_layer, cosine, u8
from test_gpu_layer import interleave_gu

pytestmark = pytest.mark.gpu

WORKLOADS = ["tiny", "vla_action_expert", "vla_prefix", "llm_decode", "long_prefill"]


def sample_rows(M, n=8):
    rows = sorted(set([0, M - 1] + [int(x) for x in np.linspace(0, M - 1, n)]))
    return np.array(rows, dtype=np.int64)


def layer_input(wl, layer, M, dev):
    if layer == 0:
        return synthetic.inputs(wl, device=dev)
    w2 = wl.with_(seed=wl.seed + 7919 * (layer + 1))
    r, _ = synthetic.inputs(w2, device=dev, M=M)
    return r, None


@pytest.mark.parametrize("name", WORKLOADS)
def test_full_size_workload(name):
    from realtime_transformer_gb300.ffn import FFNPlan
    wl = synthetic.WORKLOADS[name]
    dev = torch.device("cuda")
    checked = sorted(set([0, wl.L // 2, wl.L - 1]))
    rows = sample_rows(wl.M)
    rows_t = torch.from_numpy(rows).to(dev)
    r0, h0 = synthetic.inputs(wl, device=dev)
    r_rows, h_rows = bits(r0.index_select(0, rows_t)), bits(h0.index_select(0, rows_t))
    crow = min(wl.M, 64)
    cb = synthetic.calibration_batches(wl, device="cpu", M=crow)
    cal_r, cal_h = [bits(a) for a, _ in cb], [bits(b) for _, b in cb]

    plan = FFNPlan(wl.d, wl.ff, wl.act, wl.M, wl.L)
    s_x, s_h, q_kept = [], [], {}
    state, state32 = r_rows, oracle.bf16_decode(r_rows)
    for l in range(wl.L):
        w = synthetic.layer_weights(wl, l, device=dev)
        plan.load_weights(l, w["w_norm"], w["w_gate"], w["w_up"], w["w_down"], digest=False)
        hw = {k: bits(v) for k, v in w.items()}
        del w
        ql = oracle.quantize_stack([hw])[0]
        sx, sh, cal_r = oracle.calibrate_layer(cal_r, cal_h if l == 0 else None, ql.w_norm, ql.q_gu, ql.q_down,
                                               ql.s_gu, ql.s_d, wl.act_id)
        s_x.append(sx)
        s_h.append(sh)
        state = oracle.ffn_layer(state, h_rows if l == 0 else None, ql.w_norm, ql.q_gu, ql.q_down, sx, sh,
                                 ql.s_gu, ql.s_d, wl.act_id)
        state32 = oracle.ref_layer_f32(state32, oracle.bf16_decode(h_rows) if l == 0 else None, hw["w_norm"],
                                       hw["w_gate"], hw["w_up"], hw["w_down"], wl.act_id)
        if l in checked:
            q_kept[l] = ql
        del hw
    sc = plan.scales()
    for l, ql in q_kept.items():
        assert sc["s_gu"][l] == np.float32(ql.s_gu) and sc["s_down"][l] == np.float32(ql.s_d), l
    plan.set_scales(s_x, s_h)

    # free-running: the timed configuration, the whole stack as one graph at full M
    out = torch.empty_like(r0)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        plan.graph_capture(r0, h0, out, s)
        plan.graph_replay(wl.M, s)
    s.synchronize()
    plan.device_status()
    assert torch.isfinite(out.float()).all()
    got = oracle.bf16_decode(bits(out.index_select(0, rows_t))).astype(np.float64)
    ref_q = oracle.bf16_decode(state).astype(np.float64)
    ref32 = state32.astype(np.float64)
    c_q, c_gpu32, c_orc32 = cosine(got, ref_q), cosine(got, ref32), cosine(ref_q, ref32)
    print("%s free-running, %d layers, rows %s: cos(gpu, oracle) %.7f, cos(gpu, fp32) %.7f, "
          "cos(oracle, fp32) %.7f" % (name, wl.L, list(rows), c_q, c_gpu32, c_orc32))
    # Two FP8 pipelines that round different elements drift apart layer by
    # layer; each is as far from the fp32 forward as its own quantisation
    # takes it.  So: the GPU at least as close to fp32 as the oracle (within
    # 1e-3), and GPU and oracle no further apart than twice the oracle's own
    # distance from fp32 (0.999 where that is the tighter bound).
    assert c_gpu32 >= c_orc32 - 1e-3, (c_gpu32, c_orc32)
    assert c_q >= min(0.999, 1.0 - 2.0 * (1.0 - c_orc32)), (c_q, c_orc32)

    # teacher-forced sampled layers, every sampled row under the full contract
    for l in checked:
        ql = q_kept[l]
        w_gu, w_down = plan.weights(l)
        torch.cuda.synchronize()
        assert np.array_equal(u8(w_gu), interleave_gu(ql.q_gu, wl.ff)), "%s layer %d gate/up codes" % (name, l)
        assert np.array_equal(u8(w_down), ql.q_down), "%s layer %d down codes" % (name, l)
        del w_gu, w_down
        r, h = layer_input(wl, l, wl.M, dev)
        rb = bits(r.index_select(0, rows_t))
        hb = bits(h.index_select(0, rows_t)) if h is not None else None
        ref = oracle.ffn_layer(rb, hb, ql.w_norm, ql.q_gu, ql.q_down, s_x[l], s_h[l], ql.s_gu, ql.s_d, wl.act_id,
                               trace=True)
        st = check_layer(plan, l, r, h, ref, "%s layer %d" % (name, l), rows=rows)
        print("%s layer %d: q_x agree %.6f, q_h agree %.6f, out cos %.7f err %.4f (own path cos %.7f)" % (
            name, l, st["q_x"], st["q_h"], st["cos"], st["err"], st["cos_own"]))
    plan.close()
