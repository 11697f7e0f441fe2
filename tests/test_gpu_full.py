"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (full M, all layers, one captured graph per stack).

The oracle cannot run every row of the large shapes, but rows are
independent once the scales are fixed, so each sampled layer is checked
teacher-forced on sampled rows: the GPU runs the layer on the full M-row
input (the same kernels and tiling as the timed forward), the oracle runs the
same layer on a handful of those rows (spread over the token tiles, the last
row included), and the rows are compared under the parity contract.  Scales
come from the oracle calibrating each sampled layer on a seeded batch
("FlashRT docs/architecture.md", 6; itsolotime FlashRT article, 7.2)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import bits, check_bf16, check_codes, check_rows, u8

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
    layers = sorted(set([0, wl.L // 2, wl.L - 1]))
    plan = FFNPlan(wl.d, wl.ff, wl.act, wl.M, wl.L)
    host_w = {}
    for l in range(wl.L):
        w = synthetic.layer_weights(wl, l, device=dev)
        plan.load_weights(l, w["w_norm"], w["w_gate"], w["w_up"], w["w_down"])
        if l in layers:
            host_w[l] = {k: bits(v) for k, v in w.items()}
        del w
    # oracle weights and per-layer calibration of the sampled layers
    q = {l: oracle.quantize_stack([host_w[l]])[0] for l in layers}
    sc = plan.scales()
    for l in layers:
        assert sc["s_gu"][l] == np.float32(q[l].s_gu) and sc["s_down"][l] == np.float32(q[l].s_d)
    s_x, s_h = {}, {}
    crow = min(wl.M, 64)
    for l in layers:
        if l == 0:
            cb = synthetic.calibration_batches(wl, device="cpu", M=crow)
            rb, hb = [bits(a) for a, _ in cb], [bits(b) for _, b in cb]
        else:
            r_c, _ = layer_input(wl.with_(seed=wl.seed + 31), l, crow, "cpu")
            rb, hb = [bits(r_c)], None
        s_x[l], s_h[l], _ = oracle.calibrate_layer(rb, hb, q[l].w_norm, q[l].q_gu, q[l].q_down, q[l].s_gu, q[l].s_d,
                                                   wl.act_id)
    sx_all = [s_x.get(l, s_x[0]) for l in range(wl.L)]
    sh_all = [s_h.get(l, s_h[0]) for l in range(wl.L)]
    plan.set_scales(sx_all, sh_all)

    # the timed configuration: the whole stack as one graph at full M
    r0, h0 = synthetic.inputs(wl, device=dev)
    out = torch.empty_like(r0)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        plan.graph_capture(r0, h0, out, s)
        plan.graph_replay(wl.M, s)
    s.synchronize()
    plan.device_status()
    assert torch.isfinite(out.float()).all()

    rows = sample_rows(wl.M)
    rows_t = torch.from_numpy(rows).to(dev)
    for l in layers:
        r, h = layer_input(wl, l, wl.M, dev)
        tr = plan.trace_layer(l, r, h)
        torch.cuda.synchronize()
        plan.device_status()
        tr = {k: v.index_select(0, rows_t) for k, v in tr.items()}
        rb = bits(r.index_select(0, rows_t))
        hb = bits(h.index_select(0, rows_t)) if h is not None else None
        ref = oracle.ffn_layer(rb, hb, q[l].w_norm, q[l].q_gu, q[l].q_down, s_x[l], s_h[l], q[l].s_gu, q[l].s_d,
                               wl.act_id, trace=True)
        what = "%s layer %d" % (name, l)
        assert np.array_equal(bits(tr["r_prime"]), ref.r_prime), what
        qx = u8(tr["q_x"])
        check_codes(qx, ref.q_x, what + " q_x")
        same = np.all(qx == ref.q_x, axis=1)
        if same.any():
            check_bf16(bits(tr["gu"])[same], ref.gu[same], what + " gate/up")
            check_codes(u8(tr["q_h"])[same], ref.q_h[same], what + " q_h")
        c, e = check_rows(bits(tr["out"]), ref.out, same, what + " output")
        print("%s: rows %s q_x rows equal %d/%d, out cos %.7f err %.4f" % (what, list(rows), int(same.sum()),
                                                                          len(rows), c, e))
    plan.close()
