"""Stack parity, graph capture/replay and calibration against the oracle
("FlashRT docs/architecture.md", 6 Calibration Framework and 7 CUDA Graph
Capture; itsolotime FlashRT article, 4.1-4.2).

Stacks with the RMSNorm weight folded into the gate/up weights (the Pi0
layout, itsolotime article 5.2) run the same tests against the oracle's
folded quantisation.

Per-layer parity through the whole stack is teacher-forced: GPU layer l runs
on the oracle's own layer-l input (oracle values may feed the GPU, never the
reverse).  Free-running, the two pipelines round different elements across
E4M3 boundaries and drift apart like two FP8 runs with different summation
orders; there the stack is held to the cosine claim against the unquantised
forward and to cosine >= 0.999 against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import Case, bits, cosine
from test_gpu_layer import check_weight_codes, compare_layer

pytestmark = pytest.mark.gpu

WL = synthetic.WORKLOADS


# (workload, norm weight folded into the gate/up weights -- the Pi0 layout)
@pytest.fixture(scope="module", params=[(WL["tiny"], False), (WL["vla_action_expert"], False),
                                        (WL["tiny"].with_(name="deep_small", L=6, M=20, d=384, ff=1152,
                                                          act=synthetic.SWIGLU, outliers=True, n_calib=2), False),
                                        (WL["vla_action_expert"].with_(name="vla_ae", L=4), True),
                                        (WL["vla_prefix"].with_(name="tiled", M=200, d=512, ff=1024, L=2), True)],
                ids=lambda p: p[0].name + ("_folded" if p[1] else ""))
def case(request):
    c = Case(request.param[0], fold_norm=request.param[1])
    yield c
    c.close()


def test_weight_scales_match_oracle_exactly(case):
    sc = case.plan.scales()
    for l, ql in enumerate(case.q):
        assert sc["s_gu"][l] == np.float32(ql.s_gu)
        assert sc["s_down"][l] == np.float32(ql.s_d)


def test_weight_codes_match_oracle_byte_for_byte(case):
    """Plain and folded quantisers alike (the folded stacks compare against
    the oracle's folded quantisation)."""
    check_weight_codes(case.plan, case.q, case.wl.name + (" folded" if case.fold else ""))


def test_every_layer_teacher_forced(case):
    wl = case.wl
    traces = case.oracle_forward(trace=True)
    cur = bits(case.r)
    for l in range(wl.L):
        st = compare_layer(case.plan, l, cur, bits(case.h) if l == 0 else None, case.q[l], case.s_x[l],
                           case.s_h[l], wl.act_id, case.dev, "%s layer %d" % (wl.name, l))
        print("%s layer %2d: q_x %.6f q_h %.6f out cos %.7f err %.4f (own path cos %.7f)" % (
            wl.name, l, st["q_x"], st["q_h"], st["cos"], st["err"], st["cos_own"]))
        cur = traces[l].out


def test_free_running_stack(case):
    dev = case.dev
    out = case.plan.forward(case.r.to(dev), case.h.to(dev))
    torch.cuda.synchronize()
    case.plan.device_status()
    got = oracle.bf16_decode(bits(out)).astype(np.float64)
    ref_q = oracle.bf16_decode(case.oracle_forward()).astype(np.float64)
    ws = [{k: bits(v) for k, v in w.items()} for w in case.weights]
    ref32 = oracle.ref_stack_f32(ws, bits(case.r), bits(case.h), case.wl.act_id).astype(np.float64)
    c_q, c_gpu, c_orc = cosine(got, ref_q), cosine(got, ref32), cosine(ref_q, ref32)
    print("%s free-running: cos(gpu, oracle) %.7f, cos(gpu, fp32) %.7f, cos(oracle, fp32) %.7f, "
          "max|gpu-oracle|/rms %.4f" % (case.wl.name, c_q, c_gpu, c_orc,
                                        np.abs(got - ref_q).max() / np.sqrt((ref_q ** 2).mean())))
    assert c_q >= 0.999
    assert c_gpu >= c_orc - 1e-3


def test_graph_replay_equals_eager(case):
    dev = case.dev
    r = case.r.to(dev)
    h = case.h.to(dev)
    eager = case.plan.forward(r, h)
    torch.cuda.synchronize()           # the plan's scratch is shared across streams
    out = torch.empty_like(r)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        case.plan.graph_capture(r, h, out, s)
        out.zero_()
        case.plan.graph_replay(case.wl.M, s)
        case.plan.graph_replay(case.wl.M, s)
    s.synchronize()
    case.plan.device_status()
    assert torch.equal(out, eager)
    again = case.plan.forward(r, h)
    torch.cuda.synchronize()
    assert torch.equal(again, eager)


def test_gpu_calibration_matches_oracle(case):
    """Full-stack GPU calibration.  Layer 0: the mean square of each row is
    summed in a different order on each side, which moves it by at most
    d * 2^-24 relative, so s_x moves by at most half that (plus rounding).
    Later layers drift with the free-running pipelines (reported, held to 5%)."""
    dev = case.dev
    saved = case.plan.scales()
    case.plan.calibrate([a.to(dev) for a, _ in case.calib], [b.to(dev) for _, b in case.calib])
    sc = case.plan.scales()
    case.plan.set_scales(saved["s_x"], saved["s_h"])
    sx, sh = np.array(sc["s_x"]), np.array(sc["s_h"])
    rx, rh = np.array(case.s_x), np.array(case.s_h)
    rel = np.maximum(np.abs(sx - rx) / rx, np.abs(sh - rh) / rh)
    print("%s calibration rel diff per layer: %s" % (case.wl.name, np.array2string(rel, precision=2)))
    assert abs(sx[0] - rx[0]) <= (0.5 * case.wl.d + 4) * 2.0 ** -24 * rx[0]
    assert abs(sh[0] - rh[0]) <= 1e-3 * rh[0]
    assert np.all(rel <= 5e-2)


def test_calibration_teacher_forced_per_layer(case):
    """Each layer's calibration on the oracle's own calibration state for that
    layer (a one-layer plan per layer): scales within 1e-3 of the oracle's."""
    from realtime_transformer_gb300.ffn import FFNPlan
    wl = case.wl
    dev = case.dev
    rb = [bits(a) for a, _ in case.calib]
    hb = [bits(b) for _, b in case.calib]
    for l in range(wl.L):
        ql = case.q[l]
        plan = FFNPlan(wl.d, wl.ff, wl.act, wl.M, 1)
        w = case.weights[l]
        plan.load_weights(0, *(w[k].to(dev) for k in ("w_norm", "w_gate", "w_up", "w_down")), fold_norm=case.fold)
        plan.calibrate([synthetic.from_bf16_bits(x, dev) for x in rb],
                       [synthetic.from_bf16_bits(x, dev) for x in hb] if l == 0 else None)
        sc = plan.scales()
        plan.close()
        sx, sh, rb = oracle.calibrate_layer(rb, hb if l == 0 else None, ql.w_norm, ql.q_gu, ql.q_down, ql.s_gu,
                                            ql.s_d, wl.act_id)
        assert abs(sc["s_x"][0] - sx) <= 1e-3 * sx, (l, sc["s_x"][0], sx)
        assert abs(sc["s_h"][0] - sh) <= 1e-3 * sh, (l, sc["s_h"][0], sh)


@pytest.mark.parametrize("tactic", range(4))
def test_every_autotune_schedule_gives_the_eager_bits(case, monkeypatch, tactic):
    """Each schedule the autotuned capture may keep (defaults, global split-K
    exchange, single-CTA tiles, no programmatic dependent launch) replays to
    exactly the eager forward's output."""
    from realtime_transformer_gb300 import _native as N
    dev = case.dev
    r = case.r.to(dev)
    h = case.h.to(dev)
    eager = case.plan.forward(r, h)
    torch.cuda.synchronize()
    out = torch.empty_like(r)
    s = torch.cuda.Stream()
    monkeypatch.setenv("FRT_FFN_AUTOTUNE_ONLY", str(tactic))
    with torch.cuda.stream(s):
        t_us, k = case.plan.graph_autotune(r, h, out, s, n_tries=1, n_replays=2)
        out.zero_()
        case.plan.graph_replay(case.wl.M, s)
    s.synchronize()
    case.plan.device_status()
    assert k == tactic and N.GRAPH_TACTICS[k]
    assert torch.equal(out, eager)
