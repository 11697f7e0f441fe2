"""Boundary behaviour of the C ABI on the GPU: status codes, stale graphs,
empty and oversized inputs, misaligned pointers ("FlashRT
docs/architecture.md", 7: pointer-only forward, graphs with baked alpha)."""
import os

import pytest
import torch

import synthetic
from realtime_transformer_gb300 import _native as N
from realtime_transformer_gb300.ffn import FFNPlan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def loaded():
    wl = synthetic.WORKLOADS["tiny"]
    dev = torch.device("cuda")
    plan = FFNPlan(wl.d, wl.ff, wl.act, 16, 1)
    w = synthetic.layer_weights(wl, 0, device=dev)
    plan.load_weights(0, w["w_norm"], w["w_gate"], w["w_up"], w["w_down"])
    r, h = synthetic.inputs(wl, device=dev)
    yield plan, r, h
    plan.close()


def status_of(fn, *a):
    with pytest.raises(N.FrtError) as ei:
        fn(*a)
    return ei.value.name


def test_forward_before_scales_is_not_ready(loaded):
    plan, r, h = loaded
    assert status_of(plan.forward, r, h) == "FRT_ERR_NOT_READY"


def test_missing_weights_is_not_ready():
    p = FFNPlan(256, 1024, "geglu_tanh", 8, 2)
    p.set_scales([1.0, 1.0], [1.0, 1.0])
    r = torch.zeros((8, 256), dtype=torch.bfloat16, device="cuda")
    assert status_of(p.forward, r) == "FRT_ERR_NOT_READY"
    p.close()


def test_shape_and_argument_errors(loaded):
    plan, r, h = loaded
    plan.set_scales([0.01], [0.01])
    big = torch.zeros((17, 256), dtype=torch.bfloat16, device="cuda")
    assert status_of(plan.forward, big) == "FRT_ERR_SHAPE"
    raw = torch.zeros(8 * 256 + 8, dtype=torch.bfloat16, device="cuda")
    mis = raw[1:1 + 8 * 256].view(8, 256)
    assert status_of(N.frt_ffn_forward, plan.handle, mis.data_ptr(), None, r.data_ptr(), 8, 0) == \
        "FRT_ERR_INVALID_ARG"
    assert status_of(N.frt_ffn_set_scales, plan.handle, [0.0], [1.0]) == "FRT_ERR_INVALID_ARG"
    assert status_of(N.frt_ffn_load_weights, plan.handle, 3, r.data_ptr(), r.data_ptr(), r.data_ptr(),
                     r.data_ptr(), 0) == "FRT_ERR_INVALID_ARG"


def test_empty_input_is_a_no_op(loaded):
    plan, r, h = loaded
    plan.set_scales([0.01], [0.01])
    N.frt_ffn_forward(plan.handle, r.data_ptr(), None, r.data_ptr(), 0, 0)
    plan.device_status()


def test_graph_replay_errors_and_staleness(loaded):
    plan, r, h = loaded
    plan.set_scales([0.02], [0.003])
    assert status_of(plan.graph_replay, 5) == "FRT_ERR_CAPTURE"
    out = torch.empty_like(r)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.graph_capture(r, h, out, s)
        plan.graph_replay(8, s)
    s.synchronize()
    ref = plan.forward(r, h)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    plan.set_scales([0.02], [0.003])
    assert status_of(plan.graph_replay, 8, s) == "FRT_ERR_STALE_GRAPH"
    assert status_of(plan.graph_capture, r, h, out, 0) == "FRT_ERR_CAPTURE"


def test_smaller_M_than_M_max_and_repeat_calls(loaded):
    plan, r, h = loaded
    plan.set_scales([0.02], [0.003])
    full = plan.forward(r, h)
    part = plan.forward(r[:3].contiguous(), h[:3].contiguous())
    again = plan.forward(r, h)
    torch.cuda.synchronize()
    assert torch.equal(full[:3], part)
    assert torch.equal(full, again)


def test_graph_autotune_keeps_a_working_graph(loaded):
    """Tactic-stable capture: several captures, the fastest kept; its replay
    computes the forward, and it goes stale like a plain capture."""
    plan, r, h = loaded
    plan.set_scales([0.02], [0.003])
    out = torch.empty_like(r)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        best, tactic = plan.graph_autotune(r, h, out, s, n_tries=4, n_replays=5)
        out.zero_()
        plan.graph_replay(r.shape[0], s)
    s.synchronize()
    assert 0.0 < best < 1e5 and 0 <= tactic < len(N.GRAPH_TACTICS)
    ref = plan.forward(r, h)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert status_of(plan.graph_autotune, r, h, out, s, 0, 5) == "FRT_ERR_INVALID_ARG"
    plan.set_scales([0.02], [0.003])
    assert status_of(plan.graph_replay, r.shape[0], s) == "FRT_ERR_STALE_GRAPH"


def test_calibration_cache_hit_and_miss(tmp_path):
    """First plan: cache miss, calibrates and saves; a second plan with the
    same weights: hit, the same scales and the same output; other weights:
    another key, a miss."""
    wl = synthetic.WORKLOADS["tiny"]
    dev = torch.device("cuda")
    r, h = synthetic.inputs(wl, device=dev)
    cb = synthetic.calibration_batches(wl, device=dev)
    res, hid = [x for x, _ in cb], [y for _, y in cb]

    def make(seed_layer):
        p = FFNPlan(wl.d, wl.ff, wl.act, wl.M, 1)
        w = synthetic.layer_weights(wl, seed_layer, device=dev)
        p.load_weights(0, w["w_norm"], w["w_gate"], w["w_up"], w["w_down"])
        return p

    a = make(0)
    assert a.calibrate_cached(res, hid, directory=str(tmp_path), extra={"source": "test"}) is False
    assert os.listdir(tmp_path) == [a.cache_key(wl.M) + ".json"]
    b = make(0)
    assert b.cache_key(wl.M) == a.cache_key(wl.M)
    assert b.calibrate_cached(res, hid, directory=str(tmp_path)) is True
    assert a.scales() == b.scales()
    ya, yb = a.forward(r, h), b.forward(r, h)
    torch.cuda.synchronize()
    assert torch.equal(ya, yb)
    c = make(1)
    assert c.cache_key(wl.M) != a.cache_key(wl.M)
    assert c.calibrate_cached(res, hid, directory=str(tmp_path)) is False
    assert len(os.listdir(tmp_path)) == 2
    for p in (a, b, c):
        p.close()


def test_graph_profile_splits_the_replay_without_changing_the_graph():
    """The profiling replays stamp every launch: the per-launch shares are
    positive and sum to at most the replay's span, and the graph held for M
    still computes the same output afterwards."""
    wl = synthetic.WORKLOADS["vla_action_expert"].with_(L=3)
    dev = torch.device("cuda")
    plan = FFNPlan(wl.d, wl.ff, wl.act, wl.M, wl.L)
    for l in range(wl.L):
        w = synthetic.layer_weights(wl, l, device=dev)
        plan.load_weights(l, w["w_norm"], w["w_gate"], w["w_up"], w["w_down"], digest=False)
    plan.set_scales([0.02] * wl.L, [0.01] * wl.L)
    r, h = synthetic.inputs(wl, device=dev)
    out = torch.empty_like(r)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        plan.graph_capture(r, h, out, s)
        plan.graph_replay(wl.M, s)
    s.synchronize()
    first = out.clone()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(10):
            plan.graph_replay(wl.M, s)
        e1.record(s)
    s.synchronize()
    replay_us = e0.elapsed_time(e1) * 1000.0 / 10
    shares = plan.graph_profile(wl.M, n_replays=10, stream=s)
    assert len(shares) == 3 * wl.L
    assert all(x > 0 for x in shares), shares
    assert sum(shares) <= 1.5 * replay_us, (sum(shares), replay_us)
    out.zero_()
    with torch.cuda.stream(s):
        plan.graph_replay(wl.M, s)
    s.synchronize()
    assert torch.equal(out, first)
    with pytest.raises(N.FrtError) as ei:
        plan.graph_profile(7, stream=s)
    assert ei.value.name == "FRT_ERR_CAPTURE"
    plan.close()
