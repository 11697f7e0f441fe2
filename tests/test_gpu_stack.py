"""Free-running stack parity, graph capture/replay and calibration against the
oracle ("FlashRT docs/architecture.md", 6 Calibration Framework and 7 CUDA
Graph Capture; itsolotime FlashRT article, 4.1-4.2)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import Case, bits, check_bf16

pytestmark = pytest.mark.gpu

WL = synthetic.WORKLOADS


@pytest.fixture(scope="module", params=[WL["tiny"], WL["vla_action_expert"],
                                        WL["tiny"].with_(name="deep_small", L=6, M=20, d=384, ff=1152,
                                                         act=synthetic.SWIGLU, outliers=True, n_calib=2)],
                ids=lambda w: w.name)
def case(request):
    c = Case(request.param)
    yield c
    c.close()


def test_eager_forward_matches_oracle_stack(case):
    dev = case.dev
    out = case.plan.forward(case.r.to(dev), case.h.to(dev))
    torch.cuda.synchronize()
    case.plan.device_status()
    check_bf16(bits(out), case.oracle_forward(), "stack output")


def test_graph_replay_equals_eager(case):
    dev = case.dev
    r = case.r.to(dev)
    h = case.h.to(dev)
    eager = case.plan.forward(r, h)
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


def test_gpu_calibration_matches_oracle(case):
    dev = case.dev
    saved = case.plan.scales()
    case.plan.calibrate([a.to(dev) for a, _ in case.calib], [b.to(dev) for _, b in case.calib])
    sc = case.plan.scales()
    case.plan.set_scales(saved["s_x"], saved["s_h"])
    sx = np.array(sc["s_x"], np.float64)
    sh = np.array(sc["s_h"], np.float64)
    rx = np.array(case.s_x, np.float64)
    rh = np.array(case.s_h, np.float64)
    assert np.all(np.abs(sx - rx) <= 1e-3 * rx), (sx, rx)
    assert np.all(np.abs(sh - rh) <= 1e-3 * rh), (sh, rh)
    # layer 0's input scale depends only on RMSNorm: within a few fp32 ulp
    assert abs(sx[0] - rx[0]) <= 4 * np.spacing(np.float32(rx[0]))
