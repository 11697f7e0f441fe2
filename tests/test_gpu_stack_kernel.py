"""The persistent stack kernel (the whole FP8 FFN stack of at most 64 tokens
in one launch) against the oracle (itsolotime FlashRT article, 4.1 and 7.2;
"FlashRT docs/architecture.md", 7).

Every layer is checked teacher-forced under the full parity contract: the
kernel's debug instantiation takes the oracle's own layer input (from layer
1 on) and the oracle's E4M3 codes of step A1 as the GEMMs' input, so that no
allowed one-step q_x flip spreads; per layer the kernel's own q_x codes
(code contract), g/u, q_h and the output.  The product instantiation (no dumps)
computes what the tested one computes, bit for bit; its free-running output
is held to the oracle and to the per-layer kernels' result."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import Case, bits, check_bf16, check_codes, cosine, u8

pytestmark = pytest.mark.gpu

WL = synthetic.WORKLOADS
SHAPES = [
    WL["tiny"],                                                            # one CTA per cluster (d = 256)
    WL["vla_action_expert"],                                               # 32 clusters of 4, 18 layers
    WL["tiny"].with_(name="s2_m17", M=17, d=512, ff=1024, L=3, n_calib=1, seed=31),
    WL["tiny"].with_(name="s2_m64_swiglu", M=64, d=512, ff=384, L=2, act=synthetic.SWIGLU, n_calib=1, seed=32),
    WL["tiny"].with_(name="s8_m33", M=33, d=2048, ff=512, L=2, n_calib=1, seed=33),
    WL["llm_decode"].with_(name="m1_d1024", M=1, d=1024, ff=2048, L=4, seed=34),
]


@pytest.fixture(scope="module", params=SHAPES, ids=lambda w: w.name)
def case(request):
    # the stack kernel is opt-in, read at plan creation
    mp = pytest.MonkeyPatch()
    mp.setenv("FRT_FFN_STACK", "1")
    try:
        c = Case(request.param)
    finally:
        mp.undo()
    if not c.plan.uses_stack_kernel(c.wl.M):
        c.close()
        pytest.skip("the stack kernel does not take this shape on this GPU")
    yield c
    c.close()


def test_every_layer_teacher_forced(case):
    """Each layer from the oracle's own input (its residual r' from layer 1
    on, and its E4M3 codes as the GEMMs' input): the kernel's q_x under the
    code contract, g/u, q_h and the layer's output under the full contract,
    on every row."""
    wl, dev = case.wl, case.dev
    tr = case.oracle_forward(trace=True)
    qx_in = torch.from_numpy(np.stack([t.q_x for t in tr])).to(dev)
    res_in = synthetic.from_bf16_bits(np.stack([t.r_prime for t in tr]), dev)
    o = case.plan.debug_stack(case.r.to(dev), case.h.to(dev), q_x_in=qx_in, res_in=res_in)
    torch.cuda.synchronize()
    case.plan.device_status()
    qx, gu, qh, lo = u8(o["q_x"]), bits(o["gu"]), u8(o["q_h"]), bits(o["layer_out"])
    assert np.array_equal(bits(o["out"]), lo[-1])
    for l, t in enumerate(tr):
        what = "%s layer %d" % (wl.name, l)
        check_codes(qx[l], t.q_x, what + " q_x")
        check_bf16(gu[l], t.gu, what + " gate/up")
        check_codes(qh[l], t.q_h, what + " q_h")
        c, e = check_bf16(lo[l], t.out, what + " output")
        print("%s: out cos %.7f err %.4f" % (what, c, e))


def test_product_kernel_equals_the_tested_one_and_graph_replay(case):
    wl, dev = case.wl, case.dev
    r, h = case.r.to(dev), case.h.to(dev)
    eager = case.plan.forward(r, h)
    dbg = case.plan.debug_stack(r, h)
    torch.cuda.synchronize()
    case.plan.device_status()
    assert torch.equal(eager, dbg["out"])
    again = case.plan.forward(r, h)          # counters re-armed by the previous launch
    torch.cuda.synchronize()
    assert torch.equal(again, eager)
    out = torch.empty_like(r)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        case.plan.graph_capture(r, h, out, s)
        case.plan.graph_replay(wl.M, s)
        case.plan.graph_replay(wl.M, s)
    s.synchronize()
    case.plan.device_status()
    assert torch.equal(out, eager)
    shares = case.plan.graph_profile(wl.M, n_replays=3, stream=s)
    assert len(shares) == 1 and shares[0] > 0


def test_free_running_against_oracle_and_per_layer_kernels(case, monkeypatch):
    from realtime_transformer_gb300.ffn import FFNPlan
    wl, dev = case.wl, case.dev
    r, h = case.r.to(dev), case.h.to(dev)
    got = oracle.bf16_decode(bits(case.plan.forward(r, h))).astype(np.float64)
    torch.cuda.synchronize()
    ref = oracle.bf16_decode(case.oracle_forward()).astype(np.float64)
    monkeypatch.delenv("FRT_FFN_STACK", raising=False)
    p2 = FFNPlan(wl.d, wl.ff, wl.act, wl.M, wl.L)
    try:
        assert not p2.uses_stack_kernel(wl.M)
        for l, w in enumerate(case.weights):
            p2.load_weights(l, *(w[k].to(dev) for k in ("w_norm", "w_gate", "w_up", "w_down")), digest=False)
        p2.set_scales(case.s_x, case.s_h)
        per_layer = oracle.bf16_decode(bits(p2.forward(r, h))).astype(np.float64)
        torch.cuda.synchronize()
    finally:
        p2.close()
    c_orc, c_pl = cosine(got, ref), cosine(got, per_layer)
    print("%s free-running: cos(stack kernel, oracle) %.7f, cos(stack kernel, per-layer kernels) %.7f, "
          "cos(per-layer kernels, oracle) %.7f" % (wl.name, c_orc, c_pl, cosine(per_layer, ref)))
    assert c_orc >= 0.999
    assert c_pl >= 0.999
