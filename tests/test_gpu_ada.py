"""AdaRMSNorm sublayers on the GPU against the oracle (itsolotime FlashRT
article, 5.2: Pi0.5 modulates through AdaRMSNorm Dense layers): the norm
y = (r' inv)(1 + scale) + shift and the gated residual r' + gate FFN(y), with
one modulation row for all tokens or one per token.  Same inputs and scales
on both sides; teacher-forced layers held to the parity contract."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import bits, check_layer, cosine

pytestmark = pytest.mark.gpu

WL = synthetic.WORKLOADS
SHAPES = [
    (WL["tiny"].with_(L=2), True),
    (WL["tiny"].with_(name="tiny_tok", L=2), False),
    (WL["vla_action_expert"].with_(L=2), True),
    (WL["tiny"].with_(name="tiled", M=200, d=512, ff=1024, L=2, n_calib=1, seed=21), False),
    (WL["tiny"].with_(name="m1_swiglu", M=1, d=1024, ff=2048, act=synthetic.SWIGLU, L=2, n_calib=1, seed=22), True),
]


def modulation(wl, rows, layer, dev):
    g = torch.Generator().manual_seed(1000 + 17 * layer + wl.seed)
    sc = 0.1 * torch.randn(rows, wl.d, generator=g)
    sh = 0.1 * torch.randn(rows, wl.d, generator=g)
    gt = 1.0 + 0.1 * torch.randn(rows, wl.d, generator=g)
    return torch.cat([sc, sh, gt], 1).to(torch.bfloat16).to(dev)


@pytest.fixture(scope="module", params=SHAPES, ids=lambda p: p[0].name + ("_shared" if p[1] else "_per_token"))
def case(request):
    from realtime_transformer_gb300.ffn import FFNPlan
    wl, shared = request.param
    dev = torch.device("cuda")
    ws = [synthetic.layer_weights(wl, l) for l in range(wl.L)]
    r, h = synthetic.inputs(wl)
    cb = synthetic.calibration_batches(wl)
    rows = 1 if shared else wl.M
    mods = [modulation(wl, rows, l, dev) for l in range(wl.L)]
    q = oracle.quantize_stack([{k: bits(v) for k, v in w.items()} for w in ws])
    hm = [bits(m) for m in mods]
    s_x, s_h = oracle.calibrate_stack_ada(q, hm, [bits(a) for a, _ in cb], [bits(b) for _, b in cb], wl.act_id)
    plan = FFNPlan(wl.d, wl.ff, wl.act, wl.M, wl.L)
    for l, w in enumerate(ws):
        plan.load_weights(l, *(w[k].to(dev) for k in ("w_norm", "w_gate", "w_up", "w_down")))
    plan.set_modulation(mods)
    plan.set_scales(s_x, s_h)
    c = dict(wl=wl, dev=dev, r=r, h=h, cb=cb, mods=mods, hm=hm, q=q, s_x=s_x, s_h=s_h, plan=plan)
    yield c
    plan.close()


def test_layers_teacher_forced(case):
    c = case
    wl, dev = c["wl"], c["dev"]
    cur, hid = bits(c["r"]), bits(c["h"])
    for l in range(wl.L):
        hl = hid if l == 0 else None
        ql = c["q"][l]
        ref = oracle.ffn_layer_ada(cur, hl, c["hm"][l], ql.q_gu, ql.q_down, c["s_x"][l], c["s_h"][l], ql.s_gu, ql.s_d,
                                   wl.act_id, trace=True)
        st = check_layer(c["plan"], l, synthetic.from_bf16_bits(cur, dev),
                         synthetic.from_bf16_bits(hl, dev) if hl is not None else None, ref,
                         "%s layer %d" % (wl.name, l))
        print("%s layer %d: q_x %.6f q_h %.6f out cos %.7f err %.4f (own path cos %.7f)" % (
            wl.name, l, st["q_x"], st["q_h"], st["cos"], st["err"], st["cos_own"]))
        cur = ref.out


def test_free_running_stack_and_graph(case):
    c = case
    wl, dev = c["wl"], c["dev"]
    r, h = c["r"].to(dev), c["h"].to(dev)
    eager = c["plan"].forward(r, h)
    torch.cuda.synchronize()
    ref = oracle.stack_forward_ada(c["q"], c["hm"], bits(c["r"]), bits(c["h"]), c["s_x"], c["s_h"], wl.act_id)
    got = oracle.bf16_decode(bits(eager)).astype(np.float64)
    assert cosine(got, oracle.bf16_decode(ref)) >= 0.999
    out = torch.empty_like(r)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c["plan"].graph_capture(r, h, out, s)
        c["plan"].graph_replay(wl.M, s)
    s.synchronize()
    assert torch.equal(out, eager)


def test_gpu_calibration_matches_oracle(case):
    c = case
    dev = c["dev"]
    saved = c["plan"].scales()
    c["plan"].calibrate([a.to(dev) for a, _ in c["cb"]], [b.to(dev) for _, b in c["cb"]])
    sc = c["plan"].scales()
    c["plan"].set_scales(saved["s_x"], saved["s_h"])
    rx = c["s_x"][0]
    assert abs(sc["s_x"][0] - rx) <= (0.5 * c["wl"].d + 4) * 2.0 ** -24 * rx
    assert abs(sc["s_h"][0] - c["s_h"][0]) <= 1e-3 * c["s_h"][0]


def test_modulation_boundary():
    from realtime_transformer_gb300 import _native as N
    from realtime_transformer_gb300.ffn import FFNPlan
    dev = torch.device("cuda")
    p = FFNPlan(256, 1024, "geglu_tanh", 8, 2)
    good = [torch.zeros(1, 768, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    with pytest.raises(N.FrtError) as e:
        p.set_modulation([torch.zeros(3, 768, dtype=torch.bfloat16, device=dev)] * 2)  # rows not 1 or M_max
    assert e.value.name == "FRT_ERR_INVALID_ARG"
    with pytest.raises(N.FrtError) as e:
        N.frt_ffn_set_modulation(p.handle, [good[0].data_ptr(), None], 1)
    assert e.value.name == "FRT_ERR_INVALID_ARG"
    p.set_modulation(good)
    p.set_modulation(None)
    p.close()
