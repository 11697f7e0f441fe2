"""Teacher-forced parity of one layer (steps A0..A4) against the oracle: both
sides get the same layer input and the same scales; every intermediate is
compared (itsolotime FlashRT article, 7.2; agentlenshq summary, "Main
ideas": fused residual-norm-quantise)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import Case, bits, check_bf16, check_codes, u8

pytestmark = pytest.mark.gpu

WL = synthetic.WORKLOADS
# shapes spanning several tiles and ragged tails, both GEMM paths, both activations
SHAPES = [
    WL["tiny"],
    WL["vla_action_expert"].with_(L=1),
    WL["tiny"].with_(name="m1_swiglu", M=1, d=1024, ff=2048, act=synthetic.SWIGLU, outliers=False, n_calib=1),
    WL["tiny"].with_(name="m64", M=64, d=512, ff=1536, n_calib=1, seed=11),
    WL["tiny"].with_(name="m65_tiled", M=65, d=512, ff=1536, n_calib=1, seed=12),
    WL["vla_prefix"].with_(name="prefix_small", M=300, d=512, ff=2048, L=1),
    WL["long_prefill"].with_(name="prefill_small", M=257, d=640, ff=1280, L=1),
]


@pytest.fixture(scope="module", params=SHAPES, ids=lambda w: w.name)
def case(request):
    c = Case(request.param)
    yield c
    c.close()


def test_weight_scales_match_oracle_exactly(case):
    sc = case.plan.scales()
    for l, ql in enumerate(case.q):
        assert sc["s_gu"][l] == np.float32(ql.s_gu)
        assert sc["s_down"][l] == np.float32(ql.s_d)


@pytest.mark.parametrize("with_hidden", [True, False])
def test_layer_intermediates_match_oracle(case, with_hidden):
    wl = case.wl
    dev = case.dev
    h = case.h if with_hidden else None
    tr = case.plan.trace_layer(0, case.r.to(dev), h.to(dev) if h is not None else None)
    torch.cuda.synchronize()
    case.plan.device_status()
    ql = case.q[0]
    ref = oracle.ffn_layer(bits(case.r), bits(h) if h is not None else None, ql.w_norm, ql.q_gu, ql.q_down,
                           case.s_x[0], case.s_h[0], ql.s_gu, ql.s_d, wl.act_id, trace=True)
    assert np.array_equal(bits(tr["r_prime"]), ref.r_prime), "r' = bf16(r + h) must be bit-exact"
    check_codes(u8(tr["q_x"]), ref.q_x, "q_x")
    check_bf16(bits(tr["gu"]), ref.gu, "gate/up output")
    check_codes(u8(tr["q_h"]), ref.q_h, "q_h")
    check_bf16(bits(tr["out"]), ref.out, "layer output")


def test_out_may_alias_residual(case):
    dev = case.dev
    r = case.r.to(dev)
    h = case.h.to(dev)
    sep = case.plan.forward(r, h)
    buf = r.clone()
    case.plan.forward(buf, h, out=buf)
    torch.cuda.synchronize()
    assert torch.equal(sep, buf)
