"""Attention-input sublayer at the workloads' full sizes, in the launch
configuration the benchmark times (full M; on the long-prefill shape the split
+ RoPE runs in the GEMM epilogue).  Rows are independent once the scale is
fixed, so the oracle checks a handful of rows spread over the token tiles,
the last row included (agentlenshq FlashRT summary, "What it is";
itsolotime FlashRT article, 5.2 FusedQKV)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import bits, check_bf16, check_codes, u8

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["vla_action_expert", "vla_prefix", "llm_decode", "long_prefill"])
def test_full_size_qkv(name):
    from realtime_transformer_gb300.qkv import QKVPlan
    wl = synthetic.WORKLOADS[name]
    nq, nkv, hd, base = synthetic.ATTENTION[name]
    dev = torch.device("cuda")
    w = synthetic.qkv_weights(wl, 0, device=dev)
    r, h = synthetic.inputs(wl, device=dev)
    pos = synthetic.positions(wl)
    hw = {k: bits(v) for k, v in w.items()}
    codes, s_qkv = oracle.quantize_qkv_weights(hw["w_q"], hw["w_k"], hw["w_v"])
    crow = min(wl.M, 64)
    s_x = oracle.calibrate_qkv_layer([bits(r[:crow])], [bits(h[:crow])], hw["w_norm"])
    plan = QKVPlan(wl.d, nq, nkv, hd, base, wl.M, 1)
    plan.load_weights(0, w["w_norm"], w["w_q"], w["w_k"], w["w_v"])
    assert plan.scales()["s_qkv"][0] == np.float32(s_qkv)
    plan.set_scales([s_x])
    out = plan.forward(0, r, h, torch.from_numpy(pos).to(dev))
    torch.cuda.synchronize()
    plan.device_status()
    rows = np.array(sorted(set([0, wl.M - 1] + [int(x) for x in np.linspace(0, wl.M - 1, 8)])), dtype=np.int64)
    hr = bits(r)[rows]
    hh = bits(h)[rows]
    ref = oracle.qkv_layer(hr, hh, hw["w_norm"], codes, s_x, s_qkv, nq, nkv, hd, pos[rows],
                           oracle.rope_inv_freq(hd, base))
    assert np.array_equal(bits(out["r_prime"])[rows], ref.r_prime)
    rows_t = torch.from_numpy(rows).to(dev)
    w_st = plan.weights(0)
    torch.cuda.synchronize()
    assert np.array_equal(u8(w_st), codes), name + " stored weight codes"
    del w_st
    # q_x under the code contract on the sampled rows, then the GEMM and split
    # + RoPE at full M from the oracle's codes on those rows (the GPU's own
    # elsewhere): every sampled row under the full contract
    tr = plan.trace(0, r, h, torch.from_numpy(pos).to(dev))
    torch.cuda.synchronize()
    qx = tr["q_x"].index_select(0, rows_t)
    check_codes(u8(qx), ref.q_x, name + " q_x")
    feed = tr["q_x"].clone()
    feed.index_copy_(0, rows_t, torch.from_numpy(ref.q_x).to(dev))
    tq = plan.trace_from_qx(0, feed, torch.from_numpy(pos).to(dev))
    torch.cuda.synchronize()
    plan.device_status()
    check_bf16(bits(tq["qkv"].index_select(0, rows_t)), ref.qkv, name + " qkv")
    for k in ("q", "k", "v"):
        got = bits(tq[k].index_select(1, rows_t))
        check_bf16(got, getattr(ref, k), "%s %s" % (name, k))
    plan.close()
