"""Attention-input sublayer on the GPU against the oracle: residual + RMSNorm
+ E4M3 quantise, FP8 fused-QKV GEMM, QKV split + RoPE (agentlenshq FlashRT
summary, "What it is"; itsolotime FlashRT article, 5.2 FusedQKV; "FlashRT
docs/architecture.md", 8 Kernel Library).  Same inputs and scales on both
sides; q_x codes under the code contract, then the GEMM output and Q/K/V,
computed from the oracle's own q_x codes, on every row under the full
contract; the stored E4M3 weight codes byte for byte."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import bits, check_bf16, check_codes, cosine, u8

pytestmark = pytest.mark.gpu

# (name, M, d, n_q, n_kv, head_dim, rope_base, first position, hidden)
SHAPES = [
    ("tiny", 8, 256, 4, 1, 64, 1.0e4, 0, True),
    ("action_expert", 50, 1024, 8, 1, 256, 1.0e4, 0, True),
    ("decode", 1, 5120, 40, 8, 128, 1.0e6, 4096, False),
    ("ragged", 17, 384, 6, 3, 32, 1.0e4, 100, True),
    ("tiled", 300, 512, 4, 2, 64, 1.0e4, 0, False),
    ("far_positions", 3, 256, 4, 2, 32, 1.0e6, 100000, False),
    # tiled tiles without split-K that hold whole heads: split + RoPE in the GEMM epilogue
    ("fused_hd256", 1000, 512, 8, 1, 256, 1.0e4, 0, True),
    ("fused_hd128", 1280, 256, 12, 2, 128, 1.0e6, 7, False),
    # the norm weight folded into [W_q; W_k; W_v] (the Pi0 layout)
    ("folded", 50, 1024, 8, 1, 256, 1.0e4, 0, True, True),
    ("folded_tiled", 300, 512, 4, 2, 64, 1.0e4, 0, False, True),
]


def weights(d, nq, nkv, hd, seed):
    g = torch.Generator().manual_seed(seed)
    w = {"w_q": torch.randn(nq * hd, d, generator=g) * 0.02, "w_k": torch.randn(nkv * hd, d, generator=g) * 0.02,
         "w_v": torch.randn(nkv * hd, d, generator=g) * 0.02, "w_norm": 1 + 0.1 * torch.randn(d, generator=g)}
    return {k: v.to(torch.bfloat16) for k, v in w.items()}


@pytest.fixture(scope="module", params=SHAPES, ids=lambda s: s[0])
def case(request):
    from realtime_transformer_gb300.qkv import QKVPlan
    name, M, d, nq, nkv, hd, base, p0, with_h = request.param[:9]
    fold = len(request.param) > 9 and request.param[9]
    wl = synthetic.WORKLOADS["tiny"].with_(name=name, M=M, d=d, seed=31)
    r, h = synthetic.inputs(wl)
    h = h if with_h else None
    w = weights(d, nq, nkv, hd, 7 + M)
    pos = (p0 + 3 * np.arange(M)).astype(np.int32)
    if fold:
        codes, s_qkv = oracle.quantize_qkv_weights_folded(bits(w["w_q"]), bits(w["w_k"]), bits(w["w_v"]),
                                                          bits(w["w_norm"]))
        w_norm_ref = np.full(d, oracle.BF16_ONE, dtype=np.uint16)
    else:
        codes, s_qkv = oracle.quantize_qkv_weights(bits(w["w_q"]), bits(w["w_k"]), bits(w["w_v"]))
        w_norm_ref = bits(w["w_norm"])
    s_x = oracle.calibrate_qkv_layer([bits(r)], [bits(h)] if with_h else None, w_norm_ref)
    dev = torch.device("cuda")
    plan = QKVPlan(d, nq, nkv, hd, base, M, 1)
    plan.load_weights(0, *(w[k].to(dev) for k in ("w_norm", "w_q", "w_k", "w_v")), fold_norm=fold)
    plan.set_scales([s_x])
    c = dict(name=name, M=M, d=d, nq=nq, nkv=nkv, hd=hd, base=base, r=r, h=h, w=w, pos=pos, codes=codes,
             s_qkv=s_qkv, s_x=s_x, plan=plan, dev=dev, w_norm_ref=w_norm_ref)
    yield c
    plan.close()


def test_weight_scale_matches_oracle_exactly(case):
    assert case["plan"].scales()["s_qkv"][0] == np.float32(case["s_qkv"])


def test_weight_codes_match_oracle_byte_for_byte(case):
    w = case["plan"].weights(0)
    torch.cuda.synchronize()
    bad = np.argwhere(u8(w) != case["codes"])
    assert bad.size == 0, (case["name"], bad[:5])


def test_sublayer_matches_oracle(case, monkeypatch):
    c = case
    monkeypatch.setenv("FRT_QKV_FUSE", "1")  # the fused split + RoPE wherever the tiles allow it
    dev = c["dev"]
    tr = c["plan"].trace(0, c["r"].to(dev), c["h"].to(dev) if c["h"] is not None else None,
                         torch.from_numpy(c["pos"]).to(dev))
    torch.cuda.synchronize()
    c["plan"].device_status()
    ref = oracle.qkv_layer(bits(c["r"]), bits(c["h"]) if c["h"] is not None else None, c["w_norm_ref"],
                           c["codes"], c["s_x"], c["s_qkv"], c["nq"], c["nkv"], c["hd"], c["pos"],
                           oracle.rope_inv_freq(c["hd"], c["base"]))
    assert np.array_equal(bits(tr["r_prime"]), ref.r_prime), "r' = bf16(r + h) must be bit-exact"
    check_codes(u8(tr["q_x"]), ref.q_x, c["name"] + " q_x")
    # the GEMM and split + RoPE from the oracle's own codes: every row under
    # the contract (an allowed q_x flip does not reach the outputs)
    pos_d = torch.from_numpy(c["pos"]).to(dev)
    tq = c["plan"].trace_from_qx(0, torch.from_numpy(ref.q_x).to(dev), pos_d)
    torch.cuda.synchronize()
    c["plan"].device_status()
    check_bf16(bits(tq["qkv"]), ref.qkv, c["name"] + " qkv")
    for k in ("q", "k", "v"):
        got = bits(tq[k])
        assert got.shape == getattr(ref, k).shape, k
        check_bf16(got, getattr(ref, k), "%s %s" % (c["name"], k))
    # the own path's outputs hold the pages' cosine claim
    for k in ("q", "k", "v"):
        assert cosine(oracle.bf16_decode(bits(tr[k])), oracle.bf16_decode(getattr(ref, k))) > 0.999, k
    # the forward entry point computes the same as the trace (which runs the
    # split + RoPE kernel; the forward may run it in the GEMM's epilogue)
    o = c["plan"].forward(0, c["r"].to(dev), c["h"].to(dev) if c["h"] is not None else None,
                          torch.from_numpy(c["pos"]).to(dev))
    torch.cuda.synchronize()
    for k in ("q", "k", "v", "r_prime"):
        assert torch.equal(o[k], tr[k]), k
    monkeypatch.setenv("FRT_QKV_FUSE", "0")
    o2 = c["plan"].forward(0, c["r"].to(dev), c["h"].to(dev) if c["h"] is not None else None,
                           torch.from_numpy(c["pos"]).to(dev))
    torch.cuda.synchronize()
    for k in ("q", "k", "v"):
        assert torch.equal(o2[k], tr[k]), k


def test_gpu_calibration_matches_oracle(case):
    c = case
    dev = c["dev"]
    saved = c["plan"].scales()["s_x"]
    c["plan"].calibrate(0, [c["r"].to(dev)], [c["h"].to(dev)] if c["h"] is not None else None)
    got = c["plan"].scales()["s_x"][0]
    c["plan"].set_scales(saved)
    assert abs(got - c["s_x"]) <= (0.5 * c["d"] + 4) * 2.0 ** -24 * c["s_x"]


def test_forward_can_be_captured_in_a_cuda_graph(case):
    c = case
    dev = c["dev"]
    r = c["r"].to(dev)
    h = c["h"].to(dev) if c["h"] is not None else None
    pos = torch.from_numpy(c["pos"]).to(dev)
    eager = c["plan"].forward(0, r, h, pos)
    torch.cuda.synchronize()
    out = {k: torch.empty_like(v) for k, v in eager.items()}
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c["plan"].forward(0, r, h, pos, out=out, stream=s)  # warm up (tensor maps, attributes) outside capture
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            c["plan"].forward(0, r, h, pos, out=out, stream=s)
    for v in out.values():
        v.zero_()
    g.replay()
    torch.cuda.synchronize()
    for k in ("q", "k", "v"):
        assert torch.equal(out[k], eager[k]), k


def test_boundary_errors():
    from realtime_transformer_gb300 import _native as N
    from realtime_transformer_gb300.qkv import QKVPlan
    with pytest.raises(N.FrtError) as e:
        QKVPlan(256, 3, 2, 64, 1e4, 8, 1)  # 2 does not divide 3
    assert e.value.name == "FRT_ERR_INVALID_ARG"
    with pytest.raises(N.FrtError):
        QKVPlan(256, 4, 1, 60, 1e4, 8, 1)  # head_dim % 8
    dev = torch.device("cuda")
    p = QKVPlan(256, 4, 1, 64, 1e4, 8, 2)
    r = torch.zeros(8, 256, dtype=torch.bfloat16, device=dev)
    pos = torch.zeros(8, dtype=torch.int32, device=dev)
    with pytest.raises(N.FrtError) as e:
        p.forward(0, r, None, pos)
    assert e.value.name == "FRT_ERR_NOT_READY"
    w = weights(256, 4, 1, 64, 3)
    p.load_weights(1, *(w[k].to(dev) for k in ("w_norm", "w_q", "w_k", "w_v")))
    wd = {k: w[k].to(dev) for k in w}
    with pytest.raises(N.FrtError) as e:
        N.frt_qkv_load_weights_ex(p.handle, 1, wd["w_norm"].data_ptr(), wd["w_q"].data_ptr(), wd["w_k"].data_ptr(),
                                  wd["w_v"].data_ptr(), 2, None)  # unknown flag
    assert e.value.name == "FRT_ERR_INVALID_ARG"
    with pytest.raises(N.FrtError) as e:
        p.forward(1, r, None, pos)  # no activation scale yet
    assert e.value.name == "FRT_ERR_NOT_READY"
    with pytest.raises(N.FrtError) as e:
        p.set_scales([0.01, float("nan")])
    assert e.value.name == "FRT_ERR_INVALID_ARG"
    p.set_scales([0.01, 0.01])
    big = torch.zeros(9, 256, dtype=torch.bfloat16, device=dev)
    with pytest.raises(N.FrtError) as e:
        p.forward(1, big, None, torch.zeros(9, dtype=torch.int32, device=dev))
    assert e.value.name == "FRT_ERR_SHAPE"
    o = p._outs(8, dev)
    with pytest.raises(N.FrtError) as e:
        N.frt_qkv_forward(p.handle, 1, r.data_ptr(), None, None, None, o["q"].data_ptr(), o["k"].data_ptr(),
                          o["v"].data_ptr(), 8, None)
    assert e.value.name == "FRT_ERR_INVALID_ARG"
    N.frt_qkv_forward(p.handle, 1, r.data_ptr(), None, pos.data_ptr(), None, o["q"].data_ptr(), o["k"].data_ptr(),
                      o["v"].data_ptr(), 0, None)  # M == 0: nothing
    p.device_status()
    p.close()
