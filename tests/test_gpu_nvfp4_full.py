"""The NVFP4 sublayer at the workloads' full sizes (itsolotime FlashRT article,
7.2: the NVFP4 encoder FFN), in the launch configuration its benchmark times:
one layer at full M on the VLA prefix, LLM decode and long-prefill shapes,
whose GEMMs take other tilings and split-K factors than the small cases.

Rows are independent once the scales are fixed, so the oracle runs the layer
on sampled rows (spread over the token tiles, the first and last included)
while the GPU runs all of them.  Weight preparation is compared bit for bit;
the quantised activations under the tie-aware NVFP4 contract of the small
cases (tests/test_gpu_nvfp4.py), the output on rows whose quantised
activations agree under the FP8 path's contract, and all sampled rows'
outputs under its cosine bound."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import bits, check_bf16, cosine
from test_gpu_nvfp4 import check_nvfp4, canon, sf_from_tmem, unpack

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["vla_prefix", "llm_decode", "long_prefill"])
def test_full_size_nvfp4_layer(name):
    from realtime_transformer_gb300.nvfp4 import FP4Plan
    wl = synthetic.WORKLOADS[name]
    dev = torch.device("cuda")
    M, d, ff = wl.M, wl.d, wl.ff
    lw = synthetic.layer_weights(wl, 0, device=dev)
    hw = {k: bits(v) for k, v in lw.items()}
    L = oracle.quantize_layer_nvfp4(hw["w_norm"], hw["w_gate"], hw["w_up"], hw["w_down"])
    crow = min(M, 64)
    cb = synthetic.calibration_batches(wl, device="cpu", M=crow)
    sc, _ = oracle.calibrate_layer_nvfp4([bits(a) for a, _ in cb], [bits(b) for _, b in cb], L, wl.act_id)
    plan = FP4Plan(d, ff, wl.act, M, 1)
    try:
        plan.load_weights(0, lw["w_norm"], lw["w_gate"], lw["w_up"], lw["w_down"])
        del lw
        s_w = plan.scales()["weight"][0]
        for which, ref, rows_w, K, s in [("gate", L.gate, ff, d, s_w[0]), ("up", L.up, ff, d, s_w[1]),
                                         ("down", L.down, d, ff, s_w[2])]:
            codes, sf = plan.weights(0, which)
            assert np.float32(s) == np.float32(ref.s), which
            assert np.array_equal(canon(unpack(codes.cpu().numpy())), canon(ref.q)), which
            assert np.array_equal(sf_from_tmem(sf.cpu().numpy(), rows_w, K), ref.sb), which
            del codes, sf
        plan.set_scales([[sc.s_x, sc.s_g, sc.s_u, sc.s_h]])
        r, h = synthetic.inputs(wl, device=dev)
        tr = plan.trace(0, r, h)
        torch.cuda.synchronize()
        plan.device_status()
        rows = np.array(sorted(set([0, M - 1] + [int(x) for x in np.linspace(0, M - 1, 8)])), dtype=np.int64)
        ref = oracle.ffn_layer_nvfp4(bits(r)[rows], bits(h)[rows], L, sc, wl.act_id, trace=True)
        assert np.array_equal(bits(tr["r_prime"])[rows], ref.r_prime)
        xq = unpack(tr["x_codes"].cpu().numpy())[rows]
        xs = sf_from_tmem(tr["x_sf"].cpu().numpy(), M, d)[rows]
        ok = check_nvfp4(xq, xs, ref.x[0], ref.x[1], ref.y, sc.s_x, name + " x")
        gq = unpack(tr["g_codes"].cpu().numpy())[rows]
        uq = unpack(tr["u_codes"].cpu().numpy())[rows]
        gs, us = tr["g_sf"].cpu().numpy()[rows], tr["u_sf"].cpu().numpy()[rows]
        if ok.any():
            ok_g = check_nvfp4(gq[ok], gs[ok], ref.g[0][ok], ref.g[1][ok], ref.g_f32[ok], sc.s_g, name + " gate")
            ok_u = check_nvfp4(uq[ok], us[ok], ref.u[0][ok], ref.u[1][ok], ref.u_f32[ok], sc.s_u, name + " up")
            sel = np.nonzero(ok)[0]
            ok[sel[~(ok_g & ok_u)]] = False
        if ok.any():
            hq = unpack(tr["h_codes"].cpu().numpy())[rows]
            hs = sf_from_tmem(tr["h_sf"].cpu().numpy(), M, ff)[rows]
            ok_h = check_nvfp4(hq[ok], hs[ok], ref.h[0][ok], ref.h[1][ok], ref.a[ok], sc.s_h, name + " h")
            sel = np.nonzero(ok)[0]
            ok[sel[~ok_h]] = False
        got = bits(tr["out"])[rows]
        if ok.any():
            check_bf16(got[ok], ref.out[ok], name + " out")
        c = cosine(oracle.bf16_decode(got), oracle.bf16_decode(ref.out))
        print("%s NVFP4 layer: rows %s, %d with every quantised activation identical, out cosine %.7f" % (
            name, list(rows), int(ok.sum()), c))
        assert c > 0.9999, c
    finally:
        plan.close()
