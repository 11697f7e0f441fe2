"""The NVFP4 sublayer at the workloads' full sizes (itsolotime FlashRT article,
7.2: the NVFP4 encoder FFN), in the launch configuration its benchmark times:
one layer at full M on the VLA prefix, LLM decode and long-prefill shapes,
whose GEMMs take other tilings and split-K factors than the small cases.

Rows are independent once the scales are fixed, so the oracle runs the layer
on sampled rows (spread over the token tiles, the first and last included)
while the GPU runs all of them.  Weight preparation is compared bit for bit;
every step on every sampled row, from the oracle's own input to that step
(its X and A fed to the GPU GEMMs on those rows), under the contract of the
small cases (tests/test_gpu_nvfp4.py); the kernels' own path under the
cosine bound."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import bits, check_bf16, cosine
from test_gpu_nvfp4 import _sf_index as sf_index, check_nvfp4, canon, pack, sf_from_tmem, unpack

pytestmark = pytest.mark.gpu


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


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
        check_nvfp4(xq, xs, ref.x[0], ref.x[1], ref.y, sc.s_x, name + " x")
        # the GEMMs from the oracle's X and A on the sampled rows (the GPU's own elsewhere)
        x_codes, x_sf = tr["x_codes"].cpu().numpy().copy(), tr["x_sf"].cpu().numpy().copy()
        h_codes, h_sf = tr["h_codes"].cpu().numpy().copy(), tr["h_sf"].cpu().numpy().copy()
        x_codes[rows] = pack(ref.x[0])
        x_sf[sf_index(M, d)[rows]] = ref.x[1]
        h_codes[rows] = pack(ref.h[0])
        h_sf[sf_index(M, ff)[rows]] = ref.h[1]
        tf = plan.trace_from(0, r, h, x=(dev_u8(x_codes), dev_u8(x_sf)), h=(dev_u8(h_codes), dev_u8(h_sf)))
        torch.cuda.synchronize()
        plan.device_status()
        gq, gs = unpack(tf["g_codes"].cpu().numpy())[rows], tf["g_sf"].cpu().numpy()[rows]
        uq, us = unpack(tf["u_codes"].cpu().numpy())[rows], tf["u_sf"].cpu().numpy()[rows]
        check_nvfp4(gq, gs, ref.g[0], ref.g[1], ref.g_f32, sc.s_g, name + " gate")
        check_nvfp4(uq, us, ref.u[0], ref.u[1], ref.u_f32, sc.s_u, name + " up")
        a = oracle.nvfp4_gated_act((gq, gs), (uq, us), sc.s_g, sc.s_u, wl.act_id)
        h_ref = oracle.nvfp4_quantize(a, sc.s_h)
        check_nvfp4(unpack(tf["h_codes"].cpu().numpy())[rows], sf_from_tmem(tf["h_sf"].cpu().numpy(), M, ff)[rows],
                    h_ref[0], h_ref[1], a, sc.s_h, name + " h")
        check_bf16(bits(tf["out"])[rows], ref.out, name + " out")
        # the kernels' own path
        c = cosine(oracle.bf16_decode(bits(tr["out"])[rows]), oracle.bf16_decode(ref.out))
        print("%s NVFP4 layer: rows %s, every step on every sampled row; own-path out cosine %.7f" % (
            name, list(rows), c))
        assert c > 0.9999, c
    finally:
        plan.close()
