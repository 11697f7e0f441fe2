"""Shared helpers of the GPU parity tests: the tolerance contract and the
plumbing that hands the same seeded inputs to the CUDA path and the oracle.

Contract (GPU vs oracle on the same inputs and the same scales):
  * E4M3 activation codes identical on >= 99.9% of elements and never more
    than one code step apart on the monotone code line (+0 and -0 equal);
  * BF16 outputs: cosine >= 0.9999 and max |err| <= 2e-2 x RMS(oracle).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synthetic

CODE_AGREE = 0.999
COS_MIN = 0.9999
ERR_RMS = 2e-2


def code_ordinal(c):
    c = np.asarray(c, np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def check_codes(got, ref, what=""):
    got = np.asarray(got, np.uint8)
    ref = np.asarray(ref, np.uint8)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    same = float(np.mean(code_ordinal(got) == code_ordinal(ref)))
    step = int(np.abs(code_ordinal(got) - code_ordinal(ref)).max()) if got.size else 0
    assert same >= CODE_AGREE, "%s: only %.5f of codes agree" % (what, same)
    assert step <= 1, "%s: codes differ by %d steps" % (what, step)
    return same


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / np.sqrt((a @ a) * (b @ b)))


def check_bf16(got_bits, ref_bits, what=""):
    g = oracle.bf16_decode(got_bits).astype(np.float64)
    r = oracle.bf16_decode(ref_bits).astype(np.float64)
    assert g.shape == r.shape
    c = cosine(g, r)
    err = float(np.abs(g - r).max() / np.sqrt((r ** 2).mean()))
    assert c >= COS_MIN, "%s: cosine %.7f" % (what, c)
    assert err <= ERR_RMS, "%s: max|err|/rms %.4g" % (what, err)
    return c, err


def check_layer(plan, layer, r, h, ref, what="", rows=None):
    """Parity of one layer against the oracle's trace `ref` of the same input,
    on every row (or every sampled row), in two passes over the forward's
    kernels:
      1. the layer from its input (r, h: device tensors of all M rows): r'
         bit-exact, q_x codes under the code contract;
      2. the layer from the oracle's own r' and q_x codes (steps A2..A4 on
         the GPU; on rows outside `rows` the GPU's own codes), so that an
         allowed one-step q_x flip does not propagate: g/u (BF16), q_h codes
         and the layer output on all compared rows under the full contract
         (codes; cosine and max|err| / RMS).
    The own-path layer output of pass 1 is also reported and held to the
    pages' cosine claim.  rows: indices of the rows `ref` covers (None: all).
    """
    dev = r.device
    tr = plan.trace_layer(layer, r, h)
    torch.cuda.synchronize()
    plan.device_status()
    if rows is None:
        sel = lambda t: t
    else:
        rows_t = torch.as_tensor(np.asarray(rows, np.int64), device=dev)
        sel = lambda t: t.index_select(0, rows_t)
    assert np.array_equal(bits(sel(tr["r_prime"])), ref.r_prime), what + ": r' = bf16(r + h) must be bit-exact"
    agree_x = check_codes(u8(sel(tr["q_x"])), ref.q_x, what + " q_x")
    qx_feed = tr["q_x"].clone()
    ref_qx = torch.from_numpy(np.ascontiguousarray(ref.q_x)).to(dev)
    if rows is None:
        qx_feed.copy_(ref_qx)
    else:
        qx_feed.index_copy_(0, rows_t, ref_qx)
    tq = plan.trace_layer_from_qx(layer, tr["r_prime"], qx_feed)
    torch.cuda.synchronize()
    plan.device_status()
    check_bf16(bits(sel(tq["gu"])), ref.gu, what + " gate/up")
    agree_h = check_codes(u8(sel(tq["q_h"])), ref.q_h, what + " q_h")
    c, e = check_bf16(bits(sel(tq["out"])), ref.out, what + " layer output")
    own = bits(sel(tr["out"]))
    c_own = cosine(oracle.bf16_decode(own), oracle.bf16_decode(ref.out))
    assert c_own > 0.999, "%s: own-path output cosine %.7f" % (what, c_own)
    return dict(q_x=agree_x, q_h=agree_h, cos=c, err=e, cos_own=c_own, out=own, ref_out=ref.out)


def bits(t: torch.Tensor) -> np.ndarray:
    return synthetic.bf16_bits(t)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.uint8)


class Case:
    """One workload: seeded weights/inputs, oracle-quantised weights and
    oracle-calibrated scales, and a loaded GPU plan."""

    def __init__(self, wl, device="cuda", gen_device="cpu", M_max=None, calib_rows=None, fold_norm=False):
        from realtime_transformer_gb300.ffn import FFNPlan
        self.wl = wl
        self.fold = fold_norm
        self.dev = torch.device(device)
        self.weights = [synthetic.layer_weights(wl, l, device=gen_device) for l in range(wl.L)]
        self.r, self.h = synthetic.inputs(wl, device=gen_device)
        self.calib = synthetic.calibration_batches(wl, device=gen_device)
        self.q = oracle.quantize_stack([{k: bits(v) for k, v in w.items()} for w in self.weights],
                                       fold_norm=fold_norm)
        rows = slice(None) if calib_rows is None else slice(0, calib_rows)
        self.s_x, self.s_h = oracle.calibrate_stack(self.q, [bits(a[rows]) for a, _ in self.calib],
                                                    [bits(b[rows]) for _, b in self.calib], wl.act_id)
        self.plan = FFNPlan(wl.d, wl.ff, wl.act, M_max or wl.M, wl.L)
        for l, w in enumerate(self.weights):
            self.plan.load_weights(l, *(w[k].to(self.dev) for k in ("w_norm", "w_gate", "w_up", "w_down")),
                                   fold_norm=fold_norm)
        self.plan.set_scales(self.s_x, self.s_h)

    def oracle_forward(self, rows=None, trace=False):
        r = bits(self.r) if rows is None else bits(self.r)[rows]
        h = bits(self.h) if rows is None else bits(self.h)[rows]
        return oracle.stack_forward(self.q, r, h, self.s_x, self.s_h, self.wl.act_id, trace=trace)

    def close(self):
        self.plan.close()
