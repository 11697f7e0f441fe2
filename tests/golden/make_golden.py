"""Writes tests/golden/tiny_oracle.txt from the oracle alone.

The fixture records the oracle's results on the tiny workload (M=8, d=256,
ff=1024, GeGLU, 1 layer, seed 0): weight and calibrated activation scales
and a digest of every intermediate, so that any later change of the oracle's
arithmetic shows up as a test failure and has to be justified.

Run from the repository root:  python tests/golden/make_golden.py
"""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synthetic  # noqa: E402


def compute():
    wl = synthetic.WORKLOADS["tiny"]
    ws = [{k: synthetic.bf16_bits(v) for k, v in synthetic.layer_weights(wl, l).items()} for l in range(wl.L)]
    q = oracle.quantize_stack(ws)
    cb = synthetic.calibration_batches(wl)
    s_x, s_h = oracle.calibrate_stack(q, [synthetic.bf16_bits(a) for a, _ in cb],
                                      [synthetic.bf16_bits(b) for _, b in cb], wl.act_id)
    r, h = [synthetic.bf16_bits(x) for x in synthetic.inputs(wl)]
    (tr,) = oracle.stack_forward(q, r, h, s_x, s_h, wl.act_id, trace=True)
    rows = {
        "s_gu": q[0].s_gu.hex(), "s_d": q[0].s_d.hex(), "s_x": s_x[0].hex(), "s_h": s_h[0].hex(),
        "q_gu_sha256": hashlib.sha256(q[0].q_gu.tobytes()).hexdigest(),
        "q_down_sha256": hashlib.sha256(q[0].q_down.tobytes()).hexdigest(),
        "r_prime_sha256": hashlib.sha256(tr.r_prime.tobytes()).hexdigest(),
        "q_x_sha256": hashlib.sha256(tr.q_x.tobytes()).hexdigest(),
        "gu_sha256": hashlib.sha256(tr.gu.tobytes()).hexdigest(),
        "q_h_sha256": hashlib.sha256(tr.q_h.tobytes()).hexdigest(),
        "out_sha256": hashlib.sha256(tr.out.tobytes()).hexdigest(),
        "out_row0_first8": " ".join("%04x" % v for v in tr.out[0, :8]),
    }
    return rows


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.txt")
    with open(path, "w") as f:
        f.write("# oracle results on the tiny workload; written by tests/golden/make_golden.py\n")
        for k, v in compute().items():
            f.write("%s %s\n" % (k, v))
    print("wrote", path)
