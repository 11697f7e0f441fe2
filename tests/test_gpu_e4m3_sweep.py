"""The GPU's E4M3 conversion against the oracle's encoder on every one of the
2^32 fp32 bit patterns.  Every quantising kernel (weights at load time, the
norm's q_x, the activation's q_h) rounds with the hardware conversion
(cvt with round-to-nearest-even and saturation); the oracle's encoder is
written from the format's definition (OCP FP8 E4M3: bias 7, subnormals, max
448, no infinities).  The two are independent, so agreement on all inputs
pins both.  The only allowed difference is the NaN code: for a NaN input both
sides must give a NaN code (0x7F or 0xFF), the oracle drops the sign
(agentlenshq FlashRT summary, "Main ideas": FP8 E4M3 activations)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


def test_every_fp32_pattern_encodes_like_the_oracle():
    from realtime_transformer_gb300 import _native as N
    dev = torch.device("cuda")
    codes = torch.empty(CHUNK, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    mismatches = 0
    nan_inputs = 0
    for c in range((1 << 32) // CHUNK):
        start = c * CHUNK
        N.frt_debug_e4m3_encode_range(start, CHUNK, codes.data_ptr(), stream)
        pat = np.arange(start, start + CHUNK, dtype=np.uint64).astype(np.uint32)
        x = pat.view(np.float32)
        want = oracle.e4m3_encode(x)
        got = codes.cpu().numpy()
        nan = np.isnan(x)
        nan_inputs += int(nan.sum())
        assert np.all((got[nan] & 0x7F) == 0x7F), "chunk %d: NaN input without a NaN code" % c
        diff = (got != want) & ~nan
        if diff.any():
            idx = np.nonzero(diff)[0][:5]
            raise AssertionError("chunk %d: patterns %s -> gpu %s oracle %s" % (
                c, [hex(int(pat[i])) for i in idx], [hex(int(got[i])) for i in idx], [hex(int(want[i])) for i in idx]))
        mismatches += int(diff.sum())
    # 2^23 - 1 NaN mantissas per sign
    assert nan_inputs == 2 * ((1 << 23) - 1)
    assert mismatches == 0
