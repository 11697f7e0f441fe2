"""The allocation-free FP8 GEMM entry point (frt_fp8_gemm_noalloc).

It exists for callers that cannot call cudaMalloc -- code running under a
global-mode stream capture, real-time hosts that forbid allocation after
start-up, hosts that own all device memory -- and keeps its split-K scratch
in a fixed device array instead.  Checked against the plan-based
frt_fp8_gemm on the same inputs, on two calls in a row (the second call
reuses the scratch the first one left behind), within the GEMM tests'
fp32 summation bound.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x7E
    return c


def within_bound(got, ref, A, B, K, alpha):
    a = oracle.e4m3_decode(A).astype(np.float64)
    b = oracle.e4m3_decode(B).astype(np.float64)
    bound = 2 * K * 2.0 ** -24 * (np.abs(a) @ np.abs(b).T) * alpha + 2 * 2.0 ** -24 * np.abs(ref)
    return np.all(np.abs(got.astype(np.float64) - ref.astype(np.float64)) <= bound)


def test_no_alloc_gemm_matches_plan_gemm_on_two_calls():
    from realtime_transformer_gb300 import _native as N
    from realtime_transformer_gb300.ffn import FFNPlan
    dev = torch.device("cuda")
    plan = FFNPlan(256, 1024, "geglu_tanh", 64, 1)
    rng = np.random.default_rng(2024)
    stream = torch.cuda.current_stream().cuda_stream
    # first call: weight-streaming path with split-K; second: another shape,
    # reusing the scratch left by the first
    for (M, Nn, K) in [(50, 1024, 4096), (16, 2048, 1024)]:
        A = codes(rng, (M, K))
        B = codes(rng, (Nn, K))
        At = torch.from_numpy(A).to(dev)
        Bt = torch.from_numpy(B).to(dev)
        C = torch.full((M, Nn), float("nan"), dtype=torch.float32, device=dev)
        N.frt_fp8_gemm_noalloc(At.data_ptr(), Bt.data_ptr(), C.data_ptr(), M, Nn, K, 0.5, stream)
        ref = plan.gemm(At, Bt, alpha=0.5)
        torch.cuda.synchronize()
        got = C.cpu().numpy()
        want = ref.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert within_bound(got, want, A, B, K, 0.5)
        assert np.array_equal(got, want)
    plan.device_status()
    plan.close()


def test_no_alloc_gemm_rejects_shapes_beyond_its_scratch():
    from realtime_transformer_gb300 import _native as N
    dev = torch.device("cuda")
    M, Nn, K = 1000, 2048, 16384   # tiled path with split-K: more workspace than the fixed array
    A = torch.zeros((M, K), dtype=torch.uint8, device=dev)
    B = torch.zeros((Nn, K), dtype=torch.uint8, device=dev)
    C = torch.zeros((M, Nn), dtype=torch.float32, device=dev)
    with pytest.raises(N.FrtError) as ei:
        N.frt_fp8_gemm_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, Nn, K, 1.0,
                               torch.cuda.current_stream().cuda_stream)
    assert ei.value.name == "FRT_ERR_UNSUPPORTED"
    assert "scratch" in str(ei.value)
