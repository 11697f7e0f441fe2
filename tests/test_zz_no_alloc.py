"""The allocation-free FP8 GEMM entry point (frt_fp8_gemm_noalloc).

It exists for callers that cannot call cudaMalloc -- code running under a
global-mode stream capture, real-time hosts that forbid allocation after
start-up, hosts that own all device memory -- and keeps its split-K scratch
in a fixed device array instead.  Checked against the oracle's E4M3 GEMM,
not against the library's other entry points: bit for bit on exact-sum
inputs (every partial sum exact in fp32, so any summation order gives the
same bits), within the fp32 summation bound on random codes.  Each case runs
two calls in a row, the second reusing the scratch the first left behind,
and covers both exchanges of the split-K partials (inside a cluster, and
through the array's global workspace) and the tiled role.  This file is
collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def exact_sum_codes(rng, shape):
    # |v| < 1, multiples of 2^-5: products are multiples of 2^-10 below 1, so
    # sums over K <= 8192 stay within 23 significant bits (exact in fp32)
    e = rng.integers(5, 7, shape)
    m = rng.integers(0, 8, shape)
    s = rng.integers(0, 2, shape)
    return ((s << 7) | (e << 3) | m).astype(np.uint8)


def random_codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x7E
    return c


def within_bound(got, ref, A, B, K, alpha):
    a = oracle.e4m3_decode(A).astype(np.float64)
    b = oracle.e4m3_decode(B).astype(np.float64)
    bound = 2 * K * 2.0 ** -24 * (np.abs(a) @ np.abs(b).T) * abs(alpha) + 2 * 2.0 ** -24 * np.abs(ref)
    return np.all(np.abs(got.astype(np.float64) - ref.astype(np.float64)) <= bound)


def noalloc(A, B, alpha):
    from realtime_transformer_gb300 import _native as N
    dev = torch.device("cuda")
    M, K = A.shape
    Nn = B.shape[0]
    At = torch.from_numpy(A).to(dev)
    Bt = torch.from_numpy(B).to(dev)
    C = torch.full((M, Nn), float("nan"), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    N.frt_fp8_gemm_noalloc(At.data_ptr(), Bt.data_ptr(), C.data_ptr(), M, Nn, K, alpha, stream)
    N.frt_fp8_gemm_noalloc_status(stream)
    return C.cpu().numpy()


# (M, N, K, FRT_FFN_CLUSTER): weight-streaming with cluster split-K; the same
# through the array's global workspace; the tiled role with 16 splits through
# the global workspace (one 128 x 256 tile); unsplit weight streaming
CASES = [(50, 1024, 4096, None), (50, 1024, 4096, "0"), (128, 256, 8192, None), (16, 2048, 1024, None)]


@pytest.mark.parametrize("M,Nn,K,cluster", CASES)
def test_no_alloc_gemm_matches_oracle_on_two_calls(monkeypatch, M, Nn, K, cluster):
    if cluster is None:
        monkeypatch.delenv("FRT_FFN_CLUSTER", raising=False)
    else:
        monkeypatch.setenv("FRT_FFN_CLUSTER", cluster)
    rng = np.random.default_rng(M * 131 + Nn + K)
    for make, alpha in ((exact_sum_codes, 1.0), (random_codes, 0.5)):
        A = make(rng, (M, K))
        B = make(rng, (Nn, K))
        ref = oracle.gemm_e4m3(A, B) * np.float32(alpha)
        for _ in range(2):
            got = noalloc(A, B, alpha)
            assert np.all(np.isfinite(got))
            if make is exact_sum_codes:
                bad = np.argwhere(got != ref)
                assert bad.size == 0, (bad[:5], got[tuple(bad[0])], ref[tuple(bad[0])])
            else:
                assert within_bound(got, ref, A, B, K, alpha)


def test_no_alloc_gemm_reports_a_timed_out_wait_then_computes_again():
    """A kernel that gives up a bounded wait leaves its error in the fixed
    array until the status call reports it; the next call is correct."""
    from realtime_transformer_gb300 import _native as N
    stream = torch.cuda.current_stream().cuda_stream
    with pytest.raises(N.FrtError) as ei:
        N.frt_fp8_gemm_noalloc_debug_stall(stream)
    assert ei.value.name == "FRT_ERR_DEVICE_TIMEOUT"
    N.frt_fp8_gemm_noalloc_status(stream)   # reported once, then clear
    rng = np.random.default_rng(7)
    A = exact_sum_codes(rng, (50, 4096))
    B = exact_sum_codes(rng, (1024, 4096))
    assert np.array_equal(noalloc(A, B, 1.0), oracle.gemm_e4m3(A, B))


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
