"""FP8 GEMM kernels (tcgen05, both operand roles, split-K) against the oracle's
E4M3 GEMM: bit-exact on exact-sum inputs, within the fp32 summation bound on
random codes.  (Contraction of steps A2/A4: itsolotime FlashRT article, 7.2.)"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def plan():
    from realtime_transformer_gb300.ffn import FFNPlan
    p = FFNPlan(256, 1024, "geglu_tanh", 64, 1)
    yield p
    p.device_status()
    p.close()


def exact_sum_codes(rng, shape):
    e = rng.integers(5, 9, shape)
    m = rng.integers(0, 8, shape)
    s = rng.integers(0, 2, shape)
    return ((s << 7) | (e << 3) | m).astype(np.uint8)


def run(plan, A, B, path, splits, alpha=1.0):
    dev = torch.device("cuda")
    C = plan.gemm(torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev), alpha=alpha, path=path, splits=splits)
    torch.cuda.synchronize()
    plan.device_status()
    return C.cpu().numpy()


# (M, N, K, path, splits): path 1 = weight-streaming (M <= 64), 2 = tiled
CASES = [
    (1, 128, 128, 1, 1), (8, 256, 64, 1, 1), (16, 128, 256, 1, 2), (17, 384, 384, 1, 3), (50, 512, 1024, 1, 0),
    (64, 1024, 512, 1, 4), (33, 128, 16, 1, 1),
    (128, 256, 128, 2, 1), (1, 256, 256, 2, 1), (200, 512, 256, 2, 2), (300, 384, 640, 2, 0),
    (1000, 256, 1024, 2, 1), (129, 128, 48, 2, 1), (64, 1024, 384, 2, 3),
]


@pytest.mark.parametrize("M,N,K,path,splits", CASES)
def test_exact_sum_inputs_are_bit_exact(plan, M, N, K, path, splits):
    rng = np.random.default_rng(M * 7919 + N * 31 + K)
    A = exact_sum_codes(rng, (M, K))
    B = exact_sum_codes(rng, (N, K))
    got = run(plan, A, B, path, splits)
    ref = oracle.gemm_e4m3(A, B)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])], ref[tuple(bad[0])])


@pytest.mark.parametrize("M,N,K,path,splits", [(50, 1024, 1024, 1, 0), (7, 256, 4096, 1, 8), (300, 512, 2048, 2, 0),
                                               (256, 256, 5120, 2, 3),
                                               # weight-streaming with idle SMs / a ragged second wave of tiles
                                               (8, 2176, 13824, 1, 0), (4, 20480, 1536, 1, 0), (1, 7168, 5120, 1, 0)])
def test_random_codes_within_summation_bound(plan, M, N, K, path, splits):
    rng = np.random.default_rng(K + M)
    A = rng.integers(0, 256, (M, K)).astype(np.uint8)
    B = rng.integers(0, 256, (N, K)).astype(np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x7E
    B[(B & 0x7F) == 0x7F] = 0x7E
    alpha = 0.37
    got = run(plan, A, B, path, splits, alpha).astype(np.float64)
    ref = oracle.gemm_e4m3(A, B).astype(np.float64) * np.float32(alpha)
    a = oracle.e4m3_decode(A).astype(np.float64)
    b = oracle.e4m3_decode(B).astype(np.float64)
    bound = 2 * K * 2.0 ** -24 * (np.abs(a) @ np.abs(b).T) * alpha + 2 * 2.0 ** -24 * np.abs(ref)
    assert np.all(np.abs(got - ref) <= bound)


def test_split_k_is_deterministic(plan):
    rng = np.random.default_rng(5)
    A = rng.integers(0, 0x7E, (40, 2048)).astype(np.uint8)
    B = rng.integers(0, 0x7E, (512, 2048)).astype(np.uint8)
    c1 = run(plan, A, B, 1, 8)
    c2 = run(plan, A, B, 1, 8)
    assert np.array_equal(c1, c2)


@pytest.mark.parametrize("M,N,K,splits", [(40, 512, 2048, 2), (50, 1024, 4096, 8), (1, 640, 1536, 3), (17, 256, 1024, 5)])
def test_cluster_and_global_split_k_agree_bitwise(plan, monkeypatch, M, N, K, splits):
    """The two split-K exchanges (distributed shared memory inside a cluster,
    or a global workspace) reduce the same partials in the same order."""
    rng = np.random.default_rng(M + N + K)
    A = rng.integers(0, 0x7E, (M, K)).astype(np.uint8)
    B = rng.integers(0, 0x7E, (N, K)).astype(np.uint8)
    monkeypatch.delenv("FRT_FFN_CLUSTER", raising=False)
    c_cluster = run(plan, A, B, 1, splits)
    monkeypatch.setenv("FRT_FFN_CLUSTER", "0")
    c_global = run(plan, A, B, 1, splits)
    assert np.array_equal(c_cluster, c_global)


@pytest.mark.parametrize("M,N,K,splits", [(256, 256, 512, 1), (512, 512, 1024, 1), (1000, 768, 2048, 1),
                                          (1000, 512, 4096, 2), (256, 768, 2048, 0)])
def test_cta_pair_matches_single_cta(plan, monkeypatch, M, N, K, splits):
    """Tiled role on CTA pairs (cta_group::2 MMAs over 256 token rows, each
    CTA staging half of the weight tile) gives the same bits as one CTA per
    128-token tile."""
    rng = np.random.default_rng(M + 5 * N + K)
    A = rng.integers(0, 0x7E, (M, K)).astype(np.uint8)
    B = rng.integers(0, 0x7E, (N, K)).astype(np.uint8)
    monkeypatch.setenv("FRT_FFN_PAIR", "0")
    c_single = run(plan, A, B, 2, splits)
    monkeypatch.delenv("FRT_FFN_PAIR", raising=False)
    c_pair = run(plan, A, B, 2, splits)
    assert np.array_equal(c_single, c_pair)


@pytest.mark.parametrize("M,N,K,splits", [(512, 1024, 1024, 1), (768, 2048, 512, 0), (256, 768, 4096, 2)])
@pytest.mark.parametrize("policy", ["normal", "last"])
def test_weight_l2_priority_leaves_the_bits(plan, monkeypatch, M, N, K, splits, policy):
    """The weight tiles' L2 priority (a tuning switch of the tiled role) only
    changes what stays in L2, never the result."""
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    A = rng.integers(0, 0x7E, (M, K)).astype(np.uint8)
    B = rng.integers(0, 0x7E, (N, K)).astype(np.uint8)
    monkeypatch.delenv("FRT_FFN_W_EVICT", raising=False)
    c0 = run(plan, A, B, 2, splits)
    monkeypatch.setenv("FRT_FFN_W_EVICT", policy)
    assert np.array_equal(c0, run(plan, A, B, 2, splits))


def test_large_tiled_gemm_matches_the_oracle_on_sampled_rows():
    """8192 x 8192 x 8192 (token groups of the raster, CTA pairs, 8 waves):
    sampled rows against the oracle (exact-sum inputs: bit for bit)."""
    from realtime_transformer_gb300.ffn import FFNPlan
    p = FFNPlan(256, 1024, "geglu_tanh", 64, 1)
    try:
        rng = np.random.default_rng(8192)
        M = N = K = 8192
        e = rng.integers(5, 7, (M, K))      # |v| < 1, multiples of 2^-5: sums over 8192 stay exact in fp32
        A = ((rng.integers(0, 2, (M, K)) << 7) | (e << 3) | rng.integers(0, 8, (M, K))).astype(np.uint8)
        e = rng.integers(5, 7, (N, K))
        B = ((rng.integers(0, 2, (N, K)) << 7) | (e << 3) | rng.integers(0, 8, (N, K))).astype(np.uint8)
        dev = torch.device("cuda")
        C = p.gemm(torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev), path=2)
        torch.cuda.synchronize()
        p.device_status()
        rows = np.array([0, 1, 127, 128, 4095, 4096, 8190, 8191])
        got = C.index_select(0, torch.from_numpy(rows).to(dev)).cpu().numpy()
        assert np.array_equal(got, oracle.gemm_e4m3(A[rows], B))
    finally:
        p.close()
