"""Pins of the oracle's E4M3 x E4M3 -> fp32 GEMM (steps A2/A4 core: the FP8
gate/up and down GEMMs of the itsolotime FlashRT article, 7.2 "NVFP4 path"
pseudocode, and the FP8 GEMM of the agentlenshq summary, "Main ideas")."""
import numpy as np


def exact_sum_codes(rng, shape):
    """E4M3 codes whose values are multiples of 2^-5 with 2^-2 <= |v| < 4:
    exponent fields 5..8, any mantissa, any sign."""
    e = rng.integers(5, 9, shape)
    m = rng.integers(0, 8, shape)
    s = rng.integers(0, 2, shape)
    return ((s << 7) | (e << 3) | m).astype(np.uint8)


def exact_int_values(codes):
    """Values of exact-sum codes times 2^5, as int64, from the definition."""
    c = codes.astype(np.int64)
    e = (c >> 3) & 0xF
    m = c & 7
    mag = (8 + m) << (e - 5)          # (1 + m/8) 2^(e-7) * 2^5 = (8+m) 2^(e-5)
    return np.where(c & 0x80, -mag, mag) // 1


def test_exact_sum_brute_force(orc):
    """Products are multiples of 2^-10 below 16; sums of K <= 64 stay below
    2^10, so every partial sum is exact in fp32 and the oracle must equal the
    integer sum bit for bit.  Shapes are all distinct so a transposed operand
    cannot pass."""
    rng = np.random.default_rng(0)
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (8, 16, 32), (13, 29, 64), (64, 48, 64)]:
        A = exact_sum_codes(rng, (M, K))
        B = exact_sum_codes(rng, (N, K))
        acc = orc.gemm_e4m3(A, B)
        ai = exact_int_values(A)
        bi = exact_int_values(B)
        exact = ai @ bi.T                      # int64, units of 2^-10
        assert np.array_equal(acc.astype(np.float64) * 1024.0, exact.astype(np.float64)), (M, N, K)


def test_random_codes_within_fp32_summation_bound(orc):
    """Full code range (subnormals included, NaN excluded): the fp32 result is
    within K * 2^-24 * sum|p| of the fp64 dot product of the decoded values."""
    rng = np.random.default_rng(1)
    M, N, K = 17, 23, 300
    A = rng.integers(0, 256, (M, K)).astype(np.uint8)
    B = rng.integers(0, 256, (N, K)).astype(np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x7E
    B[(B & 0x7F) == 0x7F] = 0x7E
    acc = orc.gemm_e4m3(A, B).astype(np.float64)
    a = orc.e4m3_decode(A).astype(np.float64)
    b = orc.e4m3_decode(B).astype(np.float64)
    ref = a @ b.T
    bound = K * 2.0 ** -24 * (np.abs(a) @ np.abs(b).T)
    assert np.all(np.abs(acc - ref) <= bound)


def test_operand_roles(orc):
    """acc[m][n] pairs row m of A with row n of B (both K-major)."""
    A = np.zeros((2, 4), np.uint8)
    B = np.zeros((3, 4), np.uint8)
    A[1, 2] = 0x38   # 1.0
    B[2, 2] = 0x40   # 2.0
    acc = orc.gemm_e4m3(A, B)
    expect = np.zeros((2, 3), np.float32)
    expect[1, 2] = 2.0
    assert np.array_equal(acc, expect)
