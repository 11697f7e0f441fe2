// frt_f4.cuh -- NVFP4 element arithmetic shared by the NVFP4 kernels and the
// tensor-core GEMM's NVFP4 epilogues (itsolotime FlashRT article, 7.2: the
// NVFP4 encoder FFN).  Format as NVIDIA publishes it: E2M1 elements packed
// two per byte (element 2i in the low nibble), one E4M3 scale per 16
// consecutive elements along K, one fp32 tensor scale s (amax / (448 * 6)).
// A block of 16 is quantised with fp32 operations, each rounded on its own:
//   b = E4M3(amax_block * inv6)          inv6 = 1 / (6 s), from the host
//   q = E2M1(x * (1 / (dec(b) * s)))     0 where dec(b) == 0
// (round to nearest even, saturating: cvt.rn.satfinite), and decoded as
// (dec(q) * dec(b)) * s.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>
#include <cstring>

namespace frt {
namespace {

// E4M3 code of a non-negative block scale -> fp32 (exact): 2^(e-7) (1 + m/8),
// subnormals m 2^-9.
__device__ __forceinline__ float e4m3_dec(uint32_t c) {
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    return e == 0 ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}
// E2M1 code -> fp32 (exact): sign bit 3, 2^(e-1) (1 + m/2), subnormal m/2.
__device__ __forceinline__ float e2m1_dec(uint32_t c) {
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    const float v = e == 0 ? 0.5f * (float)m : __uint_as_float(((e + 126u) << 23) | (m << 22));
    return (c & 8u) ? -v : v;
}
// Eight fp32 values -> eight E2M1 codes in a 32-bit word, element 0 in the
// lowest nibble.
__device__ __forceinline__ uint32_t e2m1x8(const float *f) {
    uint32_t v;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(v)
        : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]));
    return v;
}

// One block of 16 values: returns the scale code, writes the 16 packed codes.
__device__ __forceinline__ uint32_t quant_block16(const float *v, float s, float inv6, uint2 &q) {
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
        amax = fmaxf(amax, fabsf(v[j]));
    const uint32_t b = (uint32_t)__nv_cvt_float_to_fp8(__fmul_rn(amax, inv6), __NV_SATFINITE, __NV_E4M3);
    const float den = __fmul_rn(e4m3_dec(b), s);
    const float inv = den > 0.0f ? __frcp_rn(den) : 0.0f;
    float t[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        t[j] = __fmul_rn(v[j], inv);
    q.x = e2m1x8(t);
    q.y = e2m1x8(t + 8);
    return b;
}

// Byte offset of the scale of (row, 16-element group g) of an operand with
// K elements per row in the TMEM-ready layout: per 128-row tile and 64-element
// K chunk a 512-byte block (tiles major, chunks minor), byte
// (r % 32) * 16 + (r / 32) * 4 + j holding row r of the tile, group j of the
// chunk: lane l of each TMEM lane quarter holds the block's 16 bytes at
// 16 l (rows l, l + 32, l + 64, l + 96 in its 4 columns), the replicated
// order in which a kind::mxf4nvf4 MMA with scale_vec::4X reads the scales of
// its 128 rows.
__device__ __forceinline__ size_t sf_offset(int row, int g, int K) {
    const int r = row & 127;
    return ((size_t)(row >> 7) * (size_t)(K >> 6) + (size_t)(g >> 2)) * 512u + (size_t)((r & 31) * 16 + (r >> 5) * 4 +
                                                                                        (g & 3));
}

// The 16 values of a block: (dec(q_j) * dec(b)) * s.  dec(q_j) * dec(b) is
// formed in f16 pairs: an E2M1 value (2 significant bits, 0.5 .. 6) times an
// E4M3 scale (4 significant bits, 2^-9 .. 448) has at most 6 significant bits
// and lies in [2^-10, 2688] (or is 0), so the f16 product is exact and equals
// the fp32 one; only the multiplication by s rounds.
__device__ __forceinline__ void dequant_block16(uint2 q, uint32_t b, float s, float *out) {
    const __half sbh = __float2half_rn(e4m3_dec(b));  // exact: E4M3 values are f16 values
    const __half2 sb2 = __halves2half2(sbh, sbh);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t w = i < 4 ? q.x : q.y;
        const uint32_t byte = (w >> (8 * (i & 3))) & 0xFFu;  // elements 2i (low nibble) and 2i + 1
        uint32_t h2;
        asm("{\n\t.reg .b8 c;\n\tcvt.u8.u32 c, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, c;\n\t}" : "=r"(h2) : "r"(byte));
        __half2 v;
        memcpy(&v, &h2, 4);
        v = __hmul2(v, sb2);
        out[2 * i] = __fmul_rn(__low2float(v), s);
        out[2 * i + 1] = __fmul_rn(__high2float(v), s);
    }
}

}  // namespace
}  // namespace frt
