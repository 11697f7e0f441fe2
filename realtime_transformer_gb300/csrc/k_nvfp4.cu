// k_nvfp4.cu -- the NVFP4 variant of the FFN sublayer on sm_103a (itsolotime
// FlashRT article, 7.2: gate and up as two NVFP4 GEMMs that emit packed FP4
// plus scales, a fused GeGLU kernel that requantises FP4 to FP4, an NVFP4
// down GEMM, the residual stream kept in 16 bits, AWQ pre-scaling of the
// normalised activation).
//
// Format (NVFP4 as NVIDIA publishes it): E2M1 elements packed two per byte
// (element 2i in the low nibble), one E4M3 scale per 16 consecutive elements
// along K, one fp32 scale s per tensor (amax / (448 * 6)).  A block of 16 is
// quantised with fp32 operations, each rounded on its own:
//   b = E4M3(amax_block * inv6)          inv6 = 1 / (6 s), from the host
//   q = E2M1(x * (1 / (dec(b) * s)))     0 where dec(b) == 0
// (round to nearest even, saturating: cvt.rn.satfinite).
//
// Block scales of a GEMM operand live in global memory in the order the
// tensor cores read them from TMEM: for every 128-row tile and 64-element K
// chunk one 512-byte block, byte (r % 32) * 16 + (r / 32) * 4 + j holding
// row r of the tile, 16-element group j of the chunk (tiles major, chunks
// minor).  One tcgen05.cp of shape 32x128b with warpx4 replication moves a
// block into four TMEM columns of every lane quarter, which is where a
// kind::mxf4nvf4 MMA with scale_vec::4X reads the scales of its 128 rows.
//
// GEMM: one output tile per CTA (128 x 128 tiled; 128 weight rows x <= 64
// tokens in the weight-streaming role), 192 threads -- warp 4 the producer
// (operand tiles of 256 elements along K: activations by 128B-swizzled TMA,
// weights by one bulk copy of their pre-swizzled tile, plus the two 2 KB
// scale blocks of the stage), warp 5 the MMA issuer (per stage eight
// tcgen05.cp and four MMAs of K = 64), warps 0..3 the epilogue (one TMEM lane
// per thread), with deterministic split-K for few tiles.  Every wait is
// bounded; on a timeout the CTA drains and exits with the error word set.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "frt_internal.h"
#include "frt_ptx.cuh"

namespace frt {

namespace {

constexpr int F4_BM = 128;             // MMA M: output rows of a CTA = TMEM lanes
constexpr int F4_BN = 128;             // MMA N: output columns of a CTA
constexpr int F4_BKB = 128;            // K bytes per stage (256 elements): one swizzle row
constexpr int F4_UKB = 32;             // K bytes of one MMA (64 elements)
constexpr int F4_TILE = F4_BM * F4_BKB;            // bytes of one operand tile per stage
constexpr int F4_SF_STAGE = 4 * 512;               // scale bytes of one operand per stage

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ void unpack8(const uint4 v, float *f) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
    f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
    f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}
__device__ __forceinline__ uint32_t bf16_bits(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

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
// K elements per row, in the TMEM-ready layout described above.
__device__ __forceinline__ size_t sf_offset(int row, int g, int K) {
    const int r = row & 127;
    return ((size_t)(row >> 7) * (size_t)(K >> 6) + (size_t)(g >> 2)) * 512u + (size_t)((r & 31) * 16 + (r >> 5) * 4 +
                                                                                        (g & 3));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// GELU (tanh form) and SiLU in fp32 with the library's tanhf / expf.
__device__ __forceinline__ float act_f32(int act, float g) {
    if (act == ACT_SWIGLU)
        return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
    const float g3 = __fmul_rn(__fmul_rn(g, g), g);
    const float inner = __fmul_rn(0.7978845608028654f, __fadd_rn(g, __fmul_rn(0.044715f, g3)));
    return __fmul_rn(__fmul_rn(0.5f, g), __fadd_rn(1.0f, tanhf(inner)));
}

// ------------------------------------------------------------ weights --

// amax of W[j][k] * c[k] (c null: of W) over a BF16 [rows, K] matrix.
__global__ void k_f4_amax_w(const uint4 *__restrict__ w, size_t rows, int K, const float *__restrict__ col,
                            unsigned *amax_word) {
    const size_t vpr = (size_t)K / 8, n = rows * vpr;
    float m = 0.0f;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        float f[8];
        unpack8(__ldg(w + i), f);
        const size_t k0 = (i % vpr) * 8;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            m = fmaxf(m, fabsf(col ? __fmul_rn(f[j], __ldg(col + k0 + j)) : f[j]));
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0)
        atomicMax(amax_word, __float_as_uint(m));
}

// Byte offset of the 8 codes of (row, 16-element group g) in the tiled weight
// layout: per 128-row tile and 256-element stage one 16 KB block holding the
// shared-memory image a 128-byte-swizzled TMA load of that box would write
// (row r at r * 128, its 16-byte chunk c at chunk c ^ (r % 8)); tiles major,
// stages minor.
__device__ __forceinline__ size_t w_tile_offset(int row, int g, int K) {
    const int r = row & 127, kbyte = g * 8, c = (kbyte & 127) >> 4;
    return ((size_t)(row >> 7) * (size_t)(K / 256) + (size_t)(kbyte >> 7)) * F4_TILE + (size_t)(r * 128) +
           (size_t)(((c ^ (r & 7)) << 4) | (kbyte & 15));
}

// NVFP4 codes and TMEM-ready scales of W (times c) with tensor scale s; codes
// row-major [rows, K/2] or, with tiled, in the tiled weight layout.
__global__ void k_f4_quant_w(const uint4 *__restrict__ w, int rows, int K, const float *__restrict__ col, float s,
                             float inv6, uint2 *__restrict__ q, uint8_t *__restrict__ sf, int tiled) {
    const int gpr = K / 16;
    const size_t n = (size_t)rows * gpr;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int row = (int)(i / gpr), g = (int)(i % gpr);
        float f[16];
        unpack8(__ldg(w + 2 * i), f);
        unpack8(__ldg(w + 2 * i + 1), f + 8);
        if (col) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                f[j] = __fmul_rn(f[j], __ldg(col + g * 16 + j));
        }
        uint2 c;
        const uint32_t b = quant_block16(f, s, inv6, c);
        if (tiled)
            *reinterpret_cast<uint2 *>(reinterpret_cast<uint8_t *>(q) + w_tile_offset(row, g, K)) = c;
        else
            q[i] = c;
        sf[sf_offset(row, g, K)] = (uint8_t)b;
    }
}

// ------------------------------------------- residual + norm + quantise --

// WPR warps per row (1, 2, 4 or 8), 8 / WPR rows per CTA; a thread takes
// blocks of 16 elements strided by 32 WPR.  Pass 1: r' = bf16(r + h) (stored
// if rprime), the sum of squares (per thread, a warp-shuffle tree, then the
// row's warps in order); pass 2: y = ((r' * inv) * w) [* awq_inv], then the
// amax (MEASURE) or the NVFP4 codes and TMEM-ready scales of y.
template <bool MEASURE, int WPR>
__global__ void __launch_bounds__(256) k_f4_norm_quant(const uint16_t *__restrict__ r, const uint16_t *__restrict__ h,
                                                       const uint16_t *__restrict__ w,
                                                       const float *__restrict__ awq_inv, int M, int d, float eps,
                                                       float s, float inv6, uint16_t *__restrict__ rprime,
                                                       uint8_t *__restrict__ q, uint8_t *__restrict__ sf,
                                                       unsigned *amax_word) {
    __shared__ float s_part[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tid = (warp % WPR) * 32 + lane;
    const int row = blockIdx.x * (8 / WPR) + warp / WPR;
    const bool active = row < M;
    const int ng = active ? d / 16 : 0;
    const uint4 *rv = reinterpret_cast<const uint4 *>(r + (size_t)(active ? row : 0) * d);
    const uint4 *hv = h ? reinterpret_cast<const uint4 *>(h + (size_t)(active ? row : 0) * d) : nullptr;
    const uint4 *wv = reinterpret_cast<const uint4 *>(w);
    float ss = 0.0f;
    for (int g = tid; g < ng; g += 32 * WPR) {
        float x[16];
        unpack8(rv[2 * g], x);
        unpack8(rv[2 * g + 1], x + 8);
        if (hv) {
            float hh[16];
            unpack8(hv[2 * g], hh);
            unpack8(hv[2 * g + 1], hh + 8);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                x[j] = round_bf16(__fadd_rn(x[j], hh[j]));
            if (rprime) {
                uint4 *o = reinterpret_cast<uint4 *>(rprime + (size_t)row * d) + 2 * g;
                o[0] = make_uint4(bf16_bits(x[0]) | (bf16_bits(x[1]) << 16), bf16_bits(x[2]) | (bf16_bits(x[3]) << 16),
                                  bf16_bits(x[4]) | (bf16_bits(x[5]) << 16), bf16_bits(x[6]) | (bf16_bits(x[7]) << 16));
                o[1] = make_uint4(bf16_bits(x[8]) | (bf16_bits(x[9]) << 16),
                                  bf16_bits(x[10]) | (bf16_bits(x[11]) << 16),
                                  bf16_bits(x[12]) | (bf16_bits(x[13]) << 16),
                                  bf16_bits(x[14]) | (bf16_bits(x[15]) << 16));
            }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)
            ss = __fadd_rn(ss, __fmul_rn(x[j], x[j]));
    }
    ss = warp_sum(ss);
    if (WPR > 1) {
        if (lane == 0)
            s_part[warp] = ss;
        __syncthreads();
        const int w0 = (warp / WPR) * WPR;
        ss = 0.0f;
        for (int k = 0; k < WPR; ++k)
            ss = __fadd_rn(ss, s_part[w0 + k]);
    }
    if (!active)
        return;
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)d), eps)));
    float amax = 0.0f;
    for (int g = tid; g < ng; g += 32 * WPR) {
        float x[16], wf[16];
        unpack8(rv[2 * g], x);
        unpack8(rv[2 * g + 1], x + 8);
        if (hv) {
            float hh[16];
            unpack8(hv[2 * g], hh);
            unpack8(hv[2 * g + 1], hh + 8);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                x[j] = round_bf16(__fadd_rn(x[j], hh[j]));
        }
        unpack8(__ldg(wv + 2 * g), wf);
        unpack8(__ldg(wv + 2 * g + 1), wf + 8);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            x[j] = __fmul_rn(__fmul_rn(x[j], inv), wf[j]);
            if (awq_inv)
                x[j] = __fmul_rn(x[j], __ldg(awq_inv + g * 16 + j));
        }
        if (MEASURE) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                amax = fmaxf(amax, fabsf(x[j]));
        } else {
            uint2 c;
            const uint32_t b = quant_block16(x, s, inv6, c);
            reinterpret_cast<uint2 *>(q + (size_t)row * (d / 2))[g] = c;
            sf[sf_offset(row, g, d)] = (uint8_t)b;
        }
    }
    if (MEASURE) {
        amax = warp_max(amax);
        if (lane == 0)
            atomicMax(amax_word, __float_as_uint(amax));
    }
}

// ------------------------------------------------ GeGLU FP4 -> FP4 --

// E2M1 code of one fp32 value (low nibble of a pair conversion with 0).
__device__ __forceinline__ uint32_t e2m1_one(float x) {
    uint32_t v;
    asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %2, %1;\n\tcvt.u32.u8 %0, b;\n\t}"
        : "=r"(v)
        : "f"(x), "f"(0.0f));
    return v & 15u;
}

// a = act(dec G) * dec U per element, then the amax (MEASURE) or the NVFP4
// codes and TMEM-ready scales of a.  G and U: codes [M, ff/2], row-major
// block scales [M, ff/16], tensor scales s_g, s_u.  One thread per element,
// a block of 16 on 16 lanes: its amax by shuffles, the codes of lane pairs
// combined into bytes.  The element count M ff is a multiple of 16, so a
// half-warp is a whole block or wholly past the end.
// One thread per block of 16 (many blocks: enough threads to fill the GPU).
template <bool MEASURE>
__global__ void k_f4_geglu_blk(const uint8_t *__restrict__ gq, const uint8_t *__restrict__ gs, float s_g,
                               const uint8_t *__restrict__ uq, const uint8_t *__restrict__ us, float s_u, int act,
                               int M, int ff, float s_h, float inv6, uint8_t *__restrict__ hq,
                               uint8_t *__restrict__ hsf, unsigned *amax_word) {
    const int gpr = ff / 16;
    const size_t n = (size_t)M * gpr;
    float amax = 0.0f;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int m = (int)(i / gpr), g = (int)(i % gpr);
        const uint2 gc = reinterpret_cast<const uint2 *>(gq)[i];
        const uint2 uc = reinterpret_cast<const uint2 *>(uq)[i];
        const float gb = e4m3_dec(gs[i]), ub = e4m3_dec(us[i]);
        float a[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint32_t gw = j < 8 ? gc.x : gc.y, uw = j < 8 ? uc.x : uc.y;
            const int sh = 4 * (j & 7);
            const float gv = __fmul_rn(__fmul_rn(e2m1_dec((gw >> sh) & 15u), gb), s_g);
            const float uv = __fmul_rn(__fmul_rn(e2m1_dec((uw >> sh) & 15u), ub), s_u);
            a[j] = __fmul_rn(act_f32(act, gv), uv);
        }
        if (MEASURE) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                amax = fmaxf(amax, fabsf(a[j]));
        } else {
            uint2 c;
            const uint32_t b = quant_block16(a, s_h, inv6, c);
            reinterpret_cast<uint2 *>(hq)[i] = c;
            hsf[sf_offset(m, g, ff)] = (uint8_t)b;
        }
    }
    if (MEASURE) {
        amax = warp_max(amax);
        if ((threadIdx.x & 31) == 0)
            atomicMax(amax_word, __float_as_uint(amax));
    }
}

// One thread per element (few blocks: sixteen times the parallelism).
template <bool MEASURE>
__global__ void k_f4_geglu(const uint8_t *__restrict__ gq, const uint8_t *__restrict__ gs, float s_g,
                           const uint8_t *__restrict__ uq, const uint8_t *__restrict__ us, float s_u, int act, int M,
                           int ff, float s_h, float inv6, uint8_t *__restrict__ hq, uint8_t *__restrict__ hsf,
                           unsigned *amax_word) {
    const int lane = threadIdx.x & 31;
    const int gpr = ff / 16;
    const size_t total = (size_t)M * ff;
    const size_t step = (size_t)gridDim.x * blockDim.x;
    float amax_all = 0.0f;
    for (size_t base = (size_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31u); base < total; base += step) {
        const size_t e = base + lane;
        const bool valid = e < total;
        const size_t i = valid ? e / 16 : 0;  // block index
        const int j = lane & 15;
        float a = 0.0f;
        if (valid) {
            const uint32_t gb = gq[e / 2], ub = uq[e / 2];
            const uint32_t gc = (j & 1) ? gb >> 4 : gb & 15u, uc = (j & 1) ? ub >> 4 : ub & 15u;
            const float gv = __fmul_rn(__fmul_rn(e2m1_dec(gc), e4m3_dec(gs[i])), s_g);
            const float uv = __fmul_rn(__fmul_rn(e2m1_dec(uc), e4m3_dec(us[i])), s_u);
            a = __fmul_rn(act_f32(act, gv), uv);
        }
        if (MEASURE) {
            amax_all = fmaxf(amax_all, fabsf(a));
            continue;
        }
        float m = fabsf(a);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const uint32_t b = (uint32_t)__nv_cvt_float_to_fp8(__fmul_rn(m, inv6), __NV_SATFINITE, __NV_E4M3);
        const float den = __fmul_rn(e4m3_dec(b), s_h);
        const float inv = den > 0.0f ? __frcp_rn(den) : 0.0f;
        const uint32_t c = e2m1_one(__fmul_rn(a, inv));
        const uint32_t hi = __shfl_xor_sync(0xffffffffu, c, 1);
        if (valid && !(j & 1))
            hq[e / 2] = (uint8_t)(c | (hi << 4));
        if (valid && j == 0) {
            const int row = (int)(i / gpr), g = (int)(i % gpr);
            hsf[sf_offset(row, g, ff)] = (uint8_t)b;
        }
    }
    if (MEASURE) {
        amax_all = warp_max(amax_all);
        if (lane == 0)
            atomicMax(amax_word, __float_as_uint(amax_all));
    }
}

// ----------------------------------------------------------------- GEMM --

// Shared-memory descriptor of a 512-byte scale block: 32 rows of 16 bytes,
// no swizzle, 8-row core matrices 128 bytes apart (leading and stride byte
// offsets both 128, so either reading of the 16-byte-wide block agrees).
__device__ __forceinline__ uint64_t smem_desc_sf(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D[tmem] (+)= (A * scale_A) (B * scale_B)^T, E2M1 operands with E4M3 scales
// per 16 elements, K = 64.
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of the block-scaled kinds: A and B E2M1 (format 1),
// both K-major, N >> 3 at bit 17, scale format UE4M3 (bit 23 clear), M >> 4
// at bit 24, scale-factor ids 0.
__host__ __device__ constexpr uint32_t idesc_nvf4(int m, int n) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// The epilogue of 16 consecutive output columns n.. of one row, v = acc * alpha.
template <int EPI>
__device__ __forceinline__ void epi_chunk(const F4GemmParams &p, int row, int n, const float *v, float &amax) {
    if constexpr (EPI == F4_EPI_F32) {
        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + (size_t)row * p.ldo + n);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    } else if constexpr (EPI == F4_EPI_AMAX) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            amax = fmaxf(amax, fabsf(v[j]));
    } else if constexpr (EPI == F4_EPI_FP4) {
        uint2 c2;
        const uint32_t b = quant_block16(v, p.s_out, p.inv6_out, c2);
        *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(p.out) + (size_t)row * p.ldo + n / 2) = c2;
        p.out_sf[(size_t)row * p.ldsf + n / 16] = (uint8_t)b;
    } else {  // F4_EPI_RESID: out = bf16(r' + acc * alpha)
        const uint4 *rr = reinterpret_cast<const uint4 *>(p.resid + (size_t)row * p.ldr + n);
        float x[16];
        unpack8(rr[0], x);
        unpack8(rr[1], x + 8);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            w[j] = bf16_bits(__fadd_rn(x[2 * j], v[2 * j])) | (bf16_bits(__fadd_rn(x[2 * j + 1], v[2 * j + 1])) << 16);
        uint4 *o = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + (size_t)row * p.ldo + n);
        o[0] = make_uint4(w[0], w[1], w[2], w[3]);
        o[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

// The epilogue of one feature f over 16 consecutive tokens t.. (weight-
// streaming role: a thread holds a feature, the lanes of a half-warp the 16
// features of one block), v = acc * alpha.  Every lane of the warp calls it.
template <int EPI>
__device__ __forceinline__ void epi_swap(const F4GemmParams &p, int f, int t, const float *v, float &amax) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int tok = t + j;
        const bool tv = tok < p.M;
        if constexpr (EPI == F4_EPI_F32) {
            if (tv)
                static_cast<float *>(p.out)[(size_t)tok * p.ldo + f] = v[j];
        } else if constexpr (EPI == F4_EPI_AMAX) {
            if (tv)
                amax = fmaxf(amax, fabsf(v[j]));
        } else if constexpr (EPI == F4_EPI_FP4) {
            float m = tv ? fabsf(v[j]) : 0.0f;
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            const uint32_t b = (uint32_t)__nv_cvt_float_to_fp8(__fmul_rn(m, p.inv6_out), __NV_SATFINITE, __NV_E4M3);
            const float den = __fmul_rn(e4m3_dec(b), p.s_out);
            const float inv = den > 0.0f ? __frcp_rn(den) : 0.0f;
            const uint32_t c = e2m1_one(__fmul_rn(v[j], inv));
            const uint32_t hi = __shfl_xor_sync(0xffffffffu, c, 1);
            if (tv && !(f & 1))
                static_cast<uint8_t *>(p.out)[(size_t)tok * p.ldo + f / 2] = (uint8_t)(c | (hi << 4));
            if (tv && !(f & 15))
                p.out_sf[(size_t)tok * p.ldsf + f / 16] = (uint8_t)b;
        } else {  // F4_EPI_RESID
            if (tv) {
                const float x = __uint_as_float((uint32_t)p.resid[(size_t)tok * p.ldr + f] << 16);
                static_cast<uint16_t *>(p.out)[(size_t)tok * p.ldo + f] = (uint16_t)bf16_bits(__fadd_rn(x, v[j]));
            }
        }
    }
}

// One GEMM variant.  Tiled role (SWAP false): 128 token rows x 128 weight
// rows per CTA.  Weight-streaming role (SWAP true, at most 64 tokens): the
// 128 weight rows are the MMA's M operand and the tokens its N = BNT
// columns, so a stage carries 16 KB of weights and BNT x 128 bytes of
// activations, and more stages fit.
// The four MMAs of a stage rotate over NACC accumulators (summed in the
// epilogue, in order), so that consecutive MMAs do not wait on each other.
template <bool SWAP, int BNT>
struct F4Cfg {
    static constexpr int NS = SWAP ? (BNT == 16 ? 9 : BNT == 32 ? 8 : 7) : 4;
    static constexpr int NACC = SWAP ? 4 : 2;
    static constexpr int B_TILE = BNT * F4_BKB;
    static constexpr int SF_COL = NACC * BNT;  // first TMEM column of the scale blocks
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t SMEM = 1024 + NS * (F4_TILE + B_TILE + 2 * F4_SF_STAGE) + 256;
    static_assert(SF_COL + NS * 32 <= TMEM_COLS, "TMEM budget");
};

// 16 accumulator columns c*16.. of this warp's lanes: the sum over the NACC
// accumulators, ((a0 + a1) + a2) + a3.
template <int NACC, int BNT>
__device__ __forceinline__ void load_acc(uint32_t tbase, int c, float *v) {
    uint32_t raw[16];
    tmem_ld_x16(tbase + (uint32_t)(c * 16), raw);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j)
        v[j] = __uint_as_float(raw[j]);
#pragma unroll
    for (int a = 1; a < NACC; ++a) {
        tmem_ld_x16(tbase + (uint32_t)(a * BNT + c * 16), raw);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
            v[j] = __fadd_rn(v[j], __uint_as_float(raw[j]));
    }
}

// Sum of the split-K partials of 16 consecutive columns in split order
// (partials `stride` floats apart), four splits' loads in flight at a time.
__device__ __forceinline__ void sum_partials(const float *src0, size_t stride, int splits, float *v) {
    const float4 *src = reinterpret_cast<const float4 *>(src0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4 t = __ldcg(src + j);
        v[4 * j] = t.x; v[4 * j + 1] = t.y; v[4 * j + 2] = t.z; v[4 * j + 3] = t.w;
    }
#pragma unroll 1
    for (int k0 = 1; k0 < splits; k0 += 4) {
        float4 t[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                t[k][j] = k0 + k < splits ? __ldcg(src + (size_t)(k0 + k) * (stride / 4) + j)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (k0 + k >= splits)
                break;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[4 * j] = __fadd_rn(v[4 * j], t[k][j].x);
                v[4 * j + 1] = __fadd_rn(v[4 * j + 1], t[k][j].y);
                v[4 * j + 2] = __fadd_rn(v[4 * j + 2], t[k][j].z);
                v[4 * j + 3] = __fadd_rn(v[4 * j + 3], t[k][j].w);
            }
        }
    }
}

template <int EPI, bool SWAP, int BNT>
__global__ void __launch_bounds__(192, 1)
    k_gemm_nvfp4(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ F4GemmParams p) {
    using C = F4Cfg<SWAP, BNT>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_last;  // split-K: this CTA reduces the tile
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = sA + NS * F4_TILE;
    uint8_t *sSF = sB + NS * C::B_TILE;  // per stage: A scales (2 KB), then B scales (2 KB)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sSF + NS * 2 * F4_SF_STAGE);
    uint64_t *full = bars;
    uint64_t *empty = bars + NS;
    uint64_t *tfull = bars + 2 * NS;
    uint64_t *drain_bar = tfull + 1;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain_bar + 1);
    volatile int *abort_f = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the tile: 128 weight rows from f0; tokens from t0 (tiled: 128 of them)
    const int f0 = blockIdx.x * 128;
    const int t0 = SWAP ? 0 : blockIdx.y * F4_BM;
    // this CTA's split of the K stages
    const int KB = p.K / 256;
    const int z = blockIdx.z;
    const int kb0 = (int)((long)z * KB / p.splits), kb1 = (int)((long)(z + 1) * KB / p.splits);
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(tfull), 1);
        mbar_init(smem_u32(drain_bar), 1);
        *abort_f = 0;
        fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 4) {
        if (lane == 0) {
            // ---- producer: weights first out of L2, activations last
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_x = l2_policy_evict_last();
            const int a_row = p.a_row0 + (SWAP ? f0 : t0), b_row = p.b_row0 + (SWAP ? 0 : f0);
            const uint8_t *sfa = p.sfa + (size_t)((SWAP ? f0 : t0) / 128) * (size_t)(p.K / 64) * 512u;
            const uint8_t *sfb = p.sfb + (size_t)((SWAP ? 0 : f0) / 128) * (size_t)(p.K / 64) * 512u;
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_par = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_f, p.err)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&full[stage]);
                mbar_arrive_expect_tx(fb, (uint32_t)(F4_TILE + C::B_TILE + 2 * F4_SF_STAGE));
                issued |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                if (p.w_tiles) {
                    // weights stored in the stage's shared-memory image: one contiguous copy
                    const uint8_t *wt = p.w_tiles + ((size_t)(f0 / 128) * (size_t)KB + (size_t)kb) * F4_TILE;
                    if constexpr (SWAP) {
                        bulk_load(smem_u32(sA + stage * F4_TILE), wt, F4_TILE, fb);
                        tma_load_2d(smem_u32(sB + stage * C::B_TILE), &tmB, fb, kb * F4_BKB, b_row, pol_x);
                    } else {
                        tma_load_2d(smem_u32(sA + stage * F4_TILE), &tmA, fb, kb * F4_BKB, a_row, pol_x);
                        bulk_load(smem_u32(sB + stage * C::B_TILE), wt, F4_TILE, fb);
                    }
                } else {
                    tma_load_2d(smem_u32(sA + stage * F4_TILE), &tmA, fb, kb * F4_BKB, a_row, SWAP ? pol_w : pol_x);
                    tma_load_2d(smem_u32(sB + stage * C::B_TILE), &tmB, fb, kb * F4_BKB, b_row, SWAP ? pol_x : pol_w);
                }
                bulk_load(smem_u32(sSF + stage * 2 * F4_SF_STAGE), sfa + (size_t)kb * F4_SF_STAGE, F4_SF_STAGE, fb);
                bulk_load(smem_u32(sSF + stage * 2 * F4_SF_STAGE + F4_SF_STAGE), sfb + (size_t)kb * F4_SF_STAGE,
                          F4_SF_STAGE, fb);
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                for (int s = 0; s < NS; ++s)
                    if (issued & (1u << s))
                        mbar_wait_for(smem_u32(&full[s]), (issued_par >> s) & 1u, 100000000ull);
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0) {
            // ---- MMA issuer
            constexpr uint32_t idesc = idesc_nvf4(128, BNT);
            int stage = 0;
            uint32_t phase = 0;
            bool issued_any = false, ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(smem_u32(&full[stage]), phase, abort_f, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t t_sf = tmem_base + (uint32_t)(C::SF_COL + stage * 32);
                const uint32_t s_sf = smem_u32(sSF + stage * 2 * F4_SF_STAGE);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    tmem_cp_sf(t_sf + 4 * j, smem_desc_sf(s_sf + 512 * j));
                    tmem_cp_sf(t_sf + 16 + 4 * j, smem_desc_sf(s_sf + F4_SF_STAGE + 512 * j));
                }
                const uint32_t aA = smem_u32(sA + stage * F4_TILE), aB = smem_u32(sB + stage * C::B_TILE);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_nvf4(tmem_base + (uint32_t)((j % C::NACC) * BNT), smem_desc_k128(aA + j * F4_UKB),
                             smem_desc_k128(aB + j * F4_UKB), idesc, t_sf + 4 * j, t_sf + 16 + 4 * j,
                             (kb > kb0 || j >= C::NACC) ? 1u : 0u);
                issued_any = true;
                mma_commit(smem_u32(&empty[stage]));
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) {
                mma_commit(smem_u32(tfull));
            } else if (issued_any) {
                mma_commit(smem_u32(drain_bar));
                mbar_wait_for(smem_u32(drain_bar), 0, 100000000ull);
            }
        }
        __syncwarp();
    } else {
        // ---- epilogue: thread = TMEM lane r.  Tiled: token row t0 + r over
        // 128 feature columns; weight-streaming: feature f0 + r over BNT tokens.
        int ok = 0;
        if (lane == 0)
            ok = mbar_wait(smem_u32(tfull), 0, abort_f, p.err) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        const int r = warp * 32 + lane;
        constexpr int NCH = SWAP ? BNT / 16 : F4_BN / 16;  // 16-column chunks of the accumulator
        constexpr int ROWLEN = SWAP ? BNT : F4_BN;
        float amax = 0.0f;
        if (p.splits == 1) {
            if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < NCH; ++c) {
                    float v[16];
                    __syncwarp();
                    load_acc<C::NACC, BNT>(tmem_base + ((uint32_t)(warp * 32) << 16), c, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[j] = __fmul_rn(v[j], p.alpha);
                    if constexpr (SWAP)
                        epi_swap<EPI>(p, f0 + r, c * 16, v, amax);
                    else if (t0 + r < p.M)
                        epi_chunk<EPI>(p, t0 + r, f0 + c * 16, v, amax);
                }
            }
        } else {
            // Split-K: every split stores its fp32 partial tile; the last
            // split to arrive sums the partials in split order and runs the
            // epilogue, then re-arms the tile's counter.
            const int tile = blockIdx.y * gridDim.x + blockIdx.x;
            float *ws_t = p.ws + (size_t)tile * p.splits * (F4_BM * F4_BN);
            const bool keep = SWAP || t0 + r < p.M;
            if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < NCH; ++c) {
                    float v[16];
                    __syncwarp();
                    load_acc<C::NACC, BNT>(tmem_base + ((uint32_t)(warp * 32) << 16), c, v);
                    if (keep) {
                        float4 *o =
                            reinterpret_cast<float4 *>(ws_t + (size_t)z * (F4_BM * F4_BN) + r * ROWLEN + c * 16);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            o[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    }
                }
            }
            __threadfence();
            named_bar_sync(1, 128);
            if (threadIdx.x == 0)
                s_last = atomicAdd(p.counters + tile, 1) == p.splits - 1 ? 1 : 0;
            named_bar_sync(1, 128);
            if (s_last) {
                __threadfence();
                if constexpr (SWAP) {
                    // thread = feature (the FP4 epilogue's blocks span lanes)
#pragma unroll 1
                    for (int c = 0; c < NCH; ++c) {
                        float v[16];
                        sum_partials(ws_t + r * ROWLEN + c * 16, (size_t)F4_BM * F4_BN, p.splits, v);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            v[j] = __fmul_rn(v[j], p.alpha);
                        epi_swap<EPI>(p, f0 + r, c * 16, v, amax);
                    }
                } else {
                    // (row, 16-column chunk) items over the 128 threads
                    const int rows = min(F4_BM, p.M - t0);
#pragma unroll 1
                    for (int it = threadIdx.x; it < rows * NCH; it += 128) {
                        const int rr = it / NCH, c = it % NCH;
                        float v[16];
                        sum_partials(ws_t + rr * ROWLEN + c * 16, (size_t)F4_BM * F4_BN, p.splits, v);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            v[j] = __fmul_rn(v[j], p.alpha);
                        epi_chunk<EPI>(p, t0 + rr, f0 + c * 16, v, amax);
                    }
                }
                if (threadIdx.x == 0)
                    p.counters[tile] = 0;
            }
        }
        if constexpr (EPI == F4_EPI_AMAX) {
            amax = warp_max(amax);
            if (lane == 0)
                atomicMax(p.amax, __float_as_uint(amax));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) {
        __syncwarp();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

int grid_cap() {
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0)
            sms = 148;
    }
    return sms * 8;
}

unsigned blocks_for(size_t n, int threads) {
    size_t b = (n + threads - 1) / threads;
    const size_t cap = (size_t)grid_cap();
    if (b > cap)
        b = cap;
    return (unsigned)(b ? b : 1);
}

}  // namespace

cudaError_t launch_f4_amax_w(const void *w, size_t rows, int K, const float *col, unsigned *amax_word,
                             cudaStream_t s) {
    k_f4_amax_w<<<blocks_for(rows * (size_t)(K / 8), 256), 256, 0, s>>>(static_cast<const uint4 *>(w), rows, K, col,
                                                                          amax_word);
    return cudaGetLastError();
}

cudaError_t launch_f4_quant_w(const void *w, int rows, int K, const float *col, float sc, float inv6, uint8_t *q,
                              uint8_t *sf, bool tiled, cudaStream_t s) {
    k_f4_quant_w<<<blocks_for((size_t)rows * (K / 16), 256), 256, 0, s>>>(
        static_cast<const uint4 *>(w), rows, K, col, sc, inv6, reinterpret_cast<uint2 *>(q), sf, tiled ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_f4_norm_quant(const void *r, const void *h, const void *w, const float *awq_inv, int M, int d,
                                 float eps, float sc, float inv6, void *rprime, uint8_t *q, uint8_t *sf,
                                 unsigned *amax_word, bool measure, cudaStream_t s) {
    // warps per row: enough threads for the row's blocks of 16 (at most 8 warps)
    const int ng = d / 16;
    const int wpr = ng >= 256 ? 8 : ng >= 128 ? 4 : ng >= 64 ? 2 : 1;
    const dim3 grid((M + 8 / wpr - 1) / (8 / wpr));
    const uint16_t *rr = static_cast<const uint16_t *>(r), *hh = static_cast<const uint16_t *>(h);
    const uint16_t *ww = static_cast<const uint16_t *>(w);
    uint16_t *rp = static_cast<uint16_t *>(rprime);
#define FRT_F4_NORM(MEAS, W) \
    k_f4_norm_quant<MEAS, W><<<grid, 256, 0, s>>>(rr, hh, ww, awq_inv, M, d, eps, sc, inv6, rp, q, sf, amax_word)
    switch (wpr * 2 + (measure ? 1 : 0)) {
    case 2: FRT_F4_NORM(false, 1); break;
    case 3: FRT_F4_NORM(true, 1); break;
    case 4: FRT_F4_NORM(false, 2); break;
    case 5: FRT_F4_NORM(true, 2); break;
    case 8: FRT_F4_NORM(false, 4); break;
    case 9: FRT_F4_NORM(true, 4); break;
    case 16: FRT_F4_NORM(false, 8); break;
    default: FRT_F4_NORM(true, 8); break;
    }
#undef FRT_F4_NORM
    return cudaGetLastError();
}

cudaError_t launch_f4_geglu(const uint8_t *gq, const uint8_t *gs, float s_g, const uint8_t *uq, const uint8_t *us,
                            float s_u, int act, int M, int ff, float s_h, float inv6, uint8_t *hq, uint8_t *hsf,
                            unsigned *amax_word, bool measure, cudaStream_t s) {
    const size_t nblk = (size_t)M * (ff / 16);
    if (nblk >= 65536) {
        const unsigned grid = blocks_for(nblk, 256);
        if (measure)
            k_f4_geglu_blk<true><<<grid, 256, 0, s>>>(gq, gs, s_g, uq, us, s_u, act, M, ff, s_h, inv6, hq, hsf,
                                                      amax_word);
        else
            k_f4_geglu_blk<false><<<grid, 256, 0, s>>>(gq, gs, s_g, uq, us, s_u, act, M, ff, s_h, inv6, hq, hsf,
                                                       amax_word);
    } else {
        const unsigned grid = blocks_for((size_t)M * ff, 256);
        if (measure)
            k_f4_geglu<true><<<grid, 256, 0, s>>>(gq, gs, s_g, uq, us, s_u, act, M, ff, s_h, inv6, hq, hsf, amax_word);
        else
            k_f4_geglu<false><<<grid, 256, 0, s>>>(gq, gs, s_g, uq, us, s_u, act, M, ff, s_h, inv6, hq, hsf,
                                                   amax_word);
    }
    return cudaGetLastError();
}

namespace {

template <int EPI, bool SWAP, int BNT>
cudaError_t launch_one(const CUtensorMap &a, const CUtensorMap &b, const F4GemmParams &p, dim3 grid, cudaStream_t s) {
    using C = F4Cfg<SWAP, BNT>;
    static bool attr = false;
    if (!attr) {
        const cudaError_t e =
            cudaFuncSetAttribute(k_gemm_nvfp4<EPI, SWAP, BNT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess)
            return e;
        attr = true;
    }
    k_gemm_nvfp4<EPI, SWAP, BNT><<<grid, 192, C::SMEM, s>>>(a, b, p);
    return cudaGetLastError();
}

template <bool SWAP, int BNT>
cudaError_t launch_epi(const CUtensorMap &a, const CUtensorMap &b, const F4GemmParams &p, dim3 grid, cudaStream_t s) {
    switch (p.epi) {
    case F4_EPI_F32: return launch_one<F4_EPI_F32, SWAP, BNT>(a, b, p, grid, s);
    case F4_EPI_AMAX: return launch_one<F4_EPI_AMAX, SWAP, BNT>(a, b, p, grid, s);
    case F4_EPI_FP4: return launch_one<F4_EPI_FP4, SWAP, BNT>(a, b, p, grid, s);
    case F4_EPI_RESID: return launch_one<F4_EPI_RESID, SWAP, BNT>(a, b, p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_f4_gemm(const CUtensorMap &tmA, const CUtensorMap &tmB, const F4GemmParams &p, int n_cols,
                           int swap_n, cudaStream_t s) {
    if (swap_n == 0)
        return launch_epi<false, 128>(tmA, tmB, p, dim3(n_cols / 128, (p.M + F4_BM - 1) / F4_BM, p.splits), s);
    if (p.M > swap_n)
        return cudaErrorInvalidValue;
    const dim3 grid(n_cols / 128, 1, p.splits);
    switch (swap_n) {
    case 16: return launch_epi<true, 16>(tmA, tmB, p, grid, s);
    case 32: return launch_epi<true, 32>(tmA, tmB, p, grid, s);
    case 64: return launch_epi<true, 64>(tmA, tmB, p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace frt
