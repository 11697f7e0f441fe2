// k_elementwise.cu -- the memory-bound steps of the FP8 FFN sublayer:
//   A0  per-tensor amax and E4M3 quantisation of BF16 weights
//       (itsolotime FlashRT article, 5.2: FusedGateUp + Quant, scale_into);
//   A1  residual add + RMSNorm + E4M3 quantise, one warp per row with
//       128-bit loads and a warp-shuffle reduction (agentlenshq FlashRT
//       summary, "Main ideas": fused residual-norm-quantise; itsolotime
//       article, 3.3: rms_norm kernel row);
// (A3, the gated activation + requantise, runs in the gate/up GEMM's
// epilogue, k_gemm_fp8.cu.)  The A1 kernel has a measure mode for
// calibration that records the per-tensor amax instead of writing codes
// ("FlashRT docs/architecture.md", 6 Calibration Framework).
//
// Arithmetic follows the rounding points of the method exactly: every fp32
// operation is rounded on its own (explicit __f*_rn intrinsics), the scale
// is applied as a multiplication by its fp32 reciprocal, E4M3 conversion is
// round-to-nearest-even with saturation (cvt.rn.satfinite).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "frt_internal.h"
#include "frt_ptx.cuh"

namespace frt {

namespace {

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
    f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
    f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

__device__ __forceinline__ uint32_t bf16_bits(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint4 pack8_bf16(const float (&f)[8]) {
    uint4 v;
    v.x = bf16_bits(f[0]) | (bf16_bits(f[1]) << 16);
    v.y = bf16_bits(f[2]) | (bf16_bits(f[3]) << 16);
    v.z = bf16_bits(f[4]) | (bf16_bits(f[5]) << 16);
    v.w = bf16_bits(f[6]) | (bf16_bits(f[7]) << 16);
    return v;
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ uint2 pack8_e4m3(const float (&f)[8]) {
    uint2 v;
    v.x = e4m3x2(f[0], f[1]) | (e4m3x2(f[2], f[3]) << 16);
    v.y = e4m3x2(f[4], f[5]) | (e4m3x2(f[6], f[7]) << 16);
    return v;
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

// |x| of non-negative floats orders like its bit pattern.
__device__ __forceinline__ void atomic_amax(unsigned *word, float v) {
    atomicMax(word, __float_as_uint(v));
}

// ------------------------------------------------------------------- A0 --

__global__ void k_amax_bf16(const uint4 *__restrict__ x, size_t nvec, const uint16_t *__restrict__ tail,
                            int ntail, unsigned *amax_word) {
    float m = 0.0f;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nvec; i += (size_t)gridDim.x * blockDim.x) {
        float f[8];
        unpack8(__ldg(x + i), f);
#pragma unroll
        for (int j = 0; j < 8; j++)
            m = fmaxf(m, fabsf(f[j]));
    }
    if (blockIdx.x == 0 && threadIdx.x < (unsigned)ntail)
        m = fmaxf(m, fabsf(__uint_as_float((uint32_t)tail[threadIdx.x] << 16)));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0)
        atomic_amax(amax_word, m);
}

__global__ void k_quant_bf16(const uint4 *__restrict__ x, size_t nvec, const uint16_t *__restrict__ tail,
                             int ntail, float inv_s, uint2 *__restrict__ q, uint8_t *__restrict__ qtail) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nvec; i += (size_t)gridDim.x * blockDim.x) {
        float f[8];
        unpack8(__ldg(x + i), f);
#pragma unroll
        for (int j = 0; j < 8; j++)
            f[j] = __fmul_rn(f[j], inv_s);
        q[i] = pack8_e4m3(f);
    }
    if (blockIdx.x == 0 && threadIdx.x < (unsigned)ntail) {
        float v = __fmul_rn(__uint_as_float((uint32_t)tail[threadIdx.x] << 16), inv_s);
        qtail[threadIdx.x] = (uint8_t)(e4m3x2(v, 0.0f) & 0xFF);
    }
}

// amax of W[j][k] * w[k] over a [rows, d] BF16 matrix: the RMSNorm weight
// w folded into the gate/up weights (itsolotime article, 5.2, the Pi0 spec's
// norm_fuse).  A BF16 x BF16 product is exact in fp32.  d % 8 == 0.
__global__ void k_amax_fold(const uint4 *__restrict__ x, size_t rows, int d, const uint4 *__restrict__ w,
                            unsigned *amax_word) {
    const size_t vpr = (size_t)d / 8;
    const size_t nvec = rows * vpr;
    float m = 0.0f;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nvec; i += (size_t)gridDim.x * blockDim.x) {
        float f[8], c[8];
        unpack8(__ldg(x + i), f);
        unpack8(__ldg(w + i % vpr), c);
#pragma unroll
        for (int j = 0; j < 8; j++)
            m = fmaxf(m, fabsf(__fmul_rn(f[j], c[j])));
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0)
        atomic_amax(amax_word, m);
}

// E4M3(W[j][k] * w[k] * inv_s) of a [rows, d] BF16 matrix into dst (row-major):
// a weight with the RMSNorm weight folded in.  d % 8 == 0.
__global__ void k_quant_fold(const uint4 *__restrict__ x, size_t rows, int d, const uint4 *__restrict__ w,
                             float inv_s, uint2 *__restrict__ q) {
    const size_t vpr = (size_t)d / 8;
    const size_t nvec = rows * vpr;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nvec; i += (size_t)gridDim.x * blockDim.x) {
        float f[8], c[8];
        unpack8(__ldg(x + i), f);
        unpack8(__ldg(w + i % vpr), c);
#pragma unroll
        for (int j = 0; j < 8; j++)
            f[j] = __fmul_rn(__fmul_rn(f[j], c[j]), inv_s);
        q[i] = pack8_e4m3(f);
    }
}

// [W_gate; W_up] quantised into the interleaved arena layout: blocks of 128
// rows, each 64 gate rows followed by the 64 up rows of the same features,
// so that one GEMM tile holds matching gate and up rows.  With fold != null
// every column k is first multiplied by fold[k] (the norm weight, exact in
// fp32).  d % 8 == 0, ff % 64 == 0.
__global__ void k_quant_gu_interleave(const uint16_t *__restrict__ gate, const uint16_t *__restrict__ up, int ff,
                                      int d, const uint16_t *__restrict__ fold, float inv_s,
                                      uint8_t *__restrict__ dst) {
    const size_t vpr = (size_t)d / 8;
    const size_t total = (size_t)2 * ff * vpr;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const size_t row = i / vpr;
        const size_t v = i - row * vpr;
        const size_t within = row & 127;
        const size_t srow = (row >> 7) * 64 + (within & 63);
        const uint16_t *src = (within < 64 ? gate : up) + srow * d + v * 8;
        float f[8];
        unpack8(__ldg(reinterpret_cast<const uint4 *>(src)), f);
        if (fold) {
            float c[8];
            unpack8(__ldg(reinterpret_cast<const uint4 *>(fold + v * 8)), c);
#pragma unroll
            for (int j = 0; j < 8; j++)
                f[j] = __fmul_rn(f[j], c[j]);
        }
#pragma unroll
        for (int j = 0; j < 8; j++)
            f[j] = __fmul_rn(f[j], inv_s);
        *reinterpret_cast<uint2 *>(dst + row * d + v * 8) = pack8_e4m3(f);
    }
}

// ------------------------------------------------------------------- A1 --

// WPR warps per row (1, 2, 4 or 8).  Pass 1: r' = bf16(r + h) (stored if
// rprime != null), sum of squares (per thread, then a warp-shuffle tree, then
// the warps of the row in order).  Pass 2: y = (r' * inv) * w -- or, with a
// modulation (AdaRMSNorm), y = (r' * inv) * (1 + scale) + shift from the
// row's modulation vectors -- then either amax (measure) or
// q = E4M3(y * inv_s).  d % 8 == 0.
//
// VPT > 0: each thread owns at most VPT 16-byte vectors of its row (the
// launcher guarantees d / 8 <= 32 * WPR * VPT) and issues every load of r, h
// and w before the first use, so the row costs one memory round trip; the
// values stay in registers for pass 2.  VPT == 0: any d, a strided loop that
// re-reads r (and h) in pass 2.
template <bool MEASURE, int WPR, int VPT, bool ADA>
__device__ __forceinline__ void norm_body(const uint16_t *__restrict__ r, const uint16_t *__restrict__ h,
                                          const uint16_t *__restrict__ w, int M, int d, float eps, float inv_s,
                                          uint16_t *__restrict__ rprime, uint8_t *__restrict__ qx,
                                          unsigned *amax_word, const NormMod &mod) {
    // Let the dependent GEMM launch (and stream its weights) right away; it
    // waits for this grid, and this grid waits for its own predecessor
    // before it can complete, so ordering is preserved.
    pdl_trigger();
    constexpr int ROWS_PER_CTA = 8 / WPR;
    constexpr int STRIDE = 32 * WPR;
    __shared__ float s_part[8];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = warp % WPR;                       // warp index within the row
    const int tid = sub * 32 + lane;                  // thread index within the row
    const int row = blockIdx.x * ROWS_PER_CTA + warp / WPR;
    const bool active = row < M;
    const int nv = d >> 3;
    const size_t roff = (size_t)(active ? row : 0) * d;
    const uint4 *rv = reinterpret_cast<const uint4 *>(r + roff);
    const uint4 *hv = h ? reinterpret_cast<const uint4 *>(h + roff) : nullptr;
    uint4 *rpv = rprime ? reinterpret_cast<uint4 *>(rprime + roff) : nullptr;
    const uint4 *wv = reinterpret_cast<const uint4 *>(w);
    uint2 *qv = reinterpret_cast<uint2 *>(qx + roff);
    // AdaRMSNorm: the row's scale vector (in place of the norm weight) and shift vector
    const uint4 *scv =
        ADA ? reinterpret_cast<const uint4 *>(mod.p + (size_t)(active ? row : 0) * mod.stride) : nullptr;
    const uint4 *shv = ADA ? scv + nv : nullptr;

    float ss = 0.0f;
    float x[VPT > 0 ? VPT : 1][8];
    if constexpr (VPT > 0) {
        // the norm weights (or the modulation) do not depend on the previous kernel
        uint4 wraw[VPT], shraw[ADA ? VPT : 1];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const bool in = tid + k * STRIDE < nv;
            wraw[k] = in ? __ldg((ADA ? scv : wv) + tid + k * STRIDE) : make_uint4(0, 0, 0, 0);
            if constexpr (ADA)
                shraw[k] = in ? __ldg(shv + tid + k * STRIDE) : make_uint4(0, 0, 0, 0);
        }
        pdl_wait();
        uint4 rraw[VPT], hraw[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const bool in = active && tid + k * STRIDE < nv;
            rraw[k] = in ? rv[tid + k * STRIDE] : make_uint4(0, 0, 0, 0);
            hraw[k] = (in && hv) ? hv[tid + k * STRIDE] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            unpack8(rraw[k], x[k]);
            if (hv) {
                float hh[8];
                unpack8(hraw[k], hh);
#pragma unroll
                for (int j = 0; j < 8; j++)
                    x[k][j] = __bfloat162float(__float2bfloat16_rn(__fadd_rn(x[k][j], hh[j])));
                if (rpv && active && tid + k * STRIDE < nv)
                    rpv[tid + k * STRIDE] = pack8_bf16(x[k]);
            }
#pragma unroll
            for (int j = 0; j < 8; j++)
                ss = __fadd_rn(ss, __fmul_rn(x[k][j], x[k][j]));
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
        const float ms = __fdiv_rn(ss, (float)d);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            if (tid + k * STRIDE >= nv)
                break;
            float wf[8];
            unpack8(wraw[k], wf);
            if constexpr (ADA) {
                float sh[8];
                unpack8(shraw[k], sh);
#pragma unroll
                for (int j = 0; j < 8; j++)
                    x[k][j] = __fadd_rn(__fmul_rn(__fmul_rn(x[k][j], inv), __fadd_rn(1.0f, wf[j])), sh[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    x[k][j] = __fmul_rn(__fmul_rn(x[k][j], inv), wf[j]);
            }
            if (MEASURE) {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    amax = fmaxf(amax, fabsf(x[k][j]));
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    x[k][j] = __fmul_rn(x[k][j], inv_s);
                qv[tid + k * STRIDE] = pack8_e4m3(x[k]);
            }
        }
        if (MEASURE) {
            amax = warp_max(amax);
            if (lane == 0)
                atomic_amax(amax_word, amax);
        }
        return;
    } else {
        pdl_wait();
        if (active) {
            for (int v = tid; v < nv; v += STRIDE) {
                unpack8(rv[v], x[0]);
                if (hv) {
                    float hh[8];
                    unpack8(hv[v], hh);
#pragma unroll
                    for (int j = 0; j < 8; j++)
                        x[0][j] = __bfloat162float(__float2bfloat16_rn(__fadd_rn(x[0][j], hh[j])));
                    if (rpv)
                        rpv[v] = pack8_bf16(x[0]);
                }
#pragma unroll
                for (int j = 0; j < 8; j++)
                    ss = __fadd_rn(ss, __fmul_rn(x[0][j], x[0][j]));
            }
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
        const float ms = __fdiv_rn(ss, (float)d);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
        float amax = 0.0f;
        for (int v = tid; v < nv; v += STRIDE) {
            float wf[8];
            unpack8(rv[v], x[0]);
            if (hv) {
                float hh[8];
                unpack8(hv[v], hh);
#pragma unroll
                for (int j = 0; j < 8; j++)
                    x[0][j] = __bfloat162float(__float2bfloat16_rn(__fadd_rn(x[0][j], hh[j])));
            }
            unpack8(__ldg((ADA ? scv : wv) + v), wf);
            if constexpr (ADA) {
                float sh[8];
                unpack8(__ldg(shv + v), sh);
#pragma unroll
                for (int j = 0; j < 8; j++)
                    x[0][j] = __fadd_rn(__fmul_rn(__fmul_rn(x[0][j], inv), __fadd_rn(1.0f, wf[j])), sh[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    x[0][j] = __fmul_rn(__fmul_rn(x[0][j], inv), wf[j]);
            }
            if (MEASURE) {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    amax = fmaxf(amax, fabsf(x[0][j]));
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    x[0][j] = __fmul_rn(x[0][j], inv_s);
                qv[v] = pack8_e4m3(x[0]);
            }
        }
        if (MEASURE) {
            amax = warp_max(amax);
            if (lane == 0)
                atomic_amax(amax_word, amax);
        }
    }
}

// Every thread of a CTA passes the same barriers inside the body (rows past
// M leave only after them), then the stamp's barrier here.
template <bool MEASURE, int WPR, int VPT, bool ADA>
__global__ void __launch_bounds__(256) k_norm_quant(const uint16_t *__restrict__ r, const uint16_t *__restrict__ h,
                                                    const uint16_t *__restrict__ w, int M, int d, float eps,
                                                    float inv_s, uint16_t *__restrict__ rprime,
                                                    uint8_t *__restrict__ qx, unsigned *amax_word, NormMod mod) {
    if (mod.stamp && threadIdx.x == 0)
        stamp_start(mod.stamp);
    norm_body<MEASURE, WPR, VPT, ADA>(r, h, w, M, d, eps, inv_s, rprime, qx, amax_word, mod);
    if (mod.stamp) {
        __syncthreads();
        if (threadIdx.x == 0)
            stamp_end(mod.stamp);
    }
}

// ------------------------------------------------------- QKV split + RoPE --

// qkv [M, (Hq + 2 Hkv) hd] BF16 (Q heads, then K heads, then V heads) ->
// q [Hq, M, hd], k [Hkv, M, hd] rotated by RoPE at pos[m], v [Hkv, M, hd]
// copied.  Rotate-half layout: element i of a head's first half pairs with
// element i + hd/2, angle = pos * theta_i in fp32, then in fp32
// o_i = x_i cos - x_{i+hd/2} sin, o_{i+hd/2} = x_{i+hd/2} cos + x_i sin,
// rounded to BF16.  A thread takes 4 consecutive pairs of a Q/K head (two
// 8-byte loads and stores) or 8 consecutive elements of a V head.
__global__ void __launch_bounds__(256) k_rope_split(const uint16_t *__restrict__ qkv, int M, int nq, int nkv, int hd,
                                                   const int *__restrict__ pos, const float *__restrict__ inv_freq,
                                                   uint16_t *__restrict__ q, uint16_t *__restrict__ k,
                                                   uint16_t *__restrict__ v) {
    pdl_trigger();
    pdl_wait();
    const int G = hd / 8;  // work items per head: 4 pairs, or 8 V elements
    const int H = nq + 2 * nkv;
    const size_t N = (size_t)H * hd;
    const size_t total = (size_t)M * H * G;
    for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < total; t += (size_t)gridDim.x * blockDim.x) {
        const int g = (int)(t % G);
        const size_t mh = t / G;
        const int h = (int)(mh % H);
        const int m = (int)(mh / H);
        const uint16_t *src = qkv + (size_t)m * N + (size_t)h * hd;
        if (h >= nq + nkv) {
            const int hv = h - nq - nkv;
            *reinterpret_cast<uint4 *>(v + ((size_t)hv * M + m) * hd + 8 * g) =
                __ldg(reinterpret_cast<const uint4 *>(src + 8 * g));
            continue;
        }
        const int half = hd / 2;
        const uint2 a = __ldg(reinterpret_cast<const uint2 *>(src + 4 * g));
        const uint2 b = __ldg(reinterpret_cast<const uint2 *>(src + half + 4 * g));
        const float x1[4] = {bf_lo(a.x), bf_hi(a.x), bf_lo(a.y), bf_hi(a.y)};
        const float x2[4] = {bf_lo(b.x), bf_hi(b.x), bf_lo(b.y), bf_hi(b.y)};
        const float p = (float)__ldg(pos + m);
        uint32_t o1[2], o2[2];
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            float r1[2], r2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float sn, cs;
                sincosf(__fmul_rn(p, __ldg(inv_freq + 4 * g + j + e)), &sn, &cs);
                r1[e] = __fsub_rn(__fmul_rn(x1[j + e], cs), __fmul_rn(x2[j + e], sn));
                r2[e] = __fadd_rn(__fmul_rn(x2[j + e], cs), __fmul_rn(x1[j + e], sn));
            }
            o1[j / 2] = bf16_bits(r1[0]) | (bf16_bits(r1[1]) << 16);
            o2[j / 2] = bf16_bits(r2[0]) | (bf16_bits(r2[1]) << 16);
        }
        uint16_t *dst = h < nq ? q + ((size_t)h * M + m) * hd : k + ((size_t)(h - nq) * M + m) * hd;
        *reinterpret_cast<uint2 *>(dst + 4 * g) = make_uint2(o1[0], o1[1]);
        *reinterpret_cast<uint2 *>(dst + half + 4 * g) = make_uint2(o2[0], o2[1]);
    }
}

// (cos, sin) of angle pos[m] * theta_i for every token and pair: the table the
// GEMM epilogue's fused split + RoPE reads (the same sincosf of the same fp32
// angle as k_rope_split, so both give the same bits).
__global__ void __launch_bounds__(256) k_rope_table(const int *__restrict__ pos, const float *__restrict__ inv_freq,
                                                   int M, int half, float2 *__restrict__ cs) {
    pdl_trigger();
    pdl_wait();
    const size_t total = (size_t)M * half;
    for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < total; t += (size_t)gridDim.x * blockDim.x) {
        const int i = (int)(t % half);
        const int m = (int)(t / half);
        float sn, c;
        sincosf(__fmul_rn((float)__ldg(pos + m), __ldg(inv_freq + i)), &sn, &c);
        cs[t] = make_float2(c, sn);
    }
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0)
            n = 1;
    }
    return n;
}

}  // namespace

cudaError_t launch_amax_bf16(const void *x, size_t n, unsigned *amax_word, cudaStream_t s) {
    const size_t nvec = n / 8;
    const int ntail = (int)(n - nvec * 8);
    const uint16_t *tail = static_cast<const uint16_t *>(x) + nvec * 8;
    size_t blocks = (nvec + 255) / 256;
    const size_t cap = (size_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    k_amax_bf16<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint4 *>(x), nvec, tail, ntail, amax_word);
    return cudaGetLastError();
}

cudaError_t launch_quant_bf16(const void *x, size_t n, float inv_s, uint8_t *q, cudaStream_t s) {
    const size_t nvec = n / 8;
    const int ntail = (int)(n - nvec * 8);
    const uint16_t *tail = static_cast<const uint16_t *>(x) + nvec * 8;
    size_t blocks = (nvec + 255) / 256;
    const size_t cap = (size_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    k_quant_bf16<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint4 *>(x), nvec, tail, ntail, inv_s,
                                                   reinterpret_cast<uint2 *>(q), q + nvec * 8);
    return cudaGetLastError();
}

cudaError_t launch_quant_gu_interleave(const void *gate, const void *up, int ff, int d, const void *fold,
                                      float inv_s, uint8_t *dst, cudaStream_t s) {
    const size_t total = (size_t)2 * ff * (d / 8);
    size_t blocks = (total + 255) / 256;
    const size_t cap = (size_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    k_quant_gu_interleave<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint16_t *>(gate),
                                                            static_cast<const uint16_t *>(up), ff, d,
                                                            static_cast<const uint16_t *>(fold), inv_s, dst);
    return cudaGetLastError();
}

cudaError_t launch_amax_fold(const void *x, size_t rows, int d, const void *w, unsigned *amax_word, cudaStream_t s) {
    const size_t nvec = rows * (size_t)(d / 8);
    size_t blocks = (nvec + 255) / 256;
    const size_t cap = (size_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    k_amax_fold<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint4 *>(x), rows, d,
                                                  static_cast<const uint4 *>(w), amax_word);
    return cudaGetLastError();
}

namespace {

template <bool MEASURE, int WPR, int VPT, bool ADA>
cudaError_t norm_launch(NormMod mod, int M, bool pdl, cudaStream_t s, const uint16_t *r, const uint16_t *h,
                        const uint16_t *w,
                        int d, float eps, float inv_s, uint16_t *rp, uint8_t *qx, unsigned *amax_word) {
    // the largest shared-memory carve-out, like the GEMMs, so that GEMM CTAs
    // can start on an SM while this kernel's CTAs run there
    static bool attr_set = false;
    if (!attr_set) {
        const cudaError_t e = cudaFuncSetAttribute(k_norm_quant<MEASURE, WPR, VPT, ADA>,
                                                   cudaFuncAttributePreferredSharedMemoryCarveout,
                                                   (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    const dim3 grid((unsigned)((M + 8 / WPR - 1) / (8 / WPR)));
    return launch_ex(k_norm_quant<MEASURE, WPR, VPT, ADA>, grid, dim3(256), 0, s, pdl, 1u, r, h, w, M, d, eps, inv_s,
                     rp, qx, amax_word, mod);
}

template <bool MEASURE>
cudaError_t norm_dispatch(NormMod mod, int M, bool pdl, cudaStream_t s, const uint16_t *r, const uint16_t *h,
                          const uint16_t *w, int d, float eps, float inv_s, uint16_t *rp, uint8_t *qx,
                          unsigned *amax_word) {
    const int nv = d / 8;
    // Few rows: spread each row over enough warps that a thread holds one
    // vector (latency first).  Many rows: a warp per row, up to four vectors
    // a thread, widening the row only as d requires (throughput first).
    int wpr = 1;
    if (M <= 256) {
        while (wpr < 8 && nv > 32 * wpr)
            wpr *= 2;
    } else {
        while (wpr < 8 && nv > 32 * wpr * 4)
            wpr *= 2;
    }
    const int per = 32 * wpr;
    const int vpt = (nv + per - 1) / per;
#define FRT_NORM(W, V)                                                                                \
    return mod.p ? norm_launch<MEASURE, W, V, true>(mod, M, pdl, s, r, h, w, d, eps, inv_s, rp, qx, amax_word) \
                 : norm_launch<MEASURE, W, V, false>(mod, M, pdl, s, r, h, w, d, eps, inv_s, rp, qx, amax_word)
    if (vpt > 4) {
        FRT_NORM(8, 0);
    }
    switch (wpr) {
    case 1: if (vpt == 1) FRT_NORM(1, 1); FRT_NORM(1, 4);
    case 2: if (vpt == 1) FRT_NORM(2, 1); FRT_NORM(2, 4);
    case 4: if (vpt == 1) FRT_NORM(4, 1); FRT_NORM(4, 4);
    default: if (vpt == 1) FRT_NORM(8, 1); FRT_NORM(8, 4);
    }
#undef FRT_NORM
}

}  // namespace

cudaError_t launch_norm_quant(const void *r, const void *h, const void *w, int M, int d, float eps, float inv_s,
                              void *rprime, uint8_t *qx, unsigned *amax_word, bool measure, cudaStream_t s,
                              bool pdl, NormMod mod) {
    auto rr = static_cast<const uint16_t *>(r);
    auto hh = static_cast<const uint16_t *>(h);
    auto ww = static_cast<const uint16_t *>(w);
    auto rp = static_cast<uint16_t *>(rprime);
    if (measure)
        return norm_dispatch<true>(mod, M, pdl, s, rr, hh, ww, d, eps, inv_s, rp, qx, amax_word);
    return norm_dispatch<false>(mod, M, pdl, s, rr, hh, ww, d, eps, inv_s, rp, qx, amax_word);
}

cudaError_t launch_rope_split(const void *qkv, int M, int nq, int nkv, int hd, const int *pos, const float *inv_freq,
                              void *q, void *k, void *v, cudaStream_t s, bool pdl) {
    const size_t total = (size_t)M * (nq + 2 * nkv) * (hd / 8);
    size_t blocks = (total + 255) / 256;
    const size_t cap = (size_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    return launch_ex(k_rope_split, dim3((unsigned)blocks), dim3(256), 0, s, pdl, 1u,
                     static_cast<const uint16_t *>(qkv), M, nq, nkv, hd, pos, inv_freq, static_cast<uint16_t *>(q),
                     static_cast<uint16_t *>(k), static_cast<uint16_t *>(v));
}

cudaError_t launch_rope_table(const int *pos, const float *inv_freq, int M, int half, float2 *cs, cudaStream_t s,
                              bool pdl) {
    const size_t total = (size_t)M * half;
    size_t blocks = (total + 255) / 256;
    const size_t cap = (size_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    return launch_ex(k_rope_table, dim3((unsigned)blocks), dim3(256), 0, s, pdl, 1u, pos, inv_freq, M, half, cs);
}

cudaError_t launch_quant_fold(const void *x, size_t rows, int d, const void *w, float inv_s, uint8_t *q,
                              cudaStream_t s) {
    const size_t nvec = rows * (size_t)(d / 8);
    size_t blocks = (nvec + 255) / 256;
    const size_t cap = (size_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    k_quant_fold<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint4 *>(x), rows, d,
                                                   static_cast<const uint4 *>(w), inv_s, reinterpret_cast<uint2 *>(q));
    return cudaGetLastError();
}

// Diagnostics: the E4M3 encoding of a range of fp32 bit patterns,
// q[i] = E4M3(float with bits start + i), eight patterns a thread, by the
// same conversion (e4m3x2) every quantising kernel here uses.  n % 8 == 0.
__global__ void k_e4m3_sweep(uint32_t start, size_t n, uint2 *__restrict__ q) {
    const size_t nv = n / 8;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nv; i += (size_t)gridDim.x * blockDim.x) {
        const uint32_t b = start + (uint32_t)(i * 8);
        float f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            f[j] = __uint_as_float(b + (uint32_t)j);
        q[i] = pack8_e4m3(f);
    }
}

cudaError_t launch_e4m3_sweep(uint32_t start, size_t n, uint8_t *q, cudaStream_t s) {
    size_t blocks = (n / 8 + 255) / 256;
    const size_t cap = (size_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    k_e4m3_sweep<<<(unsigned)blocks, 256, 0, s>>>(start, n, reinterpret_cast<uint2 *>(q));
    return cudaGetLastError();
}

}  // namespace frt
