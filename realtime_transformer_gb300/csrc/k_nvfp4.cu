// k_nvfp4.cu -- the elementwise kernels of the NVFP4 variant of the FFN
// sublayer on sm_103a (itsolotime FlashRT article, 7.2: the NVFP4 encoder
// FFN, the residual stream kept in 16 bits, AWQ pre-scaling of the
// normalised activation): weight preparation (amax, NVFP4 codes and
// TMEM-ready block scales, gate and up rows interleaved for the fused
// gate/up GEMM) and the residual add + RMSNorm + AWQ divide + NVFP4 quantise
// of a layer's input.  The NVFP4 format and the TMEM-ready scale order are
// described in frt_f4.cuh; the GEMMs (the gate/up GEMM with the FP4-to-FP4
// gated activation in its epilogue, and the down GEMM + residual) run on the
// tensor-core GEMM (k_gemm_tc.cuh, k_gemm_f4.cu).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "frt_f4.cuh"
#include "frt_internal.h"
#include "frt_ptx.cuh"

namespace frt {

namespace {

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
// eight values (already BF16-exact) as eight BF16 words
__device__ __forceinline__ uint4 pack8_bf16(const float *f) {
    return make_uint4(bf16_bits(f[0]) | (bf16_bits(f[1]) << 16), bf16_bits(f[2]) | (bf16_bits(f[3]) << 16),
                      bf16_bits(f[4]) | (bf16_bits(f[5]) << 16), bf16_bits(f[6]) | (bf16_bits(f[7]) << 16));
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

// NVFP4 codes (row-major [*, K/2]) and TMEM-ready scales of W (times c)
// with tensor scale s.  ilv 0: row j of W is row j of the destination; 1 / 2:
// W is the gate / up weight of a [W_gate; W_up] arena interleaved in blocks
// of 64 rows (64 gate rows, then the 64 up rows of the same features), row j
// going to (j / 64) * 128 + (ilv == 2 ? 64 : 0) + j % 64.
__global__ void k_f4_quant_w(const uint4 *__restrict__ w, int rows, int K, const float *__restrict__ col, float s,
                             float inv6, uint2 *__restrict__ q, uint8_t *__restrict__ sf, int ilv) {
    const int gpr = K / 16;
    const size_t n = (size_t)rows * gpr;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int row = (int)(i / gpr), g = (int)(i % gpr);
        const int dst = ilv ? (row / 64) * 128 + (ilv == 2 ? 64 : 0) + row % 64 : row;
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
        q[(size_t)dst * gpr + g] = c;
        sf[sf_offset(dst, g, K)] = (uint8_t)b;
    }
}

// ------------------------------------------- residual + norm + quantise --

// WPR warps per row (1, 2, 4 or 8), 8 / WPR rows per CTA; a thread takes
// blocks of 16 elements strided by 32 WPR.  Pass 1: r' = bf16(r + h) (stored
// if rprime), the sum of squares (per thread over its blocks in order, a
// warp-shuffle tree, then the row's warps in order); pass 2: y = ((r' * inv)
// * w) [* awq_inv], then the amax (MEASURE) or the NVFP4 codes and TMEM-ready
// scales of y.  GPT > 0: a thread holds at most GPT blocks, kept in registers
// between the passes, and its norm (and AWQ) weights are read before the wait
// on the previous kernel; GPT == 0: any d, both passes read the row.  The
// arithmetic and its order are the same either way.
template <bool MEASURE, int WPR, int GPT>
__device__ __forceinline__ void f4_norm_body(const uint16_t *__restrict__ r, const uint16_t *__restrict__ h,
                                             const uint16_t *__restrict__ w, const float *__restrict__ awq_inv,
                                             int M, int d, float eps, float s, float inv6,
                                             uint16_t *__restrict__ rprime, uint8_t *__restrict__ q,
                                             uint8_t *__restrict__ sf, unsigned *amax_word) {
    __shared__ float s_part[8];
    // launched with a programmatic dependency on the previous layer: this
    // kernel reads the previous layer's output only once that grid has
    // completed; the next kernel may start launching (and stream its weights)
    // before this one's work -- at once on the register path, whose grid is
    // resident, else after the wait (a streamed grid's last wave)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tid = (warp % WPR) * 32 + lane;
    const int row = blockIdx.x * (8 / WPR) + warp / WPR;
    const bool active = row < M;
    const int ng = active ? d / 16 : 0;
    const uint4 *rv = reinterpret_cast<const uint4 *>(r + (size_t)(active ? row : 0) * d);
    const uint4 *hv = h ? reinterpret_cast<const uint4 *>(h + (size_t)(active ? row : 0) * d) : nullptr;
    const uint4 *wv = reinterpret_cast<const uint4 *>(w);
    float ss = 0.0f;
    float x[GPT > 0 ? GPT : 1][16];
    uint4 wraw[GPT > 0 ? GPT : 1][2];
    float4 aw[GPT > 0 ? GPT : 1][4];
    if constexpr (GPT > 0) {
        pdl_trigger();
        // the norm and AWQ weights do not depend on the previous kernel
#pragma unroll
        for (int k = 0; k < GPT; ++k) {
            const int g = tid + k * 32 * WPR;
            const bool in = g < ng;
            wraw[k][0] = in ? __ldg(wv + 2 * g) : make_uint4(0, 0, 0, 0);
            wraw[k][1] = in ? __ldg(wv + 2 * g + 1) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                aw[k][j] = (in && awq_inv) ? __ldg(reinterpret_cast<const float4 *>(awq_inv + g * 16) + j)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        pdl_wait();
#pragma unroll
        for (int k = 0; k < GPT; ++k) {
            const int g = tid + k * 32 * WPR;
            if (g < ng) {
                unpack8(rv[2 * g], x[k]);
                unpack8(rv[2 * g + 1], x[k] + 8);
                if (hv) {
                    float hh[16];
                    unpack8(hv[2 * g], hh);
                    unpack8(hv[2 * g + 1], hh + 8);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        x[k][j] = round_bf16(__fadd_rn(x[k][j], hh[j]));
                    if (rprime) {
                        uint4 *o = reinterpret_cast<uint4 *>(rprime + (size_t)row * d) + 2 * g;
                        o[0] = pack8_bf16(x[k]);
                        o[1] = pack8_bf16(x[k] + 8);
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    ss = __fadd_rn(ss, __fmul_rn(x[k][j], x[k][j]));
            }
        }
    } else {
        pdl_wait();
        pdl_trigger();
        for (int g = tid; g < ng; g += 32 * WPR) {
            float xl[16];
            unpack8(rv[2 * g], xl);
            unpack8(rv[2 * g + 1], xl + 8);
            if (hv) {
                float hh[16];
                unpack8(hv[2 * g], hh);
                unpack8(hv[2 * g + 1], hh + 8);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    xl[j] = round_bf16(__fadd_rn(xl[j], hh[j]));
                if (rprime) {
                    uint4 *o = reinterpret_cast<uint4 *>(rprime + (size_t)row * d) + 2 * g;
                    o[0] = pack8_bf16(xl);
                    o[1] = pack8_bf16(xl + 8);
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j)
                ss = __fadd_rn(ss, __fmul_rn(xl[j], xl[j]));
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
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)d), eps)));
    float amax = 0.0f;
    // pass 2 on one block: y, then its amax or its codes and scale
    auto finish = [&](int g, float (&y)[16], const uint4 (&wr)[2], const float4 (&awk)[4]) {
        float wf[16];
        unpack8(wr[0], wf);
        unpack8(wr[1], wf + 8);
        const float a[16] = {awk[0].x, awk[0].y, awk[0].z, awk[0].w, awk[1].x, awk[1].y, awk[1].z, awk[1].w,
                             awk[2].x, awk[2].y, awk[2].z, awk[2].w, awk[3].x, awk[3].y, awk[3].z, awk[3].w};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            y[j] = __fmul_rn(__fmul_rn(y[j], inv), wf[j]);
            if (awq_inv)
                y[j] = __fmul_rn(y[j], a[j]);
        }
        if (MEASURE) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                amax = fmaxf(amax, fabsf(y[j]));
        } else {
            uint2 c;
            const uint32_t b = quant_block16(y, s, inv6, c);
            reinterpret_cast<uint2 *>(q + (size_t)row * (d / 2))[g] = c;
            sf[sf_offset(row, g, d)] = (uint8_t)b;
        }
    };
    if constexpr (GPT > 0) {
#pragma unroll
        for (int k = 0; k < GPT; ++k) {
            const int g = tid + k * 32 * WPR;
            if (g < ng)
                finish(g, x[k], wraw[k], aw[k]);
        }
    } else {
        for (int g = tid; g < ng; g += 32 * WPR) {
            float xl[16], wf[16];
            unpack8(rv[2 * g], xl);
            unpack8(rv[2 * g + 1], xl + 8);
            if (hv) {
                float hh[16];
                unpack8(hv[2 * g], hh);
                unpack8(hv[2 * g + 1], hh + 8);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    xl[j] = round_bf16(__fadd_rn(xl[j], hh[j]));
            }
            unpack8(__ldg(wv + 2 * g), wf);
            unpack8(__ldg(wv + 2 * g + 1), wf + 8);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                xl[j] = __fmul_rn(__fmul_rn(xl[j], inv), wf[j]);
                if (awq_inv)
                    xl[j] = __fmul_rn(xl[j], __ldg(awq_inv + g * 16 + j));
            }
            if (MEASURE) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    amax = fmaxf(amax, fabsf(xl[j]));
            } else {
                uint2 c;
                const uint32_t b = quant_block16(xl, s, inv6, c);
                reinterpret_cast<uint2 *>(q + (size_t)row * (d / 2))[g] = c;
                sf[sf_offset(row, g, d)] = (uint8_t)b;
            }
        }
    }
    if (MEASURE) {
        amax = warp_max(amax);
        if (lane == 0)
            atomicMax(amax_word, __float_as_uint(amax));
    }
}

// Every thread of a CTA leaves the body (rows past M early), then meets the
// stamp's barrier here.
template <bool MEASURE, int WPR, int GPT>
__global__ void __launch_bounds__(256) k_f4_norm_quant(const uint16_t *__restrict__ r, const uint16_t *__restrict__ h,
                                                       const uint16_t *__restrict__ w,
                                                       const float *__restrict__ awq_inv, int M, int d, float eps,
                                                       float s, float inv6, uint16_t *__restrict__ rprime,
                                                       uint8_t *__restrict__ q, uint8_t *__restrict__ sf,
                                                       unsigned *amax_word, unsigned long long *stamp) {
    if (stamp && threadIdx.x == 0)
        stamp_start(stamp);
    f4_norm_body<MEASURE, WPR, GPT>(r, h, w, awq_inv, M, d, eps, s, inv6, rprime, q, sf, amax_word);
    if (stamp) {
        __syncthreads();
        if (threadIdx.x == 0)
            stamp_end(stamp);
    }
}

int num_sms() {
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0)
            sms = 148;
    }
    return sms;
}

int grid_cap() { return num_sms() * 8; }

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
                              uint8_t *sf, int ilv, cudaStream_t s) {
    k_f4_quant_w<<<blocks_for((size_t)rows * (K / 16), 256), 256, 0, s>>>(
        static_cast<const uint4 *>(w), rows, K, col, sc, inv6, reinterpret_cast<uint2 *>(q), sf, ilv);
    return cudaGetLastError();
}

cudaError_t launch_f4_norm_quant(const void *r, const void *h, const void *w, const float *awq_inv, int M, int d,
                                 float eps, float sc, float inv6, void *rprime, uint8_t *q, uint8_t *sf,
                                 unsigned *amax_word, bool measure, cudaStream_t s, bool pdl,
                                 unsigned long long *stamp) {
    // warps per row: enough threads for the row's blocks of 16 (at most 8
    // warps); blocks a thread holds in registers: 1 or 2, else the streaming
    // path (GPT 0)
    const int ng = d / 16;
    const int wpr = ng >= 256 ? 8 : ng >= 128 ? 4 : ng >= 64 ? 2 : 1;
    const int per = (ng + 32 * wpr - 1) / (32 * wpr);
    const dim3 grid((M + 8 / wpr - 1) / (8 / wpr));
    // the register path where all CTAs are resident at once (about 60
    // registers a thread for one block, 100 for two: four or two 256-thread
    // CTAs an SM); a larger grid streams, more CTAs in flight (measured on
    // 8192 rows of 5120: 45 us against 72 with two blocks in registers)
    const int gpt = (per <= 1 && grid.x <= 4u * (unsigned)num_sms()) ? 1
                    : (per <= 2 && grid.x <= 2u * (unsigned)num_sms()) ? 2 : 0;
    const uint16_t *rr = static_cast<const uint16_t *>(r), *hh = static_cast<const uint16_t *>(h);
    const uint16_t *ww = static_cast<const uint16_t *>(w);
    uint16_t *rp = static_cast<uint16_t *>(rprime);
#define FRT_F4_NORM(MEAS, W, G)                                                                              \
    return launch_ex(k_f4_norm_quant<MEAS, W, G>, grid, dim3(256), 0, s, pdl, 1u, rr, hh, ww, awq_inv, M, d, eps, \
                     sc, inv6, rp, q, sf, amax_word, stamp)
    // a thread holding at most two blocks keeps them in registers
#define FRT_F4_NORM_G(MEAS, W)                                                                                     \
    if (gpt == 1) FRT_F4_NORM(MEAS, W, 1);                                                                          \
    if (gpt == 2) FRT_F4_NORM(MEAS, W, 2);                                                                          \
    FRT_F4_NORM(MEAS, W, 0)
    switch (wpr * 2 + (measure ? 1 : 0)) {
    case 2: FRT_F4_NORM_G(false, 1);
    case 3: FRT_F4_NORM_G(true, 1);
    case 4: FRT_F4_NORM_G(false, 2);
    case 5: FRT_F4_NORM_G(true, 2);
    case 8: FRT_F4_NORM_G(false, 4);
    case 9: FRT_F4_NORM_G(true, 4);
    case 16: FRT_F4_NORM_G(false, 8);
    default: FRT_F4_NORM_G(true, 8);
    }
#undef FRT_F4_NORM_G
#undef FRT_F4_NORM
}

}  // namespace frt
