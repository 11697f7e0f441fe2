// frt_epi.cuh -- element arithmetic shared by the FP8 GEMM epilogues and the
// persistent stack kernel: BF16 packing, the gated activations (GELU-tanh and
// SiLU, itsolotime FlashRT article 7.2) and E4M3 encoding.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "frt_internal.h"

namespace frt {
namespace {

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t bf16_bits(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// GELU, tanh form: 0.5 g (1 + tanh(y)), y = sqrt(2/pi) (g + 0.044715 g^3).
// Because 1 + tanh(y) = 2 / (1 + exp(-2y)), this equals g / (1 + exp(-2y)),
// and exp(-2y) = 2^(g (c1 + c2 g^2)) with c1 = -2 sqrt(2/pi) log2(e),
// c2 = 0.044715 c1: one base-2 exponential and one reciprocal (the hardware
// approximations, a few ulp), free of branches and of the cancellation in
// 1 + tanh(y) for negative y; the E4M3 code of the result keeps 3 bits.  An
// overflowing exponential gives g * 0 = -0 for very negative g, an
// underflowing one gives g.
__device__ __forceinline__ float gelu_tanh(float g) {
    const float c1 = -2.3022081981f;  // -2 * 0.7978845608 * 1.4426950409
    const float c2 = -0.1029432396f;  // 0.044715 * c1
    const float t = __fmul_rn(g, __fadd_rn(c1, __fmul_rn(c2, __fmul_rn(g, g))));
    return __fmul_rn(g, rcp_approx(__fadd_rn(1.0f, ex2_approx(t))));
}
// SiLU: g / (1 + exp(-g)) = g / (1 + 2^(-g log2 e)), same approximations.
__device__ __forceinline__ float silu(float g) {
    const float t = __fmul_rn(g, -1.4426950409f);
    return __fmul_rn(g, rcp_approx(__fadd_rn(1.0f, ex2_approx(t))));
}

// a[j] = act(g[j]) * u[j] over a run of N elements, the activation chosen
// once for the run so the N chains interleave.
template <int N>
__device__ __forceinline__ void gated_run(int act, const float *g, const float *u, float *a) {
    if (act == ACT_SWIGLU) {
#pragma unroll
        for (int j = 0; j < N; ++j)
            a[j] = __fmul_rn(silu(g[j]), u[j]);
    } else {
#pragma unroll
        for (int j = 0; j < N; ++j)
            a[j] = __fmul_rn(gelu_tanh(g[j]), u[j]);
    }
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

}  // namespace
}  // namespace frt
