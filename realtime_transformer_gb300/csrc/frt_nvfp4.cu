// frt_nvfp4.cu -- the NVFP4 sublayer stack behind frt_nvfp4.h (itsolotime
// FlashRT article, 7.2): per layer the norm + AWQ + FP4 quantise kernel, the
// gate and up NVFP4 GEMMs with FP4 epilogues, the GeGLU FP4 -> FP4 kernel and
// the down NVFP4 GEMM with the residual epilogue (kernels in k_nvfp4.cu).
// Tensor maps of the fixed buffers are encoded once at plan creation and
// passed as kernel parameters, so a forward can be captured into a graph.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "frt_internal.h"
#include "frt_nvfp4.h"

#define FRT_API extern "C" __attribute__((visibility("default")))

using namespace frt;

namespace {

constexpr float F4_RMS_EPS = 1e-6f;  // the FFN's reading: the pages never state it
constexpr float NVFP4_RANGE = 448.0f * 6.0f;

frt_status ffail(frt_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    set_last_error(buf);
    return st;
}

frt_status fcuda_fail(cudaError_t e, const char *what) {
    return ffail(e == cudaErrorMemoryAllocation ? FRT_ERR_OOM : FRT_ERR_CUDA, "%s: %s (%s)", what,
                 cudaGetErrorString(e), cudaGetErrorName(e));
}

#define FCK(call)                                  \
    do {                                           \
        cudaError_t e_ = (call);                   \
        if (e_ != cudaSuccess)                     \
            return fcuda_fail(e_, #call);          \
    } while (0)

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor scale from an amax: amax / (448 * 6), 1 for zero.
float scale_of(float amax) { return amax > 0.0f ? amax / NVFP4_RANGE : 1.0f; }
// The block-scale multiplier 1 / (6 s).
float inv6_of(float s) {
    const float t = 6.0f * s;
    return 1.0f / t;
}
float word_to_float(unsigned w) {
    float f;
    memcpy(&f, &w, 4);
    return f;
}

}  // namespace

struct frt_fp4_plan {
    int d = 0, ff = 0, act = 0, M_max = 0, L = 0, M_alloc = 0;
    // weights: codes [L * rows, K/2], TMEM-ready scales rows * K/16 per layer
    uint8_t *wg = nullptr, *wu = nullptr, *wd = nullptr;
    uint8_t *sg = nullptr, *su = nullptr, *sd = nullptr;
    uint16_t *w_norm = nullptr;  // BF16 [L, d]
    float *awq_inv = nullptr;    // fp32 [L, d]: 1 / c
    // activations
    uint8_t *xq = nullptr, *xsf = nullptr;  // [M_alloc, d/2], TMEM-ready
    uint8_t *gq = nullptr, *gs = nullptr;   // [M_alloc, ff/2], [M_alloc, ff/16]
    uint8_t *uq = nullptr, *us = nullptr;
    uint8_t *hq = nullptr, *hsf = nullptr;  // [M_alloc, ff/2], TMEM-ready
    uint16_t *rp = nullptr;                 // r' of layer 0 [M_alloc, d]
    uint16_t *res[2] = {nullptr, nullptr};  // layer outputs between layers
    unsigned *amax = nullptr;               // [4]
    int *err = nullptr;
    int num_sms = 0;
    float *ws = nullptr;                    // split-K partial tiles: num_sms x 128 x 128 fp32
    int *counters = nullptr;                // split-K arrival counters, one per tile
    std::vector<float> s_wg, s_wu, s_wd, s_x, s_g, s_u, s_h;
    CUtensorMap tm_wg, tm_wu, tm_wd, tm_xq, tm_hq;
    CUtensorMap tm_xq_n[3], tm_hq_n[3];     // token operands of the weight-streaming role: boxes of 16 / 32 / 64 rows
    std::vector<char> loaded, has_awq;
    bool scaled = false;
};

namespace {

void free_fp4(frt_fp4_plan *P) {
    void *ptrs[] = {P->wg, P->wu,  P->wd,  P->sg,  P->su,     P->sd,     P->w_norm, P->awq_inv, P->xq,
                    P->xsf, P->gq, P->gs,  P->uq,  P->us,     P->hq,     P->hsf,    P->rp,      P->res[0],
                    P->res[1], P->amax, P->err, P->ws, P->counters};
    for (void *p : ptrs)
        if (p) cudaFree(p);
    delete P;
}

frt_status check_ready(frt_fp4_plan *P) {
    if (!P)
        return ffail(FRT_ERR_INVALID_ARG, "null plan");
    for (int l = 0; l < P->L; ++l)
        if (!P->loaded[l])
            return ffail(FRT_ERR_NOT_READY, "weights of layer %d not loaded", l);
    return FRT_OK;
}

size_t wsf_bytes(size_t rows, size_t K) { return rows * K / 16; }

constexpr int F4_MAX_TILES = 4096;

// Split-K factor of a GEMM with `tiles` output tiles and K / 256 stages:
// enough splits to put a CTA on most SMs, each split at least four stages
// long (one CTA per SM: the kernel's shared memory allows no more).
// Token tile of the weight-streaming role for M tokens (0: the tiled role).
constexpr int F4_SWAP_MAX_TOKENS = 64;
// The tiled role measured faster on every shape (the per-stage cost of the
// block-scaled pipeline does not shrink with the narrower N), so the
// weight-streaming role runs only when FRT_F4_SWAP=1 (read per launch).
int f4_swap_n(int M) {
    const char *e = getenv("FRT_F4_SWAP");
    if (M > F4_SWAP_MAX_TOKENS || !e || atoi(e) != 1)
        return 0;
    return M <= 16 ? 16 : M <= 32 ? 32 : 64;
}
int f4_swap_idx(int n) { return n == 16 ? 0 : n == 32 ? 1 : 2; }

int f4_splits(int tiles, int KB, int num_sms) {
    if (tiles > F4_MAX_TILES)
        return 1;
    int s = num_sms / tiles;
    if (s > KB / 4)
        s = KB / 4;
    return s < 1 ? 1 : s;
}

}  // namespace

FRT_API frt_status frt_fp4_plan_create(int d, int ff, int act, int M_max, int n_layers, frt_fp4_plan_t *out) {
    if (!out)
        return ffail(FRT_ERR_INVALID_ARG, "null out pointer");
    *out = nullptr;
    if (d < 256 || d % 256 || ff < 256 || ff % 256)
        return ffail(FRT_ERR_INVALID_ARG, "d=%d and ff=%d must be positive multiples of 256", d, ff);
    if (act != FRT_ACT_GEGLU_TANH && act != FRT_ACT_SWIGLU)
        return ffail(FRT_ERR_INVALID_ARG, "unknown activation %d", act);
    if (M_max < 1 || M_max > 65536 || n_layers < 1 || n_layers > 4096)
        return ffail(FRT_ERR_INVALID_ARG, "M_max=%d or n_layers=%d out of range", M_max, n_layers);
    int dev = 0, major = 0, minor = 0;
    FCK(cudaGetDevice(&dev));
    FCK(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    FCK(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    if (major != 10 || minor != 3)
        return ffail(FRT_ERR_UNSUPPORTED, "needs a compute-capability 10.3 GPU (found %d.%d)", major, minor);
    frt_fp4_plan *P = new frt_fp4_plan;
    P->d = d;
    P->ff = ff;
    P->act = act;
    P->M_max = M_max;
    P->L = n_layers;
    P->M_alloc = (M_max + 127) / 128 * 128;
    for (auto *v : {&P->s_wg, &P->s_wu, &P->s_wd, &P->s_x, &P->s_g, &P->s_u, &P->s_h})
        v->assign(n_layers, 1.0f);
    P->loaded.assign(n_layers, 0);
    P->has_awq.assign(n_layers, 0);
    const size_t L = n_layers, D = d, F = ff, MA = P->M_alloc;
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = cudaMalloc(&P->wg, L * F * D / 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->wu, L * F * D / 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->wd, L * D * F / 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->sg, L * wsf_bytes(F, D));
    if (e == cudaSuccess) e = cudaMalloc(&P->su, L * wsf_bytes(F, D));
    if (e == cudaSuccess) e = cudaMalloc(&P->sd, L * wsf_bytes(D, F));
    if (e == cudaSuccess) e = cudaMalloc(&P->w_norm, L * D * 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->awq_inv, L * D * 4);
    if (e == cudaSuccess) e = cudaMalloc(&P->xq, MA * D / 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->xsf, MA * D / 16);
    if (e == cudaSuccess) e = cudaMalloc(&P->gq, MA * F / 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->gs, MA * F / 16);
    if (e == cudaSuccess) e = cudaMalloc(&P->uq, MA * F / 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->us, MA * F / 16);
    if (e == cudaSuccess) e = cudaMalloc(&P->hq, MA * F / 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->hsf, MA * F / 16);
    if (e == cudaSuccess) e = cudaMalloc(&P->rp, MA * D * 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->res[0], MA * D * 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->res[1], MA * D * 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->amax, 16);
    if (e == cudaSuccess) e = cudaMalloc(&P->err, 4);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaMalloc(&P->ws, (size_t)P->num_sms * 128 * 128 * 4);
    if (e == cudaSuccess) e = cudaMalloc(&P->counters, F4_MAX_TILES * 4);
    if (e == cudaSuccess) e = cudaMemset(P->counters, 0, F4_MAX_TILES * 4);
    // the GEMMs read operand rows (and their scales) up to M_alloc: padding stays zero
    if (e == cudaSuccess) e = cudaMemset(P->xq, 0, MA * D / 2);
    if (e == cudaSuccess) e = cudaMemset(P->xsf, 0, MA * D / 16);
    if (e == cudaSuccess) e = cudaMemset(P->hq, 0, MA * F / 2);
    if (e == cudaSuccess) e = cudaMemset(P->hsf, 0, MA * F / 16);
    if (e == cudaSuccess) e = cudaMemset(P->err, 0, 4);
    if (e == cudaSuccess) e = encode_tmap_u8(&P->tm_wg, P->wg, L * F, D / 2, 128);
    if (e == cudaSuccess) e = encode_tmap_u8(&P->tm_wu, P->wu, L * F, D / 2, 128);
    if (e == cudaSuccess) e = encode_tmap_u8(&P->tm_wd, P->wd, L * D, F / 2, 128);
    if (e == cudaSuccess) e = encode_tmap_u8(&P->tm_xq, P->xq, MA, D / 2, 128);
    if (e == cudaSuccess) e = encode_tmap_u8(&P->tm_hq, P->hq, MA, F / 2, 128);
    for (int i = 0; i < 3; ++i) {
        if (e == cudaSuccess) e = encode_tmap_u8(&P->tm_xq_n[i], P->xq, MA, D / 2, 16u << i);
        if (e == cudaSuccess) e = encode_tmap_u8(&P->tm_hq_n[i], P->hq, MA, F / 2, 16u << i);
    }
    if (e != cudaSuccess) {
        free_fp4(P);
        return fcuda_fail(e, "frt_fp4_plan_create");
    }
    *out = P;
    return FRT_OK;
}

FRT_API frt_status frt_fp4_plan_destroy(frt_fp4_plan_t P) {
    if (!P)
        return FRT_OK;
    cudaDeviceSynchronize();
    free_fp4(P);
    return FRT_OK;
}

FRT_API frt_status frt_fp4_load_weights(frt_fp4_plan_t P, int layer, const void *w_norm, const void *w_gate,
                                        const void *w_up, const void *w_down, const float *awq,
                                        frt_stream_t stream) {
    if (!P)
        return ffail(FRT_ERR_INVALID_ARG, "null plan");
    if (layer < 0 || layer >= P->L)
        return ffail(FRT_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, P->L);
    if (!w_norm || !w_gate || !w_up || !w_down || !al16(w_norm) || !al16(w_gate) || !al16(w_up) || !al16(w_down) ||
        !al16(awq))
        return ffail(FRT_ERR_INVALID_ARG, "weight pointers must be non-null and 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t d = P->d, ff = P->ff;
    // AWQ: 1 / c rounded once (the activation is multiplied by it)
    std::vector<float> inv(d, 1.0f);
    if (awq) {
        std::vector<float> c(d);
        FCK(cudaMemcpyAsync(c.data(), awq, d * 4, cudaMemcpyDeviceToHost, s));
        FCK(cudaStreamSynchronize(s));
        for (size_t k = 0; k < d; ++k) {
            if (!(c[k] > 0.0f) || !std::isfinite(c[k]))
                return ffail(FRT_ERR_INVALID_ARG, "awq[%zu] must be finite and > 0", k);
            inv[k] = 1.0f / c[k];
        }
    }
    FCK(cudaMemcpyAsync(P->awq_inv + (size_t)layer * d, inv.data(), d * 4, cudaMemcpyHostToDevice, s));
    FCK(cudaMemcpyAsync(P->w_norm + (size_t)layer * d, w_norm, d * 2, cudaMemcpyDeviceToDevice, s));
    FCK(cudaMemsetAsync(P->amax, 0, 16, s));
    FCK(launch_f4_amax_w(w_gate, ff, (int)d, awq, P->amax + 0, s));
    FCK(launch_f4_amax_w(w_up, ff, (int)d, awq, P->amax + 1, s));
    FCK(launch_f4_amax_w(w_down, d, (int)ff, nullptr, P->amax + 2, s));
    unsigned words[4] = {0, 0, 0, 0};
    FCK(cudaMemcpyAsync(words, P->amax, 16, cudaMemcpyDeviceToHost, s));
    FCK(cudaStreamSynchronize(s));
    const float sg = scale_of(word_to_float(words[0]));
    const float su = scale_of(word_to_float(words[1]));
    const float sd = scale_of(word_to_float(words[2]));
    FCK(launch_f4_quant_w(w_gate, (int)ff, (int)d, awq, sg, inv6_of(sg), P->wg + (size_t)layer * ff * d / 2,
                          P->sg + (size_t)layer * wsf_bytes(ff, d), true, s));
    FCK(launch_f4_quant_w(w_up, (int)ff, (int)d, awq, su, inv6_of(su), P->wu + (size_t)layer * ff * d / 2,
                          P->su + (size_t)layer * wsf_bytes(ff, d), true, s));
    FCK(launch_f4_quant_w(w_down, (int)d, (int)ff, nullptr, sd, inv6_of(sd), P->wd + (size_t)layer * d * ff / 2,
                          P->sd + (size_t)layer * wsf_bytes(d, ff), true, s));
    FCK(cudaStreamSynchronize(s));
    P->s_wg[layer] = sg;
    P->s_wu[layer] = su;
    P->s_wd[layer] = sd;
    P->has_awq[layer] = awq != nullptr;
    P->loaded[layer] = 1;
    return FRT_OK;
}

namespace {

// N1: norm (+ AWQ) + NVFP4 quantise of layer l's input into the X buffers
// (measure: the amax of y into amax[0] instead).  With h, r' goes to P->rp.
cudaError_t f4_norm(frt_fp4_plan *P, int l, const void *r, const void *h, int M, bool measure, cudaStream_t s) {
    const float sx = P->s_x[l];
    return launch_f4_norm_quant(r, h, P->w_norm + (size_t)l * P->d, P->has_awq[l] ? P->awq_inv + (size_t)l * P->d
                                                                                   : nullptr,
                                M, P->d, F4_RMS_EPS, sx, inv6_of(sx), h ? P->rp : nullptr, P->xq, P->xsf,
                                P->amax, measure, s);
}

// N2: the gate (up = false) or up GEMM; epi F4_EPI_FP4 (into G / U) or
// F4_EPI_AMAX (into amax[0] / amax[1]).
cudaError_t f4_gate_up(frt_fp4_plan *P, int l, bool up, int M, int epi, cudaStream_t s) {
    const size_t d = P->d, ff = P->ff;
    const int sw = f4_swap_n(M);
    F4GemmParams p;
    memset(&p, 0, sizeof p);
    const uint8_t *wsf = (up ? P->su : P->sg) + (size_t)l * wsf_bytes(ff, d);
    p.sfa = sw ? wsf : P->xsf;
    p.sfb = sw ? P->xsf : wsf;
    p.a_row0 = sw ? l * P->ff : 0;
    p.b_row0 = sw ? 0 : l * P->ff;
    p.M = M;
    p.K = P->d;
    p.epi = epi;
    p.alpha = P->s_x[l] * (up ? P->s_wu[l] : P->s_wg[l]);
    p.s_out = up ? P->s_u[l] : P->s_g[l];
    p.inv6_out = inv6_of(p.s_out);
    p.out = up ? P->uq : P->gq;
    p.ldo = P->ff / 2;
    p.out_sf = up ? P->us : P->gs;
    p.ldsf = P->ff / 16;
    p.amax = P->amax + (up ? 1 : 0);
    p.err = P->err;
    p.splits = f4_splits((P->ff / 128) * (sw ? 1 : (M + 127) / 128), P->d / 256, P->num_sms);
    p.ws = P->ws;
    p.counters = P->counters;
    p.w_tiles = (up ? P->wu : P->wg) + (size_t)l * ff * d / 2;
    const CUtensorMap &w = up ? P->tm_wu : P->tm_wg;
    if (sw)
        return launch_f4_gemm(w, P->tm_xq_n[f4_swap_idx(sw)], p, P->ff, sw, s);
    return launch_f4_gemm(P->tm_xq, w, p, P->ff, 0, s);
}

// N3: A = NVFP4(act(G) * U) into the A buffers (measure: amax into amax[2]).
cudaError_t f4_geglu(frt_fp4_plan *P, int l, int M, bool measure, cudaStream_t s) {
    return launch_f4_geglu(P->gq, P->gs, P->s_g[l], P->uq, P->us, P->s_u[l], P->act, M, P->ff, P->s_h[l],
                           inv6_of(P->s_h[l]), P->hq, P->hsf, P->amax + 2, measure, s);
}

// N4: out = bf16(resid + acc(A, W_d') * alpha).
cudaError_t f4_down(frt_fp4_plan *P, int l, const void *resid, void *out, int M, cudaStream_t s) {
    const int sw = f4_swap_n(M);
    F4GemmParams p;
    memset(&p, 0, sizeof p);
    const uint8_t *wsf = P->sd + (size_t)l * wsf_bytes(P->d, P->ff);
    p.sfa = sw ? wsf : P->hsf;
    p.sfb = sw ? P->hsf : wsf;
    p.a_row0 = sw ? l * P->d : 0;
    p.b_row0 = sw ? 0 : l * P->d;
    p.M = M;
    p.K = P->ff;
    p.epi = F4_EPI_RESID;
    p.alpha = P->s_h[l] * P->s_wd[l];
    p.out = out;
    p.ldo = P->d;
    p.resid = static_cast<const uint16_t *>(resid);
    p.ldr = P->d;
    p.err = P->err;
    p.splits = f4_splits((P->d / 128) * (sw ? 1 : (M + 127) / 128), P->ff / 256, P->num_sms);
    p.ws = P->ws;
    p.counters = P->counters;
    p.w_tiles = P->wd + (size_t)l * P->d * P->ff / 2;
    if (sw)
        return launch_f4_gemm(P->tm_wd, P->tm_hq_n[f4_swap_idx(sw)], p, P->d, sw, s);
    return launch_f4_gemm(P->tm_hq, P->tm_wd, p, P->d, 0, s);
}

frt_status f4_layer(frt_fp4_plan *P, int l, const void *r, const void *h, void *out, int M, cudaStream_t s) {
    FCK(f4_norm(P, l, r, h, M, false, s));
    FCK(f4_gate_up(P, l, false, M, F4_EPI_FP4, s));
    FCK(f4_gate_up(P, l, true, M, F4_EPI_FP4, s));
    FCK(f4_geglu(P, l, M, false, s));
    FCK(f4_down(P, l, h ? static_cast<const void *>(P->rp) : r, out, M, s));
    return FRT_OK;
}

frt_status check_call(frt_fp4_plan *P, const void *r, const void *h, const void *out, int M) {
    frt_status st = check_ready(P);
    if (st != FRT_OK)
        return st;
    if (!P->scaled)
        return ffail(FRT_ERR_NOT_READY, "activation scales not calibrated or set");
    if (M < 0 || M > P->M_max)
        return ffail(M < 0 ? FRT_ERR_INVALID_ARG : FRT_ERR_SHAPE, "M=%d outside [0, M_max=%d]", M, P->M_max);
    if (!r || !out || !al16(r) || !al16(h) || !al16(out))
        return ffail(FRT_ERR_INVALID_ARG, "residual and out must be non-null; all pointers 16-byte aligned");
    return FRT_OK;
}

}  // namespace

FRT_API frt_status frt_fp4_forward(frt_fp4_plan_t P, const void *residual_in, const void *hidden_in, void *out,
                                   int M, frt_stream_t stream) {
    frt_status st = check_call(P, residual_in, hidden_in, out, M);
    if (st != FRT_OK || M == 0)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const void *cur = residual_in;
    for (int l = 0; l < P->L; ++l) {
        void *dst = l == P->L - 1 ? out : static_cast<void *>(P->res[l & 1]);
        st = f4_layer(P, l, cur, l == 0 ? hidden_in : nullptr, dst, M, s);
        if (st != FRT_OK)
            return st;
        cur = dst;
    }
    return FRT_OK;
}

FRT_API frt_status frt_fp4_calibrate(frt_fp4_plan_t P, const void *const *residual, const void *const *hidden,
                                     int n_batches, int M, frt_stream_t stream) {
    frt_status st = check_ready(P);
    if (st != FRT_OK)
        return st;
    if (!residual || n_batches < 1)
        return ffail(FRT_ERR_INVALID_ARG, "need at least one residual batch");
    if (M < 1 || M > P->M_max)
        return ffail(M < 1 ? FRT_ERR_INVALID_ARG : FRT_ERR_SHAPE, "M=%d outside [1, M_max=%d]", M, P->M_max);
    for (int b = 0; b < n_batches; ++b) {
        const void *h = hidden ? hidden[b] : nullptr;
        if (!residual[b] || !al16(residual[b]) || !al16(h))
            return ffail(FRT_ERR_INVALID_ARG, "batch %d: pointers must be non-null (residual) and 16-byte aligned",
                         b);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t per = (size_t)M * P->d;
    uint16_t *buf[2] = {nullptr, nullptr};
    cudaError_t e = cudaMalloc(&buf[0], per * n_batches * 2);
    if (e == cudaSuccess)
        e = cudaMalloc(&buf[1], per * n_batches * 2);
    if (e != cudaSuccess) {
        cudaFree(buf[0]);
        return fcuda_fail(e, "calibration scratch");
    }
    std::vector<const void *> cur(residual, residual + n_batches);
    auto read_amax = [&](float *out, int n) -> cudaError_t {
        unsigned w[4];
        cudaError_t e2 = cudaMemcpyAsync(w, P->amax, 16, cudaMemcpyDeviceToHost, s);
        if (e2 == cudaSuccess)
            e2 = cudaStreamSynchronize(s);
        for (int i = 0; i < n; ++i)
            out[i] = scale_of(word_to_float(w[i]));
        return e2;
    };
    st = FRT_OK;
    for (int l = 0; l < P->L && st == FRT_OK; ++l) {
        auto hid = [&](int b) -> const void * { return (l == 0 && hidden) ? hidden[b] : nullptr; };
        float sc[4];
        // s_x
        e = cudaMemsetAsync(P->amax, 0, 16, s);
        for (int b = 0; b < n_batches && e == cudaSuccess; ++b)
            e = f4_norm(P, l, cur[b], hid(b), M, true, s);
        if (e == cudaSuccess)
            e = read_amax(sc, 1);
        if (e != cudaSuccess)
            break;
        P->s_x[l] = sc[0];
        // s_g, s_u
        e = cudaMemsetAsync(P->amax, 0, 16, s);
        for (int b = 0; b < n_batches && e == cudaSuccess; ++b) {
            e = f4_norm(P, l, cur[b], hid(b), M, false, s);
            if (e == cudaSuccess)
                e = f4_gate_up(P, l, false, M, F4_EPI_AMAX, s);
            if (e == cudaSuccess)
                e = f4_gate_up(P, l, true, M, F4_EPI_AMAX, s);
        }
        if (e == cudaSuccess)
            e = read_amax(sc, 2);
        if (e != cudaSuccess)
            break;
        P->s_g[l] = sc[0];
        P->s_u[l] = sc[1];
        // s_h
        e = cudaMemsetAsync(P->amax, 0, 16, s);
        for (int b = 0; b < n_batches && e == cudaSuccess; ++b) {
            e = f4_norm(P, l, cur[b], hid(b), M, false, s);
            if (e == cudaSuccess)
                e = f4_gate_up(P, l, false, M, F4_EPI_FP4, s);
            if (e == cudaSuccess)
                e = f4_gate_up(P, l, true, M, F4_EPI_FP4, s);
            if (e == cudaSuccess)
                e = f4_geglu(P, l, M, true, s);
        }
        if (e == cudaSuccess)
            e = read_amax(sc, 3);
        if (e != cudaSuccess)
            break;
        P->s_h[l] = sc[2];
        // the layer's outputs feed the next layer
        if (l + 1 < P->L) {
            uint16_t *dst = buf[l & 1];
            for (int b = 0; b < n_batches && st == FRT_OK; ++b)
                st = f4_layer(P, l, cur[b], hid(b), dst + per * b, M, s);
            for (int b = 0; b < n_batches; ++b)
                cur[b] = dst + per * b;
        }
    }
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    cudaFree(buf[0]);
    cudaFree(buf[1]);
    if (e != cudaSuccess)
        return fcuda_fail(e, "frt_fp4_calibrate");
    if (st == FRT_OK)
        P->scaled = true;
    return st;
}

FRT_API frt_status frt_fp4_get_scales(frt_fp4_plan_t P, float *act, float *weight) {
    if (!P)
        return ffail(FRT_ERR_INVALID_ARG, "null plan");
    for (int l = 0; l < P->L; ++l) {
        if (act) {
            act[4 * l + 0] = P->s_x[l];
            act[4 * l + 1] = P->s_g[l];
            act[4 * l + 2] = P->s_u[l];
            act[4 * l + 3] = P->s_h[l];
        }
        if (weight) {
            weight[3 * l + 0] = P->s_wg[l];
            weight[3 * l + 1] = P->s_wu[l];
            weight[3 * l + 2] = P->s_wd[l];
        }
    }
    return FRT_OK;
}

FRT_API frt_status frt_fp4_set_scales(frt_fp4_plan_t P, const float *act) {
    if (!P || !act)
        return ffail(FRT_ERR_INVALID_ARG, "null plan or scales");
    for (int i = 0; i < 4 * P->L; ++i)
        if (!(act[i] > 0.0f) || !std::isfinite(act[i]))
            return ffail(FRT_ERR_INVALID_ARG, "scale %d must be finite and > 0", i);
    for (int l = 0; l < P->L; ++l) {
        P->s_x[l] = act[4 * l + 0];
        P->s_g[l] = act[4 * l + 1];
        P->s_u[l] = act[4 * l + 2];
        P->s_h[l] = act[4 * l + 3];
    }
    P->scaled = true;
    return FRT_OK;
}

FRT_API frt_status frt_fp4_debug_trace(frt_fp4_plan_t P, int layer, const void *residual_in, const void *hidden_in,
                                       void *out, void *r_prime, void *x_codes, void *x_sf, void *g_codes,
                                       void *g_sf, void *u_codes, void *u_sf, void *h_codes, void *h_sf, int M,
                                       frt_stream_t stream) {
    frt_status st = check_call(P, residual_in, hidden_in, out, M);
    if (st != FRT_OK || M == 0)
        return st;
    if (layer < 0 || layer >= P->L)
        return ffail(FRT_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, P->L);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = f4_layer(P, layer, residual_in, hidden_in, out, M, s);
    if (st != FRT_OK)
        return st;
    const size_t d = P->d, ff = P->ff, m = (size_t)M, mt = (size_t)(M + 127) / 128 * 128;
    const cudaMemcpyKind k = cudaMemcpyDeviceToDevice;
    if (r_prime && hidden_in) FCK(cudaMemcpyAsync(r_prime, P->rp, m * d * 2, k, s));
    if (x_codes) FCK(cudaMemcpyAsync(x_codes, P->xq, m * d / 2, k, s));
    if (x_sf) FCK(cudaMemcpyAsync(x_sf, P->xsf, mt * d / 16, k, s));
    if (g_codes) FCK(cudaMemcpyAsync(g_codes, P->gq, m * ff / 2, k, s));
    if (g_sf) FCK(cudaMemcpyAsync(g_sf, P->gs, m * ff / 16, k, s));
    if (u_codes) FCK(cudaMemcpyAsync(u_codes, P->uq, m * ff / 2, k, s));
    if (u_sf) FCK(cudaMemcpyAsync(u_sf, P->us, m * ff / 16, k, s));
    if (h_codes) FCK(cudaMemcpyAsync(h_codes, P->hq, m * ff / 2, k, s));
    if (h_sf) FCK(cudaMemcpyAsync(h_sf, P->hsf, mt * ff / 16, k, s));
    FCK(cudaStreamSynchronize(s));
    return FRT_OK;
}

FRT_API frt_status frt_fp4_debug_weights(frt_fp4_plan_t P, int layer, int which, void *codes, void *sf,
                                         frt_stream_t stream) {
    if (!P)
        return ffail(FRT_ERR_INVALID_ARG, "null plan");
    if (layer < 0 || layer >= P->L || which < 0 || which > 2)
        return ffail(FRT_ERR_INVALID_ARG, "layer %d / which %d out of range", layer, which);
    if (!P->loaded[layer])
        return ffail(FRT_ERR_NOT_READY, "weights of layer %d not loaded", layer);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t d = P->d, ff = P->ff, n = d * ff;
    const uint8_t *q = which == 0 ? P->wg : which == 1 ? P->wu : P->wd;
    const uint8_t *f = which == 0 ? P->sg : which == 1 ? P->su : P->sd;
    if (codes) FCK(cudaMemcpyAsync(codes, q + (size_t)layer * n / 2, n / 2, cudaMemcpyDeviceToDevice, s));
    if (sf) FCK(cudaMemcpyAsync(sf, f + (size_t)layer * n / 16, n / 16, cudaMemcpyDeviceToDevice, s));
    FCK(cudaStreamSynchronize(s));
    return FRT_OK;
}

FRT_API frt_status frt_nvfp4_gemm(const void *a_codes, const void *a_sf, const void *b_codes, const void *b_sf,
                                  int M, int N, int K, float alpha, float *out, int splits, float *ws, int *counters,
                                  int *err, frt_stream_t stream) {
    if (!a_codes || !a_sf || !b_codes || !b_sf || !out || !err || !al16(a_codes) || !al16(a_sf) ||
        !al16(b_codes) || !al16(b_sf) || !al16(out))
        return ffail(FRT_ERR_INVALID_ARG, "pointers must be non-null and 16-byte aligned");
    if (M < 1 || M > 65536 || N < 128 || N % 128 || K < 256 || K % 256)
        return ffail(FRT_ERR_INVALID_ARG, "M=%d N=%d K=%d: need 1 <= M <= 65536, N %% 128 == 0, K %% 256 == 0", M,
                     N, K);
    const int tiles = (N / 128) * (f4_swap_n(M) ? 1 : (M + 127) / 128);
    if (splits < 1 || splits > K / 256 || (splits > 1 && (!ws || !counters || !al16(ws) || tiles > F4_MAX_TILES)))
        return ffail(FRT_ERR_INVALID_ARG, "splits=%d: need 1 <= splits <= K / 256 and, above 1, ws and counters",
                     splits);
    // the plan's choice of role: weight-streaming for at most 64 tokens
    const int sw = f4_swap_n(M);
    CUtensorMap ta, tb;
    if (encode_tmap_u8(&ta, a_codes, (uint64_t)M, (uint64_t)K / 2, sw ? (uint32_t)sw : 128u) != cudaSuccess ||
        encode_tmap_u8(&tb, b_codes, (uint64_t)N, (uint64_t)K / 2, 128) != cudaSuccess)
        return ffail(FRT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    F4GemmParams p;
    memset(&p, 0, sizeof p);
    p.sfa = static_cast<const uint8_t *>(sw ? b_sf : a_sf);
    p.sfb = static_cast<const uint8_t *>(sw ? a_sf : b_sf);
    p.M = M;
    p.K = K;
    p.epi = F4_EPI_F32;
    p.alpha = alpha;
    p.out = out;
    p.ldo = N;
    p.err = err;
    p.splits = splits;
    p.ws = ws;
    p.counters = counters;
    FCK(sw ? launch_f4_gemm(tb, ta, p, N, sw, static_cast<cudaStream_t>(stream))
           : launch_f4_gemm(ta, tb, p, N, 0, static_cast<cudaStream_t>(stream)));
    return FRT_OK;
}

FRT_API frt_status frt_fp4_device_status(frt_fp4_plan_t P, frt_stream_t stream) {
    if (!P)
        return ffail(FRT_ERR_INVALID_ARG, "null plan");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int err = 0;
    FCK(cudaMemcpyAsync(&err, P->err, 4, cudaMemcpyDeviceToHost, s));
    FCK(cudaStreamSynchronize(s));
    if (err) {
        FCK(cudaMemset(P->err, 0, 4));
        return ffail(FRT_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (code %d)", err);
    }
    return FRT_OK;
}
