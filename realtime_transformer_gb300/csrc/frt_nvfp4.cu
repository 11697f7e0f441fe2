// frt_nvfp4.cu -- the NVFP4 sublayer stack behind frt_nvfp4.h (itsolotime
// FlashRT article, 7.2): per layer the norm + AWQ + FP4 quantise kernel
// (k_nvfp4.cu), the gate/up NVFP4 GEMM whose epilogue quantises G and U to
// NVFP4 and applies the FP4-to-FP4 gated activation, and the down NVFP4 GEMM
// with the residual epilogue (f4 launches of the tensor-core GEMM,
// k_gemm_tc.cuh), chained by programmatic dependent launch.  Tensor maps of
// the fixed buffers are encoded once at plan creation (host and device
// copies), so a forward can be captured into a graph.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
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
    // weights: codes row-major [L * rows, K/2], TMEM-ready scales rows * K/16
    // per layer; gate and up as one [W_gate; W_up] arena interleaved in
    // blocks of 64 rows (2 ff rows a layer), so a 128-row tile holds the gate
    // and up rows of the same 64 features
    uint8_t *wgu = nullptr, *wd = nullptr;
    uint8_t *sgu = nullptr, *sd = nullptr;
    uint16_t *w_norm = nullptr;  // BF16 [L, d]
    float *awq_inv = nullptr;    // fp32 [L, d]: 1 / c
    // activations
    uint8_t *xq = nullptr, *xsf = nullptr;  // [M_alloc, d/2], TMEM-ready
    uint8_t *hq = nullptr, *hsf = nullptr;  // [M_alloc, ff/2], TMEM-ready
    uint16_t *rp = nullptr;                 // r' of layer 0 [M_alloc, d]
    uint16_t *res[2] = {nullptr, nullptr};  // layer outputs between layers
    unsigned *amax = nullptr;               // [4]
    int *err = nullptr;
    int num_sms = 0;
    float *ws = nullptr;                    // split-K partials of the down GEMM
    size_t ws_floats = 0;
    int *counters = nullptr;                // split-K arrival counters (SPLIT_COUNTERS)
    std::vector<float> s_wg, s_wu, s_wd, s_x, s_g, s_u, s_h;
    // tensor maps of the fixed buffers (host copies for the kernel parameter,
    // device copies the kernels read), keyed by (buffer, box rows)
    std::map<std::pair<int, int>, std::pair<CUtensorMap, int>> tmaps;
    CUtensorMap *tmap_dev = nullptr;
    bool pdl = true;                        // programmatic dependent launch (FRT_FFN_NO_PDL=1 disables)
    // profiling: while set, launch 3 l + s of a forward (s: 0 norm, 1 gate/up,
    // 2 down) records its CTAs' %globaltimer span at stamps[2 (3 l + s)]
    unsigned long long *stamps = nullptr;
    bool profiling = false;
    std::vector<char> loaded, has_awq;
    bool scaled = false;
};

namespace {

enum F4Buf : int { F_WGU = 0, F_WD = 1, F_XQ = 2, F_HQ = 3 };

void free_fp4(frt_fp4_plan *P) {
    void *ptrs[] = {P->wgu, P->wd,  P->sgu,     P->sd,  P->w_norm, P->awq_inv, P->xq,       P->xsf,
                    P->hq,  P->hsf, P->rp,      P->res[0], P->res[1], P->amax,  P->err,      P->ws,
                    P->counters, P->tmap_dev, P->stamps};
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

// The role of a GEMM on M tokens: weight-streaming for at most 64 tokens,
// else tiled; FRT_F4_SWAP = 0 / 1 forces the tiled / weight-streaming role
// (the latter for at most 64 tokens; read per launch).
constexpr int F4_SWAP_MAX_TOKENS = 64;
bool f4_swap(int M) {
    const char *e = getenv("FRT_F4_SWAP");
    if (e && e[0] == '0')
        return false;
    return M <= F4_SWAP_MAX_TOKENS;
}

frt_status build_tmaps(frt_fp4_plan *P) {
    const int combos[][2] = {{F_WGU, 128}, {F_WGU, 256}, {F_WD, 128}, {F_WD, 256}, {F_XQ, 16},  {F_XQ, 32},
                             {F_XQ, 64},   {F_XQ, 128},  {F_HQ, 16},  {F_HQ, 32}, {F_HQ, 64}, {F_HQ, 128}};
    constexpr int N = sizeof(combos) / sizeof(combos[0]);
    CUtensorMap host[N];
    const uint64_t L = P->L, D = P->d, F = P->ff, MA = P->M_alloc;
    for (int i = 0; i < N; ++i) {
        const int buf = combos[i][0], box = combos[i][1];
        cudaError_t e;
        switch (buf) {
        case F_WGU: e = encode_tmap_u8(&host[i], P->wgu, L * 2 * F, D / 2, box); break;
        case F_WD: e = encode_tmap_u8(&host[i], P->wd, L * D, F / 2, box); break;
        case F_XQ: e = encode_tmap_u8(&host[i], P->xq, MA, D / 2, box); break;
        default: e = encode_tmap_u8(&host[i], P->hq, MA, F / 2, box); break;
        }
        if (e != cudaSuccess)
            return ffail(FRT_ERR_CUDA, "cuTensorMapEncodeTiled failed for buffer %d box %d", buf, box);
        P->tmaps[std::make_pair(buf, box)] = std::make_pair(host[i], i);
    }
    FCK(cudaMalloc(&P->tmap_dev, sizeof(CUtensorMap) * N));
    FCK(cudaMemcpy(P->tmap_dev, host, sizeof(CUtensorMap) * N, cudaMemcpyHostToDevice));
    return FRT_OK;
}

frt_status get_tmap(frt_fp4_plan *P, int buf, int box, CUtensorMap *out, const CUtensorMap **dev) {
    auto it = P->tmaps.find(std::make_pair(buf, box));
    if (it == P->tmaps.end())
        return ffail(FRT_ERR_UNSUPPORTED, "no tensor map for buffer %d box %d", buf, box);
    *out = it->second.first;
    *dev = P->tmap_dev + it->second.second;
    return FRT_OK;
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
    if (const char *np = getenv("FRT_FFN_NO_PDL"))
        P->pdl = !(np[0] == '1');
    const size_t L = n_layers, D = d, F = ff, MA = P->M_alloc;
    cudaError_t e = cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, dev);
    P->ws_floats = (size_t)P->num_sms * 128 * 256;
    if (e == cudaSuccess) e = cudaMalloc(&P->wgu, L * 2 * F * D / 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->wd, L * D * F / 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->sgu, L * wsf_bytes(2 * F, D));
    if (e == cudaSuccess) e = cudaMalloc(&P->sd, L * wsf_bytes(D, F));
    if (e == cudaSuccess) e = cudaMalloc(&P->w_norm, L * D * 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->awq_inv, L * D * 4);
    if (e == cudaSuccess) e = cudaMalloc(&P->xq, MA * D / 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->xsf, MA * D / 16);
    if (e == cudaSuccess) e = cudaMalloc(&P->hq, MA * F / 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->hsf, MA * F / 16);
    if (e == cudaSuccess) e = cudaMalloc(&P->rp, MA * D * 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->res[0], MA * D * 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->res[1], MA * D * 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->amax, 16);
    if (e == cudaSuccess) e = cudaMalloc(&P->err, 4);
    if (e == cudaSuccess) e = cudaMalloc(&P->ws, P->ws_floats * 4);
    if (e == cudaSuccess) e = cudaMalloc(&P->counters, (size_t)SPLIT_COUNTERS * 4);
    if (e == cudaSuccess) e = cudaMemset(P->counters, 0, (size_t)SPLIT_COUNTERS * 4);
    if (e == cudaSuccess) e = cudaMalloc(&P->stamps, L * 3 * 2 * sizeof(unsigned long long));
    // the GEMMs read operand rows (and their scales) up to the 128-row tile:
    // padding starts at zero
    if (e == cudaSuccess) e = cudaMemset(P->xq, 0, MA * D / 2);
    if (e == cudaSuccess) e = cudaMemset(P->xsf, 0, MA * D / 16);
    if (e == cudaSuccess) e = cudaMemset(P->hq, 0, MA * F / 2);
    if (e == cudaSuccess) e = cudaMemset(P->hsf, 0, MA * F / 16);
    if (e == cudaSuccess) e = cudaMemset(P->err, 0, 4);
    frt_status st = e == cudaSuccess ? build_tmaps(P) : fcuda_fail(e, "frt_fp4_plan_create");
    if (st != FRT_OK) {
        free_fp4(P);
        return st;
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
    uint8_t *q_gu = P->wgu + (size_t)layer * 2 * ff * d / 2;
    uint8_t *s_gu = P->sgu + (size_t)layer * wsf_bytes(2 * ff, d);
    FCK(launch_f4_quant_w(w_gate, (int)ff, (int)d, awq, sg, inv6_of(sg), q_gu, s_gu, 1, s));
    FCK(launch_f4_quant_w(w_up, (int)ff, (int)d, awq, su, inv6_of(su), q_gu, s_gu, 2, s));
    FCK(launch_f4_quant_w(w_down, (int)d, (int)ff, nullptr, sd, inv6_of(sd), P->wd + (size_t)layer * d * ff / 2,
                          P->sd + (size_t)layer * wsf_bytes(d, ff), 0, s));
    FCK(cudaStreamSynchronize(s));
    P->s_wg[layer] = sg;
    P->s_wu[layer] = su;
    P->s_wd[layer] = sd;
    P->has_awq[layer] = awq != nullptr;
    P->loaded[layer] = 1;
    return FRT_OK;
}

namespace {

// Layer l's step s stamp pair while profiling, else null.
unsigned long long *f4_stamp(const frt_fp4_plan *P, int l, int s) {
    return P->profiling ? P->stamps + 2 * ((size_t)3 * l + s) : nullptr;
}

// N1: norm (+ AWQ) + NVFP4 quantise of layer l's input into the X buffers
// (measure: the amax of y into amax[0] instead).  With h, r' goes to P->rp.
cudaError_t f4_norm(frt_fp4_plan *P, int l, const void *r, const void *h, int M, bool measure, cudaStream_t s) {
    const float sx = P->s_x[l];
    return launch_f4_norm_quant(r, h, P->w_norm + (size_t)l * P->d, P->has_awq[l] ? P->awq_inv + (size_t)l * P->d
                                                                                   : nullptr,
                                M, P->d, F4_RMS_EPS, sx, inv6_of(sx), h ? P->rp : nullptr, P->xq, P->xsf,
                                P->amax, measure, s, P->pdl, f4_stamp(P, l, 0));
}

// Tensor maps and row offsets of one GEMM of layer l: the weight buffer
// (rows_per_layer rows a layer) and the token buffer, in the launch's role.
frt_status f4_maps(frt_fp4_plan *P, GemmLaunch &g, int wbuf, int xbuf, int l, int rows_per_layer) {
    frt_status st;
    if (g.swap) {
        if ((st = get_tmap(P, wbuf, 128, &g.tmP, &g.p.gtm_p)) != FRT_OK) return st;
        if ((st = get_tmap(P, xbuf, g.bn, &g.tmQ, &g.p.gtm_q)) != FRT_OK) return st;
        g.p.p_row0 = l * rows_per_layer;
        g.p.q_row0 = 0;
    } else {
        if ((st = get_tmap(P, xbuf, 128, &g.tmP, &g.p.gtm_p)) != FRT_OK) return st;
        if ((st = get_tmap(P, wbuf, g.bn, &g.tmQ, &g.p.gtm_q)) != FRT_OK) return st;
        g.p.p_row0 = 0;
        g.p.q_row0 = l * rows_per_layer;
    }
    return FRT_OK;
}

// N2 + N3: the fused gate/up GEMM: G and U as NVFP4, act(dec G) * dec U
// requantised into the A buffers (epi EPI_F4_GATED), or the calibration
// amaxes (EPI_F4_AMAX_GU: amax[0], amax[1]; EPI_F4_AMAX_H: amax[2]).  dbg: G
// and U codes and row-major scales (trace), or nulls.
frt_status f4_gate_up(frt_fp4_plan *P, int l, int M, int epi, cudaStream_t s, uint8_t *const dbg[4],
                      bool stall = false) {
    GemmLaunch g;
    memset(&g.p, 0, sizeof g.p);
    plan_gemm(g, f4_swap(M), M, 2 * P->ff, P->d / 2, P->num_sms, 1, nullptr, true);
    frt_status st = f4_maps(P, g, F_WGU, F_XQ, l, 2 * P->ff);
    if (st != FRT_OK)
        return st;
    GemmParams &p = g.p;
    p.epi = epi;
    p.alpha = P->s_x[l] * P->s_wg[l];
    p.alpha_u = P->s_x[l] * P->s_wu[l];
    p.s_g = P->s_g[l];
    p.inv6_g = inv6_of(p.s_g);
    p.s_u = P->s_u[l];
    p.inv6_u = inv6_of(p.s_u);
    p.s_h = P->s_h[l];
    p.inv6_h = inv6_of(p.s_h);
    p.out = P->hq;
    p.ldo = P->ff / 2;
    p.out_sf = P->hsf;
    p.ff = P->ff;
    p.act = P->act;
    p.amax = P->amax;
    p.sf_w = P->sgu;
    p.sf_x = P->xsf;
    p.err = P->err;
    if (dbg) {
        p.dbg_gq = dbg[0];
        p.dbg_gs = dbg[1];
        p.dbg_uq = dbg[2];
        p.dbg_us = dbg[3];
    }
    p.stall_test = stall ? 1 : 0;
    p.stamp = f4_stamp(P, l, 1);
    FCK(launch_gemm(g, s, P->pdl && !stall));
    return FRT_OK;
}

// N4: out = bf16(resid + acc(A, W_d') * alpha).
frt_status f4_down(frt_fp4_plan *P, int l, const void *resid, void *out, int M, cudaStream_t s) {
    GemmLaunch g;
    memset(&g.p, 0, sizeof g.p);
    int force = 0;
    if (const char *e = getenv("FRT_F4_DOWN_SPLITS"))
        force = atoi(e);
    plan_gemm(g, f4_swap(M), M, P->d, P->ff / 2, P->num_sms, force, nullptr, true);
    frt_status st = f4_maps(P, g, F_WD, F_HQ, l, P->d);
    if (st != FRT_OK)
        return st;
    if (gemm_ws_floats(g) > P->ws_floats || (g.p.splits > 1 && gemm_tiles(g) > MAX_SPLIT_TILES))
        return ffail(FRT_ERR_UNSUPPORTED, "split-K workspace too small for M=%d", M);
    GemmParams &p = g.p;
    p.epi = EPI_RESID;
    p.alpha = P->s_h[l] * P->s_wd[l];
    p.out = out;
    p.ldo = P->d;
    p.resid = resid;
    p.ldr = P->d;
    p.sf_w = P->sd;
    p.sf_x = P->hsf;
    p.ws = P->ws;
    p.counters = split_counters(P->counters, p.splits);
    p.err = P->err;
    p.stamp = f4_stamp(P, l, 2);
    FCK(launch_gemm(g, s, P->pdl));
    return FRT_OK;
}

frt_status f4_layer(frt_fp4_plan *P, int l, const void *r, const void *h, void *out, int M, cudaStream_t s,
                    uint8_t *const dbg[4] = nullptr) {
    FCK(f4_norm(P, l, r, h, M, false, s));
    frt_status st = f4_gate_up(P, l, M, EPI_F4_GATED, s, dbg);
    if (st != FRT_OK)
        return st;
    return f4_down(P, l, h ? static_cast<const void *>(P->rp) : r, out, M, s);
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

FRT_API frt_status frt_fp4_forward_profile(frt_fp4_plan_t P, const void *residual_in, const void *hidden_in,
                                           void *out, int M, int n_replays, float *kernel_us, int *n_kernels,
                                           frt_stream_t stream) {
    frt_status st = check_call(P, residual_in, hidden_in, out, M);
    if (st != FRT_OK)
        return st;
    if (M < 1 || !kernel_us || n_replays < 1 || n_replays > 10000)
        return ffail(FRT_ERR_INVALID_ARG, "need M >= 1, kernel_us and 1 <= n_replays <= 10000");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!s)
        return ffail(FRT_ERR_INVALID_ARG, "profiling captures a graph: needs a stream other than the default");
    // the forward captured once with every launch stamping its pair
    FCK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
    P->profiling = true;
    st = frt_fp4_forward(P, residual_in, hidden_in, out, M, stream);
    P->profiling = false;
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(s, &graph);
    if (st != FRT_OK || e != cudaSuccess) {
        if (graph)
            cudaGraphDestroy(graph);
        return st != FRT_OK ? st : fcuda_fail(e, "profiling capture");
    }
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess)
        return fcuda_fail(e, "profiling graph instantiate");
    const int nk = 3 * P->L;
    std::vector<unsigned long long> h(2 * (size_t)nk);
    std::vector<std::vector<float>> dur(nk);
    for (int i = 0; i < n_replays && e == cudaSuccess; ++i) {
        if ((e = cudaMemsetAsync(P->stamps, 0, h.size() * sizeof(unsigned long long), s)) != cudaSuccess) break;
        if ((e = cudaGraphLaunch(exec, s)) != cudaSuccess) break;
        if ((e = cudaMemcpyAsync(h.data(), P->stamps, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost,
                                 s)) != cudaSuccess) break;
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess) break;
        // launch k's share: from its first CTA's start, or the end of the
        // launches before it if later, to its last CTA's end
        unsigned long long prev_end = 0;
        for (int k = 0; k < nk; ++k) {
            const unsigned long long t0 = ~h[2 * k], t1 = h[2 * k + 1];
            const unsigned long long from = std::max(t0, prev_end);
            dur[k].push_back(t1 > from ? (float)(t1 - from) * 1e-3f : 0.0f);
            prev_end = std::max(prev_end, t1);
        }
    }
    cudaGraphExecDestroy(exec);
    if (e != cudaSuccess)
        return fcuda_fail(e, "profiling replays");
    for (int k = 0; k < nk; ++k) {
        std::sort(dur[k].begin(), dur[k].end());
        kernel_us[k] = dur[k][dur[k].size() / 2];
    }
    if (n_kernels)
        *n_kernels = nk;
    return frt_fp4_device_status(P, stream);
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
    auto read_amax = [&](float *out) -> cudaError_t {
        unsigned w[4];
        cudaError_t e2 = cudaMemcpyAsync(w, P->amax, 16, cudaMemcpyDeviceToHost, s);
        if (e2 == cudaSuccess)
            e2 = cudaStreamSynchronize(s);
        for (int i = 0; i < 4; ++i)
            out[i] = scale_of(word_to_float(w[i]));
        return e2;
    };
    st = FRT_OK;
    for (int l = 0; l < P->L && st == FRT_OK && e == cudaSuccess; ++l) {
        auto hid = [&](int b) -> const void * { return (l == 0 && hidden) ? hidden[b] : nullptr; };
        float sc[4];
        // s_x
        e = cudaMemsetAsync(P->amax, 0, 16, s);
        for (int b = 0; b < n_batches && e == cudaSuccess; ++b)
            e = f4_norm(P, l, cur[b], hid(b), M, true, s);
        if (e == cudaSuccess)
            e = read_amax(sc);
        if (e != cudaSuccess)
            break;
        P->s_x[l] = sc[0];
        // s_g and s_u, then s_h with G and U quantised by them
        for (int pass = 0; pass < 2 && st == FRT_OK && e == cudaSuccess; ++pass) {
            e = cudaMemsetAsync(P->amax, 0, 16, s);
            for (int b = 0; b < n_batches && e == cudaSuccess && st == FRT_OK; ++b) {
                e = f4_norm(P, l, cur[b], hid(b), M, false, s);
                if (e == cudaSuccess)
                    st = f4_gate_up(P, l, M, pass == 0 ? EPI_F4_AMAX_GU : EPI_F4_AMAX_H, s, nullptr);
            }
            if (e == cudaSuccess && st == FRT_OK)
                e = read_amax(sc);
            if (e != cudaSuccess || st != FRT_OK)
                break;
            if (pass == 0) {
                P->s_g[l] = sc[0];
                P->s_u[l] = sc[1];
            } else {
                P->s_h[l] = sc[2];
            }
        }
        // the layer's outputs feed the next layer
        if (l + 1 < P->L && e == cudaSuccess && st == FRT_OK) {
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
    if ((g_codes || g_sf || u_codes || u_sf) && !(g_codes && g_sf && u_codes && u_sf))
        return ffail(FRT_ERR_INVALID_ARG, "g/u codes and scales: all four or none");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *const dbg[4] = {static_cast<uint8_t *>(g_codes), static_cast<uint8_t *>(g_sf),
                             static_cast<uint8_t *>(u_codes), static_cast<uint8_t *>(u_sf)};
    st = f4_layer(P, layer, residual_in, hidden_in, out, M, s, g_codes ? dbg : nullptr);
    if (st != FRT_OK)
        return st;
    const size_t d = P->d, ff = P->ff, m = (size_t)M, mt = (size_t)(M + 127) / 128 * 128;
    const cudaMemcpyKind k = cudaMemcpyDeviceToDevice;
    if (r_prime && hidden_in) FCK(cudaMemcpyAsync(r_prime, P->rp, m * d * 2, k, s));
    if (x_codes) FCK(cudaMemcpyAsync(x_codes, P->xq, m * d / 2, k, s));
    if (x_sf) FCK(cudaMemcpyAsync(x_sf, P->xsf, mt * d / 16, k, s));
    if (h_codes) FCK(cudaMemcpyAsync(h_codes, P->hq, m * ff / 2, k, s));
    if (h_sf) FCK(cudaMemcpyAsync(h_sf, P->hsf, mt * ff / 16, k, s));
    FCK(cudaStreamSynchronize(s));
    return FRT_OK;
}

FRT_API frt_status frt_fp4_debug_trace_from(frt_fp4_plan_t P, int layer, const void *residual_in,
                                           const void *hidden_in, const void *x_codes_in, const void *x_sf_in,
                                           const void *h_codes_in, const void *h_sf_in, void *out, void *g_codes,
                                           void *g_sf, void *u_codes, void *u_sf, void *h_codes, void *h_sf, int M,
                                           frt_stream_t stream) {
    frt_status st = check_call(P, residual_in, hidden_in, out, M);
    if (st != FRT_OK || M == 0)
        return st;
    if (layer < 0 || layer >= P->L)
        return ffail(FRT_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, P->L);
    if ((g_codes || g_sf || u_codes || u_sf) && !(g_codes && g_sf && u_codes && u_sf))
        return ffail(FRT_ERR_INVALID_ARG, "g/u codes and scales: all four or none");
    if (!x_codes_in != !x_sf_in || !h_codes_in != !h_sf_in)
        return ffail(FRT_ERR_INVALID_ARG, "injected codes and scales come in pairs");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t d = P->d, ff = P->ff, m = (size_t)M, mt = (size_t)(M + 127) / 128 * 128;
    const cudaMemcpyKind k = cudaMemcpyDeviceToDevice;
    uint8_t *const dbg[4] = {static_cast<uint8_t *>(g_codes), static_cast<uint8_t *>(g_sf),
                             static_cast<uint8_t *>(u_codes), static_cast<uint8_t *>(u_sf)};
    FCK(f4_norm(P, layer, residual_in, hidden_in, M, false, s));
    if (x_codes_in) {
        FCK(cudaMemcpyAsync(P->xq, x_codes_in, m * d / 2, k, s));
        FCK(cudaMemcpyAsync(P->xsf, x_sf_in, mt * d / 16, k, s));
    }
    st = f4_gate_up(P, layer, M, EPI_F4_GATED, s, g_codes ? dbg : nullptr);
    if (st != FRT_OK)
        return st;
    if (h_codes) FCK(cudaMemcpyAsync(h_codes, P->hq, m * ff / 2, k, s));
    if (h_sf) FCK(cudaMemcpyAsync(h_sf, P->hsf, mt * ff / 16, k, s));
    if (h_codes_in) {
        FCK(cudaMemcpyAsync(P->hq, h_codes_in, m * ff / 2, k, s));
        FCK(cudaMemcpyAsync(P->hsf, h_sf_in, mt * ff / 16, k, s));
    }
    st = f4_down(P, layer, hidden_in ? static_cast<const void *>(P->rp) : residual_in, out, M, s);
    if (st != FRT_OK)
        return st;
    FCK(cudaStreamSynchronize(s));
    return FRT_OK;
}

namespace {

// Byte offset of (row, 16-element group g) in the TMEM-ready scale order of
// an operand with K elements per row (as the kernels' sf_offset).
size_t sf_off(size_t row, size_t g, size_t K) {
    const size_t r = row & 127;
    return ((row >> 7) * (K >> 6) + (g >> 2)) * 512u + (r & 31) * 16 + (r >> 5) * 4 + (g & 3);
}

}  // namespace

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
    if (which == 2) {
        if (codes) FCK(cudaMemcpyAsync(codes, P->wd + (size_t)layer * n / 2, n / 2, cudaMemcpyDeviceToDevice, s));
        if (sf) FCK(cudaMemcpyAsync(sf, P->sd + (size_t)layer * n / 16, n / 16, cudaMemcpyDeviceToDevice, s));
        FCK(cudaStreamSynchronize(s));
        return FRT_OK;
    }
    // gate or up: pick its rows out of the layer's interleaved arena (host side)
    std::vector<uint8_t> arena_q(2 * n / 2), arena_s(2 * n / 16), q(n / 2), f(n / 16);
    FCK(cudaMemcpyAsync(arena_q.data(), P->wgu + (size_t)layer * 2 * n / 2, 2 * n / 2, cudaMemcpyDeviceToHost, s));
    FCK(cudaMemcpyAsync(arena_s.data(), P->sgu + (size_t)layer * 2 * n / 16, 2 * n / 16, cudaMemcpyDeviceToHost, s));
    FCK(cudaStreamSynchronize(s));
    const size_t G = d / 16;
    for (size_t j = 0; j < ff; ++j) {
        const size_t src = (j / 64) * 128 + (which == 1 ? 64 : 0) + j % 64;
        memcpy(&q[j * (d / 2)], &arena_q[src * (d / 2)], d / 2);
        for (size_t g = 0; g < G; ++g)
            f[sf_off(j, g, d)] = arena_s[sf_off(src, g, d)];
    }
    if (codes) FCK(cudaMemcpyAsync(codes, q.data(), n / 2, cudaMemcpyHostToDevice, s));
    if (sf) FCK(cudaMemcpyAsync(sf, f.data(), n / 16, cudaMemcpyHostToDevice, s));
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
    const bool swap = f4_swap(M);
    const int tiles = (N / 128) * (swap ? 1 : (M + 127) / 128);
    if (splits < 1 || splits > K / 256 || (splits > 1 && (!ws || !counters || !al16(ws) || tiles > MAX_SPLIT_TILES)))
        return ffail(FRT_ERR_INVALID_ARG, "splits=%d: need 1 <= splits <= K / 256 and, above 1, ws and counters",
                     splits);
    int dev = 0, sms = 0;
    FCK(cudaGetDevice(&dev));
    FCK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    GemmLaunch g;
    memset(&g.p, 0, sizeof g.p);
    plan_gemm(g, swap, M, N, K / 2, sms, splits, nullptr, true);
    // swap: A (the tokens) is the narrow operand, B (the weights) the 128-row one
    cudaError_t e1, e2;
    if (swap) {
        e1 = encode_tmap_u8(&g.tmP, b_codes, (uint64_t)N, (uint64_t)K / 2, 128);
        e2 = encode_tmap_u8(&g.tmQ, a_codes, (uint64_t)M, (uint64_t)K / 2, (uint32_t)g.bn);
    } else {
        e1 = encode_tmap_u8(&g.tmP, a_codes, (uint64_t)M, (uint64_t)K / 2, 128);
        e2 = encode_tmap_u8(&g.tmQ, b_codes, (uint64_t)N, (uint64_t)K / 2, (uint32_t)g.bn);
    }
    if (e1 != cudaSuccess || e2 != cudaSuccess)
        return ffail(FRT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    GemmParams &p = g.p;
    p.sf_w = static_cast<const uint8_t *>(b_sf);
    p.sf_x = static_cast<const uint8_t *>(a_sf);
    p.epi = EPI_F32;
    p.alpha = alpha;
    p.out = out;
    p.ldo = N;
    p.ws = ws;
    p.counters = counters;
    p.err = err;
    FCK(launch_gemm(g, static_cast<cudaStream_t>(stream), false));
    return FRT_OK;
}

FRT_API frt_status frt_fp4_debug_stall(frt_fp4_plan_t P, int M, frt_stream_t stream) {
    if (!P)
        return ffail(FRT_ERR_INVALID_ARG, "null plan");
    if (M < 1 || M > P->M_max)
        return ffail(M < 1 ? FRT_ERR_INVALID_ARG : FRT_ERR_SHAPE, "M=%d outside [1, M_max=%d]", M, P->M_max);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const frt_status st = f4_gate_up(P, 0, M, EPI_F4_GATED, s, nullptr, true);
    if (st != FRT_OK)
        return st;
    return frt_fp4_device_status(P, stream);
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
        // a launch that gave up may have left split-K counters mid-generation
        FCK(cudaMemset(P->counters, 0, (size_t)SPLIT_COUNTERS * 4));
        return ffail(FRT_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (code %d)", err);
    }
    return FRT_OK;
}
