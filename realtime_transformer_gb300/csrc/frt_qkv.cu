// frt_qkv.cu -- the attention-input sublayer behind frt_qkv.h: residual +
// RMSNorm + E4M3 quantise (the FFN's norm kernel), the FP8 fused-QKV GEMM
// (the FFN's GEMM kernels, BF16 epilogue), then QKV split + RoPE
// (agentlenshq FlashRT summary, "What it is"; itsolotime FlashRT article, 5.2
// FusedQKV; "FlashRT docs/architecture.md", 8 Kernel Library).
//
// Per call two or three kernels on the caller's stream, each with a
// programmatic-dependent-launch edge to its predecessor: the split + RoPE
// runs in the GEMM's epilogue where the GEMM's tiles hold whole heads and
// need no split-K (many tokens), else as a kernel of its own.  Tensor maps are encoded per
// launch on the host (kernel parameters), so a forward holds no state that a
// later call could invalidate, and it can be captured by the caller.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "frt_internal.h"
#include "frt_qkv.h"

#define FRT_API extern "C" __attribute__((visibility("default")))

using namespace frt;

namespace {

constexpr float QKV_RMS_EPS = 1e-6f;  // the FFN's reading: the pages never state it
constexpr int QKV_SWAP_MAX_TOKENS = 64;

frt_status qfail(frt_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    set_last_error(buf);
    return st;
}

frt_status qcuda_fail(cudaError_t e, const char *what) {
    return qfail(e == cudaErrorMemoryAllocation ? FRT_ERR_OOM : FRT_ERR_CUDA, "%s: %s (%s)", what,
                 cudaGetErrorString(e), cudaGetErrorName(e));
}

#define QCK(call)                                  \
    do {                                           \
        cudaError_t e_ = (call);                   \
        if (e_ != cudaSuccess)                     \
            return qcuda_fail(e_, #call);          \
    } while (0)

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

struct frt_qkv_plan {
    int d = 0, nq = 0, nkv = 0, hd = 0, M_max = 0, L = 0, N = 0;
    int num_sms = 0, M_alloc = 0;
    uint8_t *w = nullptr;        // E4M3 [L * N, d]
    uint16_t *w_norm = nullptr;  // BF16 [L, d]
    float *inv_freq = nullptr;   // fp32 [hd / 2]
    uint8_t *qx = nullptr;       // E4M3 [M_alloc, d]
    uint16_t *qkv = nullptr;     // BF16 [M_max, N]
    float2 *rope_cs = nullptr;   // (cos, sin) [M_max, hd / 2] (fused split + RoPE)
    float *ws = nullptr;
    size_t ws_floats = 0;
    int *counters = nullptr;
    unsigned *amax = nullptr;
    int *err = nullptr;
    std::vector<float> s_x, s_qkv;
    std::vector<char> loaded;
};

namespace {

void free_qkv(frt_qkv_plan *P) {
    void *ptrs[] = {P->w, P->w_norm, P->inv_freq, P->qx, P->qkv, P->rope_cs, P->ws, P->counters, P->amax, P->err};
    for (void *p : ptrs)
        if (p) cudaFree(p);
    delete P;
}

frt_status check_layer_ready(frt_qkv_plan *P, int layer) {
    if (!P)
        return qfail(FRT_ERR_INVALID_ARG, "null plan");
    if (layer < 0 || layer >= P->L)
        return qfail(FRT_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, P->L);
    if (!P->loaded[layer])
        return qfail(FRT_ERR_NOT_READY, "weights of layer %d not loaded", layer);
    return FRT_OK;
}

// The fused-QKV GEMM launch of layer l for M tokens; tensor maps encoded
// here.  Epilogue: the split + RoPE itself (tiled tiles without split-K that
// hold whole heads; outputs q, k, v) when `fuse` allows, else BF16 into the
// plan's qkv scratch for the split + RoPE kernel.  *fused tells which.
frt_status setup_qkv_gemm(frt_qkv_plan *P, GemmLaunch &g, int l, int M, bool fuse, const int *pos, void *q,
                          void *k, void *v, bool *fused) {
    const bool swap = M <= QKV_SWAP_MAX_TOKENS;
    memset(&g.p, 0, sizeof g.p);
    plan_gemm(g, swap, M, P->N, P->d, P->num_sms, 0);
    if (gemm_ws_floats(g) > P->ws_floats || (g.p.splits > 1 && gemm_tiles(g) > MAX_SPLIT_TILES))
        return qfail(FRT_ERR_UNSUPPORTED, "split-K workspace too small for M=%d", M);
    const uint8_t *wl = P->w + (size_t)l * P->N * P->d;
    cudaError_t e1, e2;
    if (swap) {
        e1 = encode_tmap_u8(&g.tmP, wl, P->N, P->d, 128);
        e2 = encode_tmap_u8(&g.tmQ, P->qx, P->M_alloc, P->d, g.bn);
    } else {
        e1 = encode_tmap_u8(&g.tmP, P->qx, P->M_alloc, P->d, 128);
        e2 = encode_tmap_u8(&g.tmQ, wl, P->N, P->d, g.bn / (g.p.pair ? 2 : 1));
    }
    if (e1 != cudaSuccess || e2 != cudaSuccess)
        return qfail(FRT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    *fused = fuse && !swap && g.p.splits == 1 && g.bn % P->hd == 0 && P->hd % 64 == 0;
    g.p.epi = *fused ? EPI_ROPE : EPI_BF16;
    g.p.alpha = P->s_x[l] * P->s_qkv[l];
    g.p.out = P->qkv;
    g.p.ldo = P->N;
    g.p.rope_cs = P->rope_cs;
    g.p.rope_hd = P->hd;
    g.p.rope_nq = P->nq;
    g.p.rope_nkv = P->nkv;
    g.p.rope_q = static_cast<uint16_t *>(q);
    g.p.rope_k = static_cast<uint16_t *>(k);
    g.p.rope_v = static_cast<uint16_t *>(v);
    g.p.ws = P->ws;
    g.p.counters = split_counters(P->counters, g.p.splits);
    g.p.err = P->err;
    return FRT_OK;
}

// qx_in != null (diagnostics): the caller's E4M3 codes take the place of the
// norm's output (r, h, rp unused), launched without dependency edges.
frt_status run_qkv(frt_qkv_plan *P, int l, const void *r, const void *h, const int *pos, void *rp, void *q, void *k,
                   void *v, int M, cudaStream_t s, void *trace_qx, void *trace_qkv, const void *qx_in = nullptr) {
    // The split + RoPE in the GEMM's epilogue where it can run there and the
    // GEMM's K is long enough to hide it behind the MMAs of the next tile
    // (measured on GB300: 5.6% faster at d = 5120, 8192 tokens; 32% slower at
    // d = 2048, 968 tokens).  FRT_QKV_FUSE=1 fuses wherever it can, 0 never.
    // A trace of the intermediates needs the GEMM's BF16 output: the kernel.
    const char *fe = getenv("FRT_QKV_FUSE");
    const bool fuse = !trace_qkv && (fe ? fe[0] == '1' : P->d >= 4096);
    GemmLaunch g;
    bool fused = false;
    frt_status st = setup_qkv_gemm(P, g, l, M, fuse, pos, q, k, v, &fused);
    if (st != FRT_OK)
        return st;
    const float inv_sx = 1.0f / P->s_x[l];
    // the fused epilogue's (cos, sin) table, ahead of the norm kernel (whose
    // dependency wait orders it before the GEMM)
    const bool pdl = qx_in == nullptr;
    if (qx_in)
        QCK(cudaMemcpyAsync(P->qx, qx_in, (size_t)M * P->d, cudaMemcpyDeviceToDevice, s));
    if (fused)
        QCK(launch_rope_table(pos, P->inv_freq, M, P->hd / 2, P->rope_cs, s, pdl));
    // r' is stored only with a hidden input (otherwise r' = r) and only if asked for
    if (!qx_in)
        QCK(launch_norm_quant(r, h, P->w_norm + (size_t)l * P->d, M, P->d, QKV_RMS_EPS, inv_sx, h ? rp : nullptr,
                              P->qx, nullptr, false, s, true));
    QCK(launch_gemm(g, s, pdl));
    if (!fused)
        QCK(launch_rope_split(P->qkv, M, P->nq, P->nkv, P->hd, pos, P->inv_freq, q, k, v, s, pdl));
    if (rp && !h && !qx_in)
        QCK(cudaMemcpyAsync(rp, r, (size_t)M * P->d * 2, cudaMemcpyDeviceToDevice, s));
    if (trace_qx)
        QCK(cudaMemcpyAsync(trace_qx, P->qx, (size_t)M * P->d, cudaMemcpyDeviceToDevice, s));
    if (trace_qkv)
        QCK(cudaMemcpyAsync(trace_qkv, P->qkv, (size_t)M * P->N * 2, cudaMemcpyDeviceToDevice, s));
    return FRT_OK;
}

}  // namespace

FRT_API frt_status frt_qkv_plan_create(int d, int n_q_heads, int n_kv_heads, int head_dim, float rope_base, int M_max,
                                       int n_layers, frt_qkv_plan_t *out) {
    if (!out)
        return qfail(FRT_ERR_INVALID_ARG, "out must be non-null");
    *out = nullptr;
    if (d <= 0 || d % 128)
        return qfail(FRT_ERR_INVALID_ARG, "d must be a positive multiple of 128 (got %d)", d);
    if (head_dim < 16 || head_dim > 512 || head_dim % 8)
        return qfail(FRT_ERR_INVALID_ARG, "head_dim must be a multiple of 8 in [16, 512] (got %d)", head_dim);
    if (n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads)
        return qfail(FRT_ERR_INVALID_ARG, "need n_q_heads >= 1, n_kv_heads >= 1, n_kv_heads | n_q_heads");
    const long long N = (long long)(n_q_heads + 2 * n_kv_heads) * head_dim;
    if (N % 128 || N > (1 << 20))
        return qfail(FRT_ERR_INVALID_ARG, "(n_q_heads + 2 n_kv_heads) head_dim must be a multiple of 128");
    if (!(rope_base > 1.0f) || !std::isfinite(rope_base))
        return qfail(FRT_ERR_INVALID_ARG, "rope_base must be finite and > 1");
    if (M_max < 1 || M_max > 65536 || n_layers < 1 || n_layers > 4096)
        return qfail(FRT_ERR_INVALID_ARG, "need 1 <= M_max <= 65536 and 1 <= n_layers <= 4096");
    int dev = 0, major = 0, minor = 0;
    QCK(cudaGetDevice(&dev));
    QCK(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    QCK(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    if (major != 10 || minor != 3)
        return qfail(FRT_ERR_UNSUPPORTED, "this build runs on compute capability 10.3 (got %d.%d)", major, minor);
    frt_qkv_plan *P = new frt_qkv_plan();
    P->d = d;
    P->nq = n_q_heads;
    P->nkv = n_kv_heads;
    P->hd = head_dim;
    P->M_max = M_max;
    P->L = n_layers;
    P->N = (int)N;
    P->M_alloc = (M_max + 127) / 128 * 128;
    P->s_x.assign(n_layers, 0.0f);
    P->s_qkv.assign(n_layers, 1.0f);
    P->loaded.assign(n_layers, 0);
    cudaError_t e = cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, dev);
    // theta_i = base^(-2i / hd) in fp64, rounded to fp32
    std::vector<float> inv(head_dim / 2);
    for (int i = 0; i < head_dim / 2; ++i)
        inv[i] = (float)std::pow((double)rope_base, -2.0 * i / head_dim);
    P->ws_floats = (size_t)P->num_sms * 128 * 256;
    const size_t wbytes = (size_t)n_layers * P->N * d;
    if (e == cudaSuccess) e = cudaMalloc(&P->w, wbytes);
    if (e == cudaSuccess) e = cudaMalloc(&P->w_norm, (size_t)n_layers * d * 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->inv_freq, inv.size() * 4);
    if (e == cudaSuccess) e = cudaMalloc(&P->qx, (size_t)P->M_alloc * d);
    if (e == cudaSuccess) e = cudaMalloc(&P->qkv, (size_t)M_max * P->N * 2);
    if (e == cudaSuccess) e = cudaMalloc(&P->rope_cs, (size_t)M_max * (head_dim / 2) * sizeof(float2));
    if (e == cudaSuccess) e = cudaMalloc(&P->ws, P->ws_floats * 4);
    if (e == cudaSuccess) e = cudaMalloc(&P->counters, (size_t)SPLIT_COUNTERS * 4);
    if (e == cudaSuccess) e = cudaMalloc(&P->amax, 4);
    if (e == cudaSuccess) e = cudaMalloc(&P->err, 4);
    if (e == cudaSuccess) e = cudaMemcpy(P->inv_freq, inv.data(), inv.size() * 4, cudaMemcpyHostToDevice);
    // the GEMM's A tiles read rows up to M_alloc: keep the padding rows zero
    if (e == cudaSuccess) e = cudaMemset(P->qx, 0, (size_t)P->M_alloc * d);
    if (e == cudaSuccess) e = cudaMemset(P->counters, 0, (size_t)SPLIT_COUNTERS * 4);
    if (e == cudaSuccess) e = cudaMemset(P->err, 0, 4);
    if (e != cudaSuccess) {
        free_qkv(P);
        return qcuda_fail(e, "frt_qkv_plan_create");
    }
    *out = P;
    return FRT_OK;
}

FRT_API frt_status frt_qkv_plan_destroy(frt_qkv_plan_t P) {
    if (!P)
        return FRT_OK;
    cudaDeviceSynchronize();
    free_qkv(P);
    return FRT_OK;
}

FRT_API frt_status frt_qkv_load_weights(frt_qkv_plan_t P, int layer, const void *w_norm, const void *w_q,
                                        const void *w_k, const void *w_v, frt_stream_t stream) {
    return frt_qkv_load_weights_ex(P, layer, w_norm, w_q, w_k, w_v, 0u, stream);
}

FRT_API frt_status frt_qkv_load_weights_ex(frt_qkv_plan_t P, int layer, const void *w_norm, const void *w_q,
                                           const void *w_k, const void *w_v, unsigned flags, frt_stream_t stream) {
    if (!P)
        return qfail(FRT_ERR_INVALID_ARG, "null plan");
    if (flags & ~(unsigned)FRT_LOAD_FOLD_NORM)
        return qfail(FRT_ERR_INVALID_ARG, "unknown load flags 0x%x", flags);
    const bool fold = (flags & FRT_LOAD_FOLD_NORM) != 0;
    if (layer < 0 || layer >= P->L)
        return qfail(FRT_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, P->L);
    if (!w_norm || !w_q || !w_k || !w_v || !al16(w_norm) || !al16(w_q) || !al16(w_k) || !al16(w_v))
        return qfail(FRT_ERR_INVALID_ARG, "weight pointers must be non-null and 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t d = P->d, nq = (size_t)P->nq * P->hd, nk = (size_t)P->nkv * P->hd;
    uint8_t *dst = P->w + (size_t)layer * P->N * d;
    // folded: the norm weight moves into [W_q; W_k; W_v] and the norm multiplies by ones
    const std::vector<uint16_t> ones(fold ? d : 0, (uint16_t)0x3F80);
    QCK(cudaMemcpyAsync(P->w_norm + (size_t)layer * d, fold ? (const void *)ones.data() : w_norm, d * 2,
                        fold ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice, s));
    // one scale over [W_q; W_k; W_v]
    QCK(cudaMemsetAsync(P->amax, 0, 4, s));
    if (fold) {
        QCK(launch_amax_fold(w_q, nq, (int)d, w_norm, P->amax, s));
        QCK(launch_amax_fold(w_k, nk, (int)d, w_norm, P->amax, s));
        QCK(launch_amax_fold(w_v, nk, (int)d, w_norm, P->amax, s));
    } else {
        QCK(launch_amax_bf16(w_q, nq * d, P->amax, s));
        QCK(launch_amax_bf16(w_k, nk * d, P->amax, s));
        QCK(launch_amax_bf16(w_v, nk * d, P->amax, s));
    }
    unsigned h_amax = 0;
    QCK(cudaMemcpyAsync(&h_amax, P->amax, 4, cudaMemcpyDeviceToHost, s));
    QCK(cudaStreamSynchronize(s));
    float a;
    memcpy(&a, &h_amax, 4);
    const float sc = a == 0.0f ? 1.0f : a / 448.0f;
    const float inv = 1.0f / sc;
    if (fold) {
        QCK(launch_quant_fold(w_q, nq, (int)d, w_norm, inv, dst, s));
        QCK(launch_quant_fold(w_k, nk, (int)d, w_norm, inv, dst + nq * d, s));
        QCK(launch_quant_fold(w_v, nk, (int)d, w_norm, inv, dst + (nq + nk) * d, s));
    } else {
        QCK(launch_quant_bf16(w_q, nq * d, inv, dst, s));
        QCK(launch_quant_bf16(w_k, nk * d, inv, dst + nq * d, s));
        QCK(launch_quant_bf16(w_v, nk * d, inv, dst + (nq + nk) * d, s));
    }
    QCK(cudaStreamSynchronize(s));
    P->s_qkv[layer] = sc;
    P->loaded[layer] = 1;
    return FRT_OK;
}

FRT_API frt_status frt_qkv_calibrate(frt_qkv_plan_t P, int layer, const void *const *residual,
                                     const void *const *hidden, int n_batches, int M, frt_stream_t stream) {
    frt_status st = check_layer_ready(P, layer);
    if (st != FRT_OK)
        return st;
    if (!residual || n_batches < 1)
        return qfail(FRT_ERR_INVALID_ARG, "need at least one residual batch");
    if (M < 1 || M > P->M_max)
        return qfail(M < 1 ? FRT_ERR_INVALID_ARG : FRT_ERR_SHAPE, "M=%d outside [1, M_max=%d]", M, P->M_max);
    for (int b = 0; b < n_batches; ++b) {
        const void *h = hidden ? hidden[b] : nullptr;
        if (!residual[b] || !al16(residual[b]) || !al16(h))
            return qfail(FRT_ERR_INVALID_ARG, "batch %d: pointers must be non-null (residual) and 16-byte aligned",
                         b);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    QCK(cudaMemsetAsync(P->amax, 0, 4, s));
    for (int b = 0; b < n_batches; ++b)
        QCK(launch_norm_quant(residual[b], hidden ? hidden[b] : nullptr, P->w_norm + (size_t)layer * P->d, M, P->d,
                              QKV_RMS_EPS, 1.0f, nullptr, P->qx, P->amax, true, s, false));
    unsigned h_amax = 0;
    QCK(cudaMemcpyAsync(&h_amax, P->amax, 4, cudaMemcpyDeviceToHost, s));
    QCK(cudaStreamSynchronize(s));
    float a;
    memcpy(&a, &h_amax, 4);
    P->s_x[layer] = a == 0.0f ? 1.0f : a / 448.0f;
    return FRT_OK;
}

FRT_API frt_status frt_qkv_get_scales(frt_qkv_plan_t P, float *s_x, float *s_qkv) {
    if (!P)
        return qfail(FRT_ERR_INVALID_ARG, "null plan");
    for (int l = 0; l < P->L; ++l) {
        if (s_x) s_x[l] = P->s_x[l];
        if (s_qkv) s_qkv[l] = P->s_qkv[l];
    }
    return FRT_OK;
}

FRT_API frt_status frt_qkv_set_scales(frt_qkv_plan_t P, const float *s_x) {
    if (!P || !s_x)
        return qfail(FRT_ERR_INVALID_ARG, "null plan or scales");
    for (int l = 0; l < P->L; ++l)
        if (!(s_x[l] > 0.0f) || !std::isfinite(s_x[l]))
            return qfail(FRT_ERR_INVALID_ARG, "s_x[%d] must be finite and > 0", l);
    for (int l = 0; l < P->L; ++l)
        P->s_x[l] = s_x[l];
    return FRT_OK;
}

FRT_API frt_status frt_qkv_debug_trace(frt_qkv_plan_t P, int layer, const void *residual_in, const void *hidden_in,
                                       const int *positions, void *r_prime_out, void *q_out, void *k_out,
                                       void *v_out, void *q_x_out, void *qkv_out, int M, frt_stream_t stream) {
    frt_status st = check_layer_ready(P, layer);
    if (st != FRT_OK)
        return st;
    if (!(P->s_x[layer] > 0.0f))
        return qfail(FRT_ERR_NOT_READY, "activation scale of layer %d not set", layer);
    if (M < 0)
        return qfail(FRT_ERR_INVALID_ARG, "M must be >= 0 (got %d)", M);
    if (M > P->M_max)
        return qfail(FRT_ERR_SHAPE, "M=%d exceeds M_max=%d", M, P->M_max);
    if (M == 0)
        return FRT_OK;
    if (!residual_in || !positions || !q_out || !k_out || !v_out)
        return qfail(FRT_ERR_INVALID_ARG, "residual_in, positions, q_out, k_out and v_out must be non-null");
    const void *ptrs[] = {residual_in, hidden_in, positions, r_prime_out, q_out, k_out, v_out, q_x_out, qkv_out};
    for (const void *p : ptrs)
        if (!al16(p))
            return qfail(FRT_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    return run_qkv(P, layer, residual_in, hidden_in, positions, r_prime_out, q_out, k_out, v_out, M,
                   static_cast<cudaStream_t>(stream), q_x_out, qkv_out);
}

FRT_API frt_status frt_qkv_forward(frt_qkv_plan_t P, int layer, const void *residual_in, const void *hidden_in,
                                   const int *positions, void *r_prime_out, void *q_out, void *k_out, void *v_out,
                                   int M, frt_stream_t stream) {
    return frt_qkv_debug_trace(P, layer, residual_in, hidden_in, positions, r_prime_out, q_out, k_out, v_out,
                               nullptr, nullptr, M, stream);
}

FRT_API frt_status frt_qkv_debug_trace_qx(frt_qkv_plan_t P, int layer, const void *q_x_in, const int *positions,
                                          void *q_out, void *k_out, void *v_out, void *qkv_out, int M,
                                          frt_stream_t stream) {
    frt_status st = check_layer_ready(P, layer);
    if (st != FRT_OK)
        return st;
    if (!(P->s_x[layer] > 0.0f))
        return qfail(FRT_ERR_NOT_READY, "activation scale of layer %d not set", layer);
    if (M < 0)
        return qfail(FRT_ERR_INVALID_ARG, "M must be >= 0 (got %d)", M);
    if (M > P->M_max)
        return qfail(FRT_ERR_SHAPE, "M=%d exceeds M_max=%d", M, P->M_max);
    if (M == 0)
        return FRT_OK;
    if (!q_x_in || !positions || !q_out || !k_out || !v_out)
        return qfail(FRT_ERR_INVALID_ARG, "q_x_in, positions, q_out, k_out and v_out must be non-null");
    const void *ptrs[] = {q_x_in, positions, q_out, k_out, v_out, qkv_out};
    for (const void *p : ptrs)
        if (!al16(p))
            return qfail(FRT_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    return run_qkv(P, layer, nullptr, nullptr, positions, nullptr, q_out, k_out, v_out, M,
                   static_cast<cudaStream_t>(stream), nullptr, qkv_out, q_x_in);
}

FRT_API frt_status frt_qkv_debug_weights(frt_qkv_plan_t P, int layer, void *w_qkv, frt_stream_t stream) {
    if (!P)
        return qfail(FRT_ERR_INVALID_ARG, "null plan");
    if (layer < 0 || layer >= P->L)
        return qfail(FRT_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, P->L);
    if (!P->loaded[layer])
        return qfail(FRT_ERR_NOT_READY, "weights of layer %d not loaded", layer);
    if (!w_qkv)
        return qfail(FRT_ERR_INVALID_ARG, "w_qkv must be non-null");
    const size_t n = (size_t)P->N * P->d;
    QCK(cudaMemcpyAsync(w_qkv, P->w + (size_t)layer * n, n, cudaMemcpyDeviceToDevice,
                        static_cast<cudaStream_t>(stream)));
    return FRT_OK;
}

FRT_API frt_status frt_qkv_device_status(frt_qkv_plan_t P, frt_stream_t stream) {
    if (!P)
        return qfail(FRT_ERR_INVALID_ARG, "null plan");
    QCK(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    int h = 0;
    QCK(cudaMemcpy(&h, P->err, 4, cudaMemcpyDeviceToHost));
    if (h) {
        QCK(cudaMemset(P->counters, 0, (size_t)SPLIT_COUNTERS * 4));
        QCK(cudaMemset(P->err, 0, 4));
        return qfail(FRT_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (code %d)", h);
    }
    return FRT_OK;
}
