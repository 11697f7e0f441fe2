// frt_ffn.cu -- the plan object behind the C ABI of include/frt_ffn.h.
//
// The plan owns everything the forward touches besides the caller's
// input/output buffers: the E4M3 weight arena (layer-major, [W_gate; W_up]
// then W_down per layer -- the flat concatenated buffers of the itsolotime
// FlashRT article, 5.2 "FlatCat"), BF16 norm weights, per-layer scales, all
// scratch sized by M_max, the split-K workspace, TMA descriptors, and the
// CUDA graphs captured per token count ("FlashRT docs/architecture.md", 7
// CUDA Graph Capture: pointer-only forward, no allocation during replay;
// "exec/": a C ABI Buffer / Graph / Plan contract).
//
// Per layer the forward launches three kernels on the caller's stream, each
// with a programmatic-dependent-launch edge to its predecessor:
//   A1 norm_quant -> A2+A3 FP8 gate/up GEMM with the gated activation and
//   requantise in its epilogue -> A4 FP8 down GEMM with the residual add
// (itsolotime article, 7.2: the FFN layer loop; the gate/up weights are
// stored interleaved in 64-row blocks so one tile holds matching rows).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <string>
#include <utility>
#include <vector>

#include "frt_ffn.h"
#include "frt_internal.h"

#define FRT_API extern "C" __attribute__((visibility("default")))

using namespace frt;

namespace {

constexpr float RMS_EPS = 1e-6f;     // reading: the pages never state the epsilon
constexpr int SWAP_MAX_TOKENS = 64;  // weight-streaming GEMM path up to this many tokens
constexpr int N_GEMM_SITES = 2;      // gate/up and down keep separate split-K counters

thread_local std::string g_last_error;

frt_status fail(frt_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

frt_status cuda_fail(cudaError_t e, const char *what) {
    return fail(e == cudaErrorMemoryAllocation ? FRT_ERR_OOM : FRT_ERR_CUDA, "%s: %s (%s)", what,
                cudaGetErrorString(e), cudaGetErrorName(e));
}

}  // namespace

// The per-thread message of the last failed call, shared by every plan type.
void frt::set_last_error(const char *msg) { g_last_error = msg; }

namespace {

#define CK(call)                                   \
    do {                                           \
        cudaError_t e_ = (call);                   \
        if (e_ != cudaSuccess)                     \
            return cuda_fail(e_, #call);           \
    } while (0)

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

float scale_from_amax(float amax) { return amax == 0.0f ? 1.0f : amax / 448.0f; }

enum Buf { B_WGU = 0, B_WDOWN = 1, B_QX = 2, B_QH = 3 };

struct GraphEntry {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    uint64_t version = 0;
    const void *r = nullptr, *h = nullptr;  // the buffers baked into the graph
    void *out = nullptr;
};

}  // namespace

struct frt_ffn_plan {
    int d = 0, ff = 0, act = 0, M_max = 0, L = 0;
    int dev = 0, num_sms = 0, M_alloc = 0;
    uint8_t *w_gu = nullptr, *w_down = nullptr;
    uint16_t *w_norm = nullptr;
    std::vector<float> s_gu, s_d, s_x, s_h;
    std::vector<char> loaded;
    bool scales_ok = false;
    uint64_t version = 1;
    uint16_t *rbuf[2] = {nullptr, nullptr};
    uint16_t *rprime = nullptr;
    uint8_t *qx = nullptr, *qh = nullptr;
    float *ws = nullptr;
    size_t ws_floats = 0;
    int *counters = nullptr;
    unsigned *amax = nullptr;  // [2]
    int *err = nullptr;
    // Tensor maps of the plan's buffers, built once at creation; a copy of
    // each also lives in device memory (tmap_dev), where the GEMM kernels
    // read it: one fixed address per map stays warm in the TMA unit's
    // descriptor cache from launch to launch, unlike a kernel parameter.
    std::map<std::pair<int, int>, std::pair<CUtensorMap, int>> tmaps;
    CUtensorMap *tmap_dev = nullptr;
    std::map<int, GraphEntry> graphs;
    int force_path = 0;        // 0 auto, 1 swap, 2 tiled (FRT_FFN_FORCE_PATH)
    bool pdl = true;           // programmatic dependent launch (FRT_FFN_NO_PDL=1 disables)
    int max_splits = 0;        // cap on split-K (FRT_FFN_MAX_SPLITS; 0 = none)
    const Tactic *tactic = nullptr;  // schedule variant of the capture being autotuned (null: defaults)
    // AdaRMSNorm modulation (frt_ffn_set_modulation): per layer a caller
    // buffer of mod_rows rows of [scale | shift | gate], each d wide, BF16
    std::vector<const uint16_t *> mod;
    int mod_rows = 0;
    // profiling (frt_ffn_graph_profile): while set, launches carry a pointer
    // to their pair of %globaltimer stamps, [layer][step][2]
    bool profiling = false;
    unsigned long long *stamps = nullptr;
    // persistent stack kernel (k_stack_fp8.cu) for at most 64 tokens, opt-in
    // (FRT_FFN_STACK=1): its exchange buffers (allocated when the shape allows
    // it), per-layer scalars, and whether it is used
    bool stack_on = false;
    uint16_t *st_R = nullptr;
    float *st_SS = nullptr, *st_P = nullptr;
    int *st_cnt = nullptr;
    float4 *st_scal = nullptr;
};

namespace {

constexpr int TMAP_SLOTS = 24;

// The map of buffer `buf` with boxes of `box_rows` rows: the host copy (for
// the kernel parameter) and its device copy.
frt_status get_tmap(frt_ffn_plan *P, int buf, int box_rows, CUtensorMap *out, const CUtensorMap **dev) {
    auto it = P->tmaps.find(std::make_pair(buf, box_rows));
    if (it == P->tmaps.end())
        return fail(FRT_ERR_UNSUPPORTED, "no tensor map for buffer %d box %d", buf, box_rows);
    *out = it->second.first;
    *dev = P->tmap_dev + it->second.second;
    return FRT_OK;
}

// Every map a launch of this plan can ask for (weights with boxes of a
// 128/256-row tile or a CTA pair's half of one, activations with the
// weight-streaming widths and 128), uploaded in one copy.
frt_status build_tmaps(frt_ffn_plan *P) {
    const int combos[][2] = {{B_WGU, 128},  {B_WGU, 256},  {B_WDOWN, 128}, {B_WDOWN, 256},
                             {B_QX, 16},    {B_QX, 32},    {B_QX, 64},    {B_QX, 128},
                             {B_QH, 16},    {B_QH, 32},    {B_QH, 64},    {B_QH, 128}};
    CUtensorMap host[TMAP_SLOTS];
    int n = 0;
    for (const auto &c : combos) {
        const int buf = c[0], box_rows = c[1];
        CUtensorMap m;
        cudaError_t e;
        switch (buf) {
        case B_WGU: e = encode_tmap_u8(&m, P->w_gu, (uint64_t)P->L * 2 * P->ff, P->d, box_rows); break;
        case B_WDOWN: e = encode_tmap_u8(&m, P->w_down, (uint64_t)P->L * P->d, P->ff, box_rows); break;
        case B_QX: e = encode_tmap_u8(&m, P->qx, P->M_alloc, P->d, box_rows); break;
        default: e = encode_tmap_u8(&m, P->qh, P->M_alloc, P->ff, box_rows); break;
        }
        if (e != cudaSuccess)
            return fail(FRT_ERR_CUDA, "cuTensorMapEncodeTiled failed for buffer %d box %d", buf, box_rows);
        host[n] = m;
        P->tmaps[std::make_pair(buf, box_rows)] = std::make_pair(m, n);
        ++n;
    }
    const cudaError_t e = cudaMemcpy(P->tmap_dev, host, sizeof(CUtensorMap) * n, cudaMemcpyHostToDevice);
    return e == cudaSuccess ? FRT_OK : cuda_fail(e, "tensor map upload");
}

bool use_swap(const frt_ffn_plan *P, int M) {
    if (P->force_path == 1)
        return M <= SWAP_MAX_TOKENS;
    if (P->force_path == 2)
        return false;
    return M <= SWAP_MAX_TOKENS;
}

// Fill a GEMM launch for one of the two sites of layer l.
frt_status setup_gemm(frt_ffn_plan *P, GemmLaunch &g, int site, int l, int M) {
    const bool swap = use_swap(P, M);
    const int N = site == 0 ? 2 * P->ff : P->d;
    const int K = site == 0 ? P->d : P->ff;
    const int wbuf = site == 0 ? B_WGU : B_WDOWN;
    const int xbuf = site == 0 ? B_QX : B_QH;
    memset(&g.p, 0, sizeof g.p);
    // tuning: FRT_FFN_GU_SPLITS / FRT_FFN_DOWN_SPLITS force one site's split-K
    int force = 0;
    if (const char *e = getenv(site == 0 ? "FRT_FFN_GU_SPLITS" : "FRT_FFN_DOWN_SPLITS"))
        force = atoi(e);
    plan_gemm(g, swap, M, N, K, P->num_sms, force, P->tactic);
    if (P->max_splits > 0 && g.p.splits > P->max_splits)
        plan_gemm(g, swap, M, N, K, P->num_sms, P->max_splits, P->tactic);
    frt_status st;
    if (swap) {
        if ((st = get_tmap(P, wbuf, 128, &g.tmP, &g.p.gtm_p)) != FRT_OK) return st;
        if ((st = get_tmap(P, xbuf, g.bn, &g.tmQ, &g.p.gtm_q)) != FRT_OK) return st;
        g.p.p_row0 = l * N;
        g.p.q_row0 = 0;
    } else {
        if ((st = get_tmap(P, xbuf, 128, &g.tmP, &g.p.gtm_p)) != FRT_OK) return st;
        // on a CTA pair each CTA loads half of the weight tile's rows
        if ((st = get_tmap(P, wbuf, g.bn / (g.p.pair ? 2 : 1), &g.tmQ, &g.p.gtm_q)) != FRT_OK) return st;
        g.p.p_row0 = 0;
        g.p.q_row0 = l * N;
    }
    if (gemm_ws_floats(g) > P->ws_floats || (g.p.splits > 1 && gemm_tiles(g) > MAX_SPLIT_TILES))
        return fail(FRT_ERR_UNSUPPORTED, "split-K workspace too small for M=%d site %d", M, site);
    g.p.ws = P->ws;
    g.p.counters = split_counters(P->counters + (size_t)site * SPLIT_COUNTERS, g.p.splits);
    g.p.err = P->err;
    return FRT_OK;
}

// Layer l's AdaRMSNorm modulation of the norm (none when unset).
NormMod norm_mod(const frt_ffn_plan *P, int l) {
    NormMod m;
    if (!P->mod.empty()) {
        m.p = P->mod[l];
        m.stride = P->mod_rows == 1 ? 0 : 3 * P->d;
    }
    return m;
}

// The persistent stack kernel's launch for M tokens, if it takes this
// forward (plain norm, shape and residency allowed).
bool stack_launch_for(frt_ffn_plan *P, int M, StackParams &sp, size_t *smem) {
    if (!P->stack_on || !P->mod.empty() || M > 64)
        return false;
    memset(&sp, 0, sizeof sp);
    int grid = 0;
    if (!plan_stack(sp, M, P->d, P->ff, P->num_sms, smem, &grid))
        return false;
    CUtensorMap dummy;
    if (get_tmap(P, B_WGU, 256, &dummy, &sp.tm_gu) != FRT_OK || get_tmap(P, B_WDOWN, 256, &dummy, &sp.tm_d) != FRT_OK)
        return false;
    sp.w_norm = P->w_norm;
    sp.scal = P->st_scal;
    sp.R = P->st_R;
    sp.SS = P->st_SS;
    sp.P = P->st_P;
    sp.cnt = P->st_cnt;
    sp.err = P->err;
    sp.L = P->L;
    sp.act = P->act;
    sp.eps = RMS_EPS;
    return true;
}

// Per-layer scalars of the stack kernel, (1/s_x, s_x s_gu, 1/s_h, s_h s_down)
// in fp32 as the per-layer launches compute them; uploaded whenever scales change.
frt_status upload_stack_scalars(frt_ffn_plan *P) {
    if (!P->st_scal || !P->scales_ok)
        return FRT_OK;
    std::vector<float4> h(P->L);
    for (int l = 0; l < P->L; ++l)
        h[l] = make_float4(1.0f / P->s_x[l], P->s_x[l] * P->s_gu[l], 1.0f / P->s_h[l], P->s_h[l] * P->s_d[l]);
    CK(cudaMemcpy(P->st_scal, h.data(), sizeof(float4) * P->L, cudaMemcpyHostToDevice));
    return FRT_OK;
}

// Layer l's step s stamp pair while profiling, else null.
unsigned long long *stamp_of(const frt_ffn_plan *P, int l, int s) {
    return P->profiling ? P->stamps + 2 * ((size_t)3 * l + s) : nullptr;
}

// Gate/up GEMM of layer l with the gated epilogue (q_h, or its amax).
frt_status setup_gate_up(frt_ffn_plan *P, GemmLaunch &g, int l, int M, int epi) {
    frt_status st = setup_gemm(P, g, 0, l, M);
    if (st != FRT_OK)
        return st;
    g.p.epi = epi;
    g.p.alpha = P->s_x[l] * P->s_gu[l];
    g.p.out = P->qh;
    g.p.ldo = P->ff;
    g.p.act = P->act;
    g.p.ff = P->ff;
    g.p.inv_s = 1.0f / P->s_h[l];
    g.p.amax = P->amax + 1;
    return FRT_OK;
}

// Down GEMM of layer l with the residual epilogue.
frt_status setup_down(frt_ffn_plan *P, GemmLaunch &g, int l, int M, const void *resid, void *out) {
    frt_status st = setup_gemm(P, g, 1, l, M);
    if (st != FRT_OK)
        return st;
    g.p.epi = EPI_RESID;
    g.p.alpha = P->s_h[l] * P->s_d[l];
    if (!P->mod.empty()) {
        // AdaRMSNorm: the update enters the residual stream scaled by the gate
        g.p.gate = P->mod[l] + 2 * (size_t)P->d;
        g.p.ldgate = P->mod_rows == 1 ? 0 : 3 * P->d;
    }
    g.p.out = out;
    g.p.ldo = P->d;
    g.p.resid = resid;
    g.p.ldr = P->d;
    return FRT_OK;
}

// One layer: A1 -> A2+A3 -> A4.  `out` receives the layer output; when
// hid != null, r' is materialised in P->rprime and used as A4's residual.
frt_status run_layer(frt_ffn_plan *P, int l, const void *in, const void *hid, void *out, int M, cudaStream_t s,
                     void *trace_rprime, void *trace_qx, void *trace_gu, void *trace_qh) {
    const int d = P->d, ff = P->ff;
    const float s_x = P->s_x[l], s_h = P->s_h[l];
    const float inv_sx = 1.0f / s_x, inv_sh = 1.0f / s_h;
    void *rp = hid ? (void *)P->rprime : nullptr;
    const bool pdl = P->pdl;
    NormMod nm = norm_mod(P, l);
    nm.stamp = stamp_of(P, l, 0);
    CK(launch_norm_quant(in, hid, P->w_norm + (size_t)l * d, M, d, RMS_EPS, inv_sx, rp, P->qx, nullptr, false, s,
                         pdl, nm));
    GemmLaunch g;
    frt_status st = setup_gate_up(P, g, l, M, EPI_GATED);
    if (st != FRT_OK)
        return st;
    g.p.dbg_gu = static_cast<uint16_t *>(trace_gu);
    g.p.stamp = stamp_of(P, l, 1);
    CK(launch_gemm(g, s, pdl));
    if (trace_qx)
        CK(cudaMemcpyAsync(trace_qx, P->qx, (size_t)M * d, cudaMemcpyDeviceToDevice, s));
    if (trace_qh)
        CK(cudaMemcpyAsync(trace_qh, P->qh, (size_t)M * ff, cudaMemcpyDeviceToDevice, s));
    if (trace_rprime)
        CK(cudaMemcpyAsync(trace_rprime, hid ? (const void *)P->rprime : in, (size_t)M * d * 2,
                           cudaMemcpyDeviceToDevice, s));
    GemmLaunch g2;
    st = setup_down(P, g2, l, M, hid ? (const void *)P->rprime : in, out);
    if (st != FRT_OK)
        return st;
    g2.p.stamp = stamp_of(P, l, 2);
    CK(launch_gemm(g2, s, pdl));
    (void)inv_sh;
    return FRT_OK;
}

frt_status run_stack(frt_ffn_plan *P, const void *r_in, const void *h_in, void *out, int M, cudaStream_t s) {
    StackParams sp;
    size_t smem = 0;
    if (stack_launch_for(P, M, sp, &smem)) {
        sp.r_in = static_cast<const uint16_t *>(r_in);
        sp.h_in = static_cast<const uint16_t *>(h_in);
        sp.out = static_cast<uint16_t *>(out);
        sp.stamp = P->profiling ? P->stamps : nullptr;
        CK(launch_stack(sp, smem, s, false));
        return FRT_OK;
    }
    const void *cur = r_in;
    for (int l = 0; l < P->L; ++l) {
        void *dst = (l == P->L - 1) ? out : (void *)P->rbuf[l & 1];
        frt_status st = run_layer(P, l, cur, l == 0 ? h_in : nullptr, dst, M, s, nullptr, nullptr, nullptr,
                                  nullptr);
        if (st != FRT_OK)
            return st;
        cur = dst;
    }
    return FRT_OK;
}

frt_status check_ready(frt_ffn_plan *P) {
    for (int l = 0; l < P->L; ++l)
        if (!P->loaded[l])
            return fail(FRT_ERR_NOT_READY, "weights of layer %d not loaded", l);
    if (!P->scales_ok)
        return fail(FRT_ERR_NOT_READY, "activation scales not calibrated or set");
    return FRT_OK;
}

frt_status check_io(frt_ffn_plan *P, const void *r, const void *h, const void *out, int M) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    if (M < 0)
        return fail(FRT_ERR_INVALID_ARG, "M must be >= 0 (got %d)", M);
    if (M > P->M_max)
        return fail(FRT_ERR_SHAPE, "M=%d exceeds M_max=%d", M, P->M_max);
    if (M > 0 && (!r || !out))
        return fail(FRT_ERR_INVALID_ARG, "residual_in and out must be non-null");
    if (!aligned16(r) || !aligned16(h) || !aligned16(out))
        return fail(FRT_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    return FRT_OK;
}

void free_plan(frt_ffn_plan *P) {
    for (auto &kv : P->graphs) {
        if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
        if (kv.second.graph) cudaGraphDestroy(kv.second.graph);
    }
    void *ptrs[] = {P->w_gu, P->w_down, P->w_norm, P->rbuf[0], P->rbuf[1], P->rprime, P->qx,
                    P->qh,   P->ws,     P->counters, P->amax, P->err,     P->tmap_dev, P->stamps,
                    P->st_R, P->st_SS,  P->st_P,     P->st_cnt, P->st_scal};
    for (void *p : ptrs)
        if (p) cudaFree(p);
    delete P;
}

}  // namespace

namespace {

// The persistent stack kernel's buffers, when it is asked for (FRT_FFN_STACK=1
// at plan creation: measured slower than the per-layer kernels on GB300, so
// not the default), the plan's shape allows the kernel at M_max tokens or
// fewer, and all its clusters fit on the GPU at once.
frt_status setup_stack(frt_ffn_plan *P) {
    const char *e = getenv("FRT_FFN_STACK");
    if (!(e && e[0] == '1'))
        return FRT_OK;
    StackParams sp;
    memset(&sp, 0, sizeof sp);
    size_t smem = 0;
    int grid = 0;
    if (!plan_stack(sp, std::min(P->M_max, 64), P->d, P->ff, P->num_sms, &smem, &grid))
        return FRT_OK;
    if (stack_max_active_clusters(sp, smem) < sp.nC)
        return FRT_OK;
    const size_t S = sp.S, nC = sp.nC, D = P->d;
    struct A { void **p; size_t bytes; } allocs[] = {
        {(void **)&P->st_R, 2 * S * 64 * 256 * 2},
        {(void **)&P->st_SS, 2 * (size_t)sp.n_own * 64 * 4},
        {(void **)&P->st_P, 2 * nC * (D / 8) * 64 * 8 * 4},
        {(void **)&P->st_cnt, (size_t)STACK_COUNTER_INTS * 4},
        {(void **)&P->st_scal, (size_t)P->L * sizeof(float4)},
    };
    for (auto &a : allocs)
        CK(cudaMalloc(a.p, a.bytes));
    CK(cudaMemset(P->st_cnt, 0, (size_t)STACK_COUNTER_INTS * 4));
    CK(cudaDeviceSynchronize());
    P->stack_on = true;
    return FRT_OK;
}

}  // namespace

// ===================================================================== ABI ==

FRT_API const char *frt_ffn_last_error(void) { return g_last_error.c_str(); }

FRT_API frt_status frt_ffn_plan_create(int d, int ff, int act, int M_max, int n_layers, frt_ffn_plan_t *out) {
    if (!out)
        return fail(FRT_ERR_INVALID_ARG, "out is null");
    *out = nullptr;
    if (d <= 0 || ff <= 0 || d % 128 || ff % 128)
        return fail(FRT_ERR_INVALID_ARG, "d and ff must be positive multiples of 128 (d=%d ff=%d)", d, ff);
    if (act != FRT_ACT_GEGLU_TANH && act != FRT_ACT_SWIGLU)
        return fail(FRT_ERR_INVALID_ARG, "unknown activation %d", act);
    if (M_max < 1 || M_max > 65536)
        return fail(FRT_ERR_INVALID_ARG, "M_max must be in [1, 65536] (got %d)", M_max);
    if (n_layers < 1 || n_layers > 4096)
        return fail(FRT_ERR_INVALID_ARG, "n_layers must be in [1, 4096] (got %d)", n_layers);
    int dev = 0;
    CK(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    CK(cudaGetDeviceProperties(&prop, dev));
    if (prop.major != 10 || prop.minor != 3)
        return fail(FRT_ERR_UNSUPPORTED, "needs a compute capability 10.3 GPU (found %d.%d, %s)", prop.major,
                    prop.minor, prop.name);
    frt_ffn_plan *P = new frt_ffn_plan();
    P->d = d;
    P->ff = ff;
    P->act = act;
    P->M_max = M_max;
    P->L = n_layers;
    P->dev = dev;
    P->num_sms = prop.multiProcessorCount;
    P->M_alloc = (M_max + 127) / 128 * 128;
    P->s_gu.assign(n_layers, 0.f);
    P->s_d.assign(n_layers, 0.f);
    P->s_x.assign(n_layers, 0.f);
    P->s_h.assign(n_layers, 0.f);
    P->loaded.assign(n_layers, 0);
    if (const char *fp = getenv("FRT_FFN_FORCE_PATH")) {
        if (!strcmp(fp, "splitk") || !strcmp(fp, "swap")) P->force_path = 1;
        if (!strcmp(fp, "tiled")) P->force_path = 2;
    }
    if (const char *np = getenv("FRT_FFN_NO_PDL"))
        P->pdl = !(np[0] == '1');
    if (const char *ms = getenv("FRT_FFN_MAX_SPLITS"))
        P->max_splits = atoi(ms);
    const size_t L = n_layers, D = d, F = ff, MA = P->M_alloc, MM = M_max;
    P->ws_floats = (size_t)P->num_sms * 128 * 256;
    struct A { void **p; size_t bytes; } allocs[] = {
        {(void **)&P->w_gu, L * 2 * F * D},
        {(void **)&P->w_down, L * D * F},
        {(void **)&P->w_norm, L * D * 2},
        {(void **)&P->rbuf[0], MM * D * 2},
        {(void **)&P->rbuf[1], MM * D * 2},
        {(void **)&P->rprime, MM * D * 2},
        {(void **)&P->qx, MA * D},
        {(void **)&P->qh, MA * F},
        {(void **)&P->ws, P->ws_floats * 4},
        {(void **)&P->counters, (size_t)(N_GEMM_SITES + 1) * SPLIT_COUNTERS * 4},
        {(void **)&P->amax, 2 * 4},
        {(void **)&P->err, 4},
        {(void **)&P->tmap_dev, TMAP_SLOTS * sizeof(CUtensorMap)},
        {(void **)&P->stamps, L * 3 * 2 * sizeof(unsigned long long)},
    };
    for (auto &a : allocs) {
        cudaError_t e = cudaMalloc(a.p, a.bytes);
        if (e != cudaSuccess) {
            frt_status st = cuda_fail(e, "cudaMalloc");
            free_plan(P);
            return st;
        }
    }
    // Padding rows of the activation tiles and every counter start at zero.
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = cudaMemset(P->qx, 0, MA * D);
    if (e == cudaSuccess) e = cudaMemset(P->qh, 0, MA * F);
    if (e == cudaSuccess) e = cudaMemset(P->counters, 0, (size_t)(N_GEMM_SITES + 1) * SPLIT_COUNTERS * 4);
    if (e == cudaSuccess) e = cudaMemset(P->err, 0, 4);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        frt_status st = cuda_fail(e, "plan initialisation");
        free_plan(P);
        return st;
    }
    frt_status st = build_tmaps(P);
    if (st != FRT_OK) {
        free_plan(P);
        return st;
    }
    if ((st = setup_stack(P)) != FRT_OK) {
        free_plan(P);
        return st;
    }
    *out = P;
    return FRT_OK;
}

FRT_API frt_status frt_ffn_plan_destroy(frt_ffn_plan_t P) {
    if (!P)
        return FRT_OK;
    cudaDeviceSynchronize();
    free_plan(P);
    return FRT_OK;
}

FRT_API frt_status frt_ffn_load_weights(frt_ffn_plan_t P, int layer, const void *w_norm, const void *w_gate,
                                        const void *w_up, const void *w_down, frt_stream_t stream) {
    return frt_ffn_load_weights_ex(P, layer, w_norm, w_gate, w_up, w_down, 0u, stream);
}

FRT_API frt_status frt_ffn_load_weights_ex(frt_ffn_plan_t P, int layer, const void *w_norm, const void *w_gate,
                                           const void *w_up, const void *w_down, unsigned flags,
                                           frt_stream_t stream) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    if (flags & ~(unsigned)FRT_LOAD_FOLD_NORM)
        return fail(FRT_ERR_INVALID_ARG, "unknown load flags 0x%x", flags);
    const bool fold = (flags & FRT_LOAD_FOLD_NORM) != 0;
    if (layer < 0 || layer >= P->L)
        return fail(FRT_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, P->L);
    if (!w_norm || !w_gate || !w_up || !w_down)
        return fail(FRT_ERR_INVALID_ARG, "weight pointers must be non-null");
    if (!aligned16(w_norm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down))
        return fail(FRT_ERR_INVALID_ARG, "weight pointers must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t D = P->d, F = P->ff;
    uint8_t *gu_dst = P->w_gu + (size_t)layer * 2 * F * D;
    uint8_t *d_dst = P->w_down + (size_t)layer * D * F;
    // folded: the norm weight moves into the gate/up weights and the norm
    // multiplies by ones (BF16 1.0 = 0x3F80)
    const std::vector<uint16_t> ones(fold ? D : 0, (uint16_t)0x3F80);
    CK(cudaMemcpyAsync(P->w_norm + (size_t)layer * D, fold ? (const void *)ones.data() : w_norm, D * 2,
                       fold ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice, s));
    // one scale for [W_gate; W_up], one for W_down
    CK(cudaMemsetAsync(P->amax, 0, 8, s));
    if (fold) {
        CK(launch_amax_fold(w_gate, F, (int)D, w_norm, P->amax, s));
        CK(launch_amax_fold(w_up, F, (int)D, w_norm, P->amax, s));
    } else {
        CK(launch_amax_bf16(w_gate, F * D, P->amax, s));
        CK(launch_amax_bf16(w_up, F * D, P->amax, s));
    }
    CK(launch_amax_bf16(w_down, D * F, P->amax + 1, s));
    unsigned h_amax[2];
    CK(cudaMemcpyAsync(h_amax, P->amax, 8, cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    float a_gu, a_d;
    memcpy(&a_gu, &h_amax[0], 4);
    memcpy(&a_d, &h_amax[1], 4);
    const float s_gu = scale_from_amax(a_gu), s_d = scale_from_amax(a_d);
    CK(launch_quant_gu_interleave(w_gate, w_up, (int)F, (int)D, fold ? w_norm : nullptr, 1.0f / s_gu, gu_dst, s));
    CK(launch_quant_bf16(w_down, D * F, 1.0f / s_d, d_dst, s));
    CK(cudaStreamSynchronize(s));
    P->s_gu[layer] = s_gu;
    P->s_d[layer] = s_d;
    P->loaded[layer] = 1;
    P->version++;
    return upload_stack_scalars(P);
}

FRT_API frt_status frt_ffn_set_modulation(frt_ffn_plan_t P, const void *const *mod, int mod_rows) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    if (!mod) {
        P->mod.clear();
        P->mod_rows = 0;
        P->version++;
        return FRT_OK;
    }
    if (mod_rows != 1 && mod_rows != P->M_max)
        return fail(FRT_ERR_INVALID_ARG, "mod_rows must be 1 or M_max=%d (got %d)", P->M_max, mod_rows);
    std::vector<const uint16_t *> ptrs(P->L);
    for (int l = 0; l < P->L; ++l) {
        if (!mod[l] || !aligned16(mod[l]))
            return fail(FRT_ERR_INVALID_ARG, "modulation of layer %d: null or misaligned pointer", l);
        ptrs[l] = static_cast<const uint16_t *>(mod[l]);
    }
    P->mod = ptrs;
    P->mod_rows = mod_rows;
    P->version++;  // captured graphs bake the previous choice
    return FRT_OK;
}

FRT_API frt_status frt_ffn_get_scales(frt_ffn_plan_t P, float *s_x, float *s_h, float *s_gu, float *s_down) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    const size_t n = P->L * sizeof(float);
    if (s_x) memcpy(s_x, P->s_x.data(), n);
    if (s_h) memcpy(s_h, P->s_h.data(), n);
    if (s_gu) memcpy(s_gu, P->s_gu.data(), n);
    if (s_down) memcpy(s_down, P->s_d.data(), n);
    return FRT_OK;
}

FRT_API frt_status frt_ffn_set_scales(frt_ffn_plan_t P, const float *s_x, const float *s_h) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    if (!s_x || !s_h)
        return fail(FRT_ERR_INVALID_ARG, "scale arrays must be non-null");
    for (int l = 0; l < P->L; ++l)
        if (!(s_x[l] > 0.f) || !(s_h[l] > 0.f) || !std::isfinite(s_x[l]) || !std::isfinite(s_h[l]))
            return fail(FRT_ERR_INVALID_ARG, "scales of layer %d must be positive and finite", l);
    P->s_x.assign(s_x, s_x + P->L);
    P->s_h.assign(s_h, s_h + P->L);
    P->scales_ok = true;
    P->version++;
    return upload_stack_scalars(P);
}

FRT_API frt_status frt_ffn_calibrate(frt_ffn_plan_t P, const void *const *residual, const void *const *hidden,
                                     int n_batches, int M, frt_stream_t stream) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    if (!residual || n_batches < 1)
        return fail(FRT_ERR_INVALID_ARG, "need at least one calibration batch");
    if (M < 1)
        return fail(FRT_ERR_INVALID_ARG, "calibration needs M >= 1");
    if (M > P->M_max)
        return fail(FRT_ERR_SHAPE, "M=%d exceeds M_max=%d", M, P->M_max);
    for (int b = 0; b < n_batches; ++b) {
        if (!residual[b] || !aligned16(residual[b]) || (hidden && !aligned16(hidden[b])))
            return fail(FRT_ERR_INVALID_ARG, "batch %d: null or misaligned pointer", b);
    }
    for (int l = 0; l < P->L; ++l)
        if (!P->loaded[l])
            return fail(FRT_ERR_NOT_READY, "weights of layer %d not loaded", l);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int d = P->d, ff = P->ff;
    const size_t row_bytes = (size_t)M * d * 2;
    uint16_t *state = nullptr;
    CK(cudaMalloc(&state, row_bytes * n_batches));
    auto st_of = [&](int b) { return reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(state) + row_bytes * b); };
    std::vector<float> sx(P->L), sh(P->L);
    frt_status result = FRT_OK;
    auto run = [&]() -> frt_status {
        unsigned h_amax;
        for (int l = 0; l < P->L; ++l) {
            const uint16_t *wn = P->w_norm + (size_t)l * d;
            // 1. amax of the gate/up GEMM input over all batches
            CK(cudaMemsetAsync(P->amax, 0, 8, s));
            for (int b = 0; b < n_batches; ++b) {
                const void *in = l == 0 ? residual[b] : (const void *)st_of(b);
                const void *hid = (l == 0 && hidden) ? hidden[b] : nullptr;
                CK(launch_norm_quant(in, hid, wn, M, d, RMS_EPS, 1.0f, nullptr, P->qx, P->amax, true, s, false,
                                     norm_mod(P, l)));
            }
            CK(cudaMemcpyAsync(&h_amax, P->amax, 4, cudaMemcpyDeviceToHost, s));
            CK(cudaStreamSynchronize(s));
            float a;
            memcpy(&a, &h_amax, 4);
            sx[l] = scale_from_amax(a);
            // 2. amax of the down GEMM input, r' of layer 0 kept in the batch state
            CK(cudaMemsetAsync(P->amax + 1, 0, 4, s));
            for (int b = 0; b < n_batches; ++b) {
                const void *in = l == 0 ? residual[b] : (const void *)st_of(b);
                const void *hid = (l == 0 && hidden) ? hidden[b] : nullptr;
                if (l == 0 && !hid)
                    CK(cudaMemcpyAsync(st_of(b), residual[b], row_bytes, cudaMemcpyDeviceToDevice, s));
                CK(launch_norm_quant(in, hid, wn, M, d, RMS_EPS, 1.0f / sx[l], hid ? (void *)st_of(b) : nullptr,
                                     P->qx, nullptr, false, s, false, norm_mod(P, l)));
                GemmLaunch g;
                P->s_x[l] = sx[l];
                P->s_h[l] = 1.0f;
                frt_status st2 = setup_gate_up(P, g, l, M, EPI_GATED_AMAX);
                if (st2 != FRT_OK)
                    return st2;
                CK(launch_gemm(g, s, false));
            }
            CK(cudaMemcpyAsync(&h_amax, P->amax + 1, 4, cudaMemcpyDeviceToHost, s));
            CK(cudaStreamSynchronize(s));
            memcpy(&a, &h_amax, 4);
            sh[l] = scale_from_amax(a);
            // 3. finish the layer for every batch with both scales
            P->s_x[l] = sx[l];
            P->s_h[l] = sh[l];
            for (int b = 0; b < n_batches; ++b) {
                frt_status st2 = run_layer(P, l, st_of(b), nullptr, st_of(b), M, s, nullptr, nullptr, nullptr,
                                           nullptr);
                if (st2 != FRT_OK)
                    return st2;
            }
        }
        CK(cudaStreamSynchronize(s));
        return FRT_OK;
    };
    result = run();
    cudaStreamSynchronize(s);
    cudaFree(state);
    if (result != FRT_OK) {
        P->scales_ok = false;
        return result;
    }
    int h_err = 0;
    CK(cudaMemcpy(&h_err, P->err, 4, cudaMemcpyDeviceToHost));
    if (h_err) {
        CK(cudaMemset(P->err, 0, 4));
        P->scales_ok = false;
        return fail(FRT_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait during calibration");
    }
    P->s_x = sx;
    P->s_h = sh;
    P->scales_ok = true;
    P->version++;
    return upload_stack_scalars(P);
}

FRT_API frt_status frt_ffn_forward(frt_ffn_plan_t P, const void *residual_in, const void *hidden_in, void *out,
                                   int M, frt_stream_t stream) {
    frt_status st = check_io(P, residual_in, hidden_in, out, M);
    if (st != FRT_OK)
        return st;
    if ((st = check_ready(P)) != FRT_OK)
        return st;
    if (M == 0)
        return FRT_OK;
    return run_stack(P, residual_in, hidden_in, out, M, static_cast<cudaStream_t>(stream));
}

namespace {

// Checks shared by the capturing entry points.
frt_status capture_checks(frt_ffn_plan *P, const void *residual_in, const void *hidden_in, void *out, int M,
                          cudaStream_t s) {
    frt_status st = check_io(P, residual_in, hidden_in, out, M);
    if (st != FRT_OK)
        return st;
    if ((st = check_ready(P)) != FRT_OK)
        return st;
    if (M == 0)
        return fail(FRT_ERR_INVALID_ARG, "cannot capture M == 0");
    if (s == nullptr)
        return fail(FRT_ERR_CAPTURE, "capture needs a non-default stream");
    cudaStreamCaptureStatus cs;
    CK(cudaStreamIsCapturing(s, &cs));
    if (cs != cudaStreamCaptureStatusNone)
        return fail(FRT_ERR_CAPTURE, "stream is already capturing");
    // Encode every tensor map the capture needs before capturing.
    for (int site = 0; site < 2; ++site) {
        GemmLaunch g;
        if ((st = setup_gemm(P, g, site, 0, M)) != FRT_OK)
            return st;
    }
    return FRT_OK;
}

// Capture the stack for M on s and instantiate it into ge.
frt_status capture_one(frt_ffn_plan *P, const void *residual_in, const void *hidden_in, void *out, int M,
                       cudaStream_t s, GraphEntry &ge) {
    CK(cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed));
    frt_status st = run_stack(P, residual_in, hidden_in, out, M, s);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(s, &graph);
    if (st != FRT_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
    }
    if (e != cudaSuccess || !graph)
        return fail(FRT_ERR_CAPTURE, "cudaStreamEndCapture: %s", cudaGetErrorString(e));
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return fail(FRT_ERR_CAPTURE, "cudaGraphInstantiate: %s", cudaGetErrorString(e));
    }
    ge.graph = graph;
    ge.exec = exec;
    ge.version = P->version;
    ge.r = residual_in;
    ge.h = hidden_in;
    ge.out = out;
    return FRT_OK;
}

void destroy_graph(GraphEntry &ge) {
    if (ge.exec) cudaGraphExecDestroy(ge.exec);
    if (ge.graph) cudaGraphDestroy(ge.graph);
    ge.exec = nullptr;
    ge.graph = nullptr;
}

// Keep ge as the plan's graph for M, releasing the one it replaces.
void install_graph(frt_ffn_plan *P, int M, const GraphEntry &ge) {
    auto it = P->graphs.find(M);
    if (it != P->graphs.end())
        destroy_graph(it->second);
    P->graphs[M] = ge;
}

// Median duration in microseconds of n replays of exec on s, each timed
// alone with events on s after one untimed replay.
frt_status time_replays(cudaGraphExec_t exec, int n, cudaStream_t s, float *median_us) {
    cudaEvent_t ev[2];
    CK(cudaEventCreate(&ev[0]));
    cudaError_t e = cudaEventCreate(&ev[1]);
    if (e != cudaSuccess) {
        cudaEventDestroy(ev[0]);
        return cuda_fail(e, "cudaEventCreate");
    }
    std::vector<float> t;
    e = cudaGraphLaunch(exec, s);
    for (int i = 0; i < n && e == cudaSuccess; ++i) {
        float ms = 0.0f;
        if ((e = cudaEventRecord(ev[0], s)) != cudaSuccess) break;
        if ((e = cudaGraphLaunch(exec, s)) != cudaSuccess) break;
        if ((e = cudaEventRecord(ev[1], s)) != cudaSuccess) break;
        if ((e = cudaEventSynchronize(ev[1])) != cudaSuccess) break;
        if ((e = cudaEventElapsedTime(&ms, ev[0], ev[1])) != cudaSuccess) break;
        t.push_back(ms * 1000.0f);
    }
    cudaEventDestroy(ev[0]);
    cudaEventDestroy(ev[1]);
    if (e != cudaSuccess)
        return cuda_fail(e, "timing graph replays");
    std::sort(t.begin(), t.end());
    *median_us = t[t.size() / 2];
    return FRT_OK;
}

}  // namespace

FRT_API frt_status frt_ffn_graph_capture(frt_ffn_plan_t P, const void *residual_in, const void *hidden_in,
                                         void *out, int M, frt_stream_t stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    frt_status st = capture_checks(P, residual_in, hidden_in, out, M, s);
    if (st != FRT_OK)
        return st;
    GraphEntry ge;
    if ((st = capture_one(P, residual_in, hidden_in, out, M, s, ge)) != FRT_OK)
        return st;
    install_graph(P, M, ge);
    return FRT_OK;
}

// Schedules tried by the autotuned capture, each giving the same results
// bit for bit: the defaults; split-K partials exchanged through global memory;
// single-CTA tiles instead of CTA pairs; launches without programmatic
// dependent launch.
constexpr int N_TACTICS = 4;

FRT_API frt_status frt_ffn_graph_autotune(frt_ffn_plan_t P, const void *residual_in, const void *hidden_in,
                                          void *out, int M, int n_tries, int n_replays, float *best_us,
                                          int *best_tactic, frt_stream_t stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (n_tries < 1 || n_tries > 64 || n_replays < 1 || n_replays > 10000)
        return fail(FRT_ERR_INVALID_ARG, "need 1 <= n_tries <= 64 and 1 <= n_replays <= 10000");
    frt_status st = capture_checks(P, residual_in, hidden_in, out, M, s);
    if (st != FRT_OK)
        return st;
    const bool pdl0 = P->pdl;
    // FRT_FFN_AUTOTUNE_ONLY=k: every capture uses schedule k (tests, tuning)
    const char *only = getenv("FRT_FFN_AUTOTUNE_ONLY");
    const int only_k = only ? atoi(only) : -1;
    GraphEntry best;
    float best_t = 0.0f;
    int best_k = 0;
    for (int i = 0; i < n_tries; ++i) {
        const int k = (only_k >= 0 && only_k < N_TACTICS) ? only_k : i % N_TACTICS;
        Tactic t;
        t.global_exchange = k == 1;
        t.no_pairs = k == 2;
        P->tactic = &t;
        P->pdl = pdl0 && k != 3;
        GraphEntry ge;
        float tm = 0.0f;
        st = capture_one(P, residual_in, hidden_in, out, M, s, ge);
        P->tactic = nullptr;
        P->pdl = pdl0;
        if (st == FRT_OK)
            st = time_replays(ge.exec, n_replays, s, &tm);
        if (st != FRT_OK) {
            destroy_graph(ge);
            destroy_graph(best);
            return st;
        }
        if (!best.exec || tm < best_t) {
            destroy_graph(best);
            best = ge;
            best_t = tm;
            best_k = k;
        } else {
            destroy_graph(ge);
        }
    }
    install_graph(P, M, best);
    if (best_us)
        *best_us = best_t;
    if (best_tactic)
        *best_tactic = best_k;
    return FRT_OK;
}

FRT_API frt_status frt_ffn_graph_replay(frt_ffn_plan_t P, int M, frt_stream_t stream) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    auto it = P->graphs.find(M);
    if (it == P->graphs.end())
        return fail(FRT_ERR_CAPTURE, "no graph captured for M=%d", M);
    if (it->second.version != P->version)
        return fail(FRT_ERR_STALE_GRAPH, "scales or weights changed since the graph for M=%d was captured", M);
    CK(cudaGraphLaunch(it->second.exec, static_cast<cudaStream_t>(stream)));
    return FRT_OK;
}

FRT_API frt_status frt_ffn_graph_profile(frt_ffn_plan_t P, int M, int n_replays, float *kernel_us, int *n_kernels,
                                         frt_stream_t stream) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    if (!kernel_us || n_replays < 1 || n_replays > 10000)
        return fail(FRT_ERR_INVALID_ARG, "need kernel_us and 1 <= n_replays <= 10000");
    auto it = P->graphs.find(M);
    if (it == P->graphs.end())
        return fail(FRT_ERR_CAPTURE, "no graph captured for M=%d", M);
    if (it->second.version != P->version)
        return fail(FRT_ERR_STALE_GRAPH, "scales or weights changed since the graph for M=%d was captured", M);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const GraphEntry base = it->second;
    frt_status st = capture_checks(P, base.r, base.h, base.out, M, s);
    if (st != FRT_OK)
        return st;
    // the same forward, captured again with every launch stamping its pair
    GraphEntry ge;
    P->profiling = true;
    st = capture_one(P, base.r, base.h, base.out, M, s, ge);
    P->profiling = false;
    if (st != FRT_OK)
        return st;
    StackParams sp_probe;
    size_t smem_probe = 0;
    const int nk = stack_launch_for(P, M, sp_probe, &smem_probe) ? 1 : 3 * P->L;
    std::vector<unsigned long long> h(2 * (size_t)nk);
    std::vector<std::vector<float>> dur(nk);
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < n_replays && e == cudaSuccess; ++i) {
        if ((e = cudaMemsetAsync(P->stamps, 0, h.size() * sizeof(unsigned long long), s)) != cudaSuccess) break;
        if ((e = cudaGraphLaunch(ge.exec, s)) != cudaSuccess) break;
        if ((e = cudaMemcpyAsync(h.data(), P->stamps, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost,
                                 s)) != cudaSuccess) break;
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess) break;
        // launch k owns the time from when it started, or its predecessor
        // ended if later, to its own end: the stack's span split with no
        // overlap between consecutive (programmatically overlapped) kernels
        unsigned long long prev_end = 0;
        for (int k = 0; k < nk; ++k) {
            const unsigned long long t0 = ~h[2 * k], t1 = h[2 * k + 1];
            const unsigned long long from = std::max(t0, prev_end);
            dur[k].push_back(t1 > from ? (float)(t1 - from) * 1e-3f : 0.0f);
            prev_end = std::max(prev_end, t1);
        }
    }
    destroy_graph(ge);
    if (e != cudaSuccess)
        return cuda_fail(e, "profiling replays");
    for (int k = 0; k < nk; ++k) {
        std::sort(dur[k].begin(), dur[k].end());
        kernel_us[k] = dur[k][dur[k].size() / 2];
    }
    if (n_kernels)
        *n_kernels = nk;
    return frt_ffn_device_status(P, stream);
}

FRT_API frt_status frt_ffn_debug_trace(frt_ffn_plan_t P, int layer, const void *residual_in, const void *hidden_in,
                                       int M, void *r_prime, void *q_x, void *gu, void *q_h, void *out,
                                       frt_stream_t stream) {
    frt_status st = check_io(P, residual_in, hidden_in, out ? out : (void *)residual_in, M);
    if (st != FRT_OK)
        return st;
    if (layer < 0 || layer >= P->L)
        return fail(FRT_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (!P->loaded[layer] || !P->scales_ok)
        return fail(FRT_ERR_NOT_READY, "layer %d not loaded or scales not set", layer);
    if (!aligned16(r_prime) || !aligned16(q_x) || !aligned16(gu) || !aligned16(q_h))
        return fail(FRT_ERR_INVALID_ARG, "trace buffers must be 16-byte aligned");
    if (M == 0)
        return FRT_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *dst = out ? out : (void *)P->rbuf[0];
    return run_layer(P, layer, residual_in, hidden_in, dst, M, s, r_prime, q_x, gu, q_h);
}

FRT_API frt_status frt_ffn_debug_trace_qx(frt_ffn_plan_t P, int layer, const void *r_prime, const void *q_x, int M,
                                          void *gu, void *q_h, void *out, frt_stream_t stream) {
    frt_status st = check_io(P, r_prime, nullptr, out, M);
    if (st != FRT_OK)
        return st;
    if (layer < 0 || layer >= P->L)
        return fail(FRT_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (!P->loaded[layer] || !P->scales_ok)
        return fail(FRT_ERR_NOT_READY, "layer %d not loaded or scales not set", layer);
    if (M > 0 && !q_x)
        return fail(FRT_ERR_INVALID_ARG, "q_x must be non-null");
    if (!aligned16(q_x) || !aligned16(gu) || !aligned16(q_h))
        return fail(FRT_ERR_INVALID_ARG, "trace buffers must be 16-byte aligned");
    if (M == 0)
        return FRT_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the caller's codes take the place of step A1's output; the rest of the
    // layer runs the forward's kernels for this M
    CK(cudaMemcpyAsync(P->qx, q_x, (size_t)M * P->d, cudaMemcpyDeviceToDevice, s));
    GemmLaunch g;
    if ((st = setup_gate_up(P, g, layer, M, EPI_GATED)) != FRT_OK)
        return st;
    g.p.dbg_gu = static_cast<uint16_t *>(gu);
    CK(launch_gemm(g, s, false));
    if (q_h)
        CK(cudaMemcpyAsync(q_h, P->qh, (size_t)M * P->ff, cudaMemcpyDeviceToDevice, s));
    GemmLaunch g2;
    if ((st = setup_down(P, g2, layer, M, r_prime, out)) != FRT_OK)
        return st;
    CK(launch_gemm(g2, s, false));
    return FRT_OK;
}

FRT_API frt_status frt_ffn_debug_weights(frt_ffn_plan_t P, int layer, void *w_gu, void *w_down,
                                         frt_stream_t stream) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    if (layer < 0 || layer >= P->L)
        return fail(FRT_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (!P->loaded[layer])
        return fail(FRT_ERR_NOT_READY, "weights of layer %d not loaded", layer);
    const size_t D = P->d, F = P->ff;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (w_gu)
        CK(cudaMemcpyAsync(w_gu, P->w_gu + (size_t)layer * 2 * F * D, 2 * F * D, cudaMemcpyDeviceToDevice, s));
    if (w_down)
        CK(cudaMemcpyAsync(w_down, P->w_down + (size_t)layer * D * F, D * F, cudaMemcpyDeviceToDevice, s));
    return FRT_OK;
}

FRT_API frt_status frt_debug_e4m3_encode_range(unsigned start, unsigned long long n, void *codes,
                                               frt_stream_t stream) {
    if (n == 0)
        return FRT_OK;
    if (!codes || !aligned16(codes))
        return fail(FRT_ERR_INVALID_ARG, "codes must be a non-null, 16-byte aligned device pointer");
    if (n % 8 || n > 0x100000000ull - start)
        return fail(FRT_ERR_INVALID_ARG, "need n %% 8 == 0 and start + n <= 2^32");
    CK(launch_e4m3_sweep(start, (size_t)n, static_cast<uint8_t *>(codes), static_cast<cudaStream_t>(stream)));
    return FRT_OK;
}

FRT_API frt_status frt_ffn_debug_stack(frt_ffn_plan_t P, const void *residual_in, const void *hidden_in, void *out,
                                       int M, const void *q_x_in, const void *res_in, void *q_x, void *gu, void *q_h,
                                       void *layer_out, void *times, frt_stream_t stream) {
    frt_status st = check_io(P, residual_in, hidden_in, out, M);
    if (st != FRT_OK)
        return st;
    if ((st = check_ready(P)) != FRT_OK)
        return st;
    if (M == 0)
        return FRT_OK;
    const void *ptrs[] = {q_x_in, res_in, q_x, gu, q_h, layer_out, times};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr))
            return fail(FRT_ERR_INVALID_ARG, "debug buffers must be 16-byte aligned");
    StackParams sp;
    size_t smem = 0;
    if (!stack_launch_for(P, M, sp, &smem))
        return fail(FRT_ERR_UNSUPPORTED, "the persistent stack kernel does not take M=%d on this plan", M);
    sp.r_in = static_cast<const uint16_t *>(residual_in);
    sp.h_in = static_cast<const uint16_t *>(hidden_in);
    sp.out = static_cast<uint16_t *>(out);
    sp.dbg_qx_in = static_cast<const uint8_t *>(q_x_in);
    sp.dbg_res_in = static_cast<const uint16_t *>(res_in);
    sp.dbg_qx = static_cast<uint8_t *>(q_x);
    sp.dbg_gu = static_cast<uint16_t *>(gu);
    sp.dbg_qh = static_cast<uint8_t *>(q_h);
    sp.dbg_out = static_cast<uint16_t *>(layer_out);
    sp.dbg_t = static_cast<unsigned long long *>(times);
    // the product instantiation when only the timeline is asked for
    const bool dumps = q_x_in || res_in || q_x || gu || q_h || layer_out;
    CK(launch_stack(sp, smem, static_cast<cudaStream_t>(stream), dumps));
    return FRT_OK;
}

FRT_API int frt_ffn_uses_stack_kernel(frt_ffn_plan_t P, int M) {
    if (!P)
        return 0;
    StackParams sp;
    size_t smem = 0;
    return stack_launch_for(P, M, sp, &smem) ? 1 : 0;
}

FRT_API frt_status frt_ffn_debug_step(frt_ffn_plan_t P, int layer, int step, int M, frt_stream_t stream) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    if (layer < 0 || layer >= P->L || step < 0 || step > 2 || M < 1)
        return fail(FRT_ERR_INVALID_ARG, "bad layer, step or M");
    if (M > P->M_max)
        return fail(FRT_ERR_SHAPE, "M=%d exceeds M_max=%d", M, P->M_max);
    if (!P->loaded[layer] || !P->scales_ok)
        return fail(FRT_ERR_NOT_READY, "layer %d not loaded or scales not set", layer);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int d = P->d, ff = P->ff;
    GemmLaunch g;
    frt_status st;
    switch (step) {
    case 0:
        CK(launch_norm_quant(P->rbuf[0], nullptr, P->w_norm + (size_t)layer * d, M, d, RMS_EPS, 1.0f / P->s_x[layer],
                             nullptr, P->qx, nullptr, false, s, false, norm_mod(P, layer)));
        break;
    case 1:
        if ((st = setup_gate_up(P, g, layer, M, EPI_GATED)) != FRT_OK)
            return st;
        CK(launch_gemm(g, s, false));
        break;
    default:
        if ((st = setup_down(P, g, layer, M, P->rbuf[0], P->rbuf[1])) != FRT_OK)
            return st;
        CK(launch_gemm(g, s, false));
        break;
    }
    (void)ff;
    return FRT_OK;
}

FRT_API frt_status frt_ffn_device_status(frt_ffn_plan_t P, frt_stream_t stream) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    CK(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    int h = 0;
    CK(cudaMemcpy(&h, P->err, 4, cudaMemcpyDeviceToHost));
    if (h) {
        // a launch that gave up may have left split-K counters mid-generation
        CK(cudaMemset(P->counters, 0, (size_t)(N_GEMM_SITES + 1) * SPLIT_COUNTERS * 4));
        if (P->st_cnt)
            CK(cudaMemset(P->st_cnt, 0, (size_t)STACK_COUNTER_INTS * 4));
        CK(cudaMemset(P->err, 0, 4));
        CK(cudaDeviceSynchronize());
        return fail(FRT_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (code %d)", h);
    }
    return FRT_OK;
}

FRT_API frt_status frt_ffn_debug_stall(frt_ffn_plan_t P, frt_stream_t stream) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    // a 64 x 256 x d weight-streaming GEMM on the plan's own scratch: q_x
    // codes against the first 256 gate/up weight rows, fp32 into the
    // split-K workspace, without split-K
    const int M = 64, N = 256, K = P->d;
    GemmLaunch g;
    memset(&g.p, 0, sizeof g.p);
    plan_gemm(g, true, M, N, K, P->num_sms, 1);
    if (encode_tmap_u8(&g.tmP, P->w_gu, N, K, 128) != cudaSuccess ||
        encode_tmap_u8(&g.tmQ, P->qx, M, K, g.bn) != cudaSuccess)
        return fail(FRT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    g.p.epi = EPI_F32;
    g.p.alpha = 1.0f;
    g.p.out = P->ws;
    g.p.ldo = N;
    g.p.ws = P->ws;
    g.p.counters = split_counters(P->counters + (size_t)N_GEMM_SITES * SPLIT_COUNTERS, g.p.splits);
    g.p.err = P->err;
    g.p.stall_test = 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CK(launch_gemm(g, s, false));
    return frt_ffn_device_status(P, stream);
}

FRT_API frt_status frt_fp8_gemm(frt_ffn_plan_t P, const void *A, const void *B, void *C, int M, int N, int K,
                                float alpha, int path, int splits, frt_stream_t stream) {
    if (!P)
        return fail(FRT_ERR_INVALID_ARG, "null plan");
    if (!A || !B || !C || !aligned16(A) || !aligned16(B) || !aligned16(C))
        return fail(FRT_ERR_INVALID_ARG, "A, B, C must be non-null and 16-byte aligned");
    if (M < 1 || M > 65536 || N < 128 || N % 128 || K < 16 || K % 16)
        return fail(FRT_ERR_INVALID_ARG, "need 1 <= M <= 65536, N % 128 == 0, K >= 16, K %% 16 == 0");
    if (path < 0 || path > 2 || splits < 0)
        return fail(FRT_ERR_INVALID_ARG, "bad path or splits");
    const bool swap = path == 1 || (path == 0 && M <= SWAP_MAX_TOKENS);
    if (swap && M > SWAP_MAX_TOKENS)
        return fail(FRT_ERR_UNSUPPORTED, "the weight-streaming path takes at most %d tokens", SWAP_MAX_TOKENS);
    GemmLaunch g;
    memset(&g.p, 0, sizeof g.p);
    plan_gemm(g, swap, M, N, K, P->num_sms, splits);
    if (gemm_ws_floats(g) > P->ws_floats || (g.p.splits > 1 && gemm_tiles(g) > MAX_SPLIT_TILES))
        return fail(FRT_ERR_UNSUPPORTED, "split-K workspace too small");
    cudaError_t e1, e2;
    if (swap) {
        e1 = encode_tmap_u8(&g.tmP, B, N, K, 128);
        e2 = encode_tmap_u8(&g.tmQ, A, M, K, g.bn);
    } else {
        e1 = encode_tmap_u8(&g.tmP, A, M, K, 128);
        e2 = encode_tmap_u8(&g.tmQ, B, N, K, g.bn / (g.p.pair ? 2 : 1));  // weight slice per CTA
    }
    if (e1 != cudaSuccess || e2 != cudaSuccess)
        return fail(FRT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    g.p.epi = EPI_F32;
    g.p.alpha = alpha;
    g.p.out = C;
    g.p.ldo = N;
    g.p.ws = P->ws;
    g.p.counters = split_counters(P->counters + (size_t)N_GEMM_SITES * SPLIT_COUNTERS, g.p.splits);
    g.p.err = P->err;
    CK(launch_gemm(g, static_cast<cudaStream_t>(stream), false));
    return FRT_OK;
}
