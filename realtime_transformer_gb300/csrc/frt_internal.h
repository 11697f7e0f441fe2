// frt_internal.h -- declarations shared by the library's translation units
// (plan / ABI, elementwise kernels, FP8 GEMM).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace frt {

enum Act : int { ACT_GEGLU_TANH = 0, ACT_SWIGLU = 1 };

// GEMM epilogues.
enum Epi : int {
    EPI_BF16 = 0,   // out[m][n] = bf16(acc * alpha)
    EPI_RESID = 1,  // out[m][n] = bf16(resid[m][n] + acc * alpha)
    EPI_F32 = 2,    // out[m][n] = acc * alpha (fp32; diagnostics)
    EPI_GATED = 3,  // out = q_h[m][f] = E4M3(act(g) * u * inv_s), g/u = bf16(acc * alpha) (interleaved rows)
    EPI_GATED_AMAX = 4,  // atomicMax(amax, |act(g) * u|) (calibration)
    EPI_ROPE = 5,   // tiled role: x = bf16(acc * alpha), split into Q/K/V heads, RoPE on Q and K (rope_* fields)
    // NVFP4 operands (f4 launches), [W_gate; W_up] interleaved as for EPI_GATED:
    // g = acc * alpha, u = acc * alpha_u; G = NVFP4(g, s_g), U = NVFP4(u, s_u);
    // a = act(dec G) * dec U
    EPI_F4_GATED = 6,    // out = codes of NVFP4(a, s_h) [m][f/2], TMEM-ready block scales into out_sf
    EPI_F4_AMAX_GU = 7,  // atomicMax(amax[0], |g|), atomicMax(amax[1], |u|) (calibration)
    EPI_F4_AMAX_H = 8,   // atomicMax(amax[2], |a|) (calibration)
};

// One GEMM launch: C[token][feature] = epilogue(sum_k X[token][k] W[feature][k]).
// The MMA's 128-row operand P and its narrow operand Q are either
// (P = X tiles, Q = W tiles) -- the tiled path -- or (P = W tiles, Q = X tiles)
// -- the weight-streaming path for few tokens ("swap").
struct GemmParams {
    const CUtensorMap *gtm_p, *gtm_q;  // tensor maps in device memory (null: the kernel parameters)
    int p_row0, q_row0;     // row offsets of the P and Q tiles in their tensor maps
    int n_tiles_p, n_tiles_q;
    int group;              // P-tiles per rasterisation group (see decode)
    int k_blocks;           // ceil(K / 128)
    int splits;             // split-K factor (1 = none)
    int stages;             // shared-memory pipeline stages of this launch
    int kb_per_split;
    int total_units;        // n_tiles_p * n_tiles_q * splits
    int epi;                // Epi
    float alpha;
    void *out;
    int ldo;                // elements
    const void *resid;      // BF16, EPI_RESID only
    int ldr;
    int m_tok;              // valid token rows
    int n_feat;             // valid feature columns
    float *ws;              // split-K partials
    int *counters;          // split-K arrival counters, one per tile, for this launch's split count
    int pair;               // tiled role on CTA pairs (cta_group::2): 256-token MMAs, half a weight tile per CTA
    int w_evict, x_evict;   // L2 priority of the weight / token tiles: 0 evict-first, 1 normal, 2 evict-last
    int cluster;            // 1: the splits of a tile are one thread-block cluster and exchange
                            //    partials in distributed shared memory (ws, counters unused)
    const uint16_t *gate;   // EPI_RESID with AdaRMSNorm: out = bf16(resid + gate * acc * alpha), BF16 gate
    int ldgate;             //   at gate[m * ldgate + n] (0: one row for all tokens); null: no gate
    int *err;               // device error word
    int stall_test;         // test hook: the MMA issuer first waits on a phase nothing completes
    unsigned long long *stamp;  // profiling (null: off): [0] = max of ~t over the CTAs' starts (so ~[0] is
                                //   the first start), [1] = max of t over their ends, t = %globaltimer ns
    // gated epilogues
    int act;                // Act
    int ff;                 // hidden width (feature count of q_h)
    float inv_s;            // 1 / s_h
    unsigned *amax;         // EPI_GATED_AMAX target
    uint16_t *dbg_gu;       // optional: BF16 [g | u] [M, 2ff] (diagnostics)
    // QKV split + RoPE epilogue (EPI_ROPE): heads of rope_hd columns, the
    // first rope_nq query heads, then rope_nkv key and rope_nkv value heads;
    // outputs head-major [H, m_tok, hd] BF16
    const float2 *rope_cs;  // (cos, sin) [m_tok, hd / 2] of each token's angles
    int rope_hd, rope_nq, rope_nkv;
    uint16_t *rope_q, *rope_k, *rope_v;
    // NVFP4 operands (f4 launches): the E4M3 block scales of the weight and
    // token operands in the TMEM-ready order (per 128-row tile and 64-element
    // K chunk a 512-byte block, tiles major), rows counted as in the tensor maps
    const uint8_t *sf_w, *sf_x;
    // NVFP4 gated epilogues (alpha: the gate rows')
    float alpha_u;
    float s_g, inv6_g, s_u, inv6_u, s_h, inv6_h;  // tensor scales s and 1 / (6 s)
    uint8_t *out_sf;        // EPI_F4_GATED: block scales of the output, TMEM-ready (K = ff)
    uint8_t *dbg_gq, *dbg_gs, *dbg_uq, *dbg_us;  // optional: G and U codes [M, ff/2], row-major scales [M, ff/16]
};

struct GemmLaunch {
    CUtensorMap tmP, tmQ;
    GemmParams p;
    int bn;                 // MMA N (Q tile rows)
    bool swap;
    bool f4;                // NVFP4 operands (k_gemm_f4)
    int grid;
    size_t min_smem;        // dynamic shared memory floor (see plan_gemm)
};

// Host side --------------------------------------------------------------

// Message returned by frt_ffn_last_error() on this host thread.
void set_last_error(const char *msg);

// Split-K arrival counters only grow, so every split count gets its own
// range of counters (a counter is shared only by launches with the same S).
constexpr int MAX_SPLIT_TILES = 2048;
constexpr int SPLIT_COUNTERS = 17 * MAX_SPLIT_TILES;  // ranges for S = 0..16
inline int *split_counters(int *base, int splits) { return base + (size_t)splits * MAX_SPLIT_TILES; }

// Encode a 2-D E4M3 tensor map: rows x cols bytes, row stride `cols` bytes,
// box of 128 bytes x box_rows rows, 128-byte swizzle.
cudaError_t encode_tmap_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows);

// Schedule variants of a GEMM launch that leave its results unchanged bit
// for bit (a "tactic"): the split-K partials exchanged through global memory
// instead of inside a cluster (same splits, same reduction order), and the
// tiled role on single CTAs instead of CTA pairs.
struct Tactic {
    bool global_exchange = false;
    bool no_pairs = false;
};

// Choose tiling / split-K for a GEMM of m_tok tokens x n_feat features and
// K bytes per operand row (E4M3: K elements; NVFP4: K / 2 of 2 elements
// each, a multiple of 128) and fill the launch (tensor maps excluded).
// swap: weight-streaming path; tactic: null for the defaults; f4: NVFP4
// operands (single-CTA tiles, N = 128 for the tiled role).
void plan_gemm(GemmLaunch &g, bool swap, int m_tok, int n_feat, int K, int num_sms, int force_splits,
               const Tactic *tactic = nullptr, bool f4 = false);
size_t gemm_ws_floats(const GemmLaunch &g);
int gemm_tiles(const GemmLaunch &g);
cudaError_t launch_gemm(const GemmLaunch &g, cudaStream_t s, bool pdl);
// The NVFP4 instantiations (k_gemm_f4.cu); launch_gemm hands f4 launches to it.
cudaError_t launch_gemm_f4(const GemmLaunch &g, cudaStream_t s, bool pdl);

cudaError_t launch_amax_bf16(const void *x, size_t n, unsigned *amax_word, cudaStream_t s);
cudaError_t launch_quant_bf16(const void *x, size_t n, float inv_s, uint8_t *q, cudaStream_t s);
cudaError_t launch_quant_gu_interleave(const void *gate, const void *up, int ff, int d, const void *fold,
                                      float inv_s, uint8_t *dst, cudaStream_t s);
cudaError_t launch_amax_fold(const void *x, size_t rows, int d, const void *w, unsigned *amax_word, cudaStream_t s);
cudaError_t launch_quant_fold(const void *x, size_t rows, int d, const void *w, float inv_s, uint8_t *q,
                              cudaStream_t s);
cudaError_t launch_rope_table(const int *pos, const float *inv_freq, int M, int half, float2 *cs, cudaStream_t s,
                              bool pdl);
cudaError_t launch_rope_split(const void *qkv, int M, int nq, int nkv, int hd, const int *pos, const float *inv_freq,
                              void *q, void *k, void *v, cudaStream_t s, bool pdl);
// Diagnostics: q[i] = E4M3 of the fp32 whose bits are start + i (n % 8 == 0).
cudaError_t launch_e4m3_sweep(uint32_t start, size_t n, uint8_t *q, cudaStream_t s);
// AdaRMSNorm modulation of the norm: row m's scale vector at p + m * stride
// (its shift vector d elements after it); stride 0 = one row for all tokens.
struct NormMod {
    const uint16_t *p = nullptr;
    int stride = 0;
    unsigned long long *stamp = nullptr;  // profiling: see GemmParams::stamp
};
cudaError_t launch_norm_quant(const void *r, const void *h, const void *w, int M, int d, float eps, float inv_s,
                              void *rprime, uint8_t *qx, unsigned *amax_word, bool measure, cudaStream_t s,
                              bool pdl, NormMod mod = NormMod());

// ------------------------------------------------- persistent stack kernel --
// The whole FP8 FFN stack for at most 64 tokens in one launch (k_stack_fp8.cu):
// ff / 128 clusters of d / 256 CTAs, one CTA per SM, all resident together.
struct StackParams {
    const CUtensorMap *tm_gu, *tm_d;  // weight maps (device copies), boxes of 128 bytes x 256 rows
    const uint16_t *w_norm;           // [L][d] BF16
    const float4 *scal;               // [L]: (1/s_x, s_x s_gu, 1/s_h, s_h s_down)
    const uint16_t *r_in, *h_in;      // [M][d] BF16; h_in may be null (added before layer 0)
    uint16_t *out;                    // [M][d] BF16 (may alias r_in)
    uint16_t *R;                      // [2][d/256][64][256] BF16: the layer input, K-quarter major
    float *SS;                        // [2][n_own * 64]: per owner and token, sum of squares of its columns
    float *P;                         // [2][d/8][ff/128][M][8]: down partials per column group and K-slice
    int *cnt;                         // monotonic counters (see k_stack_fp8.cu), zero between launches
    int *err;                         // device error word
    unsigned long long *stamp;        // profiling stamps (null: off)
    // diagnostics (DEBUG instantiation): injected per layer (null: computed) q_x [L][M][d] and the
    // input residual of layers >= 1 [L][M][d] BF16; dumps of q_x [L][M][d], g/u [L][M][2ff] BF16,
    // q_h [L][M][ff] and each layer's output [L][M][d] BF16
    const uint8_t *dbg_qx_in;
    const uint16_t *dbg_res_in;
    uint8_t *dbg_qx;
    uint16_t *dbg_gu;
    uint8_t *dbg_qh;
    uint16_t *dbg_out;
    unsigned long long *dbg_t;        // per-CTA timeline [CTAs][L][16] (%globaltimer)
    int M, d, ff, L, act;
    int S, nC, n_own;                 // cluster size d/256, clusters ff/128, column-group owners
    uint32_t x_bytes;                 // size of the kernel's staging region
    int res_groups;                   // most 8-column groups an owner holds
    float eps;
};
constexpr int STACK_COUNTER_INTS = 32 * 10;  // residual, 8 N-tile and exit counters, 128 bytes apart
// Fill the shape fields of p for M tokens; false if the stack kernel does not
// take this shape.  *smem_bytes, *grid: the launch's dynamic shared memory and CTAs.
bool plan_stack(StackParams &p, int M, int d, int ff, int num_sms, size_t *smem_bytes, int *grid);
size_t smem_max_stack();
// Clusters of the stack kernel that fit on the GPU at once (0 on error).
int stack_max_active_clusters(const StackParams &p, size_t smem);
cudaError_t launch_stack(const StackParams &p, size_t smem, cudaStream_t s, bool debug);

// ---------------------------------------------------------------- NVFP4 --
// Elementwise kernels of the NVFP4 sublayer (k_nvfp4.cu); its GEMMs are f4
// launches of the tensor-core GEMM (plan_gemm / launch_gemm).
cudaError_t launch_f4_amax_w(const void *w, size_t rows, int K, const float *col, unsigned *amax_word,
                             cudaStream_t s);
// ilv: 0 plain rows; 1 / 2 the gate / up rows of a [W_gate; W_up] arena
// interleaved in blocks of 64 rows (q and sf: the layer's arena).
cudaError_t launch_f4_quant_w(const void *w, int rows, int K, const float *col, float sc, float inv6, uint8_t *q,
                              uint8_t *sf, int ilv, cudaStream_t s);
cudaError_t launch_f4_norm_quant(const void *r, const void *h, const void *w, const float *awq_inv, int M, int d,
                                 float eps, float sc, float inv6, void *rprime, uint8_t *q, uint8_t *sf,
                                 unsigned *amax_word, bool measure, cudaStream_t s, bool pdl,
                                 unsigned long long *stamp = nullptr);  // profiling stamps (null: off)

}  // namespace frt

namespace frt {

// cudaLaunchKernelEx with an optional programmatic-dependent-launch edge to
// the previous work on the stream and an optional 1-D cluster shape.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             bool pdl, unsigned cluster, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace frt
