// k_gemm_fp8.cu -- planning and launch of the tensor-core GEMM (k_gemm_tc.cuh)
// and its E4M3 instantiations.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "k_gemm_tc.cuh"

namespace frt {

// ---------------------------------------------------------------- host --

typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                      const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                      CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                      CUtensorMapFloatOOBfill);

static PFN_encodeTiled_t encode_fn() {
    static PFN_encodeTiled_t fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_encodeTiled_t>(ptr);
    }
    return fn;
}

cudaError_t encode_tmap_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    PFN_encodeTiled_t fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {cols};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

struct StageInfo {
    size_t stage_bytes, fixed_bytes, xbuf_bytes;  // fixed_bytes without the gate/up exchange buffer
    int max_stages;
};

template <int BN, bool SWAP, bool PAIR = false, bool F4 = false>
StageInfo stage_info() {
    using C = Cfg<BN, SWAP, PAIR, F4>;
    return {C::STAGE_BYTES, C::smem_bytes(0, false), C::XBUF_BYTES, C::STAGES};
}

StageInfo stage_info_for(int bn, bool swap, bool pair = false, bool f4 = false) {
    if (f4) {
        if (swap)
            return bn == 16 ? stage_info<16, true, false, true>()
                            : (bn == 32 ? stage_info<32, true, false, true>() : stage_info<64, true, false, true>());
        return bn == 256 ? stage_info<256, false, false, true>() : stage_info<128, false, false, true>();
    }
    if (swap)
        return bn == 16 ? stage_info<16, true>() : (bn == 32 ? stage_info<32, true>() : stage_info<64, true>());
    if (pair)
        return stage_info<256, false, true>();
    return bn == 128 ? stage_info<128, false>() : stage_info<256, false>();
}

// Shared memory a short launch may use so that CTAs of two consecutive
// GEMMs fit on one SM (228 KB) and the later one can prefetch its weights.
constexpr size_t COHABIT_SMEM = 112 * 1024;
// Just over half of an SM's 228 KB of shared memory (less the 1 KB each
// resident CTA reserves).
constexpr size_t SPREAD_SMEM = 115 * 1024;

}  // namespace

void plan_gemm(GemmLaunch &g, bool swap, int m_tok, int n_feat, int K, int num_sms, int force_splits,
               const Tactic *tactic, bool f4) {
    GemmParams &p = g.p;
    g.swap = swap;
    g.f4 = f4;
    p.k_blocks = (K + BK - 1) / BK;
    // cluster split-K (weight-streaming tiles): the splits of a tile form one
    // portable cluster of at most 8 CTAs and exchange partials in
    // distributed shared memory; FRT_FFN_CLUSTER=0 selects the global-memory
    // exchange (up to 16 splits) instead
    const char *cl_env = getenv("FRT_FFN_CLUSTER");
    const bool cluster_on = swap && !(cl_env && cl_env[0] == '0');
    constexpr int CLUSTER_MAX = 8;
    if (swap) {
        g.bn = m_tok <= 16 ? 16 : (m_tok <= 32 ? 32 : 64);
        p.n_tiles_p = (n_feat + BM - 1) / BM;
        p.n_tiles_q = (m_tok + g.bn - 1) / g.bn;
    } else {
        // NVFP4: 256-wide tiles have one accumulator (beside the stages'
        // scales), so a tile's epilogue runs between its MMAs and the next
        // tile's; with at most 8 k-blocks a tile that costs more than the
        // doubled MACs a k-block gain, and 128-wide tiles (two accumulators)
        // are used (measured: VLA prefix 92.2 against 95.9 us/layer; long
        // prefill, 20 k-blocks, 1164 against 1337 with 128-wide gate/up
        // tiles).  FRT_F4_BN=128 keeps 128 everywhere.
        const char *fb = f4 ? getenv("FRT_F4_BN") : nullptr;
        g.bn = (n_feat % 256 == 0 && !(fb && atoi(fb) == 128) && !(f4 && p.k_blocks <= 8)) ? 256 : 128;
        p.n_tiles_p = (m_tok + BM - 1) / BM;
        p.n_tiles_q = (n_feat + g.bn - 1) / g.bn;
    }
    const int tiles = p.n_tiles_p * p.n_tiles_q;
    int splits = 1;
    if (force_splits > 0)
        splits = force_splits;
    else if (tiles < num_sms)
        splits = num_sms / tiles;
    // cooperative split-K: every split of a tile resident at once, and at
    // most 16 partials per element
    splits = std::min(splits, std::max(1, num_sms / tiles));
    splits = std::max(1, std::min(std::min(splits, 16), p.k_blocks));
    if (cluster_on && force_splits == 0)
        splits = std::min(splits, CLUSTER_MAX);
    // weight-streaming tiles whose whole K fits the stage ring: no split-K
    // (each CTA prefetches its entire weight panel; no partials to exchange),
    // as long as there are enough tiles to spread the weight stream
    if (swap && force_splits == 0 && tiles >= 16 && p.k_blocks <= stage_info_for(g.bn, swap, false, f4).max_stages)
        splits = 1;
    p.kb_per_split = (p.k_blocks + splits - 1) / splits;
    p.splits = (p.k_blocks + p.kb_per_split - 1) / p.kb_per_split;
    p.total_units = tiles * p.splits;
    g.grid = std::min(p.total_units, num_sms);
    // persistent weight-streaming launches: the fewest CTAs that keep the
    // number of waves (272 tiles on 152 SMs: 136 CTAs of two tiles instead of
    // 120 of two and 32 of one, the same makespan), which leaves the other SMs
    // to the next kernel's early start (decode layer: 48.5 against 49.0 us)
    if (swap && p.splits == 1 && p.total_units > num_sms) {
        const int waves = (p.total_units + num_sms - 1) / num_sms;
        g.grid = (p.total_units + waves - 1) / waves;
    }
    // tiled role on CTA pairs (FRT_FFN_PAIR=0 disables): 256-token tiles
    // computed by two CTAs with cta_group::2 MMAs, each staging its own 128
    // tokens and half of the 256-row weight tile -- half the weight traffic
    // per CTA and 7 pipeline stages instead of 4; 256-wide tiles on an even
    // number of token tiles
    p.pair = 0;
    // (NVFP4 tiles stay on single CTAs: measured faster than pairs of
    // 256 x 128 tiles, whose two CTAs' epilogues run in lockstep)
    if (!swap && !f4 && g.bn == 256 && p.n_tiles_p % 2 == 0 && !(tactic && tactic->no_pairs)) {
        const char *e = getenv("FRT_FFN_PAIR");
        if (!(e && e[0] == '0')) {
            p.pair = 1;
            g.grid = g.grid / 2 * 2;
        }
    }
    // L2 priorities: the weight tiles evict-first, the token tiles evict-last
    // (a weight-streaming launch reads each weight byte once; a tiled launch
    // keeps its token tiles for every weight tile of a wave).  On the long
    // prefill shape normal priority for the weights
    // (FRT_FFN_W_EVICT = normal | last) brings the gate/up GEMM's DRAM
    // traffic from 1.8x to 1.04x the algorithmic bytes and the down GEMM's
    // from 4.3x to 2.3x, but the stack measured about 1% slower (compute
    // bound, 87% tensor pipe), so evict-first stays the default.
    p.w_evict = 0;
    p.x_evict = 2;
    if (!swap) {
        if (const char *e = getenv("FRT_FFN_W_EVICT"))
            p.w_evict = !strcmp(e, "normal") ? 1 : !strcmp(e, "last") ? 2 : 0;
    }
    // rasterisation: all P-tiles at once if the P operand of a wave fits
    // comfortably in L2 (for weight streaming P is the weights, each read
    // once anyway); else groups of P-tiles whose rows take about 32 MB
    {
        const size_t p_tile_bytes = (size_t)BM * (size_t)p.k_blocks * BK;
        const size_t budget = (size_t)32 << 20;
        int grp = (int)std::max<size_t>(1, budget / p_tile_bytes);
        if (swap || (size_t)p.n_tiles_p * p_tile_bytes <= ((size_t)48 << 20))
            grp = p.n_tiles_p;
        p.group = std::max(1, std::min(grp, p.n_tiles_p));
    }
    // pipeline depth: short launches keep a small footprint (see COHABIT_SMEM),
    // long ones take every stage they can
    const StageInfo si = stage_info_for(g.bn, swap, p.pair != 0, f4);
    const int units_per_cta = (p.total_units + g.grid - 1) / g.grid;
    const int kb_cta = p.kb_per_split * units_per_cta;
    // the gate/up exchange buffer is only in unsplit weight-streaming launches
    const size_t fixed = si.fixed_bytes + (swap && p.splits == 1 ? si.xbuf_bytes : 0);
    int cohabit = (int)((COHABIT_SMEM - fixed) / si.stage_bytes);
    cohabit = std::max(2, std::min(cohabit, si.max_stages));
    p.stages = kb_cta <= 2 * cohabit ? std::min(cohabit, std::max(2, kb_cta)) : si.max_stages;
    // CTA pairs: 5 of the 7 stages that fit measured fastest on the long
    // prefill shape (1237 against 1286 us a layer; 4: 1316, 6: 1257), the
    // VLA prefix shape alike at 5 to 7
    if (p.pair)
        p.stages = std::min(p.stages, 5);
    if (const char *e = getenv("FRT_FFN_STAGES")) {
        const int v = atoi(e);
        if (v >= 2)
            p.stages = std::min(v, si.max_stages);
    }
    // NVFP4 weight-streaming launches keep their TMEM (accumulators plus 32
    // scale columns a stage) within 256 columns, so that two of their CTAs
    // on one SM never wait for each other's TMEM
    if (f4 && swap)
        p.stages = std::max(2, std::min(p.stages, (256 - 2 * g.bn) / 32));
    p.cluster = (cluster_on && p.splits >= 2 && p.splits <= CLUSTER_MAX && !(tactic && tactic->global_exchange))
                    ? 1 : 0;

    if (p.cluster)
        g.grid = p.total_units;
    // A cluster launch of at most one wave is spread one CTA per SM: more
    // than half an SM's shared memory keeps two of its CTAs off one SM (the
    // cluster scheduler would otherwise pack them), while a CTA of another
    // launch still fits beside it.
    g.min_smem = 0;
    if (p.cluster && p.total_units <= num_sms) {
        const char *e = getenv("FRT_FFN_SPREAD");
        if (!(e && e[0] == '0'))
            g.min_smem = SPREAD_SMEM;
    }
    // an NVFP4 tiled CTA takes all 512 TMEM columns: one such CTA per SM
    if (f4 && !swap)
        g.min_smem = SPREAD_SMEM;
    if (p.splits > 1) {
        // the stage buffers receive this CTA's slice of all S partials (at most
        // the whole tile plus one column/row and 16 bytes of padding per split)
        // and, for cluster split-K, stage this CTA's whole partial after them
        const size_t need = red_floats(g.bn, p.splits) * 4 + (p.cluster ? (size_t)BM * g.bn * 4 : 0);
        while ((size_t)p.stages * si.stage_bytes < need && p.stages < si.max_stages)
            ++p.stages;
        if ((size_t)p.stages * si.stage_bytes < need)
            p.cluster = 0, g.grid = std::min(p.total_units, num_sms);
    }
    p.m_tok = m_tok;
    p.n_feat = n_feat;
}

size_t gemm_ws_floats(const GemmLaunch &g) {
    if (g.p.splits <= 1 || g.p.cluster)
        return 0;
    return (size_t)g.p.total_units * BM * (size_t)g.bn;
}

int gemm_tiles(const GemmLaunch &g) { return g.p.n_tiles_p * g.p.n_tiles_q; }

cudaError_t launch_gemm(const GemmLaunch &g, cudaStream_t s, bool pdl) {
    if (g.f4)
        return launch_gemm_f4(g, s, pdl);
    if (g.swap) {
        // the layer's two weight-streaming launches run kernels compiled for
        // their epilogue alone
        const bool gated = g.p.epi == EPI_GATED || g.p.epi == EPI_GATED_AMAX;
        const int role = (g.p.splits == 1 && gated) ? ROLE_GATED_TILE
                         : (g.p.cluster && !gated)  ? (g.p.gate ? ROLE_CLUSTER_GATE : ROLE_CLUSTER_PLAIN)
                                                    : ROLE_ANY;
        switch (g.bn * 8 + role) {
        case 16 * 8 + ROLE_ANY: return run<16, true, false, ROLE_ANY>(g, s, pdl);
        case 16 * 8 + ROLE_GATED_TILE: return run<16, true, false, ROLE_GATED_TILE>(g, s, pdl);
        case 16 * 8 + ROLE_CLUSTER_PLAIN: return run<16, true, false, ROLE_CLUSTER_PLAIN>(g, s, pdl);
        case 16 * 8 + ROLE_CLUSTER_GATE: return run<16, true, false, ROLE_CLUSTER_GATE>(g, s, pdl);
        case 32 * 8 + ROLE_ANY: return run<32, true, false, ROLE_ANY>(g, s, pdl);
        case 32 * 8 + ROLE_GATED_TILE: return run<32, true, false, ROLE_GATED_TILE>(g, s, pdl);
        case 32 * 8 + ROLE_CLUSTER_PLAIN: return run<32, true, false, ROLE_CLUSTER_PLAIN>(g, s, pdl);
        case 32 * 8 + ROLE_CLUSTER_GATE: return run<32, true, false, ROLE_CLUSTER_GATE>(g, s, pdl);
        case 64 * 8 + ROLE_ANY: return run<64, true, false, ROLE_ANY>(g, s, pdl);
        case 64 * 8 + ROLE_GATED_TILE: return run<64, true, false, ROLE_GATED_TILE>(g, s, pdl);
        case 64 * 8 + ROLE_CLUSTER_PLAIN: return run<64, true, false, ROLE_CLUSTER_PLAIN>(g, s, pdl);
        case 64 * 8 + ROLE_CLUSTER_GATE: return run<64, true, false, ROLE_CLUSTER_GATE>(g, s, pdl);
        default: return cudaErrorInvalidValue;
        }
    }
    if (g.p.epi == EPI_ROPE) {
        switch (g.bn) {
        case 128: return run<128, false, false, ROLE_ROPE>(g, s, pdl);
        case 256: return g.p.pair ? run<256, false, true, ROLE_ROPE>(g, s, pdl) : run<256, false, false, ROLE_ROPE>(g, s, pdl);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (g.bn) {
    case 128: return run<128, false>(g, s, pdl);
    case 256: return g.p.pair ? run<256, false, true>(g, s, pdl) : run<256, false>(g, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace frt
