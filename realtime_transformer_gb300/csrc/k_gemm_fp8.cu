// k_gemm_fp8.cu -- FP8 (E4M3 x E4M3 -> fp32) GEMM on sm_103a tensor cores
// with the epilogues of the FFN sublayer's steps A2 and A4 (itsolotime FlashRT
// article, 7.2: gate/up GEMM, down GEMM + residual add; "FlashRT
// docs/architecture.md", 6: alpha = act_scale x weight_scale applied in the
// GEMM as a host scalar).
//
// One persistent kernel template, 192 threads per CTA, one CTA per SM:
//   warp 4      TMA producer: streams 128-byte-wide K slices of the two
//               operands into a ring of shared-memory stages (128B swizzle);
//   warp 5      MMA issuer: one thread issues tcgen05.mma (kind::f8f6f4,
//               M = 128, N = BN, K = 32) into a double-buffered TMEM
//               accumulator and commits to mbarriers;
//   warps 0..3  epilogue: tcgen05.ld of the accumulator (one TMEM lane per
//               thread), scale by alpha, optional residual add, BF16 store;
//               with split-K, fp32 partials go to a workspace and the last
//               CTA to arrive on a tile sums them in split order
//               (deterministic) and runs the epilogue.
// Two operand roles:
//   tiled  (P = token tiles of 128 rows, Q = weight tiles of BN rows) for
//          many tokens;
//   swap   (P = weight tiles of 128 rows, Q = the <= 64 tokens padded to BN)
//          for few tokens: the layer is then bound by streaming the weights
//          from HBM, and split-K spreads that stream over all SMs.
// Weight tiles are requested before griddepcontrol.wait, so with
// programmatic dependent launch they stream in while the previous kernel of
// the layer finishes; activation tiles are requested after it.
// Every wait is bounded (frt_ptx.cuh); on a timeout the CTA drains its
// in-flight copies and MMAs, frees TMEM and exits with the error word set.
#include <cuda_bf16.h>

#include <algorithm>

#include "frt_internal.h"
#include "frt_ptx.cuh"

namespace frt {

namespace {

constexpr int BM = 128;        // MMA M = rows of the P tile = TMEM lanes
constexpr int BK = 128;        // K bytes per stage = one 128-byte swizzle row
constexpr int UK = 32;         // K of one tcgen05.mma for 8-bit operands
constexpr int NTHREADS = 192;  // 4 epilogue warps + producer warp + MMA warp
constexpr int SMEM_STAGE_BUDGET = 196608;

template <int BN>
struct Cfg {
    static constexpr uint32_t P_BYTES = BM * BK;
    static constexpr uint32_t Q_BYTES = BN * BK;
    static constexpr uint32_t STAGE_BYTES = P_BYTES + Q_BYTES;
    static constexpr int STAGES = (SMEM_STAGE_BUDGET / (int)STAGE_BYTES) > 10 ? 10
                                                                             : (SMEM_STAGE_BUDGET / (int)STAGE_BYTES);
    static constexpr uint32_t TMEM_COLS = (2 * BN <= 32)    ? 32
                                          : (2 * BN <= 64)  ? 64
                                          : (2 * BN <= 128) ? 128
                                          : (2 * BN <= 256) ? 256
                                                            : 512;
    static constexpr int CH = BN < 32 ? 16 : 32;  // accumulator columns per tcgen05.ld
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + 256;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
    static_assert(Q_BYTES % 1024 == 0, "tiles must stay 1024-byte aligned");
};

struct Unit {
    int tp, tq, kb0, kb1, tile, split;
};

__device__ __forceinline__ Unit decode(const GemmParams &p, int u) {
    Unit w;
    w.split = u % p.splits;
    w.tile = u / p.splits;
    w.tp = w.tile % p.n_tiles_p;
    w.tq = w.tile / p.n_tiles_p;
    w.kb0 = w.split * p.kb_per_split;
    w.kb1 = min(p.k_blocks, w.kb0 + p.kb_per_split);
    return w;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t bf16_bits(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// ------------------------------------------------------------ producer --
template <int BN, bool SWAP>
__device__ void producer(const CUtensorMap *tmP, const CUtensorMap *tmQ, const GemmParams &p, uint8_t *sP,
                         uint8_t *sQ, uint64_t *full, uint64_t *empty, volatile int *abort_f) {
    using C = Cfg<BN>;
    const uint64_t pol_w = l2_policy_evict_first();  // weights: read once per launch
    const uint64_t pol_x = l2_policy_evict_last();   // activations: re-read by many CTAs
    int stage = 0;
    uint32_t phase = 0;
    bool waited = false;
    int n_def = 0;
    int def_stage[C::STAGES], def_kb[C::STAGES], def_row[C::STAGES];
    uint32_t issued = 0, issued_par = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
        const Unit w = decode(p, u);
        const int prow = p.p_row0 + w.tp * BM;
        const int qrow = p.q_row0 + w.tq * BN;
        const int wrow = SWAP ? prow : qrow;
        const int xrow = SWAP ? qrow : prow;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
            if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_f, p.err))
                goto drain;
            {
                const uint32_t fb = smem_u32(&full[stage]);
                mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                issued |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                const uint32_t dP = smem_u32(sP + (size_t)stage * C::P_BYTES);
                const uint32_t dQ = smem_u32(sQ + (size_t)stage * C::Q_BYTES);
                const uint32_t dW = SWAP ? dP : dQ;
                const uint32_t dX = SWAP ? dQ : dP;
                const CUtensorMap *mW = SWAP ? tmP : tmQ;
                const CUtensorMap *mX = SWAP ? tmQ : tmP;
                tma_load_2d(dW, mW, fb, kb * BK, wrow, pol_w);
                if (waited) {
                    tma_load_2d(dX, mX, fb, kb * BK, xrow, pol_x);
                } else {
                    def_stage[n_def] = stage;
                    def_kb[n_def] = kb;
                    def_row[n_def] = xrow;
                    ++n_def;
                    if (n_def == C::STAGES || kb + 1 == w.kb1) {
                        pdl_wait();
                        waited = true;
                        for (int i = 0; i < n_def; ++i) {
                            const uint32_t fbi = smem_u32(&full[def_stage[i]]);
                            const uint32_t dst = SWAP ? smem_u32(sQ + (size_t)def_stage[i] * C::Q_BYTES)
                                                      : smem_u32(sP + (size_t)def_stage[i] * C::P_BYTES);
                            tma_load_2d(dst, mX, fbi, def_kb[i] * BK, def_row[i], pol_x);
                        }
                        n_def = 0;
                    }
                }
            }
            if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!waited)
        pdl_wait();
    return;
drain:
    // Give copies in flight a bounded time to land before the CTA exits.
    for (int s = 0; s < C::STAGES; ++s)
        if (issued & (1u << s))
            mbar_wait_for(smem_u32(&full[s]), (issued_par >> s) & 1u, 100000000ull);
}

// ---------------------------------------------------------- MMA issuer --
template <int BN>
__device__ void mma_issuer(const GemmParams &p, uint8_t *sP, uint8_t *sQ, uint64_t *full, uint64_t *empty,
                           uint64_t *tfull, uint64_t *tempty, uint64_t *drain_bar, uint32_t tmem_base,
                           volatile int *abort_f) {
    using C = Cfg<BN>;
    constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
    int stage = 0;
    uint32_t phase = 0;
    int abuf = 0;
    uint32_t aphase = 0;
    bool issued_any = false;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
        const Unit w = decode(p, u);
        if (!mbar_wait(smem_u32(&tempty[abuf]), aphase ^ 1u, abort_f, p.err))
            goto drain;
        tc_fence_after();
        {
            const uint32_t dt = tmem_base + (uint32_t)(abuf * BN);
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                if (!mbar_wait(smem_u32(&full[stage]), phase, abort_f, p.err))
                    goto drain;
                tc_fence_after();
                const uint32_t aP = smem_u32(sP + (size_t)stage * C::P_BYTES);
                const uint32_t aQ = smem_u32(sQ + (size_t)stage * C::Q_BYTES);
#pragma unroll
                for (int k = 0; k < BK / UK; ++k)
                    mma_f8f6f4(dt, smem_desc_k128(aP + k * UK), smem_desc_k128(aQ + k * UK), idesc,
                               (kb > w.kb0 || k > 0) ? 1u : 0u);
                issued_any = true;
                mma_commit(smem_u32(&empty[stage]));  // frees the stage when these MMAs finish
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        mma_commit(smem_u32(&tfull[abuf]));  // accumulator ready for the epilogue
        if (++abuf == 2) {
            abuf = 0;
            aphase ^= 1u;
        }
    }
    return;
drain:
    if (issued_any) {
        mma_commit(smem_u32(drain_bar));
        mbar_wait_for(smem_u32(drain_bar), 0, 100000000ull);
    }
}

// ------------------------------------------------------------ epilogue --
template <int CH>
__device__ __forceinline__ void tmem_load_chunk(uint32_t taddr, float (&v)[CH]) {
    uint32_t r[CH];
    __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp, converged
    if constexpr (CH == 16)
        tmem_ld_x16(taddr, r);
    else
        tmem_ld_x32(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < CH; ++j)
        v[j] = __uint_as_float(r[j]);
}

// Store CH accumulator columns c .. c+CH-1 of P-row r of this unit's tile.
template <int BN, bool SWAP, int CH>
__device__ __forceinline__ void store_chunk(const GemmParams &p, const Unit &w, int r, int c, const float (&v)[CH]) {
    if constexpr (!SWAP) {
        const int m = w.tp * BM + r;  // token
        if (m >= p.m_tok)
            return;
        const int n0 = w.tq * BN + c;  // first feature
        if (p.epi == EPI_F32) {
            float *o = static_cast<float *>(p.out) + (size_t)m * p.ldo + n0;
#pragma unroll
            for (int j = 0; j < CH; j += 4) {
                if (n0 + j >= p.n_feat)
                    break;
                *reinterpret_cast<float4 *>(o + j) =
                    make_float4(__fmul_rn(v[j], p.alpha), __fmul_rn(v[j + 1], p.alpha),
                                __fmul_rn(v[j + 2], p.alpha), __fmul_rn(v[j + 3], p.alpha));
            }
            return;
        }
        uint16_t *o = static_cast<uint16_t *>(p.out) + (size_t)m * p.ldo + n0;
#pragma unroll
        for (int j = 0; j < CH; j += 8) {
            if (n0 + j >= p.n_feat)
                break;
            float f[8];
#pragma unroll
            for (int t = 0; t < 8; ++t)
                f[t] = __fmul_rn(v[j + t], p.alpha);
            if (p.epi == EPI_RESID) {
                const uint4 rv = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.resid) +
                                                                 (size_t)m * p.ldr + n0 + j);
                f[0] = __fadd_rn(bf_lo(rv.x), f[0]);
                f[1] = __fadd_rn(bf_hi(rv.x), f[1]);
                f[2] = __fadd_rn(bf_lo(rv.y), f[2]);
                f[3] = __fadd_rn(bf_hi(rv.y), f[3]);
                f[4] = __fadd_rn(bf_lo(rv.z), f[4]);
                f[5] = __fadd_rn(bf_hi(rv.z), f[5]);
                f[6] = __fadd_rn(bf_lo(rv.w), f[6]);
                f[7] = __fadd_rn(bf_hi(rv.w), f[7]);
            }
            uint4 ov;
            ov.x = bf16_bits(f[0]) | (bf16_bits(f[1]) << 16);
            ov.y = bf16_bits(f[2]) | (bf16_bits(f[3]) << 16);
            ov.z = bf16_bits(f[4]) | (bf16_bits(f[5]) << 16);
            ov.w = bf16_bits(f[6]) | (bf16_bits(f[7]) << 16);
            *reinterpret_cast<uint4 *>(o + j) = ov;
        }
    } else {
        const int n = w.tp * BM + r;  // feature
        if (n >= p.n_feat)
            return;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const int m = w.tq * BN + c + j;  // token
            if (m >= p.m_tok)
                break;
            float f = __fmul_rn(v[j], p.alpha);
            if (p.epi == EPI_F32) {
                static_cast<float *>(p.out)[(size_t)m * p.ldo + n] = f;
            } else {
                if (p.epi == EPI_RESID) {
                    const uint16_t rb = static_cast<const uint16_t *>(p.resid)[(size_t)m * p.ldr + n];
                    f = __fadd_rn(__uint_as_float((uint32_t)rb << 16), f);
                }
                static_cast<uint16_t *>(p.out)[(size_t)m * p.ldo + n] = (uint16_t)bf16_bits(f);
            }
        }
    }
}

template <int BN, bool SWAP>
__device__ void epilogue(const GemmParams &p, uint64_t *tfull, uint64_t *tempty, uint32_t tmem_base,
                         volatile int *abort_f, volatile int *s_ok, volatile int *s_last) {
    using C = Cfg<BN>;
    constexpr int CH = C::CH;
    const int warp = threadIdx.x >> 5;
    const int r = threadIdx.x;  // P-tile row = TMEM lane (warps 0..3)
    pdl_wait();
    int abuf = 0;
    uint32_t aphase = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
        const Unit w = decode(p, u);
        // One thread waits (bounded) and tells the others, so that all 128
        // threads leave the loop together if the wait gives up.
        if (threadIdx.x == 0)
            s_ok[abuf] = mbar_wait(smem_u32(&tfull[abuf]), aphase, abort_f, p.err) ? 1 : 0;
        named_bar_sync(1, 128);
        if (!s_ok[abuf])
            break;
        tc_fence_after();
        const uint32_t tbase = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(abuf * BN);
        if (p.splits == 1) {
#pragma unroll 1
            for (int c = 0; c < BN; c += CH) {
                float v[CH];
                tmem_load_chunk<CH>(tbase + c, v);
                store_chunk<BN, SWAP, CH>(p, w, r, c, v);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&tempty[abuf]));
        } else {
            float *mine = p.ws + ((size_t)w.tile * p.splits + w.split) * (size_t)(BM * BN);
#pragma unroll 1
            for (int c = 0; c < BN; c += CH) {
                float v[CH];
                tmem_load_chunk<CH>(tbase + c, v);
#pragma unroll
                for (int j = 0; j < CH; ++j)
                    mine[(size_t)(c + j) * BM + r] = v[j];
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&tempty[abuf]));
            __threadfence();
            named_bar_sync(1, 128);
            if (threadIdx.x == 0) {
                const int prev = atomicAdd(&p.counters[w.tile], 1);
                s_last[abuf] = (prev == p.splits - 1) ? 1 : 0;
            }
            named_bar_sync(1, 128);
            if (s_last[abuf]) {
                __threadfence();
                const float *tile_ws = p.ws + (size_t)w.tile * p.splits * (size_t)(BM * BN);
#pragma unroll 1
                for (int c = 0; c < BN; c += CH) {
                    float v[CH];
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        float s = 0.0f;
                        for (int sp = 0; sp < p.splits; ++sp)
                            s = __fadd_rn(s, ld_cg_f32(tile_ws + (size_t)sp * (BM * BN) + (size_t)(c + j) * BM + r));
                        v[j] = s;
                    }
                    store_chunk<BN, SWAP, CH>(p, w, r, c, v);
                }
                if (threadIdx.x == 0)
                    p.counters[w.tile] = 0;  // ready for the next launch
            }
        }
        if (++abuf == 2) {
            abuf = 0;
            aphase ^= 1u;
        }
    }
}

// -------------------------------------------------------------- kernel --
template <int BN, bool SWAP>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_gemm_fp8(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
               const GemmParams p) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sP = smem;
    uint8_t *sQ = smem + (size_t)C::STAGES * C::P_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sQ + (size_t)C::STAGES * C::Q_BYTES);
    uint64_t *full = bars;
    uint64_t *empty = bars + C::STAGES;
    uint64_t *tfull = bars + 2 * C::STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain_bar = tempty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain_bar + 1);
    volatile int *abort_f = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *s_ok = abort_f + 1;    // [2]
    volatile int *s_last = s_ok + 2;     // [2]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), 128);
        }
        mbar_init(smem_u32(drain_bar), 1);
        *abort_f = 0;
        fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmP);
        prefetch_tmap(&tmQ);
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_trigger();

    if (warp < 4) {
        epilogue<BN, SWAP>(p, tfull, tempty, tmem_base, abort_f, s_ok, s_last);
    } else if (warp == 4) {
        if (lane == 0)
            producer<BN, SWAP>(&tmP, &tmQ, p, sP, sQ, full, empty, abort_f);
    } else {
        if (lane == 0)
            mma_issuer<BN>(p, sP, sQ, full, empty, tfull, tempty, drain_bar, tmem_base, abort_f);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) {
        __syncwarp();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int BN, bool SWAP>
cudaError_t run(const GemmLaunch &g, cudaStream_t s, bool pdl) {
    using C = Cfg<BN>;
    static int attr_done = 0;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_fp8<BN, SWAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::SMEM);
        if (e != cudaSuccess)
            return e;
        attr_done = 1;
    }
    return launch_ex(k_gemm_fp8<BN, SWAP>, dim3((unsigned)g.grid), dim3(NTHREADS), C::SMEM, s, pdl, g.tmP, g.tmQ,
                     g.p);
}

}  // namespace

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

void plan_gemm(GemmLaunch &g, bool swap, int m_tok, int n_feat, int K, int num_sms, int force_splits) {
    GemmParams &p = g.p;
    g.swap = swap;
    p.k_blocks = (K + BK - 1) / BK;
    if (swap) {
        g.bn = m_tok <= 16 ? 16 : (m_tok <= 32 ? 32 : 64);
        p.n_tiles_p = (n_feat + BM - 1) / BM;
        p.n_tiles_q = (m_tok + g.bn - 1) / g.bn;
    } else {
        g.bn = (n_feat % 256 == 0) ? 256 : 128;
        p.n_tiles_p = (m_tok + BM - 1) / BM;
        p.n_tiles_q = (n_feat + g.bn - 1) / g.bn;
    }
    const int tiles = p.n_tiles_p * p.n_tiles_q;
    int splits = 1;
    if (force_splits > 0)
        splits = force_splits;
    else if (tiles < num_sms)
        splits = num_sms / tiles;
    splits = std::max(1, std::min(splits, p.k_blocks));
    p.kb_per_split = (p.k_blocks + splits - 1) / splits;
    p.splits = (p.k_blocks + p.kb_per_split - 1) / p.kb_per_split;
    p.total_units = tiles * p.splits;
    g.grid = std::min(p.total_units, num_sms);
    p.m_tok = m_tok;
    p.n_feat = n_feat;
}

size_t gemm_ws_floats(const GemmLaunch &g) {
    if (g.p.splits <= 1)
        return 0;
    return (size_t)g.p.total_units * BM * (size_t)g.bn;
}

int gemm_tiles(const GemmLaunch &g) { return g.p.n_tiles_p * g.p.n_tiles_q; }

cudaError_t launch_gemm(const GemmLaunch &g, cudaStream_t s, bool pdl) {
    if (g.swap) {
        switch (g.bn) {
        case 16: return run<16, true>(g, s, pdl);
        case 32: return run<32, true>(g, s, pdl);
        case 64: return run<64, true>(g, s, pdl);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (g.bn) {
    case 128: return run<128, false>(g, s, pdl);
    case 256: return run<256, false>(g, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace frt
