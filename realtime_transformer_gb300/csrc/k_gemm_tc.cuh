// k_gemm_tc.cuh -- the tensor-core GEMM behind the FFN sublayer's GEMM steps
// (itsolotime FlashRT article, 7.2: gate/up GEMM, down GEMM + residual add;
// "FlashRT docs/architecture.md", 6: alpha = act_scale x weight_scale applied
// in the GEMM as a host scalar), for E4M3 operands (tcgen05.mma
// kind::f8f6f4) and NVFP4 operands (kind::mxf4nvf4 with E4M3 block scales,
// the pages' NVFP4 encoder FFN).  Included by the translation units that
// instantiate it: k_gemm_fp8.cu (E4M3) and k_gemm_f4.cu (NVFP4).
#pragma once
//
// One persistent kernel template, 192 threads per CTA (320 with NVFP4 operands):
//   warp 4      TMA producer: streams 128-byte-wide K slices of the two
//               operands into a ring of shared-memory stages (128B swizzle);
//   warp 5      MMA issuer: one thread issues tcgen05.mma (kind::f8f6f4,
//               M = 128, N = BN, K = 32) into a double-buffered TMEM
//               accumulator and commits to mbarriers;
//   warps 0..3  epilogue: tcgen05.ld of the accumulator (one TMEM lane per
//               thread), scale by alpha, gated activation + E4M3 requantise
//               or residual add + BF16 store;
//   warps 6..9  (NVFP4 only) scale warps: each stage's E4M3 block scales
//               from shared memory into TMEM (tcgen05.st) for the MMAs.
// Split-K is cooperative (one unit per CTA): each split stages its fp32
// partial, the S partials of a tile are exchanged -- over distributed shared
// memory inside a thread-block cluster, or through a global workspace --
// and every split reduces a 1/S slice of the tile in split order
// (deterministic) and runs the epilogue for it.
// Two operand roles:
//   tiled  (P = token tiles of 128 rows, Q = weight tiles of BN rows) for
//          many tokens;
//   swap   (P = weight tiles of 128 rows, Q = the <= 64 tokens padded to BN)
//          for few tokens: the layer is then bound by streaming the weights
//          from HBM, spread over the SMs by the tile count and split-K.
// Weight tiles are requested before griddepcontrol.wait, so with
// programmatic dependent launch they stream in while the previous kernel of
// the layer finishes (a short launch keeps a small shared-memory footprint so
// that its CTAs share SMs with the previous kernel's); activation tiles are
// requested after it.
// Every wait is bounded (frt_ptx.cuh); on a timeout the CTA drains its
// in-flight copies and MMAs, frees TMEM and exits with the error word set.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "frt_epi.cuh"
#include "frt_f4.cuh"
#include "frt_internal.h"
#include "frt_ptx.cuh"

namespace frt {

namespace {

constexpr int BM = 128;        // MMA M = rows of the P tile = TMEM lanes
constexpr int BK = 128;        // K bytes per stage = one 128-byte swizzle row
constexpr int UK = 32;         // K of one tcgen05.mma for 8-bit operands
constexpr int NTHREADS = 192;  // 4 epilogue warps + producer warp + MMA warp
constexpr int NTHREADS_F4 = 320;  // NVFP4: and 4 scale warps (warps 6..9)
constexpr int GATED_TOKENS = 4;  // tokens per step of the weight-streaming gated epilogue
constexpr uint32_t SMEM_LIMIT = 232448;  // largest dynamic shared memory of one CTA (227 KB)

// PAIR: the tiled role on a CTA pair (cta_group::2): each CTA stages its own
// token tile and half of the weight tile.
// F4: NVFP4 operands.  A stage's 128 bytes of K then hold 256 E2M1 elements,
// and the stage also carries both operands' E4M3 block scales in the
// TMEM-ready order: per 128 rows four 512-byte blocks (one per 64-element K
// chunk), the P tile's 2 KB then the Q tile's 2 KB per 128 of its rows (the
// weight-streaming role's <= 64 tokens are the first rows of their 128-row
// block).  In TMEM a chunk's scales take 4 columns per 128 rows (row r at
// lane r % 32 of every lane quarter, column r / 32).  A 256-row Q tile
// leaves room for one accumulator only (the epilogue of a tile then runs
// between its MMAs and the next tile's).  Four scale warps, one per TMEM lane quarter, write a
// stage's scales into 32 TMEM columns of their own (tcgen05.st, each quarter
// a copy: the replicated order kind::mxf4nvf4 reads) and signal the MMA
// thread, so the tensor pipe issues MMAs only.
template <int BN, bool SWAP = false, bool PAIR = false, bool F4 = false>
struct Cfg {
    static_assert(!(PAIR && SWAP), "CTA pairs serve the tiled role");
    static_assert(!(F4 && PAIR), "NVFP4 tiles: single CTAs");
    static constexpr uint32_t P_BYTES = BM * BK;
    static constexpr uint32_t Q_BYTES = (PAIR ? BN / 2 : BN) * BK;
    static constexpr int SF_QB = F4 ? (BN + 127) / 128 : 0;  // 128-row scale blocks of the Q tile
    static constexpr uint32_t SF_BYTES = F4 ? 2048u * (1 + SF_QB) : 0;  // block scales of a stage (P's, then Q's)
    static constexpr uint32_t STAGE_BYTES = P_BYTES + Q_BYTES + SF_BYTES;
    static constexpr int SF_COLS = 16 + 16 * SF_QB;  // TMEM columns of a stage's block scales (F4)
    static constexpr int ACC_BUFS = (F4 && BN > 128) ? 1 : 2;  // TMEM accumulators
    static constexpr uint32_t BAR_BYTES = F4 ? 512 : 256;  // mbarriers and flags after the stages
    static constexpr int CH = BN < 32 ? 16 : 32;  // accumulator columns per tcgen05.ld
    static constexpr uint32_t XBUF_BYTES = SWAP ? BN * (128 + 4) * 4 : 0;  // gate/up exchange, whole tile
    static constexpr int STAGES_FIT =
        (int)((SMEM_LIMIT - 1024 - BAR_BYTES - XBUF_BYTES) / STAGE_BYTES);
    static constexpr int STAGES_TMEM = F4 ? (512 - ACC_BUFS * BN) / SF_COLS : 64;  // scale columns within TMEM
    static constexpr int STAGES_CAP = STAGES_FIT < STAGES_TMEM ? STAGES_FIT : STAGES_TMEM;
    static constexpr int STAGES = STAGES_CAP > 10 ? 10 : STAGES_CAP;  // most stages a launch may ask for
    static constexpr uint32_t TMEM_COLS = (2 * BN <= 32)    ? 32
                                          : (2 * BN <= 64)  ? 64
                                          : (2 * BN <= 128) ? 128
                                          : (2 * BN <= 256) ? 256
                                                            : 512;
    // TMEM columns of a launch with `stages` stages: the accumulators, then
    // (F4) the stages' scale columns; a power of two
    __host__ __device__ static uint32_t tmem_cols(int stages) {
        if (!F4)
            return TMEM_COLS;
        const uint32_t need = (uint32_t)(ACC_BUFS * BN) + (uint32_t)(SF_COLS * stages);
        return need <= 32 ? 32u : need <= 64 ? 64u : need <= 128 ? 128u : need <= 256 ? 256u : 512u;
    }
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + BAR_BYTES + XBUF_BYTES;
    // Shared memory of a launch with `stages` pipeline stages: a small
    // footprint lets the next kernel's CTAs share the SM and start streaming
    // their weights while this one runs.
    // (the gate/up exchange buffer only for the unsplit gated epilogue)
    static size_t smem_bytes(int stages, bool xbuf) {
        return 1024 + (size_t)stages * STAGE_BYTES + BAR_BYTES + (xbuf ? XBUF_BYTES : 0);
    }
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
    static_assert(Q_BYTES % 1024 == 0, "tiles must stay 1024-byte aligned");
    static_assert(STAGES >= 2, "pipeline needs two stages");
    static_assert(SMEM <= SMEM_LIMIT, "shared memory over the per-CTA limit");
    static_assert(((F4 ? 4 : 2) * STAGES + 9) * 8 + 24 <= BAR_BYTES, "mbarriers and flags fit their block");
};

struct Unit {
    int tp, tq, kb0, kb1, tile, split;
};

// Epilogue roles a kernel is compiled for: every epilogue (ROLE_ANY), or
// only the one a launch of the layer uses -- the weight-streaming gated
// epilogue without split-K (the gate/up GEMM) or the plain cluster split-K
// epilogue (the down GEMM) -- so that the code a launch runs is compact; the
// tiled QKV split + RoPE epilogue (ROLE_ROPE) is compiled only for itself,
// and the AdaRMSNorm gate of the residual only where a launch has one
// (ROLE_CLUSTER_GATE, and the general ROLE_ANY).
enum Role : int { ROLE_ANY = 0, ROLE_GATED_TILE = 1, ROLE_CLUSTER_PLAIN = 2, ROLE_ROPE = 3, ROLE_CLUSTER_GATE = 4 };

// Tiles run in groups of p.group P-tiles: within a group the P-tile index
// changes fastest, so a wave of CTAs covers a block of group x (SMs / group)
// tiles whose operands stay in L2 together.
__device__ __forceinline__ Unit decode(const GemmParams &p, int u) {
    Unit w;
    if (!p.pair) {
        w.split = u % p.splits;
        w.tile = u / p.splits;
        const int per_group = p.group * p.n_tiles_q;
        const int grp = w.tile / per_group;
        const int rem = w.tile - grp * per_group;
        const int gsize = min(p.group, p.n_tiles_p - grp * p.group);
        w.tp = grp * p.group + rem % gsize;
        w.tq = rem / gsize;
    } else {
        // CTA pair: the two CTAs of a cluster (consecutive units) take two
        // consecutive P-tiles of the same weight tile and split; the raster
        // runs over blocks of two P-tiles
        constexpr int C = 2;
        const int rank = u % C;
        const int v = u / C;
        w.split = v % p.splits;
        const int t = v / p.splits;
        const int nblk = p.n_tiles_p / C;
        const int group = max(1, p.group / C);
        const int per_group = group * p.n_tiles_q;
        const int grp = t / per_group;
        const int rem = t - grp * per_group;
        const int gsize = min(group, nblk - grp * group);
        w.tp = (grp * group + rem % gsize) * C + rank;
        w.tq = rem / gsize;
        w.tile = w.tq * p.n_tiles_p + w.tp;
    }
    w.kb0 = w.split * p.kb_per_split;
    w.kb1 = min(p.k_blocks, w.kb0 + p.kb_per_split);
    return w;
}

// ------------------------------------------------------------ producer --
template <int BN, bool SWAP, bool PAIR, bool F4>
__device__ void producer(const CUtensorMap *tmP, const CUtensorMap *tmQ, const GemmParams &p, uint8_t *sP,
                         uint8_t *sQ, uint8_t *sSF, uint64_t *full, uint64_t *empty, uint64_t *sffull,
                         volatile int *abort_f) {
    using C = Cfg<BN, SWAP, PAIR, F4>;
    // F4: a stage's 2 KB of block scales of the 128-row tile holding `row`
    // (K / 64 blocks of 512 bytes per 128 rows, tiles major); weight scales
    // are requested before the weight tile, token scales before the token
    // tile (P's first in the stage's scale area), all completing on the
    // stage's own scale barrier, so the scale warps can move them into TMEM
    // while the operand tiles are still in flight
    const size_t sf_tile = (size_t)p.k_blocks * 2048u;
    const uint32_t sf_w_off = SWAP ? 0u : 2048u, sf_x_off = SWAP ? 2048u : 0u;
    // CTA pair: both CTAs' copies complete on the even CTA's stage barrier,
    // which alone is armed (with both CTAs' bytes)
    const uint32_t rank = PAIR ? (blockIdx.x & 1u) : 0u;
    // weights first out of L2, activations last (on GB300 this measured best
    // for the tiled role too, where weight tiles are reused within a wave)
    const uint64_t pol_w = p.w_evict == 1 ? l2_policy_evict_normal()
                           : p.w_evict == 2 ? l2_policy_evict_last() : l2_policy_evict_first();
    const uint64_t pol_x = p.x_evict == 1 ? l2_policy_evict_normal()
                           : p.x_evict == 0 ? l2_policy_evict_first() : l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    bool waited = false;
    const int NS = p.stages;
    // activation loads deferred until the previous grid has completed: a run
    // of consecutive k-blocks of one unit in consecutive stages (registers,
    // not an indexed array: local memory would cost a trip to L2 after the
    // dependency wait)
    int n_def = 0, def_kb = 0, def_stage = 0, def_row = 0;
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
                const uint32_t fb = PAIR ? mapa_shared(smem_u32(&full[stage]), 0u) : smem_u32(&full[stage]);
                const uint32_t sfb = F4 ? smem_u32(&sffull[stage]) : 0u;
                if constexpr (F4) {
                    mbar_arrive_expect_tx(sfb, C::SF_BYTES);
                    mbar_arrive_expect_tx(fb, C::P_BYTES + C::Q_BYTES);
                } else if (!PAIR) {
                    mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                } else if (rank == 0) {
                    mbar_arrive_expect_tx(smem_u32(&full[stage]), 2u * C::STAGE_BYTES);
                }
                issued |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                const uint32_t dP = smem_u32(sP + (size_t)stage * C::P_BYTES);
                const uint32_t dQ = smem_u32(sQ + (size_t)stage * C::Q_BYTES);
                const uint32_t dW = SWAP ? dP : dQ;
                const uint32_t dX = SWAP ? dQ : dP;
                const CUtensorMap *mW = SWAP ? tmP : tmQ;
                const CUtensorMap *mX = SWAP ? tmQ : tmP;
                if constexpr (F4) {
                    constexpr int WB = SWAP ? 1 : C::SF_QB;  // 128-row blocks of the weight tile
#pragma unroll
                    for (int i = 0; i < WB; ++i)
                        bulk_load(smem_u32(sSF + (size_t)stage * C::SF_BYTES + sf_w_off + 2048u * i),
                                  p.sf_w + (size_t)(wrow / BM + i) * sf_tile + (size_t)kb * 2048u, 2048u, sfb);
                }
                if constexpr (PAIR) {
                    // this CTA's half of the weight tile
                    tma_load_2d_pair(dW, mW, fb, kb * BK, wrow + (int)rank * (BN / 2), pol_w);
                } else {
                    tma_load_2d(dW, mW, fb, kb * BK, wrow, pol_w);
                }
                if (waited) {
                    if constexpr (F4)
                        bulk_load(smem_u32(sSF + (size_t)stage * C::SF_BYTES + sf_x_off),
                                  p.sf_x + (size_t)(xrow / BM) * sf_tile + (size_t)kb * 2048u, 2048u, sfb);
                    if constexpr (PAIR)
                        tma_load_2d_pair(dX, mX, fb, kb * BK, xrow, pol_x);
                    else
                        tma_load_2d(dX, mX, fb, kb * BK, xrow, pol_x);
                } else {
                    if (n_def == 0) {
                        def_kb = kb;
                        def_stage = stage;
                        def_row = xrow;
                    }
                    ++n_def;
                    if (n_def == NS || kb + 1 == w.kb1) {
                        pdl_wait();
                        waited = true;
                        int st = def_stage;
                        for (int i = 0; i < n_def; ++i) {
                            const uint32_t fbi =
                                PAIR ? mapa_shared(smem_u32(&full[st]), 0u) : smem_u32(&full[st]);
                            const uint32_t dst = SWAP ? smem_u32(sQ + (size_t)st * C::Q_BYTES)
                                                      : smem_u32(sP + (size_t)st * C::P_BYTES);
                            if constexpr (F4)
                                bulk_load(smem_u32(sSF + (size_t)st * C::SF_BYTES + sf_x_off),
                                          p.sf_x + (size_t)(def_row / BM) * sf_tile + (size_t)(def_kb + i) * 2048u,
                                          2048u, smem_u32(&sffull[st]));
                            if constexpr (PAIR)
                                tma_load_2d_pair(dst, mX, fbi, (def_kb + i) * BK, def_row, pol_x);
                            else
                                tma_load_2d(dst, mX, fbi, (def_kb + i) * BK, def_row, pol_x);
                            if (++st == NS)
                                st = 0;
                        }
                        n_def = 0;
                    }
                }
            }
            if (++stage == NS) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!waited)
        pdl_wait();
    return;
drain:
    // Give copies in flight a bounded time to land before the CTA exits (a
    // pair's odd CTA has no armed stage barrier of its own; the pair's
    // closing cluster barrier holds it until the even one is done).
    for (int s = 0; s < NS; ++s)
        if (issued & (1u << s)) {
            if (!PAIR || rank == 0)
                mbar_wait_for(smem_u32(&full[s]), (issued_par >> s) & 1u, 100000000ull);
            if constexpr (F4)
                mbar_wait_for(smem_u32(&sffull[s]), (issued_par >> s) & 1u, 100000000ull);
        }
}

// ---------------------------------------------------------- MMA issuer --
template <int BN, bool SWAP, bool PAIR, bool F4>
__device__ void mma_issuer(const GemmParams &p, uint8_t *sP, uint8_t *sQ, uint64_t *full, uint64_t *empty,
                           uint64_t *sfull, uint64_t *tfull, uint64_t *tempty, uint64_t *drain_bar,
                           uint32_t tmem_base, volatile int *abort_f) {
    using C = Cfg<BN, SWAP, PAIR, F4>;
    // a pair's MMAs (issued by the even CTA only) cover 256 token rows
    constexpr uint32_t idesc = F4 ? idesc_nvf4(BM, BN) : idesc_e4m3_f32(PAIR ? 2 * BM : BM, BN);
    int stage = 0;
    uint32_t phase = 0;
    int abuf = 0;
    uint32_t aphase = 0;
    bool issued_any = false;
    // Test hook for the failure path: wait for a phase of the drain barrier,
    // which nothing completes before an MMA is issued.  The bounded wait gives
    // up, sets the abort flag and the error word, and every role drains.
    if (p.stall_test && !mbar_wait(smem_u32(drain_bar), 0, abort_f, p.err))
        goto drain;
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
                if constexpr (F4) {
                    // the stage's block scales, in its own TMEM columns after
                    // the accumulators (per 64-element chunk j the P tile's at
                    // +4j, the Q tile's at +16+4j), once the scale warps have
                    // written them
                    if (!mbar_wait(smem_u32(&sfull[stage]), phase, abort_f, p.err))
                        goto drain;
                    tc_fence_after();
                    const uint32_t t_sf = tmem_base + (uint32_t)(C::ACC_BUFS * BN + C::SF_COLS * stage);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_nvf4(dt, smem_desc_k128(aP + k * UK), smem_desc_k128(aQ + k * UK), idesc, t_sf + 4 * k,
                                 t_sf + 16 + 4 * C::SF_QB * k, (kb > w.kb0 || k > 0) ? 1u : 0u);
                } else {
#pragma unroll
                for (int k = 0; k < BK / UK; ++k) {
                    if constexpr (PAIR)
                        mma_f8f6f4_pair(dt, smem_desc_k128(aP + k * UK), smem_desc_k128(aQ + k * UK), idesc,
                                        (kb > w.kb0 || k > 0) ? 1u : 0u);
                    else
                        mma_f8f6f4(dt, smem_desc_k128(aP + k * UK), smem_desc_k128(aQ + k * UK), idesc,
                                   (kb > w.kb0 || k > 0) ? 1u : 0u);
                }
                }
                issued_any = true;
                // frees the stage when these MMAs finish (on a CTA pair: in
                // both CTAs, each of which writes into it)
                if constexpr (PAIR)
                    mma_commit_pair(smem_u32(&empty[stage]), 0x3);
                else
                    mma_commit(smem_u32(&empty[stage]));
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // accumulator ready for the epilogue (of both CTAs of a pair)
        if constexpr (PAIR)
            mma_commit_pair(smem_u32(&tfull[abuf]), 0x3);
        else
            mma_commit(smem_u32(&tfull[abuf]));
        if (++abuf == C::ACC_BUFS) {
            abuf = 0;
            aphase ^= 1u;
        }
    }
    return;
drain:
    if (issued_any) {
        if constexpr (PAIR)
            mma_commit_pair(smem_u32(drain_bar), 0x1);
        else
            mma_commit(smem_u32(drain_bar));
        mbar_wait_for(smem_u32(drain_bar), 0, 100000000ull);
    }
}

// -------------------------------------------------------- scale warps --
// NVFP4: warps 6..9, one per TMEM lane quarter (warp id % 4).  For each stage
// in the MMA thread's order: wait until its scale copies have landed, read its
// 512-byte scale blocks (lane l: bytes 16 l .. 16 l + 15 of each, i.e. rows
// l, l + 32, l + 64, l + 96 of the block's 128), write them to this quarter's
// lanes of the stage's scale columns (P's chunk j at columns 4 j .. 4 j + 3;
// the Q tile's chunk j from 16 + 4 QB j, its 128-row blocks i at + 4 i), wait
// for the stores, and count the warp in on the stage's scales-ready barrier.  The columns of a stage are rewritten only after its
// refill, i.e. after the MMAs that read them completed.
template <int BN, bool SWAP>
__device__ void scale_feeder(const GemmParams &p, uint8_t *sSF, uint64_t *sffull, uint64_t *sfull,
                             uint32_t tmem_base, volatile int *abort_f) {
    using C = Cfg<BN, SWAP, false, true>;
    const int lane = threadIdx.x & 31;
    const uint32_t quarter = (threadIdx.x >> 5) & 3u;
    const uint32_t t_lane = tmem_base + ((quarter * 32u) << 16);
    int stage = 0;
    uint32_t phase = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
        const Unit w = decode(p, u);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
            // every lane waits itself (the blocks were written by the async proxy)
            const bool ok = mbar_wait(smem_u32(&sffull[stage]), phase, abort_f, p.err);
            if (!__all_sync(0xffffffffu, ok))
                return;
            const uint8_t *src = sSF + (size_t)stage * C::SF_BYTES + lane * 16;
            constexpr int QB = C::SF_QB;
            uint32_t v[C::SF_COLS];
#pragma unroll
            for (int b = 0; b < 4 + 4 * QB; ++b) {
                // smem block b: P's chunk b (b < 4), else the Q tile's 128-row
                // block i = (b - 4) / 4, chunk j = (b - 4) % 4
                const int col = b < 4 ? 4 * b : 16 + 4 * QB * ((b - 4) % 4) + 4 * ((b - 4) / 4);
                const uint4 q = *reinterpret_cast<const uint4 *>(src + 512 * b);
                v[col] = q.x;
                v[col + 1] = q.y;
                v[col + 2] = q.z;
                v[col + 3] = q.w;
            }
            const uint32_t t_st = t_lane + (uint32_t)(C::ACC_BUFS * BN + C::SF_COLS * stage);
            tmem_st_x32(t_st, *reinterpret_cast<const uint32_t(*)[32]>(&v[0]));
            if constexpr (C::SF_COLS == 48)
                tmem_st_x16(t_st + 32, *reinterpret_cast<const uint32_t(*)[16]>(&v[32]));
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&sfull[stage]));
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
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

// This thread's row of a weight-streaming accumulator, columns [0, BN),
// handed to put(c, v) 16 columns at a time; every TMEM load is in flight
// before the wait.
template <int BN, typename Put>
__device__ __forceinline__ void unit_row(uint32_t tbase, Put &&put) {
    __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp, converged
    uint32_t a[BN];
#pragma unroll
    for (int c = 0; c < BN; c += 16)
        tmem_ld_x16(tbase + c, *reinterpret_cast<uint32_t(*)[16]>(&a[c]));
    tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < BN; c += 16) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            v[j] = __uint_as_float(a[c + j]);
        put(c, v);
    }
}

// Store CH accumulator columns c .. c+CH-1 of P-row r (plain epilogues).
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
        // residual vectors of the whole chunk first (out may alias resid)
        uint4 rvs[CH / 8];
#pragma unroll
        for (int j = 0; j < CH; j += 8) {
            rvs[j / 8] = make_uint4(0, 0, 0, 0);
            if (p.epi == EPI_RESID && n0 + j < p.n_feat)
                rvs[j / 8] = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.resid) +
                                                             (size_t)m * p.ldr + n0 + j);
        }
        const uint16_t *gt = p.gate ? p.gate + (size_t)m * p.ldgate + n0 : nullptr;
#pragma unroll
        for (int j = 0; j < CH; j += 8) {
            if (n0 + j >= p.n_feat)
                break;
            float f[8];
#pragma unroll
            for (int t = 0; t < 8; ++t)
                f[t] = __fmul_rn(v[j + t], p.alpha);
            if (gt) {
                const uint4 gv = *reinterpret_cast<const uint4 *>(gt + j);
                f[0] = __fmul_rn(f[0], bf_lo(gv.x));
                f[1] = __fmul_rn(f[1], bf_hi(gv.x));
                f[2] = __fmul_rn(f[2], bf_lo(gv.y));
                f[3] = __fmul_rn(f[3], bf_hi(gv.y));
                f[4] = __fmul_rn(f[4], bf_lo(gv.z));
                f[5] = __fmul_rn(f[5], bf_hi(gv.z));
                f[6] = __fmul_rn(f[6], bf_lo(gv.w));
                f[7] = __fmul_rn(f[7], bf_hi(gv.w));
            }
            if (p.epi == EPI_RESID) {
                const uint4 rv = rvs[j / 8];
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
        const int m0 = w.tq * BN + c;  // first token of the chunk
        const int nv = min(CH, p.m_tok - m0);
        if (nv <= 0)
            return;
        if (p.epi == EPI_F32) {
#pragma unroll
            for (int j = 0; j < CH; ++j)
                if (j < nv)
                    static_cast<float *>(p.out)[(size_t)(m0 + j) * p.ldo + n] = __fmul_rn(v[j], p.alpha);
            return;
        }
        // Read every residual of the chunk before the first store: out may
        // alias resid, and loads issued after stores would serialise.
        float res[CH];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            res[j] = 0.0f;
            if (p.epi == EPI_RESID && j < nv)
                res[j] = __uint_as_float((uint32_t)static_cast<const uint16_t *>(p.resid)[(size_t)(m0 + j) * p.ldr + n]
                                         << 16);
        }
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            if (j < nv) {
                float f = __fmul_rn(v[j], p.alpha);
                if (p.gate)
                    f = __fmul_rn(f, __uint_as_float((uint32_t)p.gate[(size_t)(m0 + j) * p.ldgate + n] << 16));
                if (p.epi == EPI_RESID)
                    f = __fadd_rn(res[j], f);
                static_cast<uint16_t *>(p.out)[(size_t)(m0 + j) * p.ldo + n] = (uint16_t)bf16_bits(f);
            }
        }
    }
}

// --- gated epilogue (step A3 fused into the gate/up GEMM) -----------------
// The weight arena holds [W_gate; W_up] interleaved in blocks of 64 rows
// (64 gate rows, then the 64 up rows of the same features), so every tile
// holds matching gate and up rows.  g and u are rounded to BF16 (where the
// unfused method stores them), then a = act(g) * u and q_h = E4M3(a / s_h).

__device__ __forceinline__ void dbg_store_gu(const GemmParams &p, int m, int f, bool up, float val) {
    if (p.dbg_gu)
        p.dbg_gu[(size_t)m * 2 * p.ff + (up ? p.ff : 0) + f] = (uint16_t)bf16_bits(val);
}

// Weight-streaming path, whole tile at once: TMEM lanes 0..63 are gate rows,
// 64..127 the up rows of the same 64 features; columns are tokens.  Every
// thread parks its row (rounded to BF16) in xbuf, token-major (a token's 128
// rows are contiguous), and frees the accumulator; then thread t takes
// features 4(t % 16) .. +3 of tokens 8(t / 16) .. +7, reading each token's
// four gate and four up values with one 16-byte load each, and stores the
// four activations of a token as one 4-byte word of E4M3 codes.  Called by
// all 128 epilogue threads; returns after a barrier, so xbuf is free again.
template <int BN>
__device__ __forceinline__ void gated_swap_tile(const GemmParams &p, const Unit &w, int r, uint32_t tbase,
                                                uint64_t *tempty_b, float *xbuf, float &amax) {
    constexpr int LD = 128 + 4;  // floats per token
    const int m0 = w.tq * BN;    // first token of the tile
    const int ncols = min(BN, p.m_tok - m0);
    const float alpha = p.alpha;
    unit_row<BN>(tbase, [&](int c, const float (&v)[16]) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            xbuf[(c + j) * LD + r] = round_bf16(__fmul_rn(v[j], alpha));
    });
    tc_fence_before();
    mbar_arrive(smem_u32(tempty_b));  // the accumulator is read: the next unit's MMAs may start
    named_bar_sync(1, 128);
    if (p.dbg_gu) {
        const int f = w.tp * (BM / 2) + (r & 63);
        for (int c = 0; c < ncols; ++c)
            dbg_store_gu(p, m0 + c, f, r >= 64, xbuf[c * LD + r]);
    }
    constexpr int TG = BN / 8;  // tokens per thread
    constexpr int TS = TG < GATED_TOKENS ? TG : GATED_TOKENS;  // tokens per step
    const int fq = r & 15;      // feature quad
    const int c0 = (r >> 4) * TG;
    const bool meas = p.epi == EPI_GATED_AMAX;
    uint8_t *qh = static_cast<uint8_t *>(p.out) + (size_t)w.tp * (BM / 2) + 4 * fq;
    const float inv_s = p.inv_s;
    // TS tokens per step: short code, 4 TS independent activations in flight
#pragma unroll 1
    for (int i0 = 0; i0 < TG; i0 += TS) {
        float g[4 * TS], u[4 * TS], a[4 * TS];
#pragma unroll
        for (int i = 0; i < TS; ++i) {
            const float4 gv = *reinterpret_cast<const float4 *>(xbuf + (c0 + i0 + i) * LD + 4 * fq);
            const float4 uv = *reinterpret_cast<const float4 *>(xbuf + (c0 + i0 + i) * LD + 64 + 4 * fq);
            g[4 * i] = gv.x; g[4 * i + 1] = gv.y; g[4 * i + 2] = gv.z; g[4 * i + 3] = gv.w;
            u[4 * i] = uv.x; u[4 * i + 1] = uv.y; u[4 * i + 2] = uv.z; u[4 * i + 3] = uv.w;
        }
        gated_run<4 * TS>(p.act, g, u, a);
#pragma unroll
        for (int i = 0; i < TS; ++i) {
            if (c0 + i0 + i >= ncols)
                continue;
            if (meas) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    amax = fmaxf(amax, fabsf(a[4 * i + j]));
            } else {
                *reinterpret_cast<uint32_t *>(qh + (size_t)(m0 + c0 + i0 + i) * p.ldo) =
                    e4m3x2(__fmul_rn(a[4 * i], inv_s), __fmul_rn(a[4 * i + 1], inv_s)) |
                    (e4m3x2(__fmul_rn(a[4 * i + 2], inv_s), __fmul_rn(a[4 * i + 3], inv_s)) << 16);
            }
        }
    }
    named_bar_sync(1, 128);
}

// Tiled path: TMEM lanes are tokens; columns [128q, 128q+64) are gate and
// [128q+64, 128q+128) the up rows of the same 64 features.
template <int CH>
__device__ __forceinline__ void gated_tiled_chunk(const GemmParams &p, int m, int f0, const float (&g)[CH],
                                                  const float (&u)[CH], float &amax) {
    if (m >= p.m_tok)
        return;
    float gb[CH], ub[CH], a[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
        gb[j] = round_bf16(__fmul_rn(g[j], p.alpha));
        ub[j] = round_bf16(__fmul_rn(u[j], p.alpha));
    }
    if (p.dbg_gu) {
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            dbg_store_gu(p, m, f0 + j, false, gb[j]);
            dbg_store_gu(p, m, f0 + j, true, ub[j]);
        }
    }
    gated_run<CH>(p.act, gb, ub, a);
    if (p.epi == EPI_GATED_AMAX) {
#pragma unroll
        for (int j = 0; j < CH; ++j)
            amax = fmaxf(amax, fabsf(a[j]));
        return;
    }
    uint8_t *q = static_cast<uint8_t *>(p.out) + (size_t)m * p.ldo + f0;
#pragma unroll
    for (int j = 0; j < CH; j += 16) {
        uint4 ov;
        ov.x = e4m3x2(__fmul_rn(a[j + 0], p.inv_s), __fmul_rn(a[j + 1], p.inv_s)) |
               (e4m3x2(__fmul_rn(a[j + 2], p.inv_s), __fmul_rn(a[j + 3], p.inv_s)) << 16);
        ov.y = e4m3x2(__fmul_rn(a[j + 4], p.inv_s), __fmul_rn(a[j + 5], p.inv_s)) |
               (e4m3x2(__fmul_rn(a[j + 6], p.inv_s), __fmul_rn(a[j + 7], p.inv_s)) << 16);
        ov.z = e4m3x2(__fmul_rn(a[j + 8], p.inv_s), __fmul_rn(a[j + 9], p.inv_s)) |
               (e4m3x2(__fmul_rn(a[j + 10], p.inv_s), __fmul_rn(a[j + 11], p.inv_s)) << 16);
        ov.w = e4m3x2(__fmul_rn(a[j + 12], p.inv_s), __fmul_rn(a[j + 13], p.inv_s)) |
               (e4m3x2(__fmul_rn(a[j + 14], p.inv_s), __fmul_rn(a[j + 15], p.inv_s)) << 16);
        *reinterpret_cast<uint4 *>(q + j) = ov;
    }
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// --- NVFP4 gated epilogue (the gate and up GEMMs' FP4 outputs and the
// FP4-to-FP4 gated activation of the NVFP4 encoder FFN, fused) -------------
__host__ __device__ __forceinline__ bool f4_gated(int epi) {
    return epi == EPI_F4_GATED || epi == EPI_F4_AMAX_GU || epi == EPI_F4_AMAX_H;
}

// NB consecutive blocks of 16 features f0 .. f0 + 16 NB - 1 of token m: g
// and u (acc * alpha applied, fp32) -> G = NVFP4(g, s_g), U = NVFP4(u, s_u)
// -> a = act(dec G) dec U -> NVFP4(a, s_h) (codes at out[m][f0/2], the block
// scales TMEM-ready in out_sf), or the calibration amaxes: |g| into am0 and
// |u| into am1 (EPI_F4_AMAX_GU), |a| into am0 (EPI_F4_AMAX_H).  Each step
// runs over all NB blocks, so their chains interleave.
template <int NB>
__device__ __forceinline__ void f4_gated_blocks(const GemmParams &p, int m, int f0, const float (&g)[16 * NB],
                                                const float (&u)[16 * NB], float &am0, float &am1) {
    if (p.epi == EPI_F4_AMAX_GU) {
#pragma unroll
        for (int j = 0; j < 16 * NB; ++j) {
            am0 = fmaxf(am0, fabsf(g[j]));
            am1 = fmaxf(am1, fabsf(u[j]));
        }
        return;
    }
    uint2 qg[NB], qu[NB];
    uint32_t bg[NB], bu[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) {
        bg[k] = quant_block16(g + 16 * k, p.s_g, p.inv6_g, qg[k]);
        bu[k] = quant_block16(u + 16 * k, p.s_u, p.inv6_u, qu[k]);
    }
    if (p.dbg_gq) {
#pragma unroll
        for (int k = 0; k < NB; ++k) {
            const int f = f0 + 16 * k;
            *reinterpret_cast<uint2 *>(p.dbg_gq + (size_t)m * (p.ff / 2) + f / 2) = qg[k];
            *reinterpret_cast<uint2 *>(p.dbg_uq + (size_t)m * (p.ff / 2) + f / 2) = qu[k];
            p.dbg_gs[(size_t)m * (p.ff / 16) + f / 16] = (uint8_t)bg[k];
            p.dbg_us[(size_t)m * (p.ff / 16) + f / 16] = (uint8_t)bu[k];
        }
    }
    float gd[16 * NB], ud[16 * NB], a[16 * NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) {
        dequant_block16(qg[k], bg[k], p.s_g, gd + 16 * k);
        dequant_block16(qu[k], bu[k], p.s_u, ud + 16 * k);
    }
    gated_run<16 * NB>(p.act, gd, ud, a);
    if (p.epi == EPI_F4_AMAX_H) {
#pragma unroll
        for (int j = 0; j < 16 * NB; ++j)
            am0 = fmaxf(am0, fabsf(a[j]));
        return;
    }
    uint2 qh[NB];
    uint32_t bh[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k)
        bh[k] = quant_block16(a + 16 * k, p.s_h, p.inv6_h, qh[k]);
#pragma unroll
    for (int k = 0; k < NB; ++k) {
        const int f = f0 + 16 * k;
        *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(p.out) + (size_t)m * p.ldo + f / 2) = qh[k];
        p.out_sf[sf_offset(m, f / 16, p.ff)] = (uint8_t)bh[k];
    }
}

// The calibration amaxes of an NVFP4 gated epilogue into amax[0..2].
__device__ __forceinline__ void f4_flush_amax(const GemmParams &p, float am0, float am1) {
    if (p.epi == EPI_F4_AMAX_GU) {
        am0 = warp_max_f(am0);
        am1 = warp_max_f(am1);
        if ((threadIdx.x & 31) == 0) {
            atomicMax(p.amax, __float_as_uint(am0));
            atomicMax(p.amax + 1, __float_as_uint(am1));
        }
    } else if (p.epi == EPI_F4_AMAX_H) {
        am0 = warp_max_f(am0);
        if ((threadIdx.x & 31) == 0)
            atomicMax(p.amax + 2, __float_as_uint(am0));
    }
}

// Weight-streaming path, whole tile at once: TMEM lanes 0..63 are gate rows,
// 64..127 the up rows of the same 64 features; columns are tokens.  Every
// thread parks its row (times its alpha) in xbuf, token-major, and frees the
// accumulator; then the (token, block of 16 features) items go round the 128
// threads, each reading its block's 16 gate and 16 up values with 16-byte
// loads.  Called by all 128 epilogue threads; returns after a barrier.
template <int BN>
__device__ __forceinline__ void f4_gated_swap_tile(const GemmParams &p, const Unit &w, int r, uint32_t tbase,
                                                   uint64_t *tempty_b, float *xbuf, float &am0, float &am1) {
    constexpr int LD = 128 + 4;  // floats per token
    const int m0 = w.tq * BN;    // first token of the tile
    const int ncols = min(BN, p.m_tok - m0);
    const float alpha = r < 64 ? p.alpha : p.alpha_u;
    unit_row<BN>(tbase, [&](int c, const float (&v)[16]) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            xbuf[(c + j) * LD + r] = __fmul_rn(v[j], alpha);
    });
    tc_fence_before();
    mbar_arrive(smem_u32(tempty_b));  // the accumulator is read: the next unit's MMAs may start
    named_bar_sync(1, 128);
    const int fbase = w.tp * (BM / 2);
#pragma unroll 1
    for (int it = r; it < ncols * 4; it += 128) {
        const int c = it >> 2, b = it & 3;
        float g[16], u[16];
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            const float4 gv = *reinterpret_cast<const float4 *>(xbuf + c * LD + 16 * b + j);
            const float4 uv = *reinterpret_cast<const float4 *>(xbuf + c * LD + 64 + 16 * b + j);
            g[j] = gv.x; g[j + 1] = gv.y; g[j + 2] = gv.z; g[j + 3] = gv.w;
            u[j] = uv.x; u[j + 1] = uv.y; u[j + 2] = uv.z; u[j + 3] = uv.w;
        }
        f4_gated_blocks<1>(p, m0 + c, fbase + 16 * b, g, u, am0, am1);
    }
    named_bar_sync(1, 128);
}

// Consume one unit's accumulator from TMEM: the tiled gated epilogue, or a
// plain one (the weight-streaming gated epilogue is gated_swap_tile).
template <int BN, bool SWAP, bool ROPE = false, bool F4 = false>
__device__ __forceinline__ void consume_unit(const GemmParams &p, const Unit &w, uint32_t tbase) {
    using C = Cfg<BN, SWAP>;
    constexpr int CH = C::CH;
    const int r = threadIdx.x;
    const bool gated_epi = p.epi == EPI_GATED || p.epi == EPI_GATED_AMAX;
    float amax = 0.0f;
    if constexpr (F4 && !SWAP) {
        if (f4_gated(p.epi)) {
            // NVFP4 gated, tiled: TMEM lanes are tokens; columns [128q, 128q+64)
            // are gate and [128q+64, 128q+128) the up rows of the same 64
            // features, a block of 16 features per step
            // two blocks of 16 features a step
            const int m = w.tp * BM + r;
            float am0 = 0.0f, am1 = 0.0f;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 128) {
#pragma unroll 1
                for (int sub = 0; sub < 64; sub += 32) {
                    float g[32], u[32];
                    tmem_load_chunk<32>(tbase + c0 + sub, g);
                    tmem_load_chunk<32>(tbase + c0 + 64 + sub, u);
                    if (m < p.m_tok) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            g[j] = __fmul_rn(g[j], p.alpha);
                            u[j] = __fmul_rn(u[j], p.alpha_u);
                        }
                        f4_gated_blocks<2>(p, m, w.tq * (BN / 2) + c0 / 2 + sub, g, u, am0, am1);
                    }
                }
            }
            f4_flush_amax(p, am0, am1);
            return;
        }
    }
    if constexpr (!SWAP && ROPE) {
        // QKV split + RoPE of a token row (the tile's heads whole: BN % hd == 0,
        // hd % 64 == 0): element i of a head's first half pairs with i + hd/2;
        // x = bf16(acc * alpha), (cos, sin) of the token's angle pos * theta_i
        // from rope_cs [m_tok, hd/2], then in fp32 x_i cos - x_{i+hd/2} sin and
        // x_{i+hd/2} cos + x_i sin, rounded to BF16
        const int m = w.tp * BM + r;
        const bool live = m < p.m_tok;
        const int hd = p.rope_hd, half = hd / 2;
        const float2 *cs_row = p.rope_cs + (size_t)(live ? m : 0) * half;
#pragma unroll 1
        for (int hc = 0; hc < BN; hc += hd) {
            const int head = (w.tq * BN + hc) / hd;
            const bool rot = head < p.rope_nq + p.rope_nkv;
            uint16_t *dst = head < p.rope_nq ? p.rope_q + ((size_t)head * p.m_tok + m) * hd
                            : rot ? p.rope_k + ((size_t)(head - p.rope_nq) * p.m_tok + m) * hd
                                  : p.rope_v + ((size_t)(head - p.rope_nq - p.rope_nkv) * p.m_tok + m) * hd;
#pragma unroll 1
            for (int j = 0; j < half; j += CH) {
                float a[CH], b[CH];
                tmem_load_chunk<CH>(tbase + hc + j, a);
                tmem_load_chunk<CH>(tbase + hc + half + j, b);
                if (!live)
                    continue;
#pragma unroll
                for (int e = 0; e < CH; ++e) {
                    const float x1 = round_bf16(__fmul_rn(a[e], p.alpha));
                    const float x2 = round_bf16(__fmul_rn(b[e], p.alpha));
                    if (rot) {
                        const float2 t = cs_row[j + e];
                        a[e] = __fsub_rn(__fmul_rn(x1, t.x), __fmul_rn(x2, t.y));
                        b[e] = __fadd_rn(__fmul_rn(x2, t.x), __fmul_rn(x1, t.y));
                    } else {
                        a[e] = x1;
                        b[e] = x2;
                    }
                }
#pragma unroll
                for (int e = 0; e < CH; e += 8) {
                    uint4 o1, o2;
                    o1.x = bf16_bits(a[e]) | (bf16_bits(a[e + 1]) << 16);
                    o1.y = bf16_bits(a[e + 2]) | (bf16_bits(a[e + 3]) << 16);
                    o1.z = bf16_bits(a[e + 4]) | (bf16_bits(a[e + 5]) << 16);
                    o1.w = bf16_bits(a[e + 6]) | (bf16_bits(a[e + 7]) << 16);
                    o2.x = bf16_bits(b[e]) | (bf16_bits(b[e + 1]) << 16);
                    o2.y = bf16_bits(b[e + 2]) | (bf16_bits(b[e + 3]) << 16);
                    o2.z = bf16_bits(b[e + 4]) | (bf16_bits(b[e + 5]) << 16);
                    o2.w = bf16_bits(b[e + 6]) | (bf16_bits(b[e + 7]) << 16);
                    *reinterpret_cast<uint4 *>(dst + j + e) = o1;
                    *reinterpret_cast<uint4 *>(dst + half + j + e) = o2;
                }
            }
        }
    } else if (gated_epi && !SWAP) {
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 128) {
#pragma unroll 1
            for (int sub = 0; sub < 64; sub += CH) {
                float g[CH], u[CH];
                tmem_load_chunk<CH>(tbase + c0 + sub, g);
                tmem_load_chunk<CH>(tbase + c0 + 64 + sub, u);
                gated_tiled_chunk<CH>(p, w.tp * BM + r, w.tq * (BN / 2) + c0 / 2 + sub, g, u, amax);
            }
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += CH) {
            float v[CH];
            tmem_load_chunk<CH>(tbase + c, v);
            store_chunk<BN, SWAP, CH>(p, w, r, c, v);
        }
    }
    if (p.epi == EPI_GATED_AMAX) {
        amax = warp_max_f(amax);
        if ((threadIdx.x & 31) == 0)
            atomicMax(p.amax, __float_as_uint(amax));
    }
}

// Split-K, cooperative.  Every split CTA of a tile parks its fp32 partial in
// the workspace, counts itself in on the tile's arrival counter (release),
// waits until all S splits have arrived (acquire, bounded), then reduces one
// 1/S slice of the tile's elements over all partials in split order
// (deterministic) and runs the epilogue for that slice.  All splits of a tile
// must be resident at once: the planner keeps tiles x splits <= SMs, one unit
// per CTA, and a dependent kernel only launches once every CTA of this one is
// resident.
// Partial layout: weight-streaming [column][row] (a warp writes 32
// consecutive rows), tiled [row][column] (staged in shared memory, then
// copied out with contiguous whole-warp stores).
// Wait until the counter has reached `target` (wrap-around safe).
__device__ __forceinline__ bool spin_until_geq(const int *addr, unsigned target, volatile int *abort_f, int *err) {
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 0;; ++i) {
        if ((int)((unsigned)ld_acquire_gpu(addr) - target) >= 0)
            return true;
        if ((i & 15u) == 15u) {
            if (*abort_f)
                return false;
            if (globaltimer() - t0 > WAIT_TIMEOUT_NS) {
                *abort_f = 1;
                atomicExch(err, DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Index range [lo, hi) of one partial that holds everything the slice of
// split `k` needs, and the element range [e0, e1) of that slice.  Elements
// are enumerated so that a slice covers whole accumulator columns (weight-
// streaming) or rows (tiled) when gated, so the range is contiguous.
struct Slice {
    int e0, e1, lo, hi;
};

template <int BN, bool SWAP>
__device__ __forceinline__ Slice slice_of(int k, int S, int ncols, int nrows, bool gated_epi) {
    Slice sl;
    if (SWAP) {
        const int inner = gated_epi ? BM / 2 : BM;
        const int E = ncols * inner;
        // whole columns per split when gated, else 4-element (16 B) granules
        const int gran = gated_epi ? inner : 4;
        const int per = ((E + S - 1) / S + gran - 1) / gran * gran;
        sl.e0 = min(E, k * per);
        sl.e1 = min(E, sl.e0 + per);
        if (gated_epi) {
            sl.lo = (sl.e0 / inner) * BM;
            sl.hi = ((sl.e1 + inner - 1) / inner) * BM;
        } else {
            sl.lo = sl.e0;
            sl.hi = (sl.e1 + 3) & ~3;
        }
    } else {
        const int inner = gated_epi ? BN / 2 : BN;
        const int E = nrows * inner;
        const int gran = gated_epi ? inner : 4;
        const int per = ((E + S - 1) / S + gran - 1) / gran * gran;
        sl.e0 = min(E, k * per);
        sl.e1 = min(E, sl.e0 + per);
        if (gated_epi) {
            sl.lo = (sl.e0 / inner) * BN;
            sl.hi = ((sl.e1 + inner - 1) / inner) * BN;
        } else {
            sl.lo = sl.e0;
            sl.hi = (sl.e1 + 3) & ~3;
        }
    }
    return sl;
}

// Element e of a slice -> its offsets in the staged partials (a, and b for
// the up half when gated) and its output coordinates (token m, feature n).
template <int BN, bool SWAP, bool GATED>
__device__ __forceinline__ void elem_map(const Unit &w, const Slice &sl, int e, int &ia, int &ib, int &m, int &n) {
    if constexpr (SWAP) {
        constexpr int inner = GATED ? BM / 2 : BM;
        const int col = e / inner, row = e - col * inner;
        m = w.tq * BN + col;
        ia = col * BM + row - sl.lo;
        ib = ia + BM / 2;
        n = GATED ? w.tp * (BM / 2) + row : w.tp * BM + row;
    } else {
        constexpr int inner = GATED ? BN / 2 : BN;
        const int row = e / inner, col = e - row * inner;
        m = w.tp * BM + row;
        if constexpr (GATED) {
            ia = row * BN + (col >> 6) * 128 + (col & 63) - sl.lo;
            ib = ia + 64;
            n = w.tq * (BN / 2) + col;
        } else {
            ia = row * BN + col - sl.lo;
            ib = ia;
            n = w.tq * BN + col;
        }
    }
}

constexpr int RED_Q = 2;        // plain epilogues: quads (4 elements) per thread per batch
constexpr int RED_Q_GATED = 4;  // gated epilogue: a whole gate/up slice in one batch
constexpr int RED_Q_TILED = 8;  // plain epilogue of a tiled slice (half a 128 x 256 tile and up)

// Reduce this CTA's slice over the S staged partials (split order) and run
// the epilogue.  A thread takes quads: 4 consecutive elements of one token,
// i.e. 4 consecutive features, which sit next to each other in the staged
// partials (one 16-byte shared load per partial) and in the output (one
// 4-, 8- or 16-byte store).  Each step -- index math, accumulations, every
// element's math, stores -- is a straight run over the thread's quads with
// the launch-uniform choices (activation, epilogue kind, diagnostics) taken
// once around it, so the elements' instruction chains interleave.  Quads
// past the slice end repeat its last quad -- the same values to the same
// addresses -- so no store needs a predicate.  Output coordinates are
// recomputed at the store rather than held.  res0: residuals of the first
// batch, loaded early.
template <int BN, bool SWAP, bool GATED, bool RESID_GATE = true>
__device__ __forceinline__ float reduce_slice(const GemmParams &p, const Unit &w, const Slice &sl, const float *red,
                                              int span, const uint2 (&res0)[RED_Q]) {
    constexpr int NQ = GATED ? RED_Q_GATED : (SWAP ? RED_Q : RED_Q_TILED);
    constexpr int UP = SWAP ? BM / 2 : 64;  // offset of an element's up partner (gated)
    // partials per batch (registers allowing)
    constexpr int KU = (GATED ? 2 : 1) * NQ <= 4 ? 2 : 1;
    const int r = threadIdx.x;
    const int S = p.splits;
    const int epi = p.epi;
    const float alpha = p.alpha;
    const int q0 = sl.e0 >> 2, q1 = sl.e1 >> 2;
    float amax = 0.0f;
    bool first = true;
    auto coords = [&](int base, int i, int &m, int &n) {
        int ia, ib;
        elem_map<BN, SWAP, GATED>(w, sl, 4 * min(base + i * 128, q1 - 1), ia, ib, m, n);
    };
#pragma unroll 1
    for (int base = q0 + r; base < q1; base += 128 * NQ) {
        int ia[NQ];
        float acc[NQ][4], acc2[NQ][4];
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            int ib, m, n;
            elem_map<BN, SWAP, GATED>(w, sl, 4 * min(base + i * 128, q1 - 1), ia[i], ib, m, n);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[i][j] = 0.0f;
                acc2[i][j] = 0.0f;
            }
        }
        uint2 res[NQ];
        if constexpr (!GATED) {
            if (epi == EPI_RESID) {
                if (first && NQ == RED_Q) {
#pragma unroll
                    for (int i = 0; i < NQ; ++i)
                        res[i] = res0[i % RED_Q];
                } else {
#pragma unroll
                    for (int i = 0; i < NQ; ++i) {
                        int m, n;
                        coords(base, i, m, n);
                        res[i] = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p.resid) +
                                                                  (size_t)m * p.ldr + n);
                    }
                }
            }
        }
        // KU partials at a time: all their loads first, then the additions
        // in split order (the same order for every KU)
#pragma unroll 1
        for (int k0 = 0; k0 < S; k0 += KU) {
            float4 v[KU][NQ], uv[KU][NQ];
#pragma unroll
            for (int kk = 0; kk < KU; ++kk) {
                if (k0 + kk < S) {
                    const float *rk = red + (size_t)(k0 + kk) * span;
#pragma unroll
                    for (int i = 0; i < NQ; ++i) {
                        v[kk][i] = *reinterpret_cast<const float4 *>(rk + ia[i]);
                        if (GATED)
                            uv[kk][i] = *reinterpret_cast<const float4 *>(rk + ia[i] + UP);
                    }
                }
            }
#pragma unroll
            for (int kk = 0; kk < KU; ++kk) {
                if (k0 + kk < S) {
#pragma unroll
                    for (int i = 0; i < NQ; ++i) {
                        acc[i][0] = __fadd_rn(acc[i][0], v[kk][i].x);
                        acc[i][1] = __fadd_rn(acc[i][1], v[kk][i].y);
                        acc[i][2] = __fadd_rn(acc[i][2], v[kk][i].z);
                        acc[i][3] = __fadd_rn(acc[i][3], v[kk][i].w);
                        if (GATED) {
                            acc2[i][0] = __fadd_rn(acc2[i][0], uv[kk][i].x);
                            acc2[i][1] = __fadd_rn(acc2[i][1], uv[kk][i].y);
                            acc2[i][2] = __fadd_rn(acc2[i][2], uv[kk][i].z);
                            acc2[i][3] = __fadd_rn(acc2[i][3], uv[kk][i].w);
                        }
                    }
                }
            }
        }
        if constexpr (GATED) {
            float g[4 * NQ], u[4 * NQ], a[4 * NQ];
#pragma unroll
            for (int i = 0; i < NQ; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    g[4 * i + j] = round_bf16(__fmul_rn(acc[i][j], alpha));
                    u[4 * i + j] = round_bf16(__fmul_rn(acc2[i][j], alpha));
                }
            gated_run<4 * NQ>(p.act, g, u, a);
            if (p.dbg_gu) {
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    int m, n;
                    coords(base, i, m, n);
                    uint16_t *row = p.dbg_gu + (size_t)m * 2 * p.ff + n;
                    *reinterpret_cast<uint2 *>(row) =
                        make_uint2(bf16_bits(g[4 * i]) | (bf16_bits(g[4 * i + 1]) << 16),
                                   bf16_bits(g[4 * i + 2]) | (bf16_bits(g[4 * i + 3]) << 16));
                    *reinterpret_cast<uint2 *>(row + p.ff) =
                        make_uint2(bf16_bits(u[4 * i]) | (bf16_bits(u[4 * i + 1]) << 16),
                                   bf16_bits(u[4 * i + 2]) | (bf16_bits(u[4 * i + 3]) << 16));
                }
            }
            if (epi == EPI_GATED_AMAX) {
#pragma unroll
                for (int i = 0; i < 4 * NQ; ++i)
                    amax = fmaxf(amax, fabsf(a[i]));
            } else {
                uint8_t *out = static_cast<uint8_t *>(p.out);
                const float inv_s = p.inv_s;
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    int m, n;
                    coords(base, i, m, n);
                    *reinterpret_cast<uint32_t *>(out + (size_t)m * p.ldo + n) =
                        e4m3x2(__fmul_rn(a[4 * i], inv_s), __fmul_rn(a[4 * i + 1], inv_s)) |
                        (e4m3x2(__fmul_rn(a[4 * i + 2], inv_s), __fmul_rn(a[4 * i + 3], inv_s)) << 16);
                }
            }
        } else {
            if (epi == EPI_F32) {
                float *out = static_cast<float *>(p.out);
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    int m, n;
                    coords(base, i, m, n);
                    *reinterpret_cast<float4 *>(out + (size_t)m * p.ldo + n) =
                        make_float4(__fmul_rn(acc[i][0], alpha), __fmul_rn(acc[i][1], alpha),
                                    __fmul_rn(acc[i][2], alpha), __fmul_rn(acc[i][3], alpha));
                }
            } else {
                uint16_t *out = static_cast<uint16_t *>(p.out);
#pragma unroll
                for (int i = 0; i < NQ; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        acc[i][j] = __fmul_rn(acc[i][j], alpha);
                if (RESID_GATE && p.gate) {
#pragma unroll
                    for (int i = 0; i < NQ; ++i) {
                        int m, n;
                        coords(base, i, m, n);
                        const uint2 gv = *reinterpret_cast<const uint2 *>(p.gate + (size_t)m * p.ldgate + n);
                        acc[i][0] = __fmul_rn(acc[i][0], bf_lo(gv.x));
                        acc[i][1] = __fmul_rn(acc[i][1], bf_hi(gv.x));
                        acc[i][2] = __fmul_rn(acc[i][2], bf_lo(gv.y));
                        acc[i][3] = __fmul_rn(acc[i][3], bf_hi(gv.y));
                    }
                }
                if (epi == EPI_RESID) {
#pragma unroll
                    for (int i = 0; i < NQ; ++i) {
                        acc[i][0] = __fadd_rn(bf_lo(res[i].x), acc[i][0]);
                        acc[i][1] = __fadd_rn(bf_hi(res[i].x), acc[i][1]);
                        acc[i][2] = __fadd_rn(bf_lo(res[i].y), acc[i][2]);
                        acc[i][3] = __fadd_rn(bf_hi(res[i].y), acc[i][3]);
                    }
                }
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    int m, n;
                    coords(base, i, m, n);
                    *reinterpret_cast<uint2 *>(out + (size_t)m * p.ldo + n) =
                        make_uint2(bf16_bits(acc[i][0]) | (bf16_bits(acc[i][1]) << 16),
                                   bf16_bits(acc[i][2]) | (bf16_bits(acc[i][3]) << 16));
                }
            }
        }
        first = false;
    }
    return amax;
}

template <int BN, bool SWAP>
__device__ bool coop_split_unit(const GemmParams &p, const Unit &w, uint32_t tbase, uint64_t *tempty_b,
                                uint64_t *red_bar, float *red, volatile int *abort_f, volatile int *s_flag) {
    constexpr int CH = Cfg<BN, SWAP>::CH;
    const int r = threadIdx.x;
    const int S = p.splits;
    const int ncols = SWAP ? min(BN, p.m_tok - w.tq * BN) : BN;
    const int nrows = SWAP ? BM : min(BM, p.m_tok - w.tp * BM);
    const float *tile_ws = p.ws + (size_t)w.tile * S * (size_t)(BM * BN);
    float *mine = p.ws + ((size_t)w.tile * S + w.split) * (size_t)(BM * BN);
    // 1. this split's partial (weight-streaming: every TMEM load in flight at
    //    once, then the stores)
    if constexpr (SWAP) {
        unit_row<BN>(tbase, [&](int c, const float (&v)[16]) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (c + j < ncols)
                    mine[(size_t)(c + j) * BM + r] = v[j];
        });
    } else {
        // Tiled: a thread holds a whole row (BN floats); written straight to
        // global memory a warp's 16-byte stores would land 4*BN bytes apart.
        // Stage the tile row-major in the (now idle) pipeline stages instead,
        // 16-byte chunks XOR-swizzled by row so 8 consecutive rows hit all 32
        // banks, then copy it out with whole-warp contiguous 16-byte stores.
        float *stg = red;  // the slices arrive here only after the copy-out
        constexpr int CPR = BN / 4;  // 16-byte chunks per row
#pragma unroll 1
        for (int c = 0; c < BN; c += CH) {
            float v[CH];
            tmem_load_chunk<CH>(tbase + c, v);
#pragma unroll
            for (int j = 0; j < CH; j += 4) {
                const int ch = (c + j) >> 2;
                *reinterpret_cast<float4 *>(stg + (size_t)r * BN + 4 * (ch ^ (r & 7))) =
                    make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
        }
        tc_fence_before();
        // (a CTA pair's accumulator barrier counts one arrival per CTA; with
        // one unit per CTA nothing waits on it again, so pairs skip it)
        if (!p.pair)
            mbar_arrive(smem_u32(tempty_b));
        named_bar_sync(1, 128);
#pragma unroll 4
        for (int i = r; i < nrows * CPR; i += 128) {
            const int row = i / CPR, ch = i - row * CPR;
            *reinterpret_cast<float4 *>(mine + (size_t)row * BN + 4 * ch) =
                *reinterpret_cast<const float4 *>(stg + (size_t)row * BN + 4 * (ch ^ (row & 7)));
        }
    }
    if constexpr (SWAP) {
        tc_fence_before();
        mbar_arrive(smem_u32(tempty_b));
    }
    named_bar_sync(1, 128);
    // 2. count in, wait for every split of the tile, pull this CTA's slice of
    //    every partial into shared memory with bulk copies.  The counter only
    //    grows: the S splits of one launch fetch S consecutive values, which
    //    name their generation, and wait for the generation's last arrival.
    int *arrive = p.counters + w.tile;
    const bool gated_epi = p.epi == EPI_GATED || p.epi == EPI_GATED_AMAX;
    const Slice sl = slice_of<BN, SWAP>(w.split, S, ncols, nrows, gated_epi);
    const int span = sl.hi - sl.lo;
    // the first batch's residuals do not depend on the other splits: load
    // them now so their latency hides behind the wait
    uint2 res0[RED_Q];
#pragma unroll
    for (int i = 0; i < RED_Q; ++i)
        res0[i] = make_uint2(0u, 0u);
    if (p.epi == EPI_RESID && sl.e1 > sl.e0) {
        const int q0 = sl.e0 >> 2, q1 = sl.e1 >> 2;
#pragma unroll
        for (int i = 0; i < RED_Q; ++i) {
            int ia, ib, m, n;
            elem_map<BN, SWAP, false>(w, sl, 4 * min(q0 + r + i * 128, q1 - 1), ia, ib, m, n);
            res0[i] = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p.resid) + (size_t)m * p.ldr + n);
        }
    }
    if (threadIdx.x == 0) {
        const unsigned old = (unsigned)atomic_add_release_gpu(arrive, 1);
        const unsigned target = (old / (unsigned)S + 1u) * (unsigned)S;
        bool ok = spin_until_geq(arrive, target, abort_f, p.err);
        if (ok && span > 0) {
            fence_proxy_async_global();
            mbar_arrive_expect_tx(smem_u32(red_bar), (uint32_t)(S * span * 4));
            for (int k = 0; k < S; ++k)
                bulk_load(smem_u32(red + (size_t)k * span), tile_ws + (size_t)k * (BM * BN) + sl.lo,
                          (uint32_t)span * 4u, smem_u32(red_bar));
            ok = mbar_wait(smem_u32(red_bar), 0, abort_f, p.err);
        }
        *s_flag = ok ? 1 : 0;
    }
    named_bar_sync(1, 128);
    if (!*s_flag)
        return false;
    // 3. reduce the slice and run the epilogue
    const float amax = gated_epi ? reduce_slice<BN, SWAP, true>(p, w, sl, red, span, res0)
                                 : reduce_slice<BN, SWAP, false>(p, w, sl, red, span, res0);
    if (p.epi == EPI_GATED_AMAX) {
        const float m = warp_max_f(amax);
        if ((threadIdx.x & 31) == 0)
            atomicMax(p.amax, __float_as_uint(m));
    }
    return true;
}

// Split-K inside one thread-block cluster (weight-streaming tiles): the S
// splits of a tile are the S CTAs of a cluster, CTA rank = split.  Each CTA
// stages its whole partial in its own shared memory and bulk-copies slice j
// of it into CTA j's shared memory over the cluster's distributed shared
// memory; CTA j then reduces the S copies of its slice in split order, the
// same arithmetic as the global-memory path, so results are identical.
// A CTA's pipeline stages receive the copies, so each CTA first tells the
// others (remote mbarrier arrivals) that its last MMA has completed; and a
// CTA leaves only once every CTA it copied to has reported the copy landed.
template <int BN, bool SWAP, bool PLAIN_ONLY, bool RESID_GATE = true>
__device__ bool coop_cluster_unit(const GemmParams &p, const Unit &w, uint32_t tbase, uint64_t *tempty_b,
                                  uint64_t *free_bar, uint64_t *data_bar, uint64_t *sent_bar, float *red, float *stg,
                                  volatile int *abort_f, volatile int *s_flag) {
    static_assert(SWAP, "cluster split-K stages partials in weight-streaming order");
    const int r = threadIdx.x;
    const int S = p.splits;
    const int k = w.split;  // == cluster rank
    const int ncols = min(BN, p.m_tok - w.tq * BN);
    const bool gated_epi = !PLAIN_ONLY && (p.epi == EPI_GATED || p.epi == EPI_GATED_AMAX);
    const Slice sl = slice_of<BN, SWAP>(k, S, ncols, BM, gated_epi);
    const int span = sl.hi - sl.lo;
    // 1. expect this slice from every split; free this CTA's stages for them
    //    (no ordering needed: the MMAs that read the stages have completed,
    //    which the wait on the accumulator barrier established)
    //    Lane j of warp 0 handles CTA j; the expected bytes may land before
    //    lane 0 declares them (the phase needs lane 0's arrival to complete).
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        if (lane == 0)
            mbar_arrive_expect_tx(smem_u32(data_bar), (uint32_t)(S * span * 4));
        if (lane < S && lane != k)
            mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(free_bar), (uint32_t)lane));
    }
    // residuals of the first batch: independent of the other splits
    uint2 res0[RED_Q];
#pragma unroll
    for (int i = 0; i < RED_Q; ++i)
        res0[i] = make_uint2(0u, 0u);
    if (p.epi == EPI_RESID && sl.e1 > sl.e0) {
        const int q0 = sl.e0 >> 2, q1 = sl.e1 >> 2;
#pragma unroll
        for (int i = 0; i < RED_Q; ++i) {
            int ia, ib, m, n;
            elem_map<BN, SWAP, false>(w, sl, 4 * min(q0 + r + i * 128, q1 - 1), ia, ib, m, n);
            res0[i] = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p.resid) + (size_t)m * p.ldr + n);
        }
    }
    // 2. stage the partial in partial-index order (column-major, lane = row):
    //    every TMEM load in flight at once, then the stores
    unit_row<BN>(tbase, [&](int c, const float (&v)[16]) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (c + j < ncols)
                stg[(c + j) * BM + r] = v[j];
    });
    fence_proxy_async_shared();
    tc_fence_before();
    mbar_arrive(smem_u32(tempty_b));
    named_bar_sync(1, 128);
    // 3. once every CTA of the cluster has freed its stages, send slice j of
    //    this partial to CTA j, into row k of its slice buffer; then wait for
    //    this CTA's slice from all S splits
    //    (lane j of warp 0 copies to CTA j)
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int ok = 1;
        if (lane == 0)
            ok = mbar_wait_cluster(smem_u32(free_bar), 0, abort_f, p.err) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok && lane < S) {
            const Slice sj = slice_of<BN, SWAP>(lane, S, ncols, BM, gated_epi);
            const int spj = sj.hi - sj.lo;
            if (spj > 0)
                bulk_copy_to_cta(mapa_shared(smem_u32(red + (size_t)k * spj), (uint32_t)lane), smem_u32(stg + sj.lo),
                                 (uint32_t)spj * 4u, mapa_shared(smem_u32(data_bar), (uint32_t)lane));
        }
        if (ok && lane == 0)
            ok = mbar_wait_cluster(smem_u32(data_bar), 0, abort_f, p.err) ? 1 : 0;
        if (lane == 0)
            *s_flag = ok;
    }
    named_bar_sync(1, 128);
    if (!*s_flag)
        return false;
    // 4. reduce the slice and run the epilogue
    float amax = 0.0f;
    if constexpr (PLAIN_ONLY)
        amax = reduce_slice<BN, SWAP, false, RESID_GATE>(p, w, sl, red, span, res0);
    else
        amax = gated_epi ? reduce_slice<BN, SWAP, true>(p, w, sl, red, span, res0)
                         : reduce_slice<BN, SWAP, false>(p, w, sl, red, span, res0);
    if (p.epi == EPI_GATED_AMAX) {
        const float m = warp_max_f(amax);
        if ((threadIdx.x & 31) == 0)
            atomicMax(p.amax, __float_as_uint(m));
    }
    // 5. the CTA may leave once every copy out of its staging has landed (the
    //    receivers' producer warps report it as soon as their data barrier
    //    completes; normally long done by now)
    return threadIdx.x != 0 || mbar_wait_cluster(smem_u32(sent_bar), 0, abort_f, p.err);
}

// Floats of the slice buffer at the start of shared memory: the S slices
// of a split-K tile, with the per-split rounding slack.
__host__ __device__ constexpr size_t red_floats(int bn, int splits) {
    return ((size_t)BM * bn + (size_t)splits * ((BM > bn ? BM : bn) + 4) + 31) & ~(size_t)31;
}

template <int BN, bool SWAP, bool PAIR, int ROLE, bool F4>
__device__ void epilogue(const GemmParams &p, uint64_t *tfull, uint64_t *tempty, uint32_t tmem_base,
                         volatile int *abort_f, volatile int *s_ok, volatile int *s_last, float *xbuf,
                         uint64_t *red_bar, uint64_t *free_bar, uint64_t *data_bar, uint64_t *sent_bar,
                         float *red) {
    const int warp = threadIdx.x >> 5;
    const int r = threadIdx.x;  // P-tile row = TMEM lane (warps 0..3)
    if (p.cluster)
        cluster_wait();
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
        if constexpr (ROLE == ROLE_GATED_TILE && F4) {
            float am0 = 0.0f, am1 = 0.0f;
            f4_gated_swap_tile<BN>(p, w, r, tbase, &tempty[abuf], xbuf, am0, am1);
            f4_flush_amax(p, am0, am1);
        } else if constexpr (ROLE == ROLE_GATED_TILE) {
            float amax = 0.0f;
            gated_swap_tile<BN>(p, w, r, tbase, &tempty[abuf], xbuf, amax);
            if (p.epi == EPI_GATED_AMAX) {
                amax = warp_max_f(amax);
                if ((threadIdx.x & 31) == 0)
                    atomicMax(p.amax, __float_as_uint(amax));
            }
        } else if constexpr (ROLE == ROLE_CLUSTER_PLAIN || ROLE == ROLE_CLUSTER_GATE) {
            if (!coop_cluster_unit<BN, SWAP, true, ROLE == ROLE_CLUSTER_GATE>(
                    p, w, tbase, &tempty[abuf], free_bar, data_bar, sent_bar, red, red + red_floats(BN, p.splits),
                    abort_f, &s_last[abuf])) {
                // gave up: as below
                if (threadIdx.x == 0) {
                    mbar_wait_for(smem_u32(free_bar), 0, 500000000ull);
                    mbar_wait_for(smem_u32(data_bar), 0, 500000000ull);
                    mbar_wait_for(smem_u32(sent_bar), 0, 500000000ull);
                }
                break;
            }
        } else if (p.splits == 1) {
            if (F4 && SWAP && f4_gated(p.epi)) {
                if constexpr (F4 && SWAP) {
                    float am0 = 0.0f, am1 = 0.0f;
                    f4_gated_swap_tile<BN>(p, w, r, tbase, &tempty[abuf], xbuf, am0, am1);
                    f4_flush_amax(p, am0, am1);
                }
            } else if (SWAP && (p.epi == EPI_GATED || p.epi == EPI_GATED_AMAX)) {
                if constexpr (SWAP) {
                    float amax = 0.0f;
                    gated_swap_tile<BN>(p, w, r, tbase, &tempty[abuf], xbuf, amax);
                    if (p.epi == EPI_GATED_AMAX) {
                        amax = warp_max_f(amax);
                        if ((threadIdx.x & 31) == 0)
                            atomicMax(p.amax, __float_as_uint(amax));
                    }
                }
            } else {
                consume_unit<BN, SWAP, ROLE == ROLE_ROPE, F4>(p, w, tbase);
                tc_fence_before();
                if constexpr (PAIR) {
                    // the even CTA's MMA refills both CTAs' accumulators:
                    // one arrival per CTA on its barrier
                    named_bar_sync(1, 128);
                    if (threadIdx.x == 0)
                        mbar_arrive_cluster_release(mapa_shared(smem_u32(&tempty[abuf]), 0u));
                } else {
                    mbar_arrive(smem_u32(&tempty[abuf]));
                }
            }
        } else if (SWAP && p.cluster) {
            if constexpr (SWAP) {
                if (!coop_cluster_unit<BN, SWAP, false>(p, w, tbase, &tempty[abuf], free_bar, data_bar, sent_bar,
                                                        red, red + red_floats(BN, p.splits), abort_f,
                                                        &s_last[abuf])) {
                    // gave up: other CTAs of the cluster may still be copying
                    // into or out of this one; wait for them, bounded
                    if (threadIdx.x == 0) {
                        mbar_wait_for(smem_u32(free_bar), 0, 500000000ull);
                        mbar_wait_for(smem_u32(data_bar), 0, 500000000ull);
                        mbar_wait_for(smem_u32(sent_bar), 0, 500000000ull);
                    }
                    break;
                }
            }
        } else {
            if (!coop_split_unit<BN, SWAP>(p, w, tbase, &tempty[abuf], red_bar, red, abort_f, &s_last[abuf]))
                break;
        }
        if (++abuf == (F4 ? Cfg<BN, SWAP, PAIR, F4>::ACC_BUFS : 2)) {
            abuf = 0;
            aphase ^= 1u;
        }
    }
}

// -------------------------------------------------------------- kernel --
// The body of both kernels below; tmP / tmQ are their __grid_constant__
// parameters.
template <int BN, bool SWAP, bool PAIR, int ROLE, bool F4>
__device__ __forceinline__ void gemm_body(const CUtensorMap &tmP, const CUtensorMap &tmQ, const GemmParams &p) {
    using C = Cfg<BN, SWAP, PAIR, F4>;
    if (p.stamp && threadIdx.x == 0)
        stamp_start(p.stamp);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sP = smem;
    const int NS = p.stages;
    uint8_t *sQ = smem + (size_t)NS * C::P_BYTES;
    uint8_t *sSF = sQ + (size_t)NS * C::Q_BYTES;  // F4: block scales (none otherwise)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sSF + (size_t)NS * C::SF_BYTES);
    const uint32_t tmem_cols = C::tmem_cols(NS);
    uint64_t *full = bars;
    uint64_t *empty = bars + NS;
    uint64_t *tfull = bars + 2 * NS;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain_bar = tempty + 2;
    uint64_t *red_bar = drain_bar + 1;   // split-K: slice of every partial landed in shared memory
    uint64_t *free_bar = red_bar + 1;    // cluster split-K: every other CTA's stages are free
    uint64_t *data_bar = free_bar + 1;   // cluster split-K: this CTA's slice of every partial landed
    uint64_t *sent_bar = data_bar + 1;   // cluster split-K: every copy out of this CTA landed
    uint64_t *sfull = sent_bar + 1;      // F4: a stage's scales are in TMEM (4 scale warps)
    uint64_t *sffull = sfull + (F4 ? NS : 0);  // F4: a stage's scale copies landed in shared memory
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sffull + (F4 ? NS : 0));
    volatile int *abort_f = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *s_ok = abort_f + 1;    // [2]
    volatile int *s_last = s_ok + 2;     // [2]
    float *xbuf = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(bars) + C::BAR_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1u);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), PAIR ? 2u : 128u);
        }
        mbar_init(smem_u32(drain_bar), 1);
        mbar_init(smem_u32(red_bar), 1);
        mbar_init(smem_u32(free_bar), p.cluster ? (uint32_t)(p.splits - 1) : 1u);
        mbar_init(smem_u32(data_bar), 1);
        mbar_init(smem_u32(sent_bar), p.cluster ? (uint32_t)(p.splits - 1) : 1u);
        if constexpr (F4)
            for (int s = 0; s < NS; ++s) {
                mbar_init(smem_u32(&sfull[s]), 4u);
                mbar_init(smem_u32(&sffull[s]), 1u);
            }
        *abort_f = 0;
        fence_mbar_init();
    }
    const CUtensorMap *mapP = p.gtm_p ? p.gtm_p : &tmP;
    const CUtensorMap *mapQ = p.gtm_q ? p.gtm_q : &tmQ;
    if (warp == 4 && lane == 0) {
        prefetch_tmap(mapP);
        prefetch_tmap(mapQ);
    }
    if (warp == 5) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_holder), tmem_cols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_holder), tmem_cols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the other CTAs of the cluster touch this CTA's barriers only after
    // they have been initialised: every thread arrives now, and waits before
    // its first access to another CTA (the epilogue) or at its end
    if (p.cluster)
        cluster_arrive();
    if (PAIR) {
        // a pair's copies write into, and its MMA commits arrive on, the
        // other CTA's stages and barriers from the first k-block on
        cluster_arrive();
        cluster_wait();
    }
    const uint32_t tmem_base = *tmem_holder;
    pdl_trigger();

    if (warp < 4) {
        // split-K runs one unit per CTA, so the pipeline stages are free to
        // receive the partial slices once the last MMA has completed
        epilogue<BN, SWAP, PAIR, ROLE, F4>(p, tfull, tempty, tmem_base, abort_f, s_ok, s_last, xbuf, red_bar, free_bar,
                                 data_bar, sent_bar, reinterpret_cast<float *>(smem));
    } else if (warp == 4) {
        if (lane == 0)
            producer<BN, SWAP, PAIR, F4>(mapP, mapQ, p, sP, sQ, sSF, full, empty, sffull, abort_f);
        __syncwarp();
        if (p.cluster) {
            cluster_wait();
            if constexpr (SWAP) {
                // Cluster split-K: once this CTA's slice of every split's
                // partial has landed, tell each source CTA that its staging
                // may go (it leaves only then).  The producer warp does this,
                // off the epilogue's path to the reduction.
                int ok = 0;
                if (lane == 0)
                    ok = mbar_wait_cluster(smem_u32(data_bar), 0, abort_f, p.err) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                const int k = decode(p, (int)blockIdx.x).split;  // == cluster rank
                if (ok && lane < p.splits && lane != k)
                    mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(sent_bar), (uint32_t)lane));
            }
        }
    } else if (warp == 5) {
        if (lane == 0 && (!PAIR || (blockIdx.x & 1u) == 0))
            mma_issuer<BN, SWAP, PAIR, F4>(p, sP, sQ, full, empty, sfull, tfull, tempty, drain_bar, tmem_base,
                                           abort_f);
        __syncwarp();
        if (p.cluster)
            cluster_wait();
    } else {
        if constexpr (F4)
            scale_feeder<BN, SWAP>(p, sSF, sffull, sfull, tmem_base, abort_f);
        __syncwarp();
        if (p.cluster)
            cluster_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (PAIR) {
        // no CTA leaves while another may still write into it
        cluster_arrive();
        cluster_wait();
    }
    if (warp == 5) {
        __syncwarp();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, tmem_cols);
        else
            tmem_dealloc(tmem_base, tmem_cols);
    }
    if (p.stamp && threadIdx.x == 0)
        stamp_end(p.stamp);
}

template <int BN, bool SWAP, bool PAIR, int ROLE>
__global__ void __launch_bounds__(NTHREADS, SWAP ? 2 : 1)
    k_gemm_fp8(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
               const __grid_constant__ GemmParams p) {
    gemm_body<BN, SWAP, PAIR, ROLE, false>(tmP, tmQ, p);
}

// NVFP4 operands (E2M1 codes, E4M3 block scales): single CTAs, N <= 128,
// with the four scale warps.
template <int BN, bool SWAP, int ROLE>
__global__ void __launch_bounds__(NTHREADS_F4, 1)
    k_gemm_f4(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
              const __grid_constant__ GemmParams p) {
    gemm_body<BN, SWAP, false, ROLE, true>(tmP, tmQ, p);
}

template <int BN, bool SWAP, bool PAIR, int ROLE, bool F4>
constexpr auto kernel_of() {
    if constexpr (F4)
        return k_gemm_f4<BN, SWAP, ROLE>;
    else
        return k_gemm_fp8<BN, SWAP, PAIR, ROLE>;
}

template <int BN, bool SWAP, bool PAIR = false, int ROLE = ROLE_ANY, bool F4 = false>
cudaError_t set_attrs() {
    using C = Cfg<BN, SWAP, PAIR, F4>;
    constexpr auto kern = kernel_of<BN, SWAP, PAIR, ROLE, F4>();
    static int done = 0;
    if (!done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
        if (e != cudaSuccess)
            return e;
        // every kernel of the layer asks for the largest shared-memory
        // carve-out, so an SM never needs to drain before a CTA of the next
        // kernel (with its own footprint) can start beside the running ones
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        done = 1;
    }
    return cudaSuccess;
}

template <int BN, bool SWAP, bool PAIR = false, int ROLE = ROLE_ANY, bool F4 = false>
cudaError_t run(const GemmLaunch &g, cudaStream_t s, bool pdl) {
    using C = Cfg<BN, SWAP, PAIR, F4>;
    cudaError_t e = set_attrs<BN, SWAP, PAIR, ROLE, F4>();
    if (e != cudaSuccess)
        return e;
    const bool xbuf = SWAP && g.p.splits == 1 &&
                      (g.p.epi == EPI_GATED || g.p.epi == EPI_GATED_AMAX || f4_gated(g.p.epi));
    const unsigned cluster = PAIR ? 2u : g.p.cluster ? (unsigned)g.p.splits : 1u;
    return launch_ex(kernel_of<BN, SWAP, PAIR, ROLE, F4>(), dim3((unsigned)g.grid), dim3(F4 ? NTHREADS_F4 : NTHREADS),
                     std::max(C::smem_bytes(g.p.stages, xbuf), g.min_smem), s, pdl, cluster, g.tmP, g.tmQ, g.p);
}

}  // namespace

}  // namespace frt
