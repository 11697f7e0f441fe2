// k_stack_fp8.cu -- the whole FP8 FFN stack for at most 64 tokens in one
// persistent kernel (steps A1..A4 of every layer; itsolotime FlashRT article,
// 4.1: at small batch the time between kernels is the workload, and 7.2: the
// FFN layer loop).
//
// Work split (d % 256 == 0, S = d / 256 <= 8, ff % 128 == 0, nC = ff / 128):
// nC thread-block clusters of S CTAs, one CTA per SM, resident together.
// Cluster c owns hidden features [128 c, 128 c + 128) -- 256 rows of the
// gate/up weights, whose 64-row gate and up blocks interleave -- and CTA j of
// it the K-quarter [256 j, 256 j + 256) of the gate/up GEMM and the N-tile
// [256 j, 256 j + 256) of the down GEMM.  Per layer:
//   (a) the layer input r' (published by its column owners, below) is read
//       from L2 with the owners' per-token partial sums of squares; the CTA
//       normalises and quantises its K-quarter of every token into the
//       tokens-as-A operand (64 rows, 128-byte swizzle);
//   (b) 8 tcgen05.mma (M = 64 tokens, N = 256 weight rows, K = 32) into TMEM;
//   (c) the four K-quarters' fp32 partials are exchanged inside the cluster
//       over distributed shared memory (bulk copies), each CTA receiving the
//       columns of its 128 / S features;
//   (d) it sums them in K order, rounds g and u to BF16, applies the gated
//       activation and quantises to E4M3 (step A3), and writes its q_h bytes
//       into the down GEMM's operand in every CTA of the cluster;
//   (e) 4 tcgen05.mma: the cluster's 128 features against the down weights of
//       its N-tile, the partial sum over this K-slice of 128 features;
//   (f) the partial goes to L2 and a release counter per N-tile is bumped;
//   (g) every CTA owns 8-column groups of d: it adds the nC partials of its
//       columns in cluster order, adds the residual, rounds to BF16 (step
//       A4), publishes the result and its per-token sum of squares for the
//       next layer's (a) and bumps the residual counter -- or, after the
//       last layer, writes the output.
// Weights of the next layer stream into shared memory as soon as this
// layer's MMAs have read the previous ones, so weight reads from HBM overlap
// the whole dependency chain.  Dependencies between CTAs are monotonic
// counters (release add / acquire poll, bounded); inside a cluster,
// mbarriers.  Every wait gives up after WAIT_TIMEOUT_NS, sets the error word,
// and the CTA drains and exits.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "frt_epi.cuh"
#include "frt_internal.h"
#include "frt_ptx.cuh"

namespace frt {

namespace {

constexpr int ST_THREADS = 320;  // warps 0-7 compute (two per TMEM lane quarter), 8 TMA producer, 9 MMA issuer
constexpr int ST_CT = 256;       // compute threads
constexpr int W_PROD = 8, W_MMA = 9;
constexpr int ST_ROWS = 64;      // token rows of the A operands (MMA M)
constexpr int ST_KQ = 256;       // gate/up K per CTA
constexpr int ST_FEAT = 128;     // features per cluster
constexpr int ST_NT = 256;       // MMA N: weight rows per tile

constexpr uint32_t OFF_WGU = 0;        // W_gu tile: 2 k-blocks x (256 rows x 128 B)
constexpr uint32_t OFF_WD = 65536;     // W_down tile: 256 rows x 128 B
constexpr uint32_t OFF_AGU = 98304;    // q_x quarter: 2 k-blocks x (64 rows x 128 B)
constexpr uint32_t OFF_AD = 114688;    // q_h of the cluster: 64 rows x 128 B
constexpr uint32_t OFF_X = 122880;     // exchange / staging region (size from the host)

enum StBar : int {
    B_WFULL_GU = 0, B_WEMPTY_GU, B_WFULL_D, B_WEMPTY_D, B_AGU_READY, B_ACC_GU, B_AD_READY, B_ACC_D,
    B_RX, B_ASTAGE, B_OWN, B_DRAIN, N_BARS
};

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void fence_proxy_async_cluster() {
    asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }
// Each thread's own global writes ordered before the release that a thread
// of its CTA makes after a CTA barrier.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void red_release_gpu(int *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded acquire poll of a monotonic counter: true once *c >= target; gives
// up when this CTA aborted, another kernel CTA set the error word, or after
// WAIT_TIMEOUT_NS (then it sets the error word itself).
__device__ __forceinline__ bool wait_count(const int *c, int target, volatile int *abort_f, int *err) {
    if (ld_acquire_gpu(c) >= target)
        return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (ld_acquire_gpu(c) >= target)
            return true;
        if ((i & 15u) == 0) {
            if (*abort_f || *reinterpret_cast<volatile int *>(err)) {
                *abort_f = 1;
                return false;
            }
            if (globaltimer() - t0 > WAIT_TIMEOUT_NS) {
                *abort_f = 1;
                atomicExch(err, DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// The eight compute warps: a named barrier over their 256 threads, and the
// same barrier returning whether any of them passed `v` -- so that a failed
// wait takes all of them out of the layer loop together.
__device__ __forceinline__ void compute_sync() { named_bar_sync(1, ST_CT); }
__device__ __forceinline__ bool compute_sync_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.or.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Byte offset of 16-byte chunk `ch` (0..7) of row r in a 128-byte-swizzled
// K-major tile (rows of 128 bytes, chunks permuted by r % 8).
__device__ __forceinline__ uint32_t sw128(int r, int ch) { return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4)); }

__device__ __forceinline__ void unpack8_bf16(uint4 v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}
__device__ __forceinline__ uint4 pack8_bf16(const float (&f)[8]) {
    return make_uint4(bf16_bits(f[0]) | (bf16_bits(f[1]) << 16), bf16_bits(f[2]) | (bf16_bits(f[3]) << 16),
                      bf16_bits(f[4]) | (bf16_bits(f[5]) << 16), bf16_bits(f[6]) | (bf16_bits(f[7]) << 16));
}

// Column of feature f (0..127 of the cluster) in the gate/up accumulator: the
// tile holds two 64-row interleave blocks, [gate 64 | up 64] each.
__device__ __forceinline__ int gate_col(int f) { return (f >> 6) * 128 + (f & 63); }

// Diagnostics: %globaltimer at point `k` of layer l in this CTA's timeline
// ([CTAs][L][32], when dbg_t is set; either instantiation).
#define ST_MARK(k)                                                                            \
    do {                                                                                      \
        if (p.dbg_t)                                                                          \
            p.dbg_t[((size_t)blockIdx.x * L + l) * 32 + (k)] = globaltimer();                 \
    } while (0)

template <bool DEBUG>
__global__ void __launch_bounds__(ST_THREADS, 1)
    k_stack_fp8(const __grid_constant__ StackParams p) {
    if (p.stamp && threadIdx.x == 0)
        stamp_start(p.stamp);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const int S = p.S, nC = p.nC, M = p.M, d = p.d, ff = p.ff, L = p.L;
    const int FPC = ST_FEAT / S;            // features of the cluster's 128 this CTA finishes
    const int j = (int)cluster_ctarank();   // K-quarter of gate/up, N-tile of down
    const int c = (int)blockIdx.x / S;      // cluster: feature slice
    const int k_own = (int)blockIdx.x;      // owner index (owners of column groups: k < n_own)
    const int Mp = (M + 3) & ~3;            // row stride of the sum-of-squares table
    const int ngrp = d / 8;                 // 8-column groups of d
    const int G = k_own < p.n_own ? (ngrp - k_own + p.n_own - 1) / p.n_own : 0;  // groups this CTA owns

    // shared memory beyond the fixed tiles
    const int RS = 2 * FPC + 4;             // row stride (floats) of the exchange buffers: +16 B per row, so
                                            // the 16 token rows of a warp fall in different banks
    const uint32_t rx_bytes = (uint32_t)((S - 1) * M * RS * 4);
    uint8_t *X = smem + OFF_X;
    float *RX = reinterpret_cast<float *>(X);                       // (c)-(d): (S-1) x [M][RS]
    float *XS = reinterpret_cast<float *>(X + rx_bytes);            // (c): (S-1) x [M][RS]
    uint16_t *RST = reinterpret_cast<uint16_t *>(X + rx_bytes);     // (a): [M][256] BF16
    float *SST = reinterpret_cast<float *>(X + rx_bytes + (uint32_t)M * 512);  // (a): [n_own][Mp]
    float *OWN = reinterpret_cast<float *>(X);                      // (g): [G][nC][M][8]
    const uint32_t res_bytes = (uint32_t)p.res_groups * 64 * 16;
    uint4 *RES = reinterpret_cast<uint4 *>(smem + OFF_X + p.x_bytes);           // [res_groups][64]: kept r' of owned groups
    float *INV = reinterpret_cast<float *>(smem + OFF_X + p.x_bytes + res_bytes);  // [64]
    uint16_t *WN = reinterpret_cast<uint16_t *>(smem + OFF_X + p.x_bytes + res_bytes + 256);  // [2][256] norm weights
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_X + p.x_bytes + res_bytes + 256 + 1024);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + N_BARS);
    volatile int *abort_f = reinterpret_cast<volatile int *>(tmem_holder + 1);
    auto bar = [&](int b) { return smem_u32(&bars[b]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    if (tid == 0) {
        mbar_init(bar(B_WFULL_GU), 1);
        mbar_init(bar(B_WEMPTY_GU), 1);
        mbar_init(bar(B_WFULL_D), 1);
        mbar_init(bar(B_WEMPTY_D), 1);
        mbar_init(bar(B_AGU_READY), 1);
        mbar_init(bar(B_ACC_GU), 1);
        mbar_init(bar(B_AD_READY), (uint32_t)S);
        mbar_init(bar(B_ACC_D), 1);
        mbar_init(bar(B_RX), 1);
        mbar_init(bar(B_ASTAGE), 1);
        mbar_init(bar(B_OWN), 1);
        mbar_init(bar(B_DRAIN), 1);
        *abort_f = 0;
        fence_mbar_init();
    }
    if (warp == W_PROD && lane == 0) {
        prefetch_tmap(p.tm_gu);
        prefetch_tmap(p.tm_d);
    }
    if (warp == W_MMA) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // peers arrive on this CTA's barriers and copy into its shared memory only
    // after every CTA of the cluster has initialised them
    if (S > 1) {
        cluster_arrive();
        cluster_wait();
    }
    const uint32_t tmem = *tmem_holder;
    const uint32_t t_gu = tmem, t_d = tmem + 256;
    int *err = p.err;
    int *cnt_R = p.cnt;
    int *cnt_P = p.cnt + 32;               // [S] counters, 32 ints apart
    int *cnt_X = p.cnt + 32 * (1 + 8);     // exit counter

    // weights issued (producer) and MMAs issued (MMA thread), for draining
    uint32_t w_issued = 0;
    bool mma_issued = false;

    if (warp == W_PROD) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            for (int l = 0; l < L && !*abort_f; ++l) {
                const uint32_t par = (uint32_t)(l & 1);
                if (l > 0 && !mbar_wait(bar(B_WEMPTY_GU), par ^ 1u, abort_f, err))
                    break;
                // the gate/up tile and this K-quarter of the layer's norm weights
                mbar_arrive_expect_tx(bar(B_WFULL_GU), 2 * ST_NT * 128 + ST_KQ * 2);
                const int row_gu = l * 2 * ff + ST_NT * c;
                tma_load_2d(sbase + OFF_WGU, p.tm_gu, bar(B_WFULL_GU), ST_KQ * j, row_gu, pol);
                tma_load_2d(sbase + OFF_WGU + ST_NT * 128, p.tm_gu, bar(B_WFULL_GU), ST_KQ * j + 128, row_gu, pol);
                bulk_load(smem_u32(WN) + (par << 9), p.w_norm + (size_t)l * d + ST_KQ * j, ST_KQ * 2,
                          bar(B_WFULL_GU));
                w_issued |= 1u;
                if (l > 0 && !mbar_wait(bar(B_WEMPTY_D), par ^ 1u, abort_f, err))
                    break;
                mbar_arrive_expect_tx(bar(B_WFULL_D), ST_NT * 128);
                tma_load_2d(sbase + OFF_WD, p.tm_d, bar(B_WFULL_D), ST_FEAT * c, l * d + ST_NT * j, pol);
                w_issued |= 2u;
            }
        }
    } else if (warp == W_MMA) {
        // -------------------------------------------------- MMA issuer --
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(ST_ROWS, ST_NT);
            for (int l = 0; l < L; ++l) {
                const uint32_t par = (uint32_t)(l & 1);
                if (!mbar_wait(bar(B_WFULL_GU), par, abort_f, err))
                    break;
                ST_MARK(13);
                if (!mbar_wait(bar(B_AGU_READY), par, abort_f, err))
                    break;
                ST_MARK(14);
                tc_fence_after();
                fence_proxy_async_shared();
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f8f6f4(t_gu, smem_desc_k128(sbase + OFF_AGU + kb * 8192 + k * 32),
                                   smem_desc_k128(sbase + OFF_WGU + kb * (ST_NT * 128) + k * 32), idesc,
                                   (kb | k) ? 1u : 0u);
                mma_issued = true;
                mma_commit(bar(B_ACC_GU));
                mma_commit(bar(B_WEMPTY_GU));
                if (!mbar_wait(bar(B_WFULL_D), par, abort_f, err) ||
                    !mbar_wait_cluster(bar(B_AD_READY), par, abort_f, err))
                    break;
                ST_MARK(15);
                tc_fence_after();
                fence_proxy_async_shared();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_f8f6f4(t_d, smem_desc_k128(sbase + OFF_AD + k * 32), smem_desc_k128(sbase + OFF_WD + k * 32),
                               idesc, k ? 1u : 0u);
                mma_commit(bar(B_ACC_D));
                mma_commit(bar(B_WEMPTY_D));
            }
        }
    } else {
        // ---------------------------------------------- compute warps --
        const int q4 = warp & 3;                         // TMEM lane quarter of this warp
        const int hw = warp >> 2;                        // which half of the columns this warp takes
        const int i16 = lane & 15;
        const int m_t = 16 * q4 + i16;                   // this thread's token in the M = 64 TMEM layout
        const bool row_ok = lane < 16 && m_t < M;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const float eps = p.eps;

        // Prologue: owners form layer 0's input r' = bf16(r + h) and publish it.
        if (G > 0) {
            if (tid < M) {
                const int m = tid;
                float ss = 0.0f;
                for (int gi = 0; gi < G; ++gi) {
                    const int g = k_own + gi * p.n_own;
                    float x[8];
                    unpack8_bf16(*reinterpret_cast<const uint4 *>(p.r_in + (size_t)m * d + 8 * g), x);
                    if (p.h_in) {
                        float h[8];
                        unpack8_bf16(*reinterpret_cast<const uint4 *>(p.h_in + (size_t)m * d + 8 * g), h);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            x[e] = round_bf16(__fadd_rn(x[e], h[e]));
                    }
                    const uint4 v = pack8_bf16(x);
                    RES[gi * 64 + m] = v;
                    *reinterpret_cast<uint4 *>(p.R + ((size_t)(g >> 5) * ST_ROWS + m) * ST_KQ + (g & 31) * 8) = v;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        ss = __fadd_rn(ss, __fmul_rn(x[e], x[e]));
                }
                p.SS[(size_t)k_own * Mp + m] = ss;   // parity 0
            }
            fence_acq_rel_gpu();
            compute_sync();
            if (tid == 0)
                red_release_gpu(cnt_R, 1);
        }

        float4 sc_next = p.scal[0];
        for (int l = 0; l < L; ++l) {
            const uint32_t par = (uint32_t)(l & 1);
            const float4 sc = sc_next;    // (1/s_x, s_x s_gu, 1/s_h, s_h s_d); the next layer's load in flight
            sc_next = p.scal[l + 1 < L ? l + 1 : l];
            // ---- (a) the layer input, normalised and quantised ----------
            if (tid == 0) {
                ST_MARK(0);
                bool w_ok = wait_count(cnt_R, p.n_own * (l + 1), abort_f, err);
                ST_MARK(1);
                if (w_ok) {
                    fence_proxy_async_global();
                    mbar_arrive_expect_tx(bar(B_ASTAGE), (uint32_t)(M * 512 + p.n_own * Mp * 4));
                    bulk_load(smem_u32(RST), p.R + ((size_t)(par * S + j) * ST_ROWS) * ST_KQ, (uint32_t)(M * 512),
                              bar(B_ASTAGE));
                    bulk_load(smem_u32(SST), p.SS + (size_t)par * p.n_own * 64, (uint32_t)(p.n_own * Mp * 4),
                              bar(B_ASTAGE));
                }
            }
            if (compute_sync_or(!mbar_wait(bar(B_ASTAGE), par, abort_f, err) ||
                                !mbar_wait(bar(B_WFULL_GU), par, abort_f, err)))
                break;
            if (tid == 0)
                ST_MARK(2);
            {
                // four threads per token: owner partials k = part (mod 4), each
                // in order, then (part 0 + part 1) + (part 2 + part 3) -- one
                // fixed order, the same in every CTA
                const int m = tid >> 2, part = tid & 3;
                float s = 0.0f;
                if (m < M) {
                    int k = part;
                    for (; k + 28 < p.n_own; k += 32) {      // eight loads in flight, added in order
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            v[e] = SST[(k + 4 * e) * Mp + m];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            s = __fadd_rn(s, v[e]);
                    }
                    for (; k < p.n_own; k += 4)
                        s = __fadd_rn(s, SST[k * Mp + m]);
                }
                const float o1 = __shfl_xor_sync(0xffffffffu, s, 1);
                const float pair = (part & 1) ? __fadd_rn(o1, s) : __fadd_rn(s, o1);
                const float o2 = __shfl_xor_sync(0xffffffffu, pair, 2);
                if (part == 0 && m < M) {
                    const float ms = __fdiv_rn(__fadd_rn(pair, o2), (float)d);
                    INV[m] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
                }
            }
            compute_sync();
            if (tid == 0)
                ST_MARK(23);
            {
                const uint16_t *wn = WN + (par << 8);
                for (int t = tid; t < M * 16; t += ST_CT) {
                    const int m = t >> 4, ch = t & 15;
                    const float inv = INV[m];
                    float x[16], w[16];
                    const uint4 *rv = reinterpret_cast<const uint4 *>(RST + m * ST_KQ + 16 * ch);
                    const uint4 *wv = reinterpret_cast<const uint4 *>(wn + 16 * ch);
                    unpack8_bf16(rv[0], *reinterpret_cast<float(*)[8]>(&x[0]));
                    unpack8_bf16(rv[1], *reinterpret_cast<float(*)[8]>(&x[8]));
                    unpack8_bf16(wv[0], *reinterpret_cast<float(*)[8]>(&w[0]));
                    unpack8_bf16(wv[1], *reinterpret_cast<float(*)[8]>(&w[8]));
                    uint32_t q[4];
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const float y0 = __fmul_rn(__fmul_rn(__fmul_rn(x[e], inv), w[e]), sc.x);
                        const float y1 = __fmul_rn(__fmul_rn(__fmul_rn(x[e + 1], inv), w[e + 1]), sc.x);
                        const float y2 = __fmul_rn(__fmul_rn(__fmul_rn(x[e + 2], inv), w[e + 2]), sc.x);
                        const float y3 = __fmul_rn(__fmul_rn(__fmul_rn(x[e + 3], inv), w[e + 3]), sc.x);
                        q[e / 4] = e4m3x2(y0, y1) | (e4m3x2(y2, y3) << 16);
                    }
                    uint4 qv = make_uint4(q[0], q[1], q[2], q[3]);
                    const size_t qoff = ((size_t)l * M + m) * d + ST_KQ * j + 16 * ch;
                    if (DEBUG && p.dbg_qx && c == 0)
                        *reinterpret_cast<uint4 *>(p.dbg_qx + qoff) = qv;
                    if (DEBUG && p.dbg_qx_in)
                        qv = *reinterpret_cast<const uint4 *>(p.dbg_qx_in + qoff);
                    *reinterpret_cast<uint4 *>(smem + OFF_AGU + (ch >> 3) * 8192 + sw128(m, ch & 7)) = qv;
                }
            }
            fence_proxy_async_shared();
            compute_sync();
            if (tid == 0) {
                ST_MARK(3);
                mbar_arrive(bar(B_AGU_READY));
                // this layer's partials from the other CTAs of the cluster
                if (S > 1)
                    mbar_arrive_expect_tx(bar(B_RX), rx_bytes);
            }
            // ---- (c) exchange of the gate/up partials in the cluster ----
            if (compute_sync_or(!mbar_wait(bar(B_ACC_GU), par, abort_f, err)))
                break;
            if (tid == 0)
                ST_MARK(4);
            tc_fence_after();
            for (int pr = 0; pr < S; ++pr) {
                if (pr == j)
                    continue;
                float *dst = XS + (size_t)(pr < j ? pr : pr - 1) * M * RS + hw * FPC;
                // this warp's half (gate or up) of the peer's columns, in runs of
                // 16, all in flight before one wait (FPC <= 64 when S > 1)
                uint32_t v[4][16];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (16 * q < FPC)
                        tmem_ld_x16(t_gu + lane_off + (uint32_t)(gate_col(FPC * pr + 16 * q) + 64 * hw), v[q]);
                tmem_ld_wait();
                if (row_ok) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (16 * q < FPC) {
                            float4 *o = reinterpret_cast<float4 *>(dst + (size_t)m_t * RS + 16 * q);
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                o[e] = make_float4(__uint_as_float(v[q][4 * e]), __uint_as_float(v[q][4 * e + 1]),
                                                   __uint_as_float(v[q][4 * e + 2]), __uint_as_float(v[q][4 * e + 3]));
                        }
                    }
                }
            }
            if (tid == 0)
                ST_MARK(16);
            fence_proxy_async_shared();
            if (tid == 0)
                ST_MARK(17);
            compute_sync();
            if (tid == 0 && S > 1) {
                const uint32_t bytes = (uint32_t)(M * RS * 4);
                for (int pr = 0; pr < S; ++pr) {
                    if (pr == j)
                        continue;
                    const int slot = j < pr ? j : j - 1;          // this CTA's slot in the receiver
                    bulk_copy_to_cta(mapa_shared(smem_u32(RX) + (uint32_t)slot * bytes, (uint32_t)pr),
                                     smem_u32(XS) + (uint32_t)(pr < j ? pr : pr - 1) * bytes, bytes,
                                     mapa_shared(bar(B_RX), (uint32_t)pr));
                }
            }
            // ---- (d) reduce, gated activation, q_h to the cluster ------
            if (tid == 0)
                ST_MARK(5);
            if (compute_sync_or(S > 1 && !mbar_wait_cluster(bar(B_RX), par, abort_f, err)))
                break;
            if (tid == 0)
                ST_MARK(6);
            for (int f0 = 16 * hw; f0 < FPC; f0 += 32) {        // this warp's runs of 16 features
                const int fl = FPC * j + f0;                    // first feature of the run, in the cluster
                uint32_t vg[16], vu[16];
                tmem_ld_x16(t_gu + lane_off + (uint32_t)gate_col(fl), vg);
                tmem_ld_x16(t_gu + lane_off + (uint32_t)(gate_col(fl) + 64), vu);
                tmem_ld_wait();
                if (row_ok) {
                    float g[16], u[16], a[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        g[e] = 0.0f;
                        u[e] = 0.0f;
                    }
                    for (int s = 0; s < S; ++s) {               // K-quarters in order
                        if (s == j) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                g[e] = __fadd_rn(g[e], __uint_as_float(vg[e]));
                                u[e] = __fadd_rn(u[e], __uint_as_float(vu[e]));
                            }
                        } else {
                            const float *src = RX + ((size_t)(s < j ? s : s - 1) * M + m_t) * RS + f0;
#pragma unroll
                            for (int e = 0; e < 16; e += 4) {
                                const float4 gg = *reinterpret_cast<const float4 *>(src + e);
                                const float4 uu = *reinterpret_cast<const float4 *>(src + FPC + e);
                                g[e] = __fadd_rn(g[e], gg.x);
                                g[e + 1] = __fadd_rn(g[e + 1], gg.y);
                                g[e + 2] = __fadd_rn(g[e + 2], gg.z);
                                g[e + 3] = __fadd_rn(g[e + 3], gg.w);
                                u[e] = __fadd_rn(u[e], uu.x);
                                u[e + 1] = __fadd_rn(u[e + 1], uu.y);
                                u[e + 2] = __fadd_rn(u[e + 2], uu.z);
                                u[e + 3] = __fadd_rn(u[e + 3], uu.w);
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        g[e] = round_bf16(__fmul_rn(g[e], sc.y));
                        u[e] = round_bf16(__fmul_rn(u[e], sc.y));
                    }
                    gated_run<16>(p.act, g, u, a);
                    uint32_t q[4];
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        q[e / 4] = e4m3x2(__fmul_rn(a[e], sc.z), __fmul_rn(a[e + 1], sc.z)) |
                                   (e4m3x2(__fmul_rn(a[e + 2], sc.z), __fmul_rn(a[e + 3], sc.z)) << 16);
                    const uint4 qv = make_uint4(q[0], q[1], q[2], q[3]);
                    const uint32_t off = OFF_AD + sw128(m_t, fl >> 4);
                    for (int pr = 0; pr < S; ++pr) {
                        if (pr == j)
                            *reinterpret_cast<uint4 *>(smem + off) = qv;
                        else
                            st_cluster_v4(mapa_shared(sbase + off, (uint32_t)pr), qv);
                    }
                    if (DEBUG) {
                        const int fg = ST_FEAT * c + fl;        // feature index in [0, ff)
                        if (p.dbg_qh)
                            *reinterpret_cast<uint4 *>(p.dbg_qh + ((size_t)l * M + m_t) * ff + fg) = qv;
                        if (p.dbg_gu) {
                            uint16_t *o = p.dbg_gu + ((size_t)l * M + m_t) * 2 * ff + fg;
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                o[e] = (uint16_t)bf16_bits(g[e]);
                                o[ff + e] = (uint16_t)bf16_bits(u[e]);
                            }
                        }
                    }
                }
            }
            if (tid == 0)
                ST_MARK(18);
            tc_fence_before();
            fence_proxy_async_cluster();
            if (tid == 0)
                ST_MARK(19);
            fence_acq_rel_cluster();
            if (tid == 0)
                ST_MARK(20);
            compute_sync();
            if (tid == 0) {
                ST_MARK(7);
                if (S == 1)
                    mbar_arrive(bar(B_AD_READY));
                else
                    for (int pr = 0; pr < S; ++pr)
                        mbar_arrive_cluster_release(mapa_shared(bar(B_AD_READY), (uint32_t)pr));
            }
            // ---- (f) the down partial of this K-slice to L2 -----------
            if (compute_sync_or(!mbar_wait(bar(B_ACC_D), par, abort_f, err)))
                break;
            if (tid == 0)
                ST_MARK(8);
            tc_fence_after();
            {
                // P[parity][group][cluster][M][8]: an owner's groups are contiguous
                float *pp = p.P + (((size_t)par * ngrp + 32 * j) * nC + c) * M * 8;
                for (int c0 = 128 * hw; c0 < 128 * hw + 128; c0 += 64) {
                    uint32_t v[2][32];
                    tmem_ld_x32(t_d + lane_off + (uint32_t)c0, v[0]);
                    tmem_ld_x32(t_d + lane_off + (uint32_t)(c0 + 32), v[1]);
                    tmem_ld_wait();
                    if (row_ok) {
#pragma unroll
                        for (int gq = 0; gq < 8; ++gq) {
                            const uint32_t *w8 = &v[gq >> 2][8 * (gq & 3)];
                            float4 *o = reinterpret_cast<float4 *>(pp + ((size_t)(c0 / 8 + gq) * nC * M + m_t) * 8);
                            o[0] = make_float4(__uint_as_float(w8[0]), __uint_as_float(w8[1]), __uint_as_float(w8[2]),
                                               __uint_as_float(w8[3]));
                            o[1] = make_float4(__uint_as_float(w8[4]), __uint_as_float(w8[5]), __uint_as_float(w8[6]),
                                               __uint_as_float(w8[7]));
                        }
                    }
                }
            }
            if (tid == 0)
                ST_MARK(21);
            tc_fence_before();
            fence_acq_rel_gpu();
            if (tid == 0)
                ST_MARK(22);
            compute_sync();
            if (tid == 0) {
                ST_MARK(9);
                red_release_gpu(cnt_P + 32 * j, 1);
            }
            // ---- (g) owners: reduce, residual, publish ----------------
            if (G > 0) {
                if (tid == 0) {
                    bool w_ok = true;
                    int last_tile = -1;
                    for (int gi = 0; gi < G && w_ok; ++gi) {
                        const int jt = (k_own + gi * p.n_own) >> 5;
                        if (jt != last_tile)
                            w_ok = wait_count(cnt_P + 32 * jt, nC * (l + 1), abort_f, err);
                        last_tile = jt;
                    }
                    ST_MARK(10);
                    if (w_ok) {
                        fence_proxy_async_global();
                        mbar_arrive_expect_tx(bar(B_OWN), (uint32_t)(G * nC * M * 32));
                        for (int gi = 0; gi < G; ++gi) {   // one copy per owned group: all clusters' partials
                            const int g = k_own + gi * p.n_own;
                            bulk_load(smem_u32(OWN + (size_t)gi * nC * M * 8),
                                      p.P + ((size_t)par * ngrp + g) * nC * M * 8, (uint32_t)(nC * M * 32), bar(B_OWN));
                        }
                    }
                }
                if (compute_sync_or(!mbar_wait(bar(B_OWN), par, abort_f, err)))
                    break;
                if (tid == 0)
                    ST_MARK(11);
                const bool last = l == L - 1;
                {
                    // four threads per token, columns 2 part and 2 part + 1 of
                    // every owned group; the token's sum of squares as
                    // (part 0 + part 1) + (part 2 + part 3)
                    const int m = tid >> 2, part = tid & 3;
                    float ss = 0.0f;
                    if (m < M) {
                        for (int gi = 0; gi < G; ++gi) {
                            const int g = k_own + gi * p.n_own;
                            float a0 = 0.0f, a1 = 0.0f;
#pragma unroll 8
                            for (int cc = 0; cc < nC; ++cc) {     // K-slices in order
                                const float2 v2 =
                                    *reinterpret_cast<const float2 *>(OWN + ((size_t)(gi * nC + cc) * M + m) * 8 + 2 * part);
                                a0 = __fadd_rn(a0, v2.x);
                                a1 = __fadd_rn(a1, v2.y);
                            }
                            uint32_t *rw = reinterpret_cast<uint32_t *>(&RES[gi * 64 + m]) + part;
                            const uint32_t rv = *rw;
                            const float x0 = round_bf16(__fadd_rn(bf_lo(rv), __fmul_rn(a0, sc.w)));
                            const float x1 = round_bf16(__fadd_rn(bf_hi(rv), __fmul_rn(a1, sc.w)));
                            uint32_t v = bf16_bits(x0) | (bf16_bits(x1) << 16);
                            const size_t col = 8 * (size_t)g + 2 * part;
                            if (DEBUG && p.dbg_out)
                                *reinterpret_cast<uint32_t *>(p.dbg_out + ((size_t)l * M + m) * d + col) = v;
                            if (last) {
                                *reinterpret_cast<uint32_t *>(p.out + (size_t)m * d + col) = v;
                            } else {
                                float y0 = x0, y1 = x1;
                                if (DEBUG && p.dbg_res_in) {
                                    // the next layer starts from the caller's residual instead
                                    v = *reinterpret_cast<const uint32_t *>(p.dbg_res_in + ((size_t)(l + 1) * M + m) * d + col);
                                    y0 = bf_lo(v);
                                    y1 = bf_hi(v);
                                }
                                *rw = v;
                                *reinterpret_cast<uint32_t *>(p.R + ((size_t)((par ^ 1u) * S + (g >> 5)) * ST_ROWS + m) * ST_KQ +
                                                              (g & 31) * 8 + 2 * part) = v;
                                ss = __fadd_rn(ss, __fmul_rn(y0, y0));
                                ss = __fadd_rn(ss, __fmul_rn(y1, y1));
                            }
                        }
                    }
                    const float o1 = __shfl_xor_sync(0xffffffffu, ss, 1);
                    const float pr2 = (part & 1) ? __fadd_rn(o1, ss) : __fadd_rn(ss, o1);
                    const float o2 = __shfl_xor_sync(0xffffffffu, pr2, 2);
                    if (!last && part == 0 && m < M)
                        p.SS[(size_t)(par ^ 1u) * p.n_own * 64 + (size_t)k_own * Mp + m] = __fadd_rn(pr2, o2);
                }
                if (tid == 0)
                    ST_MARK(24);
                fence_acq_rel_gpu();
                if (tid == 0)
                    ST_MARK(25);
                compute_sync();
                if (tid == 0) {
                    ST_MARK(12);
                    if (!last)
                        red_release_gpu(cnt_R, 1);
                }
            }
        }
    }

    // ---------------------------------------------------------- exit --
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*abort_f) {
        // copies into this CTA that may still be in flight: its own stages
        // of the layer input and of the owned partials, and the partials
        // the cluster sends (each phase waited for, bounded; a phase with
        // nothing in flight just runs out its bound)
        if (tid == 0) {
            for (int b : {(int)B_ASTAGE, (int)B_OWN, (int)B_RX})
                for (uint32_t par = 0; par < 2; ++par)
                    mbar_wait_for(bar(b), par, 20000000ull);
        }
        // drain what this CTA may still have in flight: weight copies, MMAs
        if (warp == W_PROD && lane == 0) {
            if (w_issued & 1u)
                mbar_wait_for(bar(B_WFULL_GU), 0, 100000000ull), mbar_wait_for(bar(B_WFULL_GU), 1, 100000000ull);
            if (w_issued & 2u)
                mbar_wait_for(bar(B_WFULL_D), 0, 100000000ull), mbar_wait_for(bar(B_WFULL_D), 1, 100000000ull);
        }
        if (warp == W_MMA && lane == 0 && mma_issued) {
            mma_commit(bar(B_DRAIN));
            mbar_wait_for(bar(B_DRAIN), 0, 100000000ull);
        }
    }
    __syncthreads();
    // no CTA leaves while a peer may still write into its shared memory
    if (S > 1) {
        cluster_arrive();
        cluster_wait();
    }
    if (warp == W_MMA) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0) {
        // the last CTA out re-arms the counters for the next launch (after a
        // failure they are left for the host to clear)
        if (!*abort_f && !*reinterpret_cast<volatile int *>(err)) {
            __threadfence();
            const int old = atomicAdd(cnt_X, 1);
            if (old == (int)gridDim.x - 1) {
                *reinterpret_cast<volatile int *>(cnt_R) = 0;
                for (int t = 0; t < S; ++t)
                    *reinterpret_cast<volatile int *>(cnt_P + 32 * t) = 0;
                *reinterpret_cast<volatile int *>(cnt_X) = 0;
                __threadfence();
            }
        }
        if (p.stamp)
            stamp_end(p.stamp);
    }
}

template <bool DEBUG>
cudaError_t stack_run(const StackParams &p, int grid, size_t smem, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_stack_fp8<DEBUG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem_max_stack());
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    return launch_ex(k_stack_fp8<DEBUG>, dim3((unsigned)grid), dim3(ST_THREADS), smem, s, false,
                     (unsigned)(p.S > 1 ? p.S : 1), p);
}

}  // namespace

size_t smem_max_stack() { return 232448; }

bool plan_stack(StackParams &p, int M, int d, int ff, int num_sms, size_t *smem_bytes, int *grid) {
    if (M < 1 || M > ST_ROWS || d % ST_KQ || ff % ST_FEAT)
        return false;
    const int S = d / ST_KQ, nC = ff / ST_FEAT;
    // a CTA finishes 128 / S features in runs of 16
    if ((S != 1 && S != 2 && S != 4 && S != 8) || S * nC > num_sms)
        return false;
    const int nCTA = S * nC;
    const int n_own = std::min(nCTA, d / 8);
    const int ngrp = d / 8;
    const int G = (ngrp + n_own - 1) / n_own;
    if (G > 16)
        return false;
    const int FPC = ST_FEAT / S;
    const int Mp = (M + 3) & ~3;
    const size_t rx = (size_t)(S - 1) * M * (2 * FPC + 4) * 4;
    const size_t xs = rx;
    const size_t astage = (size_t)M * 512 + (size_t)n_own * Mp * 4;
    const size_t own = (size_t)G * nC * M * 32;
    size_t x = std::max(rx + std::max(xs, astage), own);
    x = (x + 1023) / 1024 * 1024;
    const size_t total = 1024 + OFF_X + x + (size_t)G * 64 * 16 + 256 + 1024 + N_BARS * 8 + 16;
    if (total > smem_max_stack())
        return false;
    // over half an SM's shared memory: one CTA per SM, each holding all 512
    // TMEM columns (a second CTA's allocation would wait for the first)
    const size_t one_per_sm = 116 * 1024;
    p.M = M;
    p.d = d;
    p.ff = ff;
    p.S = S;
    p.nC = nC;
    p.n_own = n_own;
    p.x_bytes = (uint32_t)x;
    p.res_groups = G;
    *smem_bytes = std::max(total, one_per_sm);
    *grid = nCTA;
    return true;
}

int stack_max_active_clusters(const StackParams &p, size_t smem) {
    cudaError_t e = cudaFuncSetAttribute(k_stack_fp8<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_max_stack());
    if (e != cudaSuccess)
        return 0;
    if (p.S > 1) {
        e = cudaFuncSetAttribute(k_stack_fp8<false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
        (void)e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.S * p.nC));
    cfg.blockDim = dim3(ST_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)(p.S > 1 ? p.S : 1);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, k_stack_fp8<false>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_stack(const StackParams &p, size_t smem, cudaStream_t s, bool debug) {
    const int grid = p.S * p.nC;
    return debug ? stack_run<true>(p, grid, smem, s) : stack_run<false>(p, grid, smem, s);
}

}  // namespace frt
