/*
 * frt_nvfp4.h -- C ABI of the NVFP4 variant of the FFN sublayer in
 * libfrt_ffn.so (itsolotime FlashRT article, 7.2: the NVFP4 encoder FFN --
 * gate and up as two NVFP4 GEMMs that emit packed FP4 plus scales, a fused
 * GeGLU kernel that requantises FP4 to FP4, an NVFP4 down GEMM, the residual
 * kept in 16 bits, AWQ pre-scaling; 7.2's closing remark: the residual
 * stream stays in high precision).
 *
 * Per layer l, on M tokens (fp32 operations, each rounded):
 *   N1  r' = bf16(r + h);  y = ((r' * inv_rms) * w_norm) / c   (c: AWQ scales or 1)
 *       X = NVFP4(y, s_x)
 *   N2  G = NVFP4(acc(X, W_g') * (s_x s_wg), s_g);  U = NVFP4(acc(X, W_u') * (s_x s_wu), s_u)
 *       W_g' = NVFP4(W_g[j][k] * c[k], s_wg) and likewise W_u'
 *   N3  A = NVFP4(act(dec G) * dec U, s_h)
 *   N4  out = bf16(r' + acc(A, W_d') * (s_h s_wd));  W_d' = NVFP4(W_d, s_wd)
 * NVFP4(x, s): E2M1 codes with one E4M3 scale per 16 consecutive elements
 * along K, b = E4M3(amax_block / (6 s)), q = E2M1(x / (dec(b) s)); the
 * tensor scales s = amax / (448 * 6) -- of the weights when they are loaded,
 * of the activations by calibration (progressive, layer by layer).
 * Readings (the pages give the loop, not the format or the AWQ rule): NVFP4
 * as NVIDIA publishes it; AWQ scales supplied by the caller (the oracle's
 * awq_scales gives the activation-magnitude rule c_k = mean|y_k|^alpha).
 * Kernels: N2 and N3 run as one GEMM over [W_g'; W_u'] (stored interleaved in
 * blocks of 64 rows, so a tile holds the gate and up rows of the same
 * features) whose epilogue forms G and U as above, decodes them and
 * requantises act(dec G) * dec U -- the same operations in the same order as
 * two GEMMs and a combine kernel, without the round trip of G and U through
 * memory; three kernels per layer, chained by programmatic dependent launch.
 *
 * Layouts: codes are packed two per byte, element 2i in the low nibble,
 * row-major [rows, K/2]; the block scales of GEMM operands (X, A and the
 * weights) are stored in the tensor cores' TMEM-ready order: per 128-row tile
 * and 64-element K chunk a 512-byte block, byte (r % 32) * 16 + (r / 32) * 4 + j
 * for row r of the tile and 16-element group j of the chunk (tiles major,
 * chunks minor); the block scales of G and U (frt_fp4_debug_trace) are
 * row-major [M, ff/16].
 *
 * Conventions: as frt_ffn.h (BF16 bit patterns, 16-byte aligned device
 * pointers, frt_ffn_last_error() for messages, one host thread and one stream
 * at a time per plan).  Nothing is allocated after plan creation except by
 * frt_fp4_calibrate; frt_fp4_forward may be captured into a CUDA graph.
 */
#ifndef FRT_NVFP4_H
#define FRT_NVFP4_H

#include "frt_ffn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct frt_fp4_plan *frt_fp4_plan_t;

/*
 * Create a plan for n_layers NVFP4 sublayers of width d and hidden width ff,
 * activation act (frt_act), at most M_max tokens per call.  Allocates the
 * weight arenas (codes and scales), norm weights, AWQ reciprocals and
 * scratch.  Requires: d % 256 == 0; ff % 256 == 0; 1 <= M_max <= 65536;
 * 1 <= n_layers <= 4096; a compute-capability 10.3 GPU.
 * Errors: INVALID_ARG, UNSUPPORTED, OOM, CUDA.  *out is NULL on failure.
 */
frt_status frt_fp4_plan_create(int d, int ff, int act, int M_max, int n_layers, frt_fp4_plan_t *out);

/* Free the plan and its device memory (synchronises the device).  NULL is accepted. */
frt_status frt_fp4_plan_destroy(frt_fp4_plan_t plan);

/*
 * Quantise one layer's BF16 weights into the plan: w_norm [d], w_gate [ff, d],
 * w_up [ff, d], w_down [d, ff] (device, nn.Linear layout); awq: device fp32
 * [d] AWQ scales c (each > 0) applied to the gate and up weights' columns and
 * divided out of the activation, or NULL for none.  Synchronises `stream`.
 * Errors: INVALID_ARG (null/misaligned pointer, layer out of range), CUDA.
 */
frt_status frt_fp4_load_weights(frt_fp4_plan_t plan, int layer, const void *w_norm, const void *w_gate,
                                const void *w_up, const void *w_down, const float *awq, frt_stream_t stream);

/*
 * Progressive calibration over the whole stack: for layer 0..L-1 in turn,
 * s_x, then s_g and s_u, then s_h from the amax over the n_batches batches
 * (each [M, d] BF16; hidden[b] added at layer 0, hidden == NULL for none),
 * every later tensor measured with the earlier scales applied; the layer's
 * outputs are the next layer's inputs.  Allocates (and frees) 2 n_batches M d
 * BF16 of scratch.  Synchronises `stream`.
 * Errors: INVALID_ARG, NOT_READY (weights missing), SHAPE (M > M_max), OOM, CUDA.
 */
frt_status frt_fp4_calibrate(frt_fp4_plan_t plan, const void *const *residual, const void *const *hidden,
                             int n_batches, int M, frt_stream_t stream);

/* Host arrays: act [n_layers * 4] = (s_x, s_g, s_u, s_h) per layer, weight
 * [n_layers * 3] = (s_wg, s_wu, s_wd) per layer (either may be NULL). */
frt_status frt_fp4_get_scales(frt_fp4_plan_t plan, float *act, float *weight);
/* Set every layer's activation scales (host [n_layers * 4], each finite and > 0). */
frt_status frt_fp4_set_scales(frt_fp4_plan_t plan, const float *act);

/*
 * The stack on M tokens: residual_in [M, d] BF16, hidden_in [M, d] BF16 (added
 * at layer 0) or NULL, out [M, d] BF16 (may not alias the inputs).  M == 0
 * does nothing.  Three kernels per layer; no allocation.
 * Errors: INVALID_ARG, NOT_READY (weights or scales missing), SHAPE, CUDA.
 */
frt_status frt_fp4_forward(frt_fp4_plan_t plan, const void *residual_in, const void *hidden_in, void *out, int M,
                           frt_stream_t stream);

/*
 * Measurement: where the time of the stack goes, kernel by kernel, when it
 * runs as one replayed graph ("FlashRT docs/architecture.md", 7).  Captures
 * frt_fp4_forward on these buffers into a graph with every launch recording
 * %globaltimer at its CTAs' starts and ends, replays it n_replays times
 * (synchronising after each), and writes to kernel_us[k] the median over
 * replays of launch k's share of the replay: from its first CTA's start, or
 * the end of the launches before it if later, to its last CTA's end -- so the
 * shares of launches that overlap (programmatic dependent launch) do not
 * overlap.  Launch k = 3 l + s for layer l and step s (0 norm + quantise,
 * 1 gate/up GEMM with the gated FP4 epilogue, 2 down GEMM with the residual);
 * kernel_us must hold 3 n_layers floats and *n_kernels (may be NULL)
 * receives that count.  The replays write `out` like frt_fp4_forward.  The
 * graph is freed before returning.  `stream` must not be the legacy default
 * stream (a graph is captured on it).  Synchronises.
 * Errors: INVALID_ARG (M < 1, counts, default stream), NOT_READY, SHAPE,
 * CUDA, DEVICE_TIMEOUT.
 */
frt_status frt_fp4_forward_profile(frt_fp4_plan_t plan, const void *residual_in, const void *hidden_in, void *out,
                                   int M, int n_replays, float *kernel_us, int *n_kernels, frt_stream_t stream);

/*
 * Test/diagnostic: layer `layer` alone on its input, with the same kernels,
 * copying the intermediates to caller buffers (any may be NULL): r_prime
 * [M, d] BF16 (only when hidden_in is given), x_codes [M, d/2] and x_sf
 * (TMEM-ready, ceil(M/128) * 128 * d/16 bytes), g/u codes [M, ff/2] and
 * row-major scales [M, ff/16], h_codes [M, ff/2] and h_sf (TMEM-ready,
 * ceil(M/128) * 128 * ff/16 bytes).  G and U are written by the gate/up
 * GEMM's epilogue as it forms them (the four g/u buffers: all or none).
 * Synchronises `stream`.
 */
frt_status frt_fp4_debug_trace(frt_fp4_plan_t plan, int layer, const void *residual_in, const void *hidden_in,
                               void *out, void *r_prime, void *x_codes, void *x_sf, void *g_codes, void *g_sf,
                               void *u_codes, void *u_sf, void *h_codes, void *h_sf, int M, frt_stream_t stream);

/*
 * Test/diagnostic: layer `layer` step by step, each GEMM optionally started
 * from caller-supplied quantised inputs (so that a test can feed the
 * oracle's X and A and compare every row of each step alone): x_codes_in
 * [M, d/2] with x_sf_in (TMEM-ready, ceil(M/128) * 128 * d/16 bytes) replace
 * the norm's X for the gate/up GEMM; h_codes_in [M, ff/2] with h_sf_in
 * (TMEM-ready) replace the gate/up epilogue's A for the down GEMM; either
 * pair may be NULL (the kernels' own).  Copies out G and U (as
 * frt_fp4_debug_trace; all four or none), A as the gate/up GEMM produced it
 * (h_codes, h_sf; before any injection) and the layer output (out).
 * Synchronises `stream`.
 */
frt_status frt_fp4_debug_trace_from(frt_fp4_plan_t plan, int layer, const void *residual_in, const void *hidden_in,
                                   const void *x_codes_in, const void *x_sf_in, const void *h_codes_in,
                                   const void *h_sf_in, void *out, void *g_codes, void *g_sf, void *u_codes,
                                   void *u_sf, void *h_codes, void *h_sf, int M, frt_stream_t stream);

/*
 * Test/diagnostic: copy a layer's quantised weight (which: 0 gate, 1 up,
 * 2 down) -- codes row-major [rows, K/2] and TMEM-ready scales (rows * K/16
 * bytes) of that weight's own rows (gate and up taken out of the interleaved
 * arena on the host).  Synchronises `stream`.
 */
frt_status frt_fp4_debug_weights(frt_fp4_plan_t plan, int layer, int which, void *codes, void *sf,
                                 frt_stream_t stream);

/*
 * Test/diagnostic: out[m][n] = alpha * sum_k A[m][k] B[n][k] over NVFP4
 * operands (codes [M, K/2] and [N, K/2]; TMEM-ready scales sized for
 * ceil(M/128) and N/128 tiles), fp32 [M, N] out.  N % 128 == 0, K % 256 == 0,
 * 1 <= M <= 65536.  Runs the role the plan's GEMMs run: weight-streaming
 * (the weights as the 128-row operand) for M <= 64, else tiled; FRT_F4_SWAP=0
 * forces the tiled role.  splits: the split-K factor asked for (1 <= splits
 * <= K / 256; the planner may take fewer, never more); weight-streaming
 * splits of a tile exchange partials inside a thread-block cluster, tiled
 * ones through ws (fp32, tiles * splits * 128 * 128; tiles = N/128, or N/128
 * * ceil(M/128) tiled; at most 2048) with one arrival counter per tile in
 * counters (zeroed before the first call; each call advances a tile's counter
 * by its split count, so counters may be reused only with the same splits).
 * The partials are summed in split order.  err: a device int the kernel sets
 * on a timed-out wait.
 */
frt_status frt_nvfp4_gemm(const void *a_codes, const void *a_sf, const void *b_codes, const void *b_sf, int M, int N,
                          int K, float alpha, float *out, int splits, float *ws, int *counters, int *err,
                          frt_stream_t stream);

/* Synchronise `stream` and report a kernel that gave up a bounded wait
 * (DEVICE_TIMEOUT; the plan's error word and split-K counters are then
 * cleared). */
frt_status frt_fp4_device_status(frt_fp4_plan_t plan, frt_stream_t stream);

/*
 * Test hook for the failure path (no counterpart in the pages): launch layer
 * 0's gate/up GEMM for M tokens (the weight-streaming role for M <= 64, else
 * the tiled one) whose MMA thread first waits for a barrier phase that
 * nothing completes.  The bounded wait gives up after about 2 s, sets the
 * plan's error word, and every role of the kernel -- the scale warps
 * included -- drains its copies, frees its tensor memory and exits; the call
 * then returns what frt_fp4_device_status reports -- DEVICE_TIMEOUT -- and the
 * plan (and the CUDA context) stay usable.  Overwrites the plan's activation
 * scratch.  Errors: INVALID_ARG, SHAPE, CUDA, DEVICE_TIMEOUT.
 */
frt_status frt_fp4_debug_stall(frt_fp4_plan_t plan, int M, frt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FRT_NVFP4_H */
