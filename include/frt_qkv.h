/*
 * frt_qkv.h -- C ABI of the attention-input sublayer of libfrt_ffn.so: the
 * projections on the other side of the residual stream from the FFN.
 *
 *   A1  r' = bf16(r + h);  y = r' / sqrt(mean(r'^2) + eps) * w_norm;
 *       q_x = E4M3(y / s_x)                                (as the FFN's A1)
 *   P2  qkv = bf16((q_x . W_qkv^T) * s_x * s_qkv)          (FP8 GEMM)
 *       W_qkv = [W_q; W_k; W_v], one per-tensor scale s_qkv
 *   P3  split qkv into Hq query, Hkv key and Hkv value heads of head_dim
 *       (columns: Q heads, then K heads, then V heads) and rotate Q and K
 *       by RoPE at each token's position; outputs head-major [H, M, hd]
 *
 * Passages (page title, section):
 *   - agentlenshq "flashrt-project/FlashRT" summary, "What it is": the
 *     kernel set includes fused residual-norm-quantise, RoPE and FP8 GEMM.
 *   - itsolotime FlashRT article, 5.2: the weight spec fuses q/k/v into one
 *     FusedQKV tensor quantised as one (Quant(), scale_into).
 *   - "FlashRT docs/architecture.md", 8 Kernel Library: "qkv split + RoPE"
 *     among the memory-bound kernels.
 * The pages give no formula for the split or the rotation.  Readings (the
 * usual ones): RoPE in the rotate-half layout -- element i of a head's
 * first half pairs with element i + hd/2 -- with theta_i = base^(-2i/hd)
 * (fp64, rounded to fp32), angle = fp32(pos * theta_i), and in fp32
 * o_i = x_i cos - x_{i+hd/2} sin, o_{i+hd/2} = x_{i+hd/2} cos + x_i sin,
 * each output rounded to BF16; V is copied unrotated.
 *
 * Conventions: as frt_ffn.h (row-major dense tensors, BF16 bit patterns,
 * E4M3 bytes, 16-byte aligned device pointers, frt_ffn_last_error() for
 * messages, one host thread and one stream at a time per plan).  Nothing is
 * allocated after plan creation; frt_qkv_forward is pointer-stable and may
 * be captured into a CUDA graph by the caller (Relaxed mode).
 */
#ifndef FRT_QKV_H
#define FRT_QKV_H

#include "frt_ffn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct frt_qkv_plan *frt_qkv_plan_t;

/*
 * Create a plan for n_layers attention-input sublayers of model width d with
 * n_q_heads query and n_kv_heads key/value heads of head_dim, RoPE base
 * rope_base, at most M_max tokens per call.  Allocates the E4M3 weight arena
 * (layer-major [W_q; W_k; W_v], each [(Hq + 2 Hkv) hd, d]), the BF16 norm
 * weights, and scratch sized by M_max.
 * Requires: d % 128 == 0; head_dim % 8 == 0 and 16 <= head_dim <= 512;
 * n_q_heads >= 1, n_kv_heads >= 1, n_q_heads % n_kv_heads == 0;
 * (n_q_heads + 2 n_kv_heads) head_dim % 128 == 0; rope_base > 1;
 * 1 <= M_max <= 65536; 1 <= n_layers <= 4096; a compute-capability 10.3 GPU.
 * Errors: INVALID_ARG, UNSUPPORTED, OOM, CUDA.  *out is NULL on failure.
 */
frt_status frt_qkv_plan_create(int d, int n_q_heads, int n_kv_heads, int head_dim, float rope_base, int M_max,
                               int n_layers, frt_qkv_plan_t *out);

/* Free the plan and its device memory (synchronises the device).  NULL is accepted. */
frt_status frt_qkv_plan_destroy(frt_qkv_plan_t plan);

/*
 * Quantise one layer's BF16 weights into the plan: w_norm [d], w_q [Hq hd, d],
 * w_k [Hkv hd, d], w_v [Hkv hd, d] (device, row-major nn.Linear layout);
 * s_qkv = amax([W_q; W_k; W_v]) / 448 (1 for an all-zero tensor).  The plan
 * copies what it needs.  Synchronises `stream`.
 * Errors: INVALID_ARG (null/misaligned pointer, layer out of range), CUDA.
 */
frt_status frt_qkv_load_weights(frt_qkv_plan_t plan, int layer, const void *w_norm, const void *w_q, const void *w_k,
                                const void *w_v, frt_stream_t stream);

/*
 * frt_qkv_load_weights with options.  flags FRT_LOAD_FOLD_NORM (itsolotime
 * article, 5.2: the Pi0 spec folds the RMSNorm weight into the FusedQKV
 * weight): [W_q; W_k; W_v] quantised as W'[j][k] = W[j][k] * w_norm[k] (exact
 * in fp32), one scale amax(W') / 448, and the sublayer's norm multiplies by
 * ones.  Calibrate (or set the scale) after loading.  Errors: as
 * frt_qkv_load_weights; INVALID_ARG for unknown flags.
 */
frt_status frt_qkv_load_weights_ex(frt_qkv_plan_t plan, int layer, const void *w_norm, const void *w_q,
                                   const void *w_k, const void *w_v, unsigned flags, frt_stream_t stream);

/*
 * Calibrate layer `layer`'s activation scale: s_x = amax(y) / 448 over
 * n_batches batches of M rows (residual[b] [M, d] BF16, hidden[b] the same
 * or hidden == NULL / hidden[b] == NULL for none).  Synchronises `stream`.
 * Errors: INVALID_ARG, NOT_READY (weights of the layer not loaded), SHAPE, CUDA.
 */
frt_status frt_qkv_calibrate(frt_qkv_plan_t plan, int layer, const void *const *residual, const void *const *hidden,
                             int n_batches, int M, frt_stream_t stream);

/* Host arrays of n_layers fp32 scales (either may be NULL). */
frt_status frt_qkv_get_scales(frt_qkv_plan_t plan, float *s_x, float *s_qkv);
/* Set every layer's activation scale s_x (host array of n_layers, each > 0). */
frt_status frt_qkv_set_scales(frt_qkv_plan_t plan, const float *s_x);

/*
 * Run layer `layer` on M tokens: residual_in [M, d] BF16 (+ hidden_in [M, d]
 * or NULL), positions [M] int32 (device; each >= 0); writes q_out [Hq, M, hd],
 * k_out [Hkv, M, hd], v_out [Hkv, M, hd] BF16 and, if r_prime_out is not
 * NULL, r' [M, d] BF16 (the residual for the attention's output add).  M == 0
 * does nothing.  No allocation.
 * Errors: INVALID_ARG, NOT_READY (weights or scale missing), SHAPE (M > M_max),
 * CUDA (launch errors); kernel errors surface through frt_qkv_device_status.
 */
frt_status frt_qkv_forward(frt_qkv_plan_t plan, int layer, const void *residual_in, const void *hidden_in,
                           const int *positions, void *r_prime_out, void *q_out, void *k_out, void *v_out, int M,
                           frt_stream_t stream);

/*
 * Test/diagnostic: as frt_qkv_forward, and also copy the intermediates q_x
 * [M, d] E4M3 and qkv [M, (Hq + 2 Hkv) hd] BF16 to caller buffers (either
 * may be NULL).  Same kernels.
 */
frt_status frt_qkv_debug_trace(frt_qkv_plan_t plan, int layer, const void *residual_in, const void *hidden_in,
                               const int *positions, void *r_prime_out, void *q_out, void *k_out, void *v_out,
                               void *q_x_out, void *qkv_out, int M, frt_stream_t stream);

/*
 * Test/diagnostic: the GEMM and split + RoPE steps of layer `layer` from
 * caller-supplied E4M3 codes q_x_in [M, d] (device) in place of the norm's
 * output, so that another implementation's codes can feed this library's
 * GEMM; writes q_out, k_out, v_out as frt_qkv_forward does and, if qkv_out is
 * not NULL, the GEMM's BF16 output [M, (Hq + 2 Hkv) hd].  Same kernels.
 * Errors: as frt_qkv_debug_trace.
 */
frt_status frt_qkv_debug_trace_qx(frt_qkv_plan_t plan, int layer, const void *q_x_in, const int *positions,
                                  void *q_out, void *k_out, void *v_out, void *qkv_out, int M, frt_stream_t stream);

/*
 * Test/diagnostic: copy layer `layer`'s fused E4M3 weight [W_q; W_k; W_v]
 * ([(Hq + 2 Hkv) hd, d], as the plan stores it) to a caller device buffer,
 * enqueued on `stream`.  Errors: INVALID_ARG, NOT_READY, CUDA.
 */
frt_status frt_qkv_debug_weights(frt_qkv_plan_t plan, int layer, void *w_qkv, frt_stream_t stream);

/* Synchronise `stream` and report a kernel that gave up a bounded wait
 * (DEVICE_TIMEOUT; the plan's error word is then cleared). */
frt_status frt_qkv_device_status(frt_qkv_plan_t plan, frt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FRT_QKV_H */
