/*
 * frt_ffn.h -- C ABI of the GB300 (sm_103a) FP8 FFN sublayer library
 * (libfrt_ffn.so).
 *
 * The library runs the FP8-quantised pre-norm transformer FFN sublayer,
 * stacked n_layers deep, on one GPU:
 *
 *   A1  r' = bf16(r + h);  y = r' / sqrt(mean(r'^2) + eps) * w_norm;
 *       q_x = E4M3(y / s_x)
 *   A2  [g | u] = bf16((q_x . W_gu^T) * s_x * s_gu)         (FP8 GEMM)
 *   A3  q_h = E4M3(act(g) * u / s_h)   act = GELU(tanh) or SiLU
 *   A4  out = bf16(r' + (q_h . W_down^T) * s_h * s_down)    (FP8 GEMM)
 *
 * Passages (page title, section):
 *   - agentlenshq "flashrt-project/FlashRT" summary, "Main ideas": kernels
 *     for fused residual-norm-quantise and FP8 GEMM bundled into static CUDA
 *     graphs; FP8 weights and activations with per-tensor calibration cached
 *     as JSON.
 *   - itsolotime FlashRT article, 4.1-4.2 (graph capture of a pointer-only
 *     forward, Relaxed capture mode, no allocation during replay), 5.2
 *     (FusedGateUp quantised as one tensor), 7.1 (FP8 path), 7.2 (the FFN
 *     layer loop: norm, gate/up GEMM, gated activation + requantise, down
 *     GEMM, residual add).
 *   - "FlashRT docs/architecture.md": "exec/" (a C ABI execution contract of
 *     Buffer / Graph / Plan), 6 "Calibration Framework" (amax per FP8 GEMM
 *     input; alpha = act_scale x weight_scale baked as host scalars), 7
 *     "CUDA Graph Capture" (pointer-only forward, no allocation in replay).
 *
 * Conventions for every call:
 *   - Tensors are row-major and dense.  BF16 tensors are the 16-bit bfloat16
 *     bit patterns; E4M3 tensors are OCP FP8 E4M3 ("fn") bytes.
 *   - Device pointers are pointers into the current CUDA device's memory and
 *     must be 16-byte aligned; host pointers are ordinary host memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     that take a stream enqueue work on it and return before the GPU has
 *     finished, unless a call says it synchronises.
 *   - No call throws.  Each returns an frt_status; on failure
 *     frt_ffn_last_error() gives a message (per host thread).
 *   - A plan is used from one host thread at a time, and its calls must not
 *     run concurrently on different streams: they share the plan's scratch
 *     buffers.  Order work on different streams with events.
 */
#ifndef FRT_FFN_H
#define FRT_FFN_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct frt_ffn_plan *frt_ffn_plan_t;
typedef void *frt_stream_t; /* cudaStream_t */

typedef enum {
    FRT_OK = 0,
    FRT_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size or layer index */
    FRT_ERR_UNSUPPORTED = 2,    /* shape outside what the kernels support, or wrong GPU */
    FRT_ERR_OOM = 3,            /* a device allocation failed */
    FRT_ERR_NOT_READY = 4,      /* weights not loaded or scales not calibrated/set */
    FRT_ERR_SHAPE = 5,          /* M > M_max */
    FRT_ERR_CAPTURE = 6,        /* stream capture failed, or no graph for this M */
    FRT_ERR_STALE_GRAPH = 7,    /* scales changed after the graph was captured */
    FRT_ERR_CUDA = 8,           /* a CUDA runtime call failed (message has the name) */
    FRT_ERR_DEVICE_TIMEOUT = 9  /* a kernel gave up a bounded wait (see frt_ffn_device_status) */
} frt_status;

typedef enum { FRT_ACT_GEGLU_TANH = 0, FRT_ACT_SWIGLU = 1 } frt_act;

/*
 * Create a plan for a stack of n_layers FFN sublayers of model width d and
 * hidden width ff, gated activation act, at most M_max tokens per call.
 * Allocates, on the current device, the FP8 weight arena (layer-major,
 * [W_gate; W_up] as one [2ff, d] matrix and W_down [d, ff] per layer, the
 * flat concatenated buffers of the itsolotime article, 5.2 "FlatCat"), the
 * BF16 norm weights, and all scratch sized by M_max.  Nothing is allocated
 * later by forward, capture or replay.
 * Requires: d % 128 == 0, ff % 128 == 0, 1 <= M_max <= 65536,
 * 1 <= n_layers <= 4096, a compute-capability 10.3 device.
 * Errors: INVALID_ARG, UNSUPPORTED, OOM, CUDA.  *out is NULL on failure.
 */
frt_status frt_ffn_plan_create(int d, int ff, int act, int M_max, int n_layers, frt_ffn_plan_t *out);

/* Free the plan, its device memory and its captured graphs.  Synchronises
 * the device first.  NULL is accepted. */
frt_status frt_ffn_plan_destroy(frt_ffn_plan_t plan);

/*
 * Step A0 (itsolotime article, 5.2 FusedGateUp + Quant; "scale_into"):
 * quantise one layer's BF16 master weights into the plan's E4M3 arena with
 * per-tensor scales s_gu = amax([W_gate; W_up]) / 448 and
 * s_down = amax(W_down) / 448 (an all-zero tensor gets scale 1).
 * w_norm [d], w_gate [ff, d], w_up [ff, d], w_down [d, ff]: BF16, device,
 * row-major (nn.Linear layout, so every GEMM operand is K-major).  The plan
 * copies what it needs; the caller keeps ownership of its buffers.
 * Synchronises `stream` (the scales are read back to the host).
 * Errors: INVALID_ARG (null/misaligned pointer, layer out of range), CUDA.
 */
frt_status frt_ffn_load_weights(frt_ffn_plan_t plan, int layer, const void *w_norm, const void *w_gate,
                                const void *w_up, const void *w_down, frt_stream_t stream);

/* Flags of frt_ffn_load_weights_ex. */
#define FRT_LOAD_FOLD_NORM 1u

/*
 * frt_ffn_load_weights with options.  flags 0: the same.  FRT_LOAD_FOLD_NORM
 * (itsolotime article, 5.2: the Pi0 spec folds the RMSNorm weight into the
 * fused gate/up weights; the Pi0.5 spec does not): the gate/up weights are
 * quantised as W'[j][k] = W[j][k] * w_norm[k] (the fp32 product of two BF16
 * values, exact), s_gu = amax(W') / 448, and the layer's norm multiplies by
 * ones; the layer computes the same function up to quantisation, with the
 * norm weight inside the GEMM.  Activation scales measured without the fold
 * do not apply to a folded layer: calibrate (or set scales) after loading.
 * Errors: as frt_ffn_load_weights; INVALID_ARG for unknown flags.
 */
frt_status frt_ffn_load_weights_ex(frt_ffn_plan_t plan, int layer, const void *w_norm, const void *w_gate,
                                   const void *w_up, const void *w_down, unsigned flags, frt_stream_t stream);

/*
 * Step A6 ("FlashRT docs/architecture.md", 6 Calibration Framework: amax per
 * FP8 GEMM input; "What happens when you call model.predict": run one
 * forward and record amax).  Progressive, layer by layer: for layer l the
 * amax of y over all batches gives s_x[l] = amax / 448; the batches are then
 * quantised with it and run through the gate/up GEMM and activation, whose
 * amax gives s_h[l]; the batches are finished with s_h[l] and become the
 * inputs of layer l + 1.  residual[b] and hidden[b] (hidden may be NULL, or
 * may hold NULL entries) are n_batches host arrays of device pointers to BF16
 * [M, d]; hidden is added at layer 0 only.  Needs all layers' weights.
 * Allocates temporary device memory for the batches' running residuals and
 * frees it before returning; synchronises `stream`.  Marks captured graphs
 * stale.  Errors: INVALID_ARG, NOT_READY, SHAPE, OOM, CUDA, DEVICE_TIMEOUT.
 */
frt_status frt_ffn_calibrate(frt_ffn_plan_t plan, const void *const *residual, const void *const *hidden,
                             int n_batches, int M, frt_stream_t stream);

/* Copy the scales to host arrays of n_layers floats each (any may be NULL).
 * s_x, s_h are 0 until calibrated or set.  Errors: INVALID_ARG. */
frt_status frt_ffn_get_scales(frt_ffn_plan_t plan, float *s_x, float *s_h, float *s_gu, float *s_down);

/* Set the activation scales (e.g. from a calibration cache) from host arrays
 * of n_layers positive finite floats.  Graphs captured before are stale: their
 * alpha values are baked in ("FlashRT docs/architecture.md", 6).
 * Errors: INVALID_ARG. */
frt_status frt_ffn_set_scales(frt_ffn_plan_t plan, const float *s_x, const float *s_h);

/*
 * Eager forward through all layers (steps A1..A4 per layer, step A5's stack):
 * residual_in [M, d] BF16 (device), hidden_in [M, d] BF16 or NULL (added at
 * layer 0 only), out [M, d] BF16 (device; may alias residual_in).  0 <= M <=
 * M_max; M == 0 does nothing.  Allocates nothing.
 * Errors: INVALID_ARG, NOT_READY, SHAPE, CUDA (launch errors).  Errors inside
 * kernels surface through frt_ffn_device_status.
 */
frt_status frt_ffn_forward(frt_ffn_plan_t plan, const void *residual_in, const void *hidden_in, void *out, int M,
                           frt_stream_t stream);

/*
 * AdaRMSNorm (itsolotime article, 5.2: the Pi0.5 spec modulates through
 * AdaRMSNorm Dense layers instead of a norm weight).  mod: host array of
 * n_layers device pointers, each to mod_rows rows of [scale | shift | gate]
 * (3d BF16 values a row, row-major; the Dense layers' outputs, computed by the
 * caller); mod_rows = 1 (one row for every token: per-sample conditioning)
 * or M_max (row m for token m).  While set, every layer's norm computes
 * y = (r' / sqrt(mean(r'^2) + eps)) * (1 + scale) + shift (the norm weight is
 * not used) and its down GEMM's epilogue out = bf16(r' + gate * (acc *
 * alpha_d)), each operation in fp32 in that order.  The plan keeps the
 * pointers: the buffers must stay valid, and may be rewritten between calls
 * (captured graphs read them at replay).  Calibrate after setting it (the
 * activation scales depend on it).  mod == NULL returns to the plain norm.
 * Marks captured graphs stale.  Errors: INVALID_ARG.
 */
frt_status frt_ffn_set_modulation(frt_ffn_plan_t plan, const void *const *mod, int mod_rows);

/*
 * Capture the forward for token count M into a CUDA graph owned by the plan
 * (itsolotime article, 4.1: cudaStreamBeginCapture in Relaxed mode on this
 * stream only; 4.2: stable pointers, no allocation).  The pointers are baked
 * into the graph; replay reads and writes the same buffers.  `stream` must be
 * a non-default stream that is not capturing.  Replaces a graph already held
 * for this M.  Errors: INVALID_ARG, NOT_READY, SHAPE, CAPTURE, CUDA.
 */
frt_status frt_ffn_graph_capture(frt_ffn_plan_t plan, const void *residual_in, const void *hidden_in, void *out,
                                 int M, frt_stream_t stream);

/* Launch the graph captured for M on `stream` (one cudaGraphLaunch).
 * Errors: CAPTURE (no graph for M), STALE_GRAPH (scales changed since the
 * capture), CUDA. */
frt_status frt_ffn_graph_replay(frt_ffn_plan_t plan, int M, frt_stream_t stream);

/*
 * Tactic-stable capture ("FlashRT docs/architecture.md", 7 Graph: re-capture
 * up to N times and keep the fastest schedule).  Captures the forward for M
 * n_tries times as frt_ffn_graph_capture does, cycling through the schedules
 * below (each gives the same results bit for bit), times n_replays replays of
 * each capture (CUDA events on `stream`, each replay timed alone, after one
 * untimed replay; the median counts), and keeps the fastest capture as the
 * plan's graph for M.  Schedules: 0 the defaults, 1 split-K partials
 * exchanged through global memory instead of inside a cluster, 2 single-CTA
 * tiles instead of CTA pairs (many tokens), 3 no programmatic dependent
 * launch.  The timed replays run the forward, so `out` holds its result
 * afterwards.  *best_us and *best_tactic (either may be NULL) receive the kept
 * graph's median replay time in microseconds and its schedule.  Synchronises
 * `stream`.  1 <= n_tries <= 64, 1 <= n_replays <= 10000.  Errors: as
 * frt_ffn_graph_capture, INVALID_ARG for the counts, CUDA for a failed replay
 * or timing.
 */
frt_status frt_ffn_graph_autotune(frt_ffn_plan_t plan, const void *residual_in, const void *hidden_in, void *out,
                                  int M, int n_tries, int n_replays, float *best_us, int *best_tactic,
                                  frt_stream_t stream);

/*
 * Measurement: where the time of a graph replay goes, kernel by kernel,
 * inside the stack ("FlashRT docs/architecture.md", 7: the replayed graph is
 * the unit that runs).  Captures the forward for M again, on the buffers of
 * the graph held for M, with every launch recording %globaltimer at its
 * CTAs' starts and ends; replays it n_replays times (synchronising after
 * each); and writes to kernel_us[k] the median over replays of launch k's
 * share of the replay: from its first CTA's start, or its predecessor's end
 * if later, to its last CTA's end -- so the shares of consecutive launches
 * that overlap (programmatic dependent launch) do not overlap, and they sum
 * to at most the replay's span.  Launch k = 3 l + s for layer l and step s
 * (0 norm + quantise, 1 gate/up GEMM with the gated activation, 2 down GEMM
 * with the residual) -- or, where the forward for M is the one persistent
 * stack launch (frt_ffn_uses_stack_kernel), that launch alone (k = 0);
 * *n_kernels (may be NULL) receives how many were written (kernel_us must
 * hold 3 n_layers floats).  The profiling graph is freed
 * before returning; the graph held for M is unchanged.  Synchronises.
 * Errors: INVALID_ARG, CAPTURE (no graph for M), STALE_GRAPH, CUDA,
 * DEVICE_TIMEOUT.
 */
frt_status frt_ffn_graph_profile(frt_ffn_plan_t plan, int M, int n_replays, float *kernel_us, int *n_kernels,
                                 frt_stream_t stream);

/*
 * 1 if the forward for M tokens runs as one persistent kernel over the whole
 * stack, else 0 (then three launches per layer).  That kernel takes at most
 * 64 tokens when it was asked for (FRT_FFN_STACK=1 in the environment at
 * plan creation; off by default: on GB300 it measured slower than the
 * per-layer kernels), d is 256, 512, 1024 or 2048, ff a multiple of 128, the
 * norm unmodulated (no frt_ffn_set_modulation), and its (ff/128) x (d/256)
 * CTAs -- clusters of d/256, one CTA per SM -- fit on the GPU at once.  It
 * computes the same steps with a different fp32 summation order (the
 * gate/up sum in four K-slices, the down sum in ff/128 K-slices), so its
 * results equal the per-layer kernels' within rounding, not bit for bit.
 */
int frt_ffn_uses_stack_kernel(frt_ffn_plan_t plan, int M);

/*
 * Test/diagnostic: the forward through the persistent stack kernel
 * (frt_ffn_uses_stack_kernel(plan, M) must be 1) with optional per-layer
 * inputs and dumps, all device buffers, each may be NULL.  Inputs, so that
 * another implementation's values can feed the kernel at every layer:
 * q_x_in [L][M][d] E4M3 -- layer l's GEMMs read these codes instead of its
 * own step A1 result (which is still computed and dumped); res_in [L][M][d]
 * BF16 -- layer l >= 1 starts from res_in[l] (its norm's input and its
 * residual) instead of layer l-1's output (row 0 unused).  Dumps: q_x
 * [L][M][d] E4M3, gu [L][M][2ff] BF16 (g then u, the sums rounded to BF16
 * before the activation), q_h [L][M][ff] E4M3, layer_out [L][M][d] BF16 (each
 * layer's computed output), times [CTAs][L][32] uint64 (%globaltimer
 * nanoseconds at fixed points of each layer in each CTA: 0-12 and 16-25 the
 * compute warps' phases, 13-15 the MMA issuer's waits; CTAs = (ff/128)
 * (d/256)).
 * out as frt_ffn_forward.  Errors: as frt_ffn_forward; UNSUPPORTED when the
 * stack kernel does not take M.
 */
frt_status frt_ffn_debug_stack(frt_ffn_plan_t plan, const void *residual_in, const void *hidden_in, void *out,
                               int M, const void *q_x_in, const void *res_in, void *q_x, void *gu, void *q_h,
                               void *layer_out, void *times, frt_stream_t stream);

/*
 * Test/diagnostic: run layer `layer` alone on residual_in (+ hidden_in if not
 * NULL) and copy its intermediates to caller device buffers (each may be
 * NULL): r_prime [M, d] BF16, q_x [M, d] E4M3, gu [M, 2ff] BF16 (g then u),
 * q_h [M, ff] E4M3, out [M, d] BF16.  Runs the same kernels as the forward
 * for this M.  Errors: as frt_ffn_forward.
 */
frt_status frt_ffn_debug_trace(frt_ffn_plan_t plan, int layer, const void *residual_in, const void *hidden_in,
                               int M, void *r_prime, void *q_x, void *gu, void *q_h, void *out, frt_stream_t stream);

/*
 * Test/diagnostic: steps A2..A4 of layer `layer` from caller-supplied step-A1
 * results, so that another implementation's q_x codes (e.g. a reference
 * model's) can feed this library's GEMMs: r_prime [M, d] BF16 (the residual
 * the down GEMM adds) and q_x [M, d] E4M3 (device).  Outputs, each optional
 * (NULL) except out: gu [M, 2ff] BF16 (g then u), q_h [M, ff] E4M3, out
 * [M, d] BF16.  Runs the forward's gate/up and down kernels for this M.
 * Errors: as frt_ffn_debug_trace.
 */
frt_status frt_ffn_debug_trace_qx(frt_ffn_plan_t plan, int layer, const void *r_prime, const void *q_x, int M,
                                  void *gu, void *q_h, void *out, frt_stream_t stream);

/*
 * Test/diagnostic: copy layer `layer`'s E4M3 weights as the plan stores them
 * (step A0's output) to caller device buffers (either may be NULL):
 * w_gu [2ff, d], the gate and up rows interleaved in blocks of 64 -- stored
 * row 128 b + i holds W_gate row 64 b + i and row 128 b + 64 + i holds W_up
 * row 64 b + i (0 <= i < 64) -- and w_down [d, ff].  Enqueued on `stream`.
 * Errors: INVALID_ARG, NOT_READY (layer not loaded), CUDA.
 */
frt_status frt_ffn_debug_weights(frt_ffn_plan_t plan, int layer, void *w_gu, void *w_down, frt_stream_t stream);

/*
 * Test/diagnostic: codes[i] = E4M3 encoding of the fp32 value whose bit
 * pattern is start + i, for 0 <= i < n, by the conversion every quantising
 * kernel of this library uses (round to nearest even, saturating to +-448;
 * steps A1, A3 and A0).  Lets a test sweep all 2^32 fp32 patterns against a
 * reference encoder.  codes: device, 16-byte aligned, n bytes; n % 8 == 0,
 * start + n <= 2^32.  Enqueued on `stream`.  Errors: INVALID_ARG, CUDA.
 */
frt_status frt_debug_e4m3_encode_range(unsigned start, unsigned long long n, void *codes, frt_stream_t stream);

/*
 * Diagnostics (timing single kernels): launch step `step` of layer `layer`
 * alone, for M tokens, on the plan's own scratch buffers (whatever they hold):
 * 0 = A1 residual+RMSNorm+quantise, 1 = A2 gate/up GEMM with A3 (gated
 * activation + requantise) in its epilogue, 2 = A4 down GEMM + residual.  No
 * programmatic dependency on earlier work.  Errors: INVALID_ARG, NOT_READY,
 * SHAPE, CUDA.
 */
frt_status frt_ffn_debug_step(frt_ffn_plan_t plan, int layer, int step, int M, frt_stream_t stream);

/*
 * Synchronise `stream` and report kernel-side failures: DEVICE_TIMEOUT if a
 * kernel of this plan gave up a bounded wait since the last call (the flag is
 * then cleared), else OK.  Errors: CUDA.
 */
frt_status frt_ffn_device_status(frt_ffn_plan_t plan, frt_stream_t stream);

/*
 * Test hook for the failure path (no counterpart in the pages): launch one
 * small GEMM of the plan's kernels on the plan's scratch whose MMA thread
 * first waits for a barrier phase that nothing completes.  The bounded wait
 * gives up after about 2 s, sets the plan's error word, and every role of the
 * kernel drains its copies, frees its tensor memory and exits; the call then
 * returns what frt_ffn_device_status reports -- DEVICE_TIMEOUT -- and the
 * plan (and the CUDA context) stay usable.  Overwrites the plan's split-K
 * workspace.  Errors: INVALID_ARG, CUDA.
 */
frt_status frt_ffn_debug_stall(frt_ffn_plan_t plan, frt_stream_t stream);

/*
 * Test/diagnostic: the plan's FP8 GEMM kernels on caller buffers,
 * C[m][n] = alpha * sum_k A[m][k] B[n][k] stored as fp32 (the contraction of
 * steps A2/A4, itsolotime article 7.2).  A [M, K] and B [N, K] E4M3 (device,
 * K-major, 16-byte aligned), C [M, N] fp32 (device).  path: 0 = pick as the
 * forward does, 1 = weight-streaming (B rows on the MMA's 128-row side, the M
 * tokens on its narrow side; M <= 64), 2 = tiled (128 x 256 or 128 x 128
 * tiles).  splits: 0 = pick, else the split-K factor.  Uses the plan's
 * split-K workspace and error word.  Requires K % 16 == 0, N % 128 == 0,
 * 1 <= M <= 65536, 16 <= K.  Synchronises nothing.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
frt_status frt_fp8_gemm(frt_ffn_plan_t plan, const void *A, const void *B, void *C, int M, int N, int K,
                        float alpha, int path, int splits, frt_stream_t stream);

/* Message of the last failed call on this host thread ("" if none). */
const char *frt_ffn_last_error(void);

/*
 * FP8 GEMM that allocates nothing.  The pages have no counterpart: this entry
 * point is for callers that cannot call cudaMalloc -- code running while a
 * CUDA graph is captured in global mode, embedded or real-time hosts that
 * forbid allocation after start-up, hosts that give all device memory to
 * their own pool.  It computes what frt_fp8_gemm computes with path 0 and
 * splits 0, C[m][n] = alpha * sum_k A[m][k] B[n][k] as fp32, with A [M, K],
 * B [N, K] E4M3 and C [M, N] fp32 (device, 16-byte aligned, K-major), on the
 * same kernels, but needs no plan: its split-K workspace and counters live in
 * one fixed array of 5 MiB + 136 KiB in this library's device memory, which
 * every GPU that loads the library holds until the process exits.
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress, once per device, with the device current); make
 *     that first call before any stream capture.
 *   - Every call clears the split-K counters on `stream` and then launches;
 *     no call allocates or frees.  Calls share the array, which keeps the
 *     last call's contents: calls that overlap on the GPU (different streams,
 *     different host threads) race and must be ordered by the caller.
 *   - A kernel that gives up a bounded wait (about 2 s) leaves C incomplete
 *     and sets an error word in the array; the call that launched it has
 *     already returned FRT_OK.  frt_fp8_gemm_noalloc_status reports it.
 *   - Shapes whose split-K workspace would exceed the array are rejected
 *     with FRT_ERR_UNSUPPORTED before anything is launched.
 *   - The first call's set-up is safe to race from several host threads.
 * Requires 1 <= M <= 65536, N % 128 == 0, K >= 16, K % 16 == 0.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA; the message comes from
 * frt_fp8_gemm_noalloc_last_error().
 */
frt_status frt_fp8_gemm_noalloc(const void *A, const void *B, void *C, int M, int N, int K, float alpha,
                                frt_stream_t stream);

/*
 * Synchronise `stream` and report whether an allocation-free GEMM on the
 * current device gave up a bounded wait since the last report:
 * FRT_ERR_DEVICE_TIMEOUT (its C is incomplete; the error word and the
 * split-K counters are then cleared, synchronously), else FRT_OK.  Not for
 * use while `stream` is being captured.  Allocates nothing.
 * Errors: CUDA, DEVICE_TIMEOUT.
 */
frt_status frt_fp8_gemm_noalloc_status(frt_stream_t stream);

/*
 * Test hook for that failure path (no counterpart in the pages): launch one
 * small GEMM on the fixed array whose MMA thread first waits for a barrier
 * phase that nothing completes; the wait gives up after about 2 s and every
 * role of the kernel drains and exits.  Returns what
 * frt_fp8_gemm_noalloc_status then reports: DEVICE_TIMEOUT.  Overwrites the
 * array's workspace.  Errors: CUDA, DEVICE_TIMEOUT.
 */
frt_status frt_fp8_gemm_noalloc_debug_stall(frt_stream_t stream);

/* Message of the last failed frt_fp8_gemm_noalloc* call on this host thread. */
const char *frt_fp8_gemm_noalloc_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FRT_FFN_H */
