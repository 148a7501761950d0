/*
 * moe_layer.h - C ABI of the Grok-1 top-2-of-8 Mixture-of-Experts feed-forward
 * layer on NVIDIA B300 (sm_103a).
 *
 * The layer, per token t (hidden state x_t of d_model values):
 *
 *   xn    = RMSNorm_pre(x_t)                 = x_t / sqrt(mean(x_t^2) + eps) * s_pre
 *   p     = softmax(G xn + b)                  G [E, d] router gate, b optional
 *   i0,i1 = the two largest p, ties to the lower index; weights p_i0, p_i1 (not
 *           renormalised)
 *   o_r   = W1_e (GELU_tanh(W_e xn) * (Wv_e xn)),  e = i_r
 *   y_t   = x_t + RMSNorm_post(p_i0 o_0 + p_i1 o_1)
 *
 * Sources (page title, section): "Jah-yee/grok" README, architecture diagram
 * (8 experts, top-2, GELU(x W) (*) (x Wv) then the output projection, RMSNorm);
 * "Grok-1: 314B Total Parameters, 25B Active Per Token (MoE Explained)"
 * (oneruby-dev blog), "Expert Routing Details" (softmax of the
 * gate logits, then top_k(k=2) of the softmax outputs) and "How MoE Works in
 * Practice" (gate-weighted sum of the expert outputs); "TevunahAi/Grok-1-BF16"
 * model card, "Grok-1 Specific Behaviors" (pre-MoE and post-MoE norms),
 * "Weight Verification" (tensor shapes, PyTorch [out, in] order) and
 * "Conversion Details" (int8 weights with bf16 scales).
 *
 * Conventions for every entry point:
 *  - Device pointers are CUDA global-memory addresses on the device that was
 *    current when the handle was created; host pointers are ordinary CPU memory.
 *    Each argument's comment says which.  All must be 16-byte aligned.
 *  - A stream argument is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).
 *  - Argument errors are returned synchronously, before anything is enqueued.
 *    Errors found on the device (a bounded wait that ran out, an index check of
 *    MOE_FLAG_DEVICE_CHECKS) are latched in the handle and reported by
 *    moe_layer_sync_status().  No kernel of this library traps or spins without
 *    a limit.
 *  - moe_last_error_message() gives a one-line description of the last error
 *    returned on the calling thread.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, T out of range, bad config value */
  MOE_ERR_UNSUPPORTED = 2,  /* shape or dtype this build does not implement */
  MOE_ERR_OOM = 3,          /* workspace allocation failed in moe_layer_create */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed */
  MOE_ERR_DEVICE_CHECK = 5, /* a device-side check failed (MOE_FLAG_DEVICE_CHECKS): an index out of
                               range, or an int8 layer's fp16 activation past +-65504 (saturated) */
  MOE_ERR_TIMEOUT = 6       /* a bounded device wait ran out; the kernel returned early */
} moe_status_t;

typedef enum { MOE_WEIGHT_BF16 = 0, MOE_WEIGHT_INT8 = 1 } moe_weight_dtype_t;

/* Bits of moe_config_t.flags */
#define MOE_FLAG_DEVICE_CHECKS 0x1u /* kernels validate routing indices and row maps; int8 layers
                                      also report fp16 saturation of their activations */
#define MOE_FLAG_FORCE_TC 0x2u      /* always use the tensor-core grouped GEMM path */
#define MOE_FLAG_FORCE_GEMV 0x4u    /* always use the weight-streaming decode path */
#define MOE_FLAG_DECODE_TC 0x8u     /* int8 weights at T <= 16: run the tensor-core weight-streaming
                                      kernels instead of the CUDA-core GEMV kernels */

typedef struct {
  int32_t d_model;      /* d: multiple of 128 (Grok-1: 6144) */
  int32_t d_ffn;        /* F: multiple of 128 (Grok-1: 32768) */
  int32_t num_experts;  /* E: must be 8 */
  int32_t top_k;        /* must be 2 */
  int32_t max_tokens;   /* largest T any forward call will pass (>= 1); sizes the workspace */
  float eps;            /* RMSNorm epsilon (Grok-1 configs: 1e-5) */
  int32_t weight_dtype; /* moe_weight_dtype_t */
  uint32_t flags;       /* MOE_FLAG_* */
  /* int8 only: logical scale shape (scale_experts, scale_groups, N) of every
   * expert weight ("TevunahAi/Grok-1-BF16", "Conversion Details": (8,1,N),
   * (8,8,N), (1,N), (8,N); the last two read as (1,1,N) and (1,8,N)).
   * scale_experts: 8 = one scale set per expert, 1 = one set shared by all
   * experts (0 means 8).  scale_groups: G groups along each weight's input
   * dimension, group g covering inputs [g K/G, (g+1) K/G) (0 means 1).  G > 1
   * needs d and F to be multiples of 128 G.  With G == 1 the scale multiplies
   * the fp32 result of the reduction (exact); with G > 1 it multiplies each
   * weight as it is converted on chip, rounded once to bf16 (fp16 on the T <= 16
   * tensor-core path), or, on the T <= 16 CUDA-core GEMV path, each integer
   * block sum in fp32. */
  int32_t scale_experts;
  int32_t scale_groups;
} moe_config_t;

/*
 * Layer parameters.  DEVICE pointers, BORROWED: the caller keeps them alive and
 * unchanged for the life of the handle (the library keeps TMA descriptors that
 * point into them).  Layouts are row-major, PyTorch [out, in] order for the
 * expert matrices ("TevunahAi/Grok-1-BF16", "Weight Verification").
 */
typedef struct {
  const float* gate;            /* [E, d] fp32 router gate (moe_block.gate.weight) */
  const float* gate_bias;       /* [E] fp32 added to the logits, or NULL for none */
  const void* w;                /* [E, F, d] bf16 or int8: GELU branch ("linear") */
  const void* wv;               /* [E, F, d] bf16 or int8: linear branch ("linear_v") */
  const void* w1;               /* [E, d, F] bf16 or int8: down projection ("linear_1") */
  const uint16_t* w_scale;      /* int8 only: bf16 bits [scale_experts, scale_groups, F] (per expert,
                                   group and output channel); NULL for bf16 */
  const uint16_t* wv_scale;     /* int8 only: bf16 bits [scale_experts, scale_groups, F] */
  const uint16_t* w1_scale;     /* int8 only: bf16 bits [scale_experts, scale_groups, d] */
  const float* pre_norm_scale;  /* [d] fp32 (pre_moe_norm.scale) */
  const float* post_norm_scale; /* [d] fp32 (post_moe_norm.scale) */
} moe_weights_t;

typedef struct moe_layer moe_layer_t;

/*
 * Validate cfg, take the borrowed weight pointers, build the TMA descriptors and
 * allocate the workspace for cfg->max_tokens tokens on the current device.
 * Launches no kernel.  On success *out receives the handle (owned by the caller,
 * freed by moe_layer_destroy).  Errors: MOE_ERR_INVALID_ARG (null / misaligned
 * pointer, max_tokens < 1, eps <= 0, int8 without scales, scale_experts not in
 * {0, 1, 8}), MOE_ERR_UNSUPPORTED (E != 8, top_k != 2, d or F not a multiple of
 * 128, d > 16384, scale_groups > 1 with d or F not a multiple of 128 G, device
 * not sm_103), MOE_ERR_OOM, MOE_ERR_CUDA.
 */
moe_status_t moe_layer_create(const moe_config_t* cfg, const moe_weights_t* weights, moe_layer_t** out);

/*
 * The layer on T tokens, asynchronous on `stream`.
 *   hidden        DEVICE [T, d] bf16, read only
 *   out           DEVICE [T, d] bf16, written; may equal `hidden` (in place)
 *   T             0 <= T <= max_tokens; T == 0 enqueues nothing
 *   topk_idx      DEVICE [T, 2] int32 or NULL: chosen experts in rank order
 *   topk_prob     DEVICE [T, 2] fp32 or NULL: their softmax probabilities
 *   expert_counts DEVICE [E] int32 or NULL: tokens routed to each expert
 * The host never waits on the device and reads nothing back, so the call may be
 * captured in a CUDA graph.  Calls on one handle must not overlap on the device
 * (they share the workspace): issue them on one stream, or order the streams.
 */
moe_status_t moe_layer_forward(moe_layer_t* layer, const void* hidden, void* out, int32_t T, void* stream,
                               int32_t* topk_idx, float* topk_prob, int32_t* expert_counts);

/*
 * Same layer, HOST buffers: copies hidden_host to the device, runs the layer
 * and copies the results back, then waits for `stream`.  Synchronous.
 *   hidden_host   HOST [T, d] bf16 (pinned memory gives full copy bandwidth)
 *   out_host      HOST [T, d] bf16
 *   topk_idx_host HOST [T, 2] int32 or NULL; topk_prob_host HOST [T, 2] fp32 or
 *   NULL; expert_counts_host HOST [E] int32 or NULL.
 * Uses a device staging area of the handle (allocated on first use).  Returns
 * device-side errors directly (it synchronises).
 */
moe_status_t moe_layer_forward_host(moe_layer_t* layer, const void* hidden_host, void* out_host, int32_t T,
                                    void* stream, int32_t* topk_idx_host, float* topk_prob_host,
                                    int32_t* expert_counts_host);

/*
 * Same as moe_layer_forward_host, but asynchronous, so that a caller serving a
 * stream of batches overlaps the copies of one call with the layer of another.
 * The input copy runs on an internal copy stream, the layer on `stream` (after
 * the input landed), and the output copies on a second internal copy stream.
 * Two device staging slots are used in turn (allocated with the copy streams
 * on the first call): a call reuses a slot only after the output copies of the
 * call two before it finished.  The host buffers must stay untouched until
 * moe_layer_host_wait returns (pinned memory is needed for the copies to
 * overlap anything).  Argument errors return at once; device errors are
 * reported by moe_layer_host_wait.
 */
moe_status_t moe_layer_forward_host_async(moe_layer_t* layer, const void* hidden_host, void* out_host, int32_t T,
                                          void* stream, int32_t* topk_idx_host, float* topk_prob_host,
                                          int32_t* expert_counts_host);

/* Wait for every moe_layer_forward_host_async call on this handle (their output
 * copies) and for `stream`; then as moe_layer_sync_status. */
moe_status_t moe_layer_host_wait(moe_layer_t* layer, void* stream);

/* Wait for `stream`, then return (and clear) the first device-side error any
 * earlier forward on this handle latched: MOE_OK, MOE_ERR_TIMEOUT,
 * MOE_ERR_DEVICE_CHECK or MOE_ERR_CUDA. */
moe_status_t moe_layer_sync_status(moe_layer_t* layer, void* stream);

/* Free the workspace and the handle.  Waits for the device first.  NULL is a no-op. */
moe_status_t moe_layer_destroy(moe_layer_t* layer);

/* Static string naming a status code. */
const char* moe_status_string(moe_status_t status);

/* One-line detail of the last error returned on this thread ("" if none). */
const char* moe_last_error_message(void);

/*
 * Routing diagnostics of the last forward enqueued on this handle ("Jah-yee/grok"
 * README: list "New metrics track MoE-specific grokking signals" and the --demo
 * block "[3] MoE routing (layer 0)", which prints a weight per expert and the
 * routing entropy against its maximum).  Enqueued on `stream` (one small kernel);
 * issue it on the forward's stream, after the forward, and before the next
 * forward on this handle (it reads the router's per-CTA partial sums).
 *   stats  DEVICE [10] fp32, written:
 *          stats[0..7] mean router probability of each expert over the T tokens
 *          stats[8]    routing entropy of that mean distribution, in nats (uniform: ln 8 = 2.079)
 *          stats[9]    collapse index 1 - stats[8] / ln 8 (0 uniform, 1 one expert takes all)
 * Token counts per expert come from moe_layer_forward's expert_counts.  Errors:
 * MOE_ERR_INVALID_ARG (null or misaligned pointer, no forward with T > 0 yet).
 */
moe_status_t moe_layer_router_stats(moe_layer_t* layer, float* stats, void* stream);

/* ----------------------------------------------------------- measurement */

/* Kernels of one forward, in launch order (indices of the profiling arrays). */
typedef enum {
  MOE_K_ROUTER = 0,   /* pre-norm statistics + router logits + softmax + top-2 */
  MOE_K_GROUP = 1,    /* per-expert counts, padded offsets, stable slot order, and the
                         normed rows written in expert-contiguous order */
  MOE_K_UP = 2,       /* expert up-projections W, Wv with the GeGLU epilogue */
  MOE_K_DOWN = 3,     /* expert down-projection W1, scaled by the combine weight */
  MOE_K_COMBINE = 4,  /* combine of the two expert rows + post-norm + residual */
  MOE_K_COUNT = 5
} moe_kernel_id_t;

/* Turn per-kernel CUDA-event timing of later forwards on (1) or off (0).
 * Events are recorded on the forward's stream around each kernel. */
moe_status_t moe_layer_set_profiling(moe_layer_t* layer, int32_t enable);

/* Waits for the recorded events and returns, per kernel id, the summed device
 * time in ms (ms_total[MOE_K_COUNT]) and the number of timed launches
 * (launches[MOE_K_COUNT]) since the last reset.  Either array may be NULL.
 * reset != 0 clears the sums afterwards. */
moe_status_t moe_layer_profile_read(moe_layer_t* layer, double* ms_total, int64_t* launches, int32_t reset);

/* Grid sizes (CTAs) of the grouped-GEMM launches this handle makes at large T
 * (T >= 2048; with d_ffn >= 16384 those launches pair two m-blocks per tile):
 * grid[0] up / bf16, grid[1] down / bf16, grid[2] up / int8, grid[3] down / int8.
 * Each is twice the number of CTA pairs that can be resident at once. */
moe_status_t moe_layer_gemm_grid(const moe_layer_t* layer, int32_t grid[4]);

/* Kernel launches enqueued by this handle since creation (all kernels). */
int64_t moe_layer_launch_count(const moe_layer_t* layer);

/* Workspace introspection (DEVICE pointers into the handle's workspace, valid
 * until destroy; contents are those of the last forward once it completed). */
typedef struct {
  float* rnorm;         /* [max_tokens] fp32: 1 / rms of each token's hidden row (the pre-norm's
                           scale; the normed rows themselves exist only in xn_perm) */
  int32_t* counts;      /* [E] tokens per expert */
  int32_t* row_offset;  /* [E + 1] first permuted row of each expert (multiples of 128) */
  int32_t* row_of_slot; /* [max_tokens, 2] permuted row of (token, rank) */
  void* xn_perm;        /* [rows_cap, d] bf16 (fp16 for int8 weights): normed rows in expert order,
                           (x_j r) s_pre_j rounded; zero rows for padding */
  void* act;            /* [rows_cap, F] bf16 (fp16 for int8 weights): GELU(h) * v per permuted row */
  float* y_rows;        /* [rows_cap, d] fp32: p * (W1 act) per permuted row */
  int64_t rows_cap;     /* capacity in permuted rows */
} moe_workspace_view_t;

moe_status_t moe_layer_workspace(const moe_layer_t* layer, moe_workspace_view_t* view);

/* ------------------------------------------------ allocation-free grouping */

/*
 * Groups T tokens' routed slots by expert exactly as moe_layer_forward does
 * internally, without allocating any memory.  The pages have no counterpart:
 * this is for callers that cannot call cudaMalloc, such as a serving runtime
 * that reserved all free device memory for its own pool at start-up or a plugin
 * host that gives an op only its input and output buffers (there cudaMalloc
 * fails or stalls the device mid-step).
 *   topk_idx      DEVICE [T, 2] int32, experts in [0, 8) (e.g. moe_layer_forward's
 *                 topk_idx); an out-of-range index is counted as expert 0 and
 *                 NOT reported: this entry point has no error word to latch it in
 *   topk_prob     DEVICE [T, 2] fp32, their probabilities
 *   T             0 <= T <= 16384 (larger T: MOE_ERR_INVALID_ARG); T == 0 is a no-op
 *   expert_counts DEVICE [8] int32, written: slots per expert
 *   row_of_slot   DEVICE [T, 2] int32, written: row of slot (t, r) when each
 *                 expert's slots are laid out contiguously in token order and
 *                 each expert's block is padded to a multiple of 128 rows
 *   stream        cudaStream_t (as void*), asynchronous
 * Scratch lives in one static device array of 270,592 bytes (about 264 KB) that every GPU
 * loading this library holds until the process exits.  All calls share it, so
 * calls that overlap on the GPU (other streams, other threads) race: order them.
 * The first call on a device looks up the array's device address (a one-time
 * set-up); make that first call before any CUDA stream capture.
 */
moe_status_t moe_group_slots_noalloc(const int32_t* topk_idx, const float* topk_prob, int32_t T,
                                     int32_t* expert_counts, int32_t* row_of_slot, void* stream);

/* Self-test of the bounded waits every kernel of this library uses (no device
 * memory of any layer is touched): one thread of one block waits on an
 * mbarrier phase that nothing completes.  mode 0: the spinning wait (GEMM,
 * decode and grouping kernels); mode 1: the sleeping wait (attention kernel);
 * mode 2: the spinning wait with the abort flag already raised, which must
 * return at once whatever limit_ns is.  limit_ns in [1 ms, 2 s].  Synchronous
 * (synchronises the current device).  Returns MOE_ERR_TIMEOUT when the wait gave
 * up and latched the error word, as it should, with the time it waited in
 * *elapsed_ns (HOST, may be NULL); MOE_ERR_DEVICE_CHECK if the wait returned
 * true or did not latch the error; MOE_ERR_CUDA on a CUDA error.  The GPU
 * context stays usable afterwards. */
moe_status_t moe_selftest_bounded_wait(int32_t mode, uint64_t limit_ns, uint64_t* elapsed_ns);

/* The GELU (tanh approximation; "TevunahAi/Grok-1-BF16" model card, "Grok-1
 * Specific Behaviors": GeGLU experts) that the GeGLU epilogues of the up
 * projections apply, evaluated elementwise: y[i] = GELU(x[i]) for i < n.
 *   x, y    DEVICE float buffers of n elements (caller-owned; y may equal x)
 *   n       >= 0; n = 0 launches nothing
 *   stream  cudaStream_t (as void*), asynchronous
 * Exists so the device GELU can be checked against a reference over a sweep of
 * arguments.  MOE_ERR_INVALID_ARG for n < 0 or a null buffer with n > 0. */
moe_status_t moe_selftest_gelu(const float* x, float* y, int64_t n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYER_H */
