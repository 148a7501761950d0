/*
 * attn_block.h - C ABI of the attention half of a Grok-1 decoder layer on
 * NVIDIA B300 (sm_103a): pre-attention RMSNorm, grouped-query attention with
 * rotary position embeddings and clamped logits, output projection,
 * post-attention RMSNorm and the residual add.  Together with moe_layer.h it
 * makes one whole decoder layer.
 *
 * For one causal sequence x [T, d] at positions 0..T-1, every token t:
 *
 *   xn     = x_t / sqrt(mean(x_t^2) + eps) * s_pre
 *   q_h    = RoPE_t((Wq xn)_h),  k_g,j = RoPE_j((Wk xn_j)_g),  v_g,j = (Wv xn_j)_g
 *   s_h,j  = clamp(<q_h, k_g,j> / sqrt(128), -c, c)   for j <= t,  g = h / (Hq / Hkv)
 *   ctx_h  = sum_j softmax_j(s_h) v_g,j
 *   o      = Wo concat_h ctx_h
 *   y_t    = x_t + o / sqrt(mean(o^2) + eps) * s_post
 *
 * with RoPE_t rotating each pair (2i, 2i + 1) of a 128-value head by the angle
 * t * base^(-2i / 128).
 *
 * Sources (page title, section): "Jah-yee/grok" README, architecture diagram
 * (GQA with 48 query and 8 key/value heads, rotary embeddings, RMSNorm) and its
 * references (Su et al., RoFormer, for the rotary embedding);
 * "TevunahAi/Grok-1-BF16" model card, "Grok-1 Specific Behaviors" (attention
 * logits hard-clamped to [-30, 30] before the softmax; pre- and post-attention
 * norms among the four norms of a layer) and "Weight Verification" (q_proj
 * [6144, 6144], k_proj and v_proj [1024, 6144], o_proj [6144, 6144] in PyTorch
 * [out, in] order, hence heads of 128).
 *
 * Conventions: as in moe_layer.h (status codes, device/host pointers, 16-byte
 * alignment, streams passed as void*, errors found on the device latched in
 * the handle and reported by attn_block_sync_status, moe_last_error_message
 * for the last error on the calling thread).
 */
#ifndef ATTN_BLOCK_H
#define ATTN_BLOCK_H

#include <stddef.h>
#include <stdint.h>

#include "moe_layer.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t d_model;     /* d: multiple of 256 (Grok-1: 6144) */
  int32_t n_q_heads;   /* Hq: query heads (Grok-1: 48); Hq * 128 a multiple of 256 */
  int32_t n_kv_heads;  /* Hkv: key/value heads (Grok-1: 8); divides Hq */
  int32_t head_dim;    /* must be 128 */
  int32_t max_tokens;  /* largest T any forward call will pass (1 .. 65536); sizes the workspace */
  float eps;           /* RMSNorm epsilon (1e-5) */
  float rope_base;     /* rotary base (10000) */
  float logit_clamp;   /* c of the clamp to [-c, c]; 0 < c <= 40 (Grok-1: 30) */
} attn_config_t;

typedef struct {
  const void* wq;       /* DEVICE bf16 [Hq * 128, d]   q_proj, [out, in] */
  const void* wk;       /* DEVICE bf16 [Hkv * 128, d]  k_proj */
  const void* wv;       /* DEVICE bf16 [Hkv * 128, d]  v_proj */
  const void* wo;       /* DEVICE bf16 [d, Hq * 128]   o_proj */
  const float* s_pre;   /* DEVICE fp32 [d] pre-attention RMSNorm scale */
  const float* s_post;  /* DEVICE fp32 [d] post-attention RMSNorm scale */
} attn_weights_t;

typedef struct attn_block attn_block_t;

/* Validate the configuration, copy Wq, Wk and Wv into one [(Hq + 2 Hkv) 128, d]
 * matrix owned by the handle (the caller may free its copies afterwards),
 * borrow wo, s_pre and s_post (they must stay valid until attn_block_destroy),
 * allocate the workspace for max_tokens and fill the rotation table.
 * Synchronises the current device once.  On error *out is NULL. */
moe_status_t attn_block_create(const attn_config_t* cfg, const attn_weights_t* weights, attn_block_t** out);

/* y = attention block of the causal sequence x.  x: DEVICE bf16 [T, d];
 * y: DEVICE bf16 [T, d] (may not alias x).  1 <= T <= max_tokens.  Enqueues six
 * kernels on `stream` and returns without waiting; calls on one handle must be
 * ordered (the workspace is reused). */
moe_status_t attn_block_forward(attn_block_t* block, const void* x, void* y, int32_t T, void* stream);

/* Synchronise `stream` and report (then clear) any error latched on the
 * device: MOE_ERR_TIMEOUT when a bounded wait of a kernel ran out. */
moe_status_t attn_block_sync_status(attn_block_t* block, void* stream);

/* Kernels of one forward, in launch order (indices of the profile arrays). */
typedef enum {
  ATTN_K_PRENORM = 0,   /* pre-attention RMSNorm (bf16 rows) */
  ATTN_K_QKV = 1,       /* q/k/v projections, one tensor-core GEMM */
  ATTN_K_ROPE = 2,      /* rotary embedding of q and k, per-head layouts, V transposed */
  ATTN_K_ATTN = 3,      /* causal attention with the logit clamp (tensor cores) */
  ATTN_K_OPROJ = 4,     /* output projection, tensor-core GEMM */
  ATTN_K_POST = 5,      /* post-attention RMSNorm + residual */
  ATTN_K_COUNT = 6
} attn_kernel_id_t;

/* Per-kernel timing with CUDA events recorded on the forward's stream around
 * every launch while enabled (off by default; a host-side switch).  profile_read
 * synchronises on the recorded events and returns the summed device time in ms
 * (ms_total[ATTN_K_COUNT]) and the number of timed launches
 * (launches[ATTN_K_COUNT]) since the last reset.  Either array may be NULL. */
moe_status_t attn_block_set_profiling(attn_block_t* block, int32_t enable);
moe_status_t attn_block_profile_read(attn_block_t* block, double* ms_total, int64_t* launches, int32_t reset);

/* Launches attn_block_forward makes per call (for counting). */
int32_t attn_block_launch_count(const attn_block_t* block);

/* Free the workspace and the owned q/k/v copy.  NULL is a no-op. */
moe_status_t attn_block_destroy(attn_block_t* block);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BLOCK_H */
