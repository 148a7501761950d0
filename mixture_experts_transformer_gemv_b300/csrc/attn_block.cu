// Host runtime and C ABI of the attention half of a Grok-1 decoder layer
// (declared in include/attn_block.h).
//
// attn_block_create validates the configuration, copies Wq, Wk, Wv into one
// [(Hq + 2 Hkv) 128, d] fp16 matrix so the three projections are one GEMM on the
// precision the logits need (fp16 keeps 3 more mantissa bits than bf16), allocates
// one workspace block, fills the rotation table and encodes the TMA descriptors.
// attn_block_forward enqueues, on the caller's stream and without a host wait:
//   A1 attn_prenorm_kernel   xn = RMSNorm_pre(x) (fp16), padded rows zero; GEMM schedule
//   A2 grouped_gemm<down>    qkv = xn Wqkv^T (fp16 operands, fp32 out)     (tcgen05 pairs)
//   A3 rope_layout_kernel    Q, K rotated (fp16) and V^T (bf16), per-head layouts
//   A4 attn_kernel           ctx = causal softmax(clamp(Q K^T / sqrt(128))) V   (tcgen05)
//   A5 grouped_gemm<down>    o = ctx Wo^T (fp32)                            (tcgen05 pairs)
//   A6 attn_post_kernel      y = x + RMSNorm_post(o)
// The projections reuse the MoE layer's grouped GEMM with a schedule of one
// group holding every row and row scale 1.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstring>
#include <vector>

#include "attn_block.h"
#include "common.cuh"
#include "host_util.h"
#include "k_attn.cuh"
#include "k_gemm.cuh"
#include "k_selftest.cuh"

using namespace moe;
using namespace moe_host;

struct attn_block {
  attn_config_t cfg{};
  int device = 0;
  int num_sms = 0;
  int gemm_grid = 0;
  const void* wo = nullptr;
  const float* s_pre = nullptr;
  const float* s_post = nullptr;
  void* wqkv = nullptr;  // owned [(Hq + 2 Hkv) 128, d] fp16
  int64_t rows_cap = 0;  // rows of the GEMM buffers: max_tokens rounded up to 256
  int64_t t_stride = 0;  // token rows per head of Q / K: max_tokens rounded up to 256
  int n_qkv = 0;         // (Hq + 2 Hkv) 128
  int n_ctx = 0;         // Hq 128
  void* ws = nullptr;
  __half* xn = nullptr;
  float* qkv = nullptr;
  __half* q = nullptr;
  __half* k = nullptr;
  __nv_bfloat16* vt = nullptr;
  __nv_bfloat16* ctx = nullptr;
  float* o = nullptr;
  float* ones = nullptr;
  float2* rope_cs = nullptr;
  int32_t* sched = nullptr;
  uint32_t* err = nullptr;
  CUtensorMap tm_xn{}, tm_wqkv{}, tm_ctx{}, tm_wo{}, tm_q{}, tm_k{}, tm_vt{};
  CUtensorMap tm_xn64{}, tm_ctx64{};  // 64-row A boxes of the GEMM's half tiles (row counts here are
                                      // multiples of 256, so none occur; the maps keep the launch complete)
  // per-kernel event timing (attn_block_set_profiling)
  bool profiling = false;
  std::vector<std::array<cudaEvent_t, ATTN_K_COUNT + 1>> ring;
  std::vector<bool> pending;
  int ring_next = 0;
  double prof_ms[ATTN_K_COUNT] = {};
  int64_t prof_n[ATTN_K_COUNT] = {};
};

namespace {

constexpr int kAttnLaunches = ATTN_K_COUNT;
constexpr int kAttnProfRing = 64;

void harvest(attn_block* B, int slot) {
  if (!B->pending[slot]) return;
  auto& ev = B->ring[slot];
  cudaEventSynchronize(ev[ATTN_K_COUNT]);
  for (int k = 0; k < ATTN_K_COUNT; ++k) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, ev[k], ev[k + 1]) == cudaSuccess) {
      B->prof_ms[k] += ms;
      B->prof_n[k] += 1;
    }
  }
  B->pending[slot] = false;
}

moe_status_t enqueue(attn_block* B, const void* x, void* y, int T, cudaStream_t st) {
  cudaEvent_t* ev = nullptr;
  if (B->profiling) {
    const int slot = B->ring_next;
    B->ring_next = (B->ring_next + 1) % kAttnProfRing;
    harvest(B, slot);
    ev = B->ring[slot].data();
    B->pending[slot] = true;
  }
  auto mark = [&](int k) {
    if (ev) cudaEventRecord(ev[k], st);
  };
  const int d = B->cfg.d_model, Hq = B->cfg.n_q_heads, Hkv = B->cfg.n_kv_heads;
  const int rows_pad = (int)align_up((size_t)T, kGemmBM);
  const int t_pad = (int)align_up((size_t)T, 2 * kAttnBM);  // whole pairs of query tiles
  mark(ATTN_K_PRENORM);
  attn_prenorm_kernel<<<rows_pad, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), B->s_pre, B->cfg.eps, T,
                                                rows_pad, d, B->xn, B->sched);
  mark(ATTN_K_QKV);
  {
    GemmParams p{};
    p.sched = B->sched;
    p.K = d;
    p.n_tiles = B->n_qkv / kGemmBN;
    p.b_rows_per_expert = B->n_qkv;
    p.n_out = B->n_qkv;
    p.out = B->qkv;
    p.row_scale = B->ones;
    p.scale_experts = 1;
    p.scale_groups = 1;
    p.group_kb = 1;
    p.f16_operands = 1;
    p.err = B->err;
    p.timeout_ns = kWaitLimitNs;
    grouped_gemm_kernel<kEpiDown, false><<<B->gemm_grid, kGemmThreads, kGemmSmemBytes, st>>>(
        B->tm_xn, B->tm_wqkv, B->tm_wqkv, B->tm_xn64, B->tm_wqkv, B->tm_wqkv, p);
  }
  mark(ATTN_K_ROPE);
  rope_layout_kernel<<<dim3(t_pad / 32, Hq + 2 * Hkv), 256, 0, st>>>(B->qkv, B->n_qkv, B->rope_cs, T,
                                                                     (int)B->t_stride, Hq, Hkv, B->q, B->k, B->vt);
  mark(ATTN_K_ATTN);
  {
    AttnParams p{};
    p.T = T;
    p.t_stride = (int)B->t_stride;
    p.n_q_heads = Hq;
    p.group = Hq / Hkv;
    p.n_qpairs = t_pad / (2 * kAttnBM);
    const double log2e = 1.4426950408889634;
    p.sat_scale = (float)(1.0 / (2.0 * (double)B->cfg.logit_clamp * std::sqrt((double)kAttnDh)));
    p.clamp2_log2 = (float)(2.0 * (double)B->cfg.logit_clamp * log2e);
    p.ctx = B->ctx;
    p.ctx_ld = B->n_ctx;
    p.err = B->err;
    p.timeout_ns = kWaitLimitNs;
    // persistent: one CTA per SM, each looping over pairs of query tiles
    const int grid = std::min(B->num_sms, p.n_qpairs * Hq);
    attn_kernel<<<grid, kAttnThreads, kAttnSmemBytes, st>>>(B->tm_q, B->tm_k, B->tm_vt, p);
  }
  mark(ATTN_K_OPROJ);
  {
    GemmParams p{};
    p.sched = B->sched;
    p.K = B->n_ctx;
    p.n_tiles = (d + kGemmBN - 1) / kGemmBN;
    p.b_rows_per_expert = d;
    p.n_out = d;
    p.out = B->o;
    p.row_scale = B->ones;
    p.scale_experts = 1;
    p.scale_groups = 1;
    p.group_kb = 1;
    p.err = B->err;
    p.timeout_ns = kWaitLimitNs;
    grouped_gemm_kernel<kEpiDown, false><<<B->gemm_grid, kGemmThreads, kGemmSmemBytes, st>>>(
        B->tm_ctx, B->tm_wo, B->tm_wo, B->tm_ctx64, B->tm_wo, B->tm_wo, p);
  }
  mark(ATTN_K_POST);
  attn_post_kernel<<<T, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), B->o, d, B->s_post, B->cfg.eps, d,
                                      static_cast<__nv_bfloat16*>(y));
  mark(ATTN_K_COUNT);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t attn_block_create(const attn_config_t* cfg, const attn_weights_t* w, attn_block_t** out) {
  if (!cfg || !w || !out) return fail(MOE_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  const attn_config_t c = *cfg;
  if (c.head_dim != kAttnDh) return fail(MOE_ERR_UNSUPPORTED, "head_dim must be 128 (got %d)", c.head_dim);
  if (c.d_model <= 0 || c.d_model % kGemmBN != 0)
    return fail(MOE_ERR_UNSUPPORTED, "d_model must be a positive multiple of 256 (got %d)", c.d_model);
  if (c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.n_q_heads % c.n_kv_heads != 0)
    return fail(MOE_ERR_INVALID_ARG, "n_kv_heads (%d) must divide n_q_heads (%d)", c.n_kv_heads, c.n_q_heads);
  if ((c.n_q_heads * kAttnDh) % kGemmBN != 0 || ((c.n_q_heads + 2 * c.n_kv_heads) * kAttnDh) % kGemmBN != 0)
    return fail(MOE_ERR_UNSUPPORTED, "Hq * 128 and (Hq + 2 Hkv) * 128 must be multiples of 256");
  if (c.max_tokens < 1 || c.max_tokens > 65536)
    return fail(MOE_ERR_INVALID_ARG, "max_tokens=%d outside [1, 65536]", c.max_tokens);
  if (!(c.eps > 0.f) || !(c.rope_base > 1.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be > 0 and rope_base > 1");
  // exp(-2c) must stay a normal fp32 / bf16 number (the kernel subtracts c instead of a running maximum)
  if (!(c.logit_clamp > 0.f) || c.logit_clamp > 40.f)
    return fail(MOE_ERR_UNSUPPORTED, "logit_clamp must be in (0, 40] (got %g)", (double)c.logit_clamp);
  if (!w->wq || !w->wk || !w->wv || !w->wo || !w->s_pre || !w->s_post)
    return fail(MOE_ERR_INVALID_ARG, "null weight pointer");
  if (!aligned16(w->wq) || !aligned16(w->wk) || !aligned16(w->wv) || !aligned16(w->wo) || !aligned16(w->s_pre) ||
      !aligned16(w->s_post))
    return fail(MOE_ERR_INVALID_ARG, "weight pointers must be 16-byte aligned");

  attn_block* B = new attn_block();
  B->cfg = c;
  B->wo = w->wo;
  B->s_pre = w->s_pre;
  B->s_post = w->s_post;
  moe_status_t s = MOE_OK;
  auto bail = [&](moe_status_t st) {
    const std::string msg = g_last_error;
    attn_block_destroy(B);
    g_last_error = msg;
    return st;
  };
  if (cudaGetDevice(&B->device) != cudaSuccess) return bail(fail(MOE_ERR_CUDA, "cudaGetDevice failed"));
  cudaDeviceProp prop{};
  if (cudaGetDeviceProperties(&prop, B->device) != cudaSuccess)
    return bail(fail(MOE_ERR_CUDA, "cudaGetDeviceProperties failed"));
  if (prop.major != 10 || prop.minor != 3)
    return bail(fail(MOE_ERR_UNSUPPORTED, "built for sm_103a; device is sm_%d%d", prop.major, prop.minor));
  B->num_sms = prop.multiProcessorCount;

  const int d = c.d_model, Hq = c.n_q_heads, Hkv = c.n_kv_heads;
  B->n_qkv = (Hq + 2 * Hkv) * kAttnDh;
  B->n_ctx = Hq * kAttnDh;
  B->rows_cap = (int64_t)align_up((size_t)c.max_tokens, kGemmBM);
  B->t_stride = (int64_t)align_up((size_t)c.max_tokens, 2 * kAttnBM);
  const size_t R = (size_t)B->rows_cap, TS = (size_t)B->t_stride;
  const size_t sz_wqkv = (size_t)B->n_qkv * d * 2;
  const size_t sz_xn = align_up(R * d * 2, 256), sz_qkv = align_up(R * B->n_qkv * 4, 256);
  const size_t sz_q = align_up((size_t)Hq * TS * kAttnDh * 2, 256), sz_kv = align_up((size_t)Hkv * TS * kAttnDh * 2, 256);
  const size_t sz_ctx = align_up(R * B->n_ctx * 2, 256), sz_o = align_up(R * d * 4, 256);
  const size_t sz_ones = align_up(R * 4, 256), sz_cs = align_up(TS * (kAttnDh / 2) * 8, 256);
  const size_t total = sz_xn + sz_qkv + sz_q + 2 * sz_kv + sz_ctx + sz_o + sz_ones + sz_cs + 256 + 256;
  if (cudaMalloc(&B->wqkv, sz_wqkv) != cudaSuccess || cudaMalloc(&B->ws, total) != cudaSuccess) {
    cudaGetLastError();
    return bail(fail(MOE_ERR_OOM, "workspace allocation of %zu bytes failed", total + sz_wqkv));
  }
  uint8_t* p = static_cast<uint8_t*>(B->ws);
  auto take = [&](size_t n) {
    uint8_t* r = p;
    p += n;
    return r;
  };
  B->xn = reinterpret_cast<__half*>(take(sz_xn));
  B->qkv = reinterpret_cast<float*>(take(sz_qkv));
  B->q = reinterpret_cast<__half*>(take(sz_q));
  B->k = reinterpret_cast<__half*>(take(sz_kv));
  B->vt = reinterpret_cast<__nv_bfloat16*>(take(sz_kv));
  B->ctx = reinterpret_cast<__nv_bfloat16*>(take(sz_ctx));
  B->o = reinterpret_cast<float*>(take(sz_o));
  B->ones = reinterpret_cast<float*>(take(sz_ones));
  B->rope_cs = reinterpret_cast<float2*>(take(sz_cs));
  B->sched = reinterpret_cast<int32_t*>(take(256));
  B->err = reinterpret_cast<uint32_t*>(take(256));

  const size_t wq_bytes = (size_t)Hq * kAttnDh * d * 2, wkv_bytes = (size_t)Hkv * kAttnDh * d * 2;
  uint8_t* wqkv = static_cast<uint8_t*>(B->wqkv);
  if (cudaMemcpy(wqkv, w->wq, wq_bytes, cudaMemcpyDeviceToDevice) != cudaSuccess ||
      cudaMemcpy(wqkv + wq_bytes, w->wk, wkv_bytes, cudaMemcpyDeviceToDevice) != cudaSuccess ||
      cudaMemcpy(wqkv + wq_bytes + wkv_bytes, w->wv, wkv_bytes, cudaMemcpyDeviceToDevice) != cudaSuccess)
    return bail(fail(MOE_ERR_CUDA, "copy of Wq, Wk, Wv failed: %s", cudaGetErrorString(cudaGetLastError())));
  bf16_to_f16_kernel<<<4 * B->num_sms, 256>>>(static_cast<uint32_t*>(B->wqkv), (int64_t)(sz_wqkv / 4));
  // context rows past T are read by the output projection (and discarded): keep them finite
  if (cudaMemset(B->ctx, 0, sz_ctx) != cudaSuccess || cudaMemset(B->err, 0, 256) != cudaSuccess)
    return bail(fail(MOE_ERR_CUDA, "workspace initialisation failed"));
  fill_f32_kernel<<<(unsigned)((R + 255) / 256), 256>>>(B->ones, 1.f, (int)R);
  const int n_cs = (int)TS * (kAttnDh / 2);
  rope_table_kernel<<<(n_cs + 255) / 256, 256>>>(B->rope_cs, (int)TS, (double)c.rope_base);
  if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
    return bail(fail(MOE_ERR_CUDA, "workspace initialisation kernels failed"));

  if (s == MOE_OK) s = make_tmap_bf16(&B->tm_xn, B->xn, d, R, kGemmHalfM);
  if (s == MOE_OK) s = make_tmap_bf16(&B->tm_wqkv, B->wqkv, d, (uint64_t)B->n_qkv, kGemmHalfN);
  if (s == MOE_OK) s = make_tmap_bf16(&B->tm_ctx, B->ctx, (uint64_t)B->n_ctx, R, kGemmHalfM);
  if (s == MOE_OK) s = make_tmap_bf16(&B->tm_wo, B->wo, (uint64_t)B->n_ctx, d, kGemmHalfN);
  if (s == MOE_OK) s = make_tmap_bf16(&B->tm_xn64, B->xn, d, R, kGemmBoxRows);
  if (s == MOE_OK) s = make_tmap_bf16(&B->tm_ctx64, B->ctx, (uint64_t)B->n_ctx, R, kGemmBoxRows);
  if (s == MOE_OK) s = make_tmap_bf16(&B->tm_q, B->q, kAttnDh, (uint64_t)Hq * TS, kAttnBM);
  if (s == MOE_OK) s = make_tmap_bf16(&B->tm_k, B->k, kAttnDh, (uint64_t)Hkv * TS, kAttnBN);
  if (s == MOE_OK) s = make_tmap_bf16(&B->tm_vt, B->vt, TS, (uint64_t)Hkv * kAttnDh, kAttnDh);
  if (s != MOE_OK) return bail(s);

  if (cudaFuncSetAttribute(grouped_gemm_kernel<kEpiDown, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kGemmSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttnSmemBytes) !=
          cudaSuccess)
    return bail(fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (shared memory) failed"));
  s = cluster_pair_grid(B->num_sms, (const void*)grouped_gemm_kernel<kEpiDown, false>, kGemmThreads, kGemmSmemBytes,
                        &B->gemm_grid);
  if (s != MOE_OK) return bail(s);
  B->ring.resize(kAttnProfRing);
  B->pending.assign(kAttnProfRing, false);
  for (auto& r : B->ring)
    for (auto& e : r)
      if (cudaEventCreate(&e) != cudaSuccess) {
        e = nullptr;
        return bail(fail(MOE_ERR_CUDA, "cudaEventCreate failed"));
      }
  *out = B;
  return ok();
}

moe_status_t attn_block_forward(attn_block_t* B, const void* x, void* y, int32_t T, void* stream) {
  if (!B) return fail(MOE_ERR_INVALID_ARG, "null block");
  if (T < 1 || T > B->cfg.max_tokens) return fail(MOE_ERR_INVALID_ARG, "T=%d outside [1, %d]", T, B->cfg.max_tokens);
  if (!x || !y) return fail(MOE_ERR_INVALID_ARG, "null x or y");
  if (!aligned16(x) || !aligned16(y)) return fail(MOE_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  if (x == y) return fail(MOE_ERR_INVALID_ARG, "y may not alias x");
  DeviceGuard g(B->device);
  if (!g.ok) return fail(MOE_ERR_CUDA, "cannot select the block's device");
  moe_status_t s = enqueue(B, x, y, T, static_cast<cudaStream_t>(stream));
  return s == MOE_OK ? ok() : s;
}

moe_status_t attn_block_sync_status(attn_block_t* B, void* stream) {
  if (!B) return fail(MOE_ERR_INVALID_ARG, "null block");
  DeviceGuard g(B->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_CUDA_TRY(cudaStreamSynchronize(st));
  uint32_t h = 0;
  MOE_CUDA_TRY(cudaMemcpyAsync(&h, B->err, sizeof(h), cudaMemcpyDeviceToHost, st));
  MOE_CUDA_TRY(cudaStreamSynchronize(st));
  if (h) {
    MOE_CUDA_TRY(cudaMemsetAsync(B->err, 0, sizeof(uint32_t), st));
    MOE_CUDA_TRY(cudaStreamSynchronize(st));
    if (h & kErrTimeout) return fail(MOE_ERR_TIMEOUT, "a device wait ran out of time (error word 0x%x)", h);
    return fail(MOE_ERR_DEVICE_CHECK, "a device check failed (error word 0x%x)", h);
  }
  return ok();
}

int32_t attn_block_launch_count(const attn_block_t* B) { return B ? kAttnLaunches : 0; }

moe_status_t moe_selftest_bounded_wait(int32_t mode, uint64_t limit_ns, uint64_t* elapsed_ns) {
  if (mode < 0 || mode > 2) return fail(MOE_ERR_INVALID_ARG, "mode must be 0, 1 or 2 (got %d)", mode);
  if (limit_ns < 1000000ull || limit_ns > 2000000000ull)
    return fail(MOE_ERR_INVALID_ARG, "limit_ns outside [1 ms, 2 s]");
  void* buf = nullptr;
  MOE_CUDA_TRY(cudaMalloc(&buf, 64));
  uint32_t* err = static_cast<uint32_t*>(buf);
  uint64_t* res = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(buf) + 16);
  uint64_t h[2] = {0, 0};
  uint32_t e = 0;
  cudaError_t ce = cudaMemset(buf, 0, 64);
  if (ce == cudaSuccess) {
    selftest_wait_kernel<<<1, 32>>>(mode, limit_ns, err, res);
    ce = cudaGetLastError();
  }
  if (ce == cudaSuccess) ce = cudaDeviceSynchronize();
  if (ce == cudaSuccess) ce = cudaMemcpy(h, res, sizeof(h), cudaMemcpyDeviceToHost);
  if (ce == cudaSuccess) ce = cudaMemcpy(&e, err, sizeof(e), cudaMemcpyDeviceToHost);
  cudaFree(buf);
  if (ce != cudaSuccess) return fail(MOE_ERR_CUDA, "self-test: %s", cudaGetErrorString(ce));
  if (elapsed_ns) *elapsed_ns = h[1];
  if (h[0] != 0) return fail(MOE_ERR_DEVICE_CHECK, "a wait on a phase nobody completes returned true");
  if (e & kErrTimeout) return fail(MOE_ERR_TIMEOUT, "the wait gave up after %llu ns", (unsigned long long)h[1]);
  return fail(MOE_ERR_DEVICE_CHECK, "the wait gave up but did not latch the error word");
}

moe_status_t moe_selftest_gelu(const float* x, float* y, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return fail(MOE_ERR_INVALID_ARG, "x and y must be device buffers of n >= 0 floats");
  if (n == 0) return ok();
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 4096);
  selftest_gelu_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
  MOE_CUDA_TRY(cudaGetLastError());
  return ok();
}

moe_status_t attn_block_set_profiling(attn_block_t* B, int32_t enable) {
  if (!B) return fail(MOE_ERR_INVALID_ARG, "null block");
  B->profiling = enable != 0;
  return ok();
}

moe_status_t attn_block_profile_read(attn_block_t* B, double* ms_total, int64_t* launches, int32_t reset) {
  if (!B) return fail(MOE_ERR_INVALID_ARG, "null block");
  DeviceGuard g(B->device);
  for (int s = 0; s < kAttnProfRing; ++s) harvest(B, s);
  for (int k = 0; k < ATTN_K_COUNT; ++k) {
    if (ms_total) ms_total[k] = B->prof_ms[k];
    if (launches) launches[k] = B->prof_n[k];
  }
  if (reset)
    for (int k = 0; k < ATTN_K_COUNT; ++k) {
      B->prof_ms[k] = 0.0;
      B->prof_n[k] = 0;
    }
  return ok();
}

moe_status_t attn_block_destroy(attn_block_t* B) {
  if (!B) return ok();
  DeviceGuard g(B->device);
  cudaDeviceSynchronize();
  for (auto& r : B->ring)
    for (auto& e : r)
      if (e) cudaEventDestroy(e);
  if (B->ws) cudaFree(B->ws);
  if (B->wqkv) cudaFree(B->wqkv);
  delete B;
  return ok();
}

}  // extern "C"
