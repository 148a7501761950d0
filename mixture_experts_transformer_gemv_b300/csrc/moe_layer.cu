// Host runtime and C ABI of the Grok-1 MoE layer (declared in include/moe_layer.h).
//
// moe_layer_create validates the configuration, keeps the borrowed weight
// pointers, encodes the TMA descriptors of the expert weights and of the two
// GEMM activation buffers, and allocates one workspace block.
// moe_layer_forward enqueues, on the caller's stream and without any host wait:
//   K1 router_kernel        pre-norm statistics, router logits, softmax, top-2
//   K2 group_rows_kernel    counts, padded row offsets, stable slot -> row map,
//                           and the normed rows written in expert order
//   K3 grouped_gemm<geglu>  act = GELU(A W^T) * (A Wv^T)        (tcgen05)
//   K4 grouped_gemm<down>   Y = p * (act W1^T)                   (tcgen05)
//   K5 combine_kernel       out = x + RMSNorm_post(Y[r0] + Y[r1])
// For T <= 16 (or MOE_FLAG_FORCE_GEMV) K3/K4 are replaced by the weight-streaming
// decode kernels (k_decode.cuh for bf16 weights; for int8 the CUDA-core GEMV kernels
// of k_gemv_i8.cuh, or with MOE_FLAG_DECODE_TC the tensor-core ones of k_decode_i8.cuh)
// and K5 sums their split-K partials.  int8 weights are converted to fp16 on chip and
// their per-channel scales applied in the epilogues.  The allocation-free
// grouping entry point (end of file) runs permute_kernel, K2's grouping alone.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "moe_layer.h"
#include "common.cuh"
#include "host_util.h"
#include "k_combine.cuh"
#include "k_decode.cuh"
#include "k_decode_i8.cuh"
#include "k_gemv_i8.cuh"
#include "k_gemm.cuh"
#include "k_permute.cuh"
#include "k_router.cuh"

using namespace moe;
using namespace moe_host;

namespace {

static_assert(kDecMaxSplitCombine == kDecMaxSplit, "the combine unrolls to the decode split");
static_assert(kGemmBK == kDecBK && kGemmBK == kTmapBoxInner, "every bf16 GEMM operand box is 64 elements wide");

// Row-major 2-D int8 tensor [rows, inner], box [box_rows, box_inner]: the staging
// layout the int8 converter warps read; 64-byte rows without swizzle for the
// grouped GEMMs (threads read along rows), 128-byte rows with 128-byte swizzle
// for the decode kernels (each thread reads one row).
moe_status_t make_tmap_i8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows,
                          uint32_t box_inner, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (int8) failed (%d)", (int)r);
  return MOE_OK;
}

constexpr int kProfRing = 64;

// The grouped GEMMs pair two m-blocks per tile when F >= kPairMinF and
// T >= kPairMinT.  Measured at F = 32768 and T >= 2048: faster (half the
// weight-tile traffic, and for int8 half the conversions, per MMA, and less
// power, so a higher clock under the cap).  At F = 4096 the paired kernels were
// slower (up projection 22 %: few tiles of short mainloops, each epilogue
// exposed), and at T <= 512 (at most one m-block per expert, so no pairs) the
// up projection ran 14 % slower with the paired kernel's shallower ring and
// un-overlapped epilogue.  T = 2048 gives each expert 512 rows on average: two
// full m-blocks.
constexpr int kPairMinF = 16384;
constexpr int kPairMinT = 2048;

}  // namespace

struct moe_layer {
  moe_config_t cfg{};
  moe_weights_t w{};
  int device = 0;
  int num_sms = 0;
  int gemm_grid[2][2][2] = {};  // [epilogue][int8][paired m-blocks]: CTAs of a grouped GEMM launch
  int64_t rows_cap = 0;

  void* ws = nullptr;
  float* rnorm = nullptr;  // [max_T] 1 / rms of each token's hidden row (router)
  int32_t* idx = nullptr;
  float* prob = nullptr;
  int32_t* sched = nullptr;
  int32_t* row_of_slot = nullptr;
  int32_t* token_of_row = nullptr;
  float* prob_of_row = nullptr;
  __nv_bfloat16* xn_perm = nullptr;
  __nv_bfloat16* act = nullptr;
  float* y_rows = nullptr;
  float* part = nullptr;  // decode path: [kDecMaxSplit][E][16][d] fp32 split-K partials
  float* p_part = nullptr;  // [router CTAs (<= max_T)][E] per-router-CTA sums of p
  int16_t* xq = nullptr;    // int8 GEMV path: [E * 16][max(d, F)] slot rows in 16-bit fixed point
  float* xqs = nullptr;     //                 [max(d, F) / 128][E * 16] their block scales
  int last_T = 0;           // tokens of the last forward enqueued (routing diagnostics)
  uint32_t* err = nullptr;
  int ksplit = 1;         // decode path: chunks of the down-projection reduction
  bool router_gsmem = false;     // the router's scaled gate s_pre (.) G fits one CTA's shared memory
  bool router_small = false;     // T <= kRouterSmallT and d <= 6144: router_split_kernel
  float* router_part = nullptr;  // [kRouterSmallT][32][9] per-virtual-lane sums of router_split_kernel
  int32_t* router_done = nullptr;  // [kRouterSmallT] its per-token counters (zero between forwards)
  bool pair_mblocks = false;     // F >= kPairMinF: forwards with T >= kPairMinT pair two m-blocks per tile
  int ksplit_i8 = 1;      // the same for the int8 decode kernel (128-wide k-blocks)

  CUtensorMap tm_xn_perm{}, tm_act{}, tm_w{}, tm_wv{}, tm_w1_128{};  // boxes of 128 rows x 64
  CUtensorMap tm_xn_perm64{}, tm_act64{}, tm_w64{}, tm_wv64{};       // grouped GEMMs' half tiles: 64 rows x 64
  CUtensorMap tm_xn_perm16{}, tm_act16{};                             // decode path: 16-row boxes
  CUtensorMap tm_w8{}, tm_wv8{}, tm_w18{};              // int8 weights (staging boxes of 128 rows)
  CUtensorMap tm_w8h{}, tm_wv8h{};                      // int8 weights, half tiles (64 rows)
  CUtensorMap tm_w8d{}, tm_wv8d{}, tm_w18d{};           // int8 weights, 64-byte swizzle (decode)
  CUtensorMap tm_xq_d{}, tm_xq_f{}, tm_xqs_d{}, tm_xqs_f{};  // int8 GEMV: quantised rows and scales, K = d or F

  void* host_stage = nullptr;  // device staging for moe_layer_forward_host
  size_t host_stage_bytes = 0;

  // moe_layer_forward_host_async: two device staging slots, copy streams and events
  void* async_stage[2] = {nullptr, nullptr};
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t in_ready[2] = {}, fwd_done[2] = {}, slot_free[2] = {};
  int async_slot = 0;
  bool async_pending = false;

  bool profiling = false;
  std::vector<std::array<cudaEvent_t, MOE_K_COUNT + 1>> ring;
  std::vector<bool> pending;
  int ring_next = 0;
  double prof_ms[MOE_K_COUNT] = {};
  int64_t prof_n[MOE_K_COUNT] = {};
  std::atomic<int64_t> launches{0};
};

namespace {

moe_status_t gemm_pairs(moe_layer* L, const void* kernel, int threads, size_t smem, int* grid) {
  return cluster_pair_grid(L->num_sms, kernel, threads, smem, grid);
}

void harvest(moe_layer* L, int slot) {
  if (!L->pending[slot]) return;
  auto& ev = L->ring[slot];
  cudaEventSynchronize(ev[MOE_K_COUNT]);
  for (int k = 0; k < MOE_K_COUNT; ++k) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, ev[k], ev[k + 1]) == cudaSuccess) {
      L->prof_ms[k] += ms;
      L->prof_n[k] += 1;
    }
  }
  L->pending[slot] = false;
}

// int8 GEMV path: the 2T slot rows (fp16, K wide) into 16-bit fixed point, one
// warp per slot row and 128-element block, 8 warps per CTA.
void launch_quantize_slots(moe_layer* L, int T, const void* rows, int K, cudaStream_t st) {
  const int S = 2 * T, warps = S * (K / kGv8BK);
  quantize_slots_kernel<<<(warps + 7) / 8, 256, 0, st>>>(static_cast<const uint16_t*>(rows), K, L->row_of_slot,
                                                         L->idx, L->sched, S, L->xq, L->xqs);
}

moe_status_t enqueue_forward(moe_layer* L, const void* hidden, void* out, int T, cudaStream_t st,
                             int32_t* topk_idx, float* topk_prob, int32_t* counts) {
  const int d = L->cfg.d_model, F = L->cfg.d_ffn;
  const int checks = (L->cfg.flags & MOE_FLAG_DEVICE_CHECKS) ? 1 : 0;
  cudaEvent_t* ev = nullptr;
  if (L->profiling) {
    int slot = L->ring_next;
    L->ring_next = (L->ring_next + 1) % kProfRing;
    harvest(L, slot);
    ev = L->ring[slot].data();
    L->pending[slot] = true;
  }
  auto mark = [&](int k) {
    if (ev) cudaEventRecord(ev[k], st);
  };

  const bool int8 = L->cfg.weight_dtype == MOE_WEIGHT_INT8;
  const bool decode = (L->cfg.flags & MOE_FLAG_FORCE_GEMV) || (!(L->cfg.flags & MOE_FLAG_FORCE_TC) && T <= kDecNS);
  const bool pair = L->pair_mblocks && T >= kPairMinT;  // grouped GEMMs: two m-blocks per tile
  mark(0);
  // Router: 8 warps per CTA, each warp a contiguous run of tokens.  With the
  // scaled gate in shared memory: one CTA per SM at most (the gate is staged once
  // per CTA), and one CTA per token below that, so small batches spread over as
  // many SMs as they have tokens.  Otherwise the gate is read from L2 at every
  // use, and the CTAs get 4 tokens per warp (fewer reads).
  {
    const __nv_bfloat16* xh = static_cast<const __nv_bfloat16*>(hidden);
    if (L->router_small && T <= kRouterSmallT) {
      router_split_kernel<<<dim3(T, kRouterSlices), kRouterSplitThreads, 0, st>>>(
          xh, d, L->w.gate, L->w.gate_bias, L->w.pre_norm_scale, L->cfg.eps, L->rnorm, L->idx, L->prob, topk_idx,
          topk_prob, L->p_part, L->router_part, L->router_done);
    } else if (L->router_gsmem) {
      const int grid = std::min(L->num_sms, T);
      router_kernel<true><<<grid, kRouterThreads, (size_t)kNumExperts * d * 4, st>>>(
          xh, T, d, L->w.gate, L->w.gate_bias, L->w.pre_norm_scale, L->cfg.eps, L->rnorm, L->idx, L->prob, topk_idx,
          topk_prob, L->p_part);
    } else {
      constexpr int kTokPerCta = kRouterWarps * kRouterWTok;
      const int grid = (T + kTokPerCta - 1) / kTokPerCta;
      router_kernel<false><<<grid, kRouterThreads, 0, st>>>(xh, T, d, L->w.gate, L->w.gate_bias,
                                                           L->w.pre_norm_scale, L->cfg.eps, L->rnorm, L->idx,
                                                           L->prob, topk_idx, topk_prob, L->p_part);
    }
  }
  mark(1);
  // grouping + normed rows in expert order; int8 layers multiply in fp16 (int8 ->
  // fp16 is one shuffle and one subtraction), so their activation rows are fp16
  // 4 CTAs per SM (memory parallelism for the row copies); every CTA reads all of
  // idx and does the counting, so beyond 16384 tokens one CTA per SM, and for a
  // decode-sized batch one CTA per two SMs (a few rows to copy, up to 8 x 127
  // padding rows to zero)
  const int group_grid = T <= 64 ? std::max(1, L->num_sms / 2) : (T <= 16384 ? 4 * L->num_sms : L->num_sms);
  group_rows_kernel<<<group_grid, kGroupThreads, 0, st>>>(
      L->idx, L->prob, T, static_cast<const __nv_bfloat16*>(hidden), L->rnorm, L->w.pre_norm_scale, d,
      int8 ? 1 : 0, L->sched, L->row_of_slot, L->token_of_row, L->prob_of_row, L->xn_perm, counts,
      (int)L->rows_cap, checks, L->err);
  mark(2);
  // int8 weights at T <= 16: integer dot products on the CUDA cores (k_gemv_i8.cuh)
  const bool gemv8 = decode && int8 && T <= kGv8MaxT && !(L->cfg.flags & MOE_FLAG_DECODE_TC);
  const bool grouped8 = L->cfg.scale_groups > 1;
  if (decode && int8) {
    DecI8Params p{};
    p.sched = L->sched;
    p.K = d;
    p.rows_per_expert = F;
    p.n_out = F;
    p.ksplit = 1;
    p.out = L->act;
    p.row_scale = nullptr;
    p.scale0 = L->w.w_scale;
    p.scale1 = L->w.wv_scale;
    p.scale_experts = L->cfg.scale_experts;
    p.scale_groups = L->cfg.scale_groups;
    p.group_kb = d / L->cfg.scale_groups / kDq8BK;
    p.checks = checks;
    p.err = L->err;
    p.timeout_ns = kWaitLimitNs;
    if (gemv8) launch_quantize_slots(L, T, L->xn_perm, d, st);
    if (gemv8 && grouped8)
      gemv_i8_kernel<kEpiGeglu, true><<<L->num_sms, GvI8Cfg<kEpiGeglu>::kThreads, GvI8Cfg<kEpiGeglu>::kSmemBytes,
                                        st>>>(L->tm_w8d, L->tm_wv8d, L->tm_xq_d, L->tm_xqs_d, p);
    else if (gemv8)
      gemv_i8_kernel<kEpiGeglu, false><<<L->num_sms, GvI8Cfg<kEpiGeglu>::kThreads, GvI8Cfg<kEpiGeglu>::kSmemBytes,
                                         st>>>(L->tm_w8d, L->tm_wv8d, L->tm_xq_d, L->tm_xqs_d, p);
    else
      decode_gemm_i8_kernel<kEpiGeglu><<<L->num_sms, DecI8Cfg<kEpiGeglu>::kThreads, DecI8Cfg<kEpiGeglu>::kSmemBytes,
                                         st>>>(L->tm_w8d, L->tm_wv8d, L->tm_xn_perm16, p);
  } else if (decode) {
    DecParams p{};
    p.sched = L->sched;
    p.K = d;
    p.rows_per_expert = F;
    p.n_out = F;
    p.ksplit = 1;
    p.out = L->act;
    p.row_scale = nullptr;
    p.err = L->err;
    p.timeout_ns = kWaitLimitNs;
    decode_gemm_kernel<kEpiGeglu><<<L->num_sms, kDecThreads, DecCfg<kEpiGeglu>::kSmemBytes, st>>>(
        L->tm_w, L->tm_wv, L->tm_xn_perm16, p);
  } else {
    GemmParams p{};
    p.sched = L->sched;
    p.K = d;
    p.n_tiles = F / kGemmHalfN;
    p.tile_counter = L->sched + kSchedTileCtr;  // dynamic tile schedule (zeroed by K2)
    p.b_rows_per_expert = F;
    p.n_out = F;
    p.out = L->act;
    p.row_scale = nullptr;
    p.scale0 = L->w.w_scale;
    p.scale1 = L->w.wv_scale;
    p.scale_experts = L->cfg.scale_experts;
    p.scale_groups = L->cfg.scale_groups;
    p.group_kb = d / L->cfg.scale_groups / kGemmBK;
    p.checks = checks;
    p.err = L->err;
    p.timeout_ns = kWaitLimitNs;
    if (int8 && pair)
      grouped_gemm_kernel<kEpiGeglu, true, kGemmMBPair>
          <<<L->gemm_grid[kEpiGeglu][1][1], GemmCfg<true, kGemmMBPair>::kThreads, GemmCfg<true, kGemmMBPair>::kSmemBytes,
             st>>>(L->tm_xn_perm, L->tm_w8, L->tm_wv8, L->tm_xn_perm64, L->tm_w8h, L->tm_wv8h, p);
    else if (int8)
      grouped_gemm_kernel<kEpiGeglu, true><<<L->gemm_grid[kEpiGeglu][1][0], GemmCfg<true>::kThreads,
                                             GemmCfg<true>::kSmemBytes, st>>>(
          L->tm_xn_perm, L->tm_w8, L->tm_wv8, L->tm_xn_perm64, L->tm_w8h, L->tm_wv8h, p);
    else if (pair)
      grouped_gemm_kernel<kEpiGeglu, false, kGemmMBPair>
          <<<L->gemm_grid[kEpiGeglu][0][1], GemmCfg<false, kGemmMBPair>::kThreads,
             GemmCfg<false, kGemmMBPair>::kSmemBytes, st>>>(L->tm_xn_perm, L->tm_w, L->tm_wv, L->tm_xn_perm64,
                                                            L->tm_w64, L->tm_wv64, p);
    else
      grouped_gemm_kernel<kEpiGeglu, false><<<L->gemm_grid[kEpiGeglu][0][0], kGemmThreads, kGemmSmemBytes, st>>>(
          L->tm_xn_perm, L->tm_w, L->tm_wv, L->tm_xn_perm64, L->tm_w64, L->tm_wv64, p);
  }
  mark(3);
  if (decode && int8) {
    DecI8Params p{};
    p.sched = L->sched;
    p.K = F;
    p.rows_per_expert = d;
    p.n_out = d;
    p.ksplit = L->ksplit_i8;
    p.out = L->part;
    p.row_scale = L->prob_of_row;
    p.scale0 = L->w.w1_scale;
    p.scale1 = nullptr;
    p.scale_experts = L->cfg.scale_experts;
    p.scale_groups = L->cfg.scale_groups;
    p.group_kb = F / L->cfg.scale_groups / kDq8BK;
    p.err = L->err;
    p.timeout_ns = kWaitLimitNs;
    if (gemv8) launch_quantize_slots(L, T, L->act, F, st);
    if (gemv8 && grouped8)
      gemv_i8_kernel<kEpiDown, true><<<L->num_sms, GvI8Cfg<kEpiDown>::kThreads, GvI8Cfg<kEpiDown>::kSmemBytes, st>>>(
          L->tm_w18d, L->tm_w18d, L->tm_xq_f, L->tm_xqs_f, p);
    else if (gemv8)
      gemv_i8_kernel<kEpiDown, false><<<L->num_sms, GvI8Cfg<kEpiDown>::kThreads, GvI8Cfg<kEpiDown>::kSmemBytes, st>>>(
          L->tm_w18d, L->tm_w18d, L->tm_xq_f, L->tm_xqs_f, p);
    else
      decode_gemm_i8_kernel<kEpiDown><<<L->num_sms, DecI8Cfg<kEpiDown>::kThreads, DecI8Cfg<kEpiDown>::kSmemBytes,
                                        st>>>(L->tm_w18d, L->tm_w18d, L->tm_act16, p);
  } else if (decode) {
    DecParams p{};
    p.sched = L->sched;
    p.K = F;
    p.rows_per_expert = d;
    p.n_out = d;
    p.ksplit = L->ksplit;
    p.out = L->part;
    p.row_scale = L->prob_of_row;
    p.err = L->err;
    p.timeout_ns = kWaitLimitNs;
    decode_gemm_kernel<kEpiDown><<<L->num_sms, kDecThreads, DecCfg<kEpiDown>::kSmemBytes, st>>>(
        L->tm_w1_128, L->tm_w1_128, L->tm_act16, p);
  } else {
    GemmParams p{};
    p.sched = L->sched;
    p.K = F;
    p.n_tiles = (d + kGemmBN - 1) / kGemmBN;
    p.tile_counter = L->sched + kSchedTileCtr + 1;  // dynamic tile schedule (zeroed by K2)
    p.b_rows_per_expert = d;
    p.n_out = d;
    p.out = L->y_rows;
    p.row_scale = L->prob_of_row;
    p.scale0 = L->w.w1_scale;
    p.scale1 = nullptr;
    p.scale_experts = L->cfg.scale_experts;
    p.scale_groups = L->cfg.scale_groups;
    p.group_kb = F / L->cfg.scale_groups / kGemmBK;
    p.err = L->err;
    p.timeout_ns = kWaitLimitNs;
    if (int8 && pair)
      grouped_gemm_kernel<kEpiDown, true, kGemmMBPair>
          <<<L->gemm_grid[kEpiDown][1][1], GemmCfg<true, kGemmMBPair>::kThreads, GemmCfg<true, kGemmMBPair>::kSmemBytes,
             st>>>(L->tm_act, L->tm_w18, L->tm_w18, L->tm_act64, L->tm_w18, L->tm_w18, p);
    else if (int8)
      grouped_gemm_kernel<kEpiDown, true><<<L->gemm_grid[kEpiDown][1][0], GemmCfg<true>::kThreads,
                                            GemmCfg<true>::kSmemBytes, st>>>(L->tm_act, L->tm_w18, L->tm_w18,
                                                                             L->tm_act64, L->tm_w18, L->tm_w18, p);
    else if (!pair)
      grouped_gemm_kernel<kEpiDown, false><<<L->gemm_grid[kEpiDown][0][0], kGemmThreads, kGemmSmemBytes, st>>>(
          L->tm_act, L->tm_w1_128, L->tm_w1_128, L->tm_act64, L->tm_w1_128, L->tm_w1_128, p);
    else
      grouped_gemm_kernel<kEpiDown, false, kGemmMBPair>
          <<<L->gemm_grid[kEpiDown][0][1], GemmCfg<false, kGemmMBPair>::kThreads, GemmCfg<false, kGemmMBPair>::kSmemBytes,
             st>>>(
          L->tm_act, L->tm_w1_128, L->tm_w1_128, L->tm_act64, L->tm_w1_128, L->tm_w1_128, p);
  }
  mark(4);
  {
    const __nv_bfloat16* xh = static_cast<const __nv_bfloat16*>(hidden);
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
    const int rc = (int)L->rows_cap;
    const bool wide = T < L->num_sms;  // few tokens: more threads per token hide latency
    if (decode) {
      const int ks = int8 ? L->ksplit_i8 : L->ksplit;
      if (wide)
        launch_combine<true, 1024>(T, st, L->part, L->row_of_slot, L->idx, L->sched, ks, xh, L->w.post_norm_scale,
                                   L->cfg.eps, d, rc, checks, L->err, o);
      else
        launch_combine<true, kCombineThreads>(T, st, L->part, L->row_of_slot, L->idx, L->sched, ks, xh,
                                              L->w.post_norm_scale, L->cfg.eps, d, rc, checks, L->err, o);
    } else {
      if (wide)
        launch_combine<false, 1024>(T, st, L->y_rows, L->row_of_slot, L->idx, L->sched, 1, xh,
                                    L->w.post_norm_scale, L->cfg.eps, d, rc, checks, L->err, o);
      else
        launch_combine<false, kCombineThreads>(T, st, L->y_rows, L->row_of_slot, L->idx, L->sched, 1, xh,
                                               L->w.post_norm_scale, L->cfg.eps, d, rc, checks, L->err, o);
    }
  }
  mark(5);
  L->launches += MOE_K_COUNT + (gemv8 ? 2 : 0);  // + the two row quantisations of the int8 GEMV path
  L->last_T = T;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_OOM: return "MOE_ERR_OOM";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_last_error_message(void) { return g_last_error.c_str(); }

moe_status_t moe_layer_create(const moe_config_t* cfg, const moe_weights_t* w, moe_layer_t** out) {
  if (!cfg || !w || !out) return fail(MOE_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  const moe_config_t c = *cfg;
  if (c.num_experts != kNumExperts) return fail(MOE_ERR_UNSUPPORTED, "num_experts must be 8 (got %d)", c.num_experts);
  if (c.top_k != kTopK) return fail(MOE_ERR_UNSUPPORTED, "top_k must be 2 (got %d)", c.top_k);
  if (c.d_model <= 0 || c.d_ffn <= 0 || c.d_model % 128 || c.d_ffn % 128)
    return fail(MOE_ERR_UNSUPPORTED, "d_model and d_ffn must be positive multiples of 128 (got %d, %d)", c.d_model,
                c.d_ffn);
  if (c.d_model > 4 * kCombineThreads * kCombineVec)
    return fail(MOE_ERR_UNSUPPORTED, "d_model > %d", 4 * kCombineThreads * kCombineVec);
  if ((int64_t)kNumExperts * c.d_ffn > INT32_MAX / 2)
    return fail(MOE_ERR_UNSUPPORTED, "d_ffn too large");
  if (c.max_tokens < 1 || c.max_tokens > (1 << 24)) return fail(MOE_ERR_INVALID_ARG, "max_tokens out of range");
  if (!(c.eps > 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be > 0");
  if (c.weight_dtype != MOE_WEIGHT_BF16 && c.weight_dtype != MOE_WEIGHT_INT8)
    return fail(MOE_ERR_INVALID_ARG, "unknown weight_dtype %d", c.weight_dtype);
  if (c.scale_experts != 0 && c.scale_experts != 1 && c.scale_experts != kNumExperts)
    return fail(MOE_ERR_INVALID_ARG, "scale_experts must be 0, 1 or 8 (got %d)", c.scale_experts);
  if (c.scale_groups < 0) return fail(MOE_ERR_INVALID_ARG, "scale_groups < 0");
  if (c.weight_dtype == MOE_WEIGHT_INT8 && c.scale_groups > 1 &&
      (c.d_model % (128 * c.scale_groups) || c.d_ffn % (128 * c.scale_groups)))
    return fail(MOE_ERR_UNSUPPORTED, "scale_groups = %d needs d_model and d_ffn to be multiples of %d",
                c.scale_groups, 128 * c.scale_groups);
  if ((c.flags & MOE_FLAG_FORCE_GEMV) && (c.flags & MOE_FLAG_FORCE_TC))
    return fail(MOE_ERR_INVALID_ARG, "MOE_FLAG_FORCE_GEMV and MOE_FLAG_FORCE_TC are exclusive");
  const void* req[] = {w->gate, w->w, w->wv, w->w1, w->pre_norm_scale, w->post_norm_scale};
  for (const void* p : req)
    if (!p || !aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "weight pointer null or not 16-byte aligned");
  if (w->gate_bias && !aligned4(w->gate_bias)) return fail(MOE_ERR_INVALID_ARG, "gate_bias misaligned");
  if (c.weight_dtype == MOE_WEIGHT_INT8) {
    const void* sc[] = {w->w_scale, w->wv_scale, w->w1_scale};
    for (const void* p : sc)
      if (!p || !aligned16(p))
        return fail(MOE_ERR_INVALID_ARG, "int8 weights need w_scale, wv_scale, w1_scale (16-byte aligned)");
  }

  int dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  MOE_CUDA_TRY(cudaGetDeviceProperties(&prop, dev));
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(MOE_ERR_UNSUPPORTED, "built for sm_103a; device is sm_%d%d", prop.major, prop.minor);
  const size_t smem_need =
      std::max(std::max(std::max(kGemmSmemBytes, GemmCfg<true>::kSmemBytes),
                        std::max(GemmCfg<false, kGemmMBPair>::kSmemBytes, GemmCfg<true, kGemmMBPair>::kSmemBytes)),
               std::max(std::max(DecCfg<kEpiGeglu>::kSmemBytes, DecCfg<kEpiDown>::kSmemBytes),
                        std::max(std::max(DecI8Cfg<kEpiGeglu>::kSmemBytes, DecI8Cfg<kEpiDown>::kSmemBytes),
                                 std::max(GvI8Cfg<kEpiGeglu>::kSmemBytes, GvI8Cfg<kEpiDown>::kSmemBytes))));
  if (prop.sharedMemPerBlockOptin < smem_need)
    return fail(MOE_ERR_UNSUPPORTED, "device offers %zu B shared memory per block, need %zu",
                (size_t)prop.sharedMemPerBlockOptin, smem_need);

  auto* L = new (std::nothrow) moe_layer();
  if (!L) return fail(MOE_ERR_OOM, "host allocation failed");
  L->cfg = c;
  if (L->cfg.scale_experts == 0) L->cfg.scale_experts = kNumExperts;
  if (L->cfg.scale_groups == 0) L->cfg.scale_groups = 1;
  L->w = *w;
  L->device = dev;
  L->num_sms = prop.multiProcessorCount;
  const int64_t T = c.max_tokens, d = c.d_model, F = c.d_ffn;
  L->rows_cap = (int64_t)align_up((size_t)(2 * T), kRowPad) + (int64_t)kNumExperts * kRowPad;
  const int64_t R = L->rows_cap;

  // one workspace block, every buffer 1 KB aligned
  const int64_t kq = std::max(d, F);
  const bool i8 = c.weight_dtype == MOE_WEIGHT_INT8;
  size_t offs[16], total = 0;
  const size_t sizes[16] = {(size_t)(T * 4), (size_t)(T * 2 * 4), (size_t)(T * 2 * 4), 256,
                            (size_t)(T * 2 * 4), (size_t)(R * 4),     (size_t)(R * 4),     (size_t)(R * d * 2),
                            (size_t)(R * F * 2), (size_t)(R * d * 4), 256,
                            (size_t)kDecMaxSplit * kNumExperts * kDecNS * d * 4,
                            (size_t)T * kNumExperts * 4,
                            i8 ? (size_t)kGv8QRows * kq * 2 : 0,
                            i8 ? (size_t)(kq / kGv8BK) * kGv8QRows * 4 : 0,
                            (size_t)kRouterSmallT * (kRouterPartFloats + 1) * 4};
  for (int i = 0; i < 16; ++i) {
    offs[i] = total;
    total = align_up(total + sizes[i], 1024);
  }
  cudaError_t e = cudaMalloc(&L->ws, total);
  if (e != cudaSuccess) {
    delete L;
    cudaGetLastError();
    return fail(MOE_ERR_OOM, "workspace of %zu bytes: %s", total, cudaGetErrorString(e));
  }
  char* b = static_cast<char*>(L->ws);
  L->rnorm = reinterpret_cast<float*>(b + offs[0]);
  L->idx = reinterpret_cast<int32_t*>(b + offs[1]);
  L->prob = reinterpret_cast<float*>(b + offs[2]);
  L->sched = reinterpret_cast<int32_t*>(b + offs[3]);
  L->row_of_slot = reinterpret_cast<int32_t*>(b + offs[4]);
  L->token_of_row = reinterpret_cast<int32_t*>(b + offs[5]);
  L->prob_of_row = reinterpret_cast<float*>(b + offs[6]);
  L->xn_perm = reinterpret_cast<__nv_bfloat16*>(b + offs[7]);
  L->act = reinterpret_cast<__nv_bfloat16*>(b + offs[8]);
  L->y_rows = reinterpret_cast<float*>(b + offs[9]);
  L->err = reinterpret_cast<uint32_t*>(b + offs[10]);
  L->part = reinterpret_cast<float*>(b + offs[11]);
  L->p_part = reinterpret_cast<float*>(b + offs[12]);
  L->xq = reinterpret_cast<int16_t*>(b + offs[13]);
  L->xqs = reinterpret_cast<float*>(b + offs[14]);
  L->router_part = reinterpret_cast<float*>(b + offs[15]);
  L->router_done = reinterpret_cast<int32_t*>(L->router_part + (size_t)kRouterSmallT * kRouterPartFloats);
  // decode-path split of the F reduction: up to kDecMaxSplit chunks of whole 64-wide blocks
  L->ksplit = kDecMaxSplit;
  while (L->ksplit > 1 && (F / kDecBK) % L->ksplit) L->ksplit /= 2;
  L->ksplit_i8 = kDecMaxSplit;
  while (L->ksplit_i8 > 1 && (F / kDq8BK) % L->ksplit_i8) L->ksplit_i8 /= 2;
  moe_status_t s = MOE_OK;
  if (cudaMemset(L->ws, 0, total) != cudaSuccess) s = fail(MOE_ERR_CUDA, "workspace memset failed");
  if (s == MOE_OK) s = make_tmap_bf16(&L->tm_xn_perm, L->xn_perm, d, R, kGemmHalfM);
  if (s == MOE_OK) s = make_tmap_bf16(&L->tm_act, L->act, F, R, kGemmHalfM);
  if (s == MOE_OK) s = make_tmap_bf16(&L->tm_xn_perm64, L->xn_perm, d, R, kGemmBoxRows);
  if (s == MOE_OK) s = make_tmap_bf16(&L->tm_act64, L->act, F, R, kGemmBoxRows);
  if (c.weight_dtype == MOE_WEIGHT_BF16) {
    static_assert(kGemmHalfN == kDecBM, "the GEMM and decode paths share the 128-row weight boxes");
    if (s == MOE_OK) s = make_tmap_bf16(&L->tm_w, w->w, d, kNumExperts * F, kGemmHalfN);
    if (s == MOE_OK) s = make_tmap_bf16(&L->tm_wv, w->wv, d, kNumExperts * F, kGemmHalfN);
    if (s == MOE_OK) s = make_tmap_bf16(&L->tm_w1_128, w->w1, F, kNumExperts * d, kGemmHalfN);
    if (s == MOE_OK) s = make_tmap_bf16(&L->tm_w64, w->w, d, kNumExperts * F, kGemmBoxRows);
    if (s == MOE_OK) s = make_tmap_bf16(&L->tm_wv64, w->wv, d, kNumExperts * F, kGemmBoxRows);
  } else {
    if (s == MOE_OK) s = make_tmap_i8(&L->tm_w8, w->w, d, kNumExperts * F, kGemmHalfN, kGemmBK);
    if (s == MOE_OK) s = make_tmap_i8(&L->tm_wv8, w->wv, d, kNumExperts * F, kGemmHalfN, kGemmBK);
    if (s == MOE_OK) s = make_tmap_i8(&L->tm_w18, w->w1, F, kNumExperts * d, kGemmHalfN, kGemmBK);
    if (s == MOE_OK) s = make_tmap_i8(&L->tm_w8h, w->w, d, kNumExperts * F, kGemmBoxRows, kGemmBK);
    if (s == MOE_OK) s = make_tmap_i8(&L->tm_wv8h, w->wv, d, kNumExperts * F, kGemmBoxRows, kGemmBK);
    if (s == MOE_OK) s = make_tmap_i8(&L->tm_w8d, w->w, d, kNumExperts * F, kDecBM, kDq8BK, CU_TENSOR_MAP_SWIZZLE_128B);
    if (s == MOE_OK)
      s = make_tmap_i8(&L->tm_wv8d, w->wv, d, kNumExperts * F, kDecBM, kDq8BK, CU_TENSOR_MAP_SWIZZLE_128B);
    if (s == MOE_OK)
      s = make_tmap_i8(&L->tm_w18d, w->w1, F, kNumExperts * d, kDecBM, kDq8BK, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (i8) {  // int8 GEMV: a slot group's 8 quantised rows of a block (256 B each) and their 8 scales
    if (s == MOE_OK)
      s = make_tmap_2d(&L->tm_xq_d, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, L->xq, d, kGv8QRows, kGv8BK, kGv8NS);
    if (s == MOE_OK)
      s = make_tmap_2d(&L->tm_xq_f, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, L->xq, F, kGv8QRows, kGv8BK, kGv8NS);
    if (s == MOE_OK)
      s = make_tmap_2d(&L->tm_xqs_d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, L->xqs, kGv8QRows, d / kGv8BK, kGv8NS, 1);
    if (s == MOE_OK)
      s = make_tmap_2d(&L->tm_xqs_f, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, L->xqs, kGv8QRows, F / kGv8BK, kGv8NS, 1);
  }
  if (s == MOE_OK) s = make_tmap_bf16(&L->tm_xn_perm16, L->xn_perm, d, R, kDecNS);
  if (s == MOE_OK) s = make_tmap_bf16(&L->tm_act16, L->act, F, R, kDecNS);
  L->router_small = d <= 32 * 8 * kRouterSmallK;  // small batches: router_split_kernel
  {
    // the router keeps the scaled gate (32 d bytes) in shared memory where it fits
    const size_t gsm = (size_t)kNumExperts * d * 4;
    if (gsm + 1024 <= (size_t)prop.sharedMemPerBlockOptin) {
      if (cudaFuncSetAttribute(router_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gsm) ==
          cudaSuccess)
        L->router_gsmem = true;
      else
        cudaGetLastError();
    }
  }
  if (s == MOE_OK &&
      cudaFuncSetAttribute(grouped_gemm_kernel<kEpiGeglu, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kGemmSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (up GEMM, one m-block per tile) failed");
  if (s == MOE_OK &&
      cudaFuncSetAttribute(grouped_gemm_kernel<kEpiGeglu, false, kGemmMBPair>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)GemmCfg<false, kGemmMBPair>::kSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (up GEMM) failed");
  if (s == MOE_OK &&
      cudaFuncSetAttribute(grouped_gemm_kernel<kEpiDown, false, kGemmMBPair>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)GemmCfg<false, kGemmMBPair>::kSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (down GEMM) failed");
  if (s == MOE_OK &&
      cudaFuncSetAttribute(grouped_gemm_kernel<kEpiGeglu, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)GemmCfg<true>::kSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (int8 up GEMM, one m-block per tile) failed");
  if (s == MOE_OK &&
      cudaFuncSetAttribute(grouped_gemm_kernel<kEpiGeglu, true, kGemmMBPair>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)GemmCfg<true, kGemmMBPair>::kSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (int8 up GEMM) failed");
  if (s == MOE_OK &&
      cudaFuncSetAttribute(grouped_gemm_kernel<kEpiDown, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kGemmSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (down GEMM, one m-block per tile) failed");
  if (s == MOE_OK &&
      cudaFuncSetAttribute(grouped_gemm_kernel<kEpiDown, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)GemmCfg<true>::kSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (int8 down GEMM, one m-block per tile) failed");
  if (s == MOE_OK &&
      cudaFuncSetAttribute(grouped_gemm_kernel<kEpiDown, true, kGemmMBPair>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)GemmCfg<true, kGemmMBPair>::kSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (int8 down GEMM) failed");
  if (s == MOE_OK &&
      cudaFuncSetAttribute(decode_gemm_kernel<kEpiGeglu>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)DecCfg<kEpiGeglu>::kSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (decode up) failed");
  if (s == MOE_OK &&
      cudaFuncSetAttribute(decode_gemm_kernel<kEpiDown>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)DecCfg<kEpiDown>::kSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (decode down) failed");
  if (s == MOE_OK &&
      cudaFuncSetAttribute(decode_gemm_i8_kernel<kEpiGeglu>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)DecI8Cfg<kEpiGeglu>::kSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (int8 decode up) failed");
  if (s == MOE_OK &&
      cudaFuncSetAttribute(decode_gemm_i8_kernel<kEpiDown>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)DecI8Cfg<kEpiDown>::kSmemBytes) != cudaSuccess)
    s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (int8 decode down) failed");
  {
    const struct {
      const void* k;
      size_t smem;
    } gv[4] = {{(const void*)gemv_i8_kernel<kEpiGeglu, false>, GvI8Cfg<kEpiGeglu>::kSmemBytes},
               {(const void*)gemv_i8_kernel<kEpiGeglu, true>, GvI8Cfg<kEpiGeglu>::kSmemBytes},
               {(const void*)gemv_i8_kernel<kEpiDown, false>, GvI8Cfg<kEpiDown>::kSmemBytes},
               {(const void*)gemv_i8_kernel<kEpiDown, true>, GvI8Cfg<kEpiDown>::kSmemBytes}};
    for (const auto& k : gv)
      if (s == MOE_OK &&
          cudaFuncSetAttribute(k.k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k.smem) != cudaSuccess)
        s = fail(MOE_ERR_CUDA, "cudaFuncSetAttribute (int8 GEMV) failed");
  }
  // Grouped GEMMs run one CTA pair per two SMs, persistent: launch as many
  // pairs as can be resident at once (whole clusters only), at most one per SM pair.
  L->pair_mblocks = F >= kPairMinF;
  {
    struct {
      const void* k;
      int threads;
      size_t smem;
      int* grid;
    } g[8] = {
        {(const void*)grouped_gemm_kernel<kEpiGeglu, false>, kGemmThreads, kGemmSmemBytes, &L->gemm_grid[0][0][0]},
        {(const void*)grouped_gemm_kernel<kEpiDown, false>, kGemmThreads, kGemmSmemBytes, &L->gemm_grid[1][0][0]},
        {(const void*)grouped_gemm_kernel<kEpiGeglu, true>, GemmCfg<true>::kThreads, GemmCfg<true>::kSmemBytes,
         &L->gemm_grid[0][1][0]},
        {(const void*)grouped_gemm_kernel<kEpiDown, true>, GemmCfg<true>::kThreads, GemmCfg<true>::kSmemBytes,
         &L->gemm_grid[1][1][0]},
        {(const void*)grouped_gemm_kernel<kEpiGeglu, false, kGemmMBPair>, GemmCfg<false, kGemmMBPair>::kThreads,
         GemmCfg<false, kGemmMBPair>::kSmemBytes, &L->gemm_grid[0][0][1]},
        {(const void*)grouped_gemm_kernel<kEpiDown, false, kGemmMBPair>, GemmCfg<false, kGemmMBPair>::kThreads,
         GemmCfg<false, kGemmMBPair>::kSmemBytes, &L->gemm_grid[1][0][1]},
        {(const void*)grouped_gemm_kernel<kEpiGeglu, true, kGemmMBPair>, GemmCfg<true, kGemmMBPair>::kThreads,
         GemmCfg<true, kGemmMBPair>::kSmemBytes, &L->gemm_grid[0][1][1]},
        {(const void*)grouped_gemm_kernel<kEpiDown, true, kGemmMBPair>, GemmCfg<true, kGemmMBPair>::kThreads,
         GemmCfg<true, kGemmMBPair>::kSmemBytes, &L->gemm_grid[1][1][1]},
    };
    for (int i = 0; i < 8 && s == MOE_OK; ++i) s = gemm_pairs(L, g[i].k, g[i].threads, g[i].smem, g[i].grid);
  }
  if (s == MOE_OK) {
    L->ring.resize(kProfRing);
    L->pending.assign(kProfRing, false);
    for (auto& r : L->ring)
      for (auto& ev : r)
        if (s == MOE_OK && cudaEventCreate(&ev) != cudaSuccess) s = fail(MOE_ERR_CUDA, "cudaEventCreate failed");
  }
  if (s != MOE_OK) {
    std::string msg = g_last_error;
    moe_layer_destroy(L);
    g_last_error = msg;
    return s;
  }
  *out = L;
  return ok();
}

moe_status_t moe_layer_destroy(moe_layer_t* L) {
  if (!L) return ok();
  DeviceGuard g(L->device);
  cudaDeviceSynchronize();
  for (auto& r : L->ring)
    for (auto& ev : r)
      if (ev) cudaEventDestroy(ev);
  if (L->ws) cudaFree(L->ws);
  if (L->host_stage) cudaFree(L->host_stage);
  for (int i = 0; i < 2; ++i) {
    if (L->async_stage[i]) cudaFree(L->async_stage[i]);
    if (L->in_ready[i]) cudaEventDestroy(L->in_ready[i]);
    if (L->fwd_done[i]) cudaEventDestroy(L->fwd_done[i]);
    if (L->slot_free[i]) cudaEventDestroy(L->slot_free[i]);
  }
  if (L->copy_in) cudaStreamDestroy(L->copy_in);
  if (L->copy_out) cudaStreamDestroy(L->copy_out);
  delete L;
  return ok();
}

moe_status_t moe_layer_forward(moe_layer_t* L, const void* hidden, void* out, int32_t T, void* stream,
                               int32_t* topk_idx, float* topk_prob, int32_t* expert_counts) {
  if (!L) return fail(MOE_ERR_INVALID_ARG, "null layer");
  if (T < 0 || T > L->cfg.max_tokens) return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, %d]", T, L->cfg.max_tokens);
  if (T == 0) return ok();
  if (!hidden || !out || !aligned16(hidden) || !aligned16(out))
    return fail(MOE_ERR_INVALID_ARG, "hidden/out null or not 16-byte aligned");
  if ((L->cfg.flags & MOE_FLAG_FORCE_GEMV) && T > kDecNS)
    return fail(MOE_ERR_INVALID_ARG, "MOE_FLAG_FORCE_GEMV handles T <= %d (got %d)", kDecNS, T);
  if ((topk_idx && !aligned4(topk_idx)) || (topk_prob && !aligned4(topk_prob)) ||
      (expert_counts && !aligned4(expert_counts)))
    return fail(MOE_ERR_INVALID_ARG, "optional output pointer misaligned");
  DeviceGuard g(L->device);
  if (!g.ok) return fail(MOE_ERR_CUDA, "cannot select device %d", L->device);
  return enqueue_forward(L, hidden, out, T, static_cast<cudaStream_t>(stream), topk_idx, topk_prob, expert_counts);
}

moe_status_t moe_layer_sync_status(moe_layer_t* L, void* stream) {
  if (!L) return fail(MOE_ERR_INVALID_ARG, "null layer");
  DeviceGuard g(L->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_CUDA_TRY(cudaStreamSynchronize(st));
  uint32_t h = 0;
  MOE_CUDA_TRY(cudaMemcpyAsync(&h, L->err, sizeof(h), cudaMemcpyDeviceToHost, st));
  MOE_CUDA_TRY(cudaStreamSynchronize(st));
  if (h) {
    MOE_CUDA_TRY(cudaMemsetAsync(L->err, 0, sizeof(uint32_t), st));
    MOE_CUDA_TRY(cudaStreamSynchronize(st));
    if (h & kErrTimeout) return fail(MOE_ERR_TIMEOUT, "a device wait ran out of time (error word 0x%x)", h);
    if (h & kErrCheck) return fail(MOE_ERR_DEVICE_CHECK, "a device index check failed (error word 0x%x)", h);
    return fail(MOE_ERR_DEVICE_CHECK,
                "an fp16 activation of an int8 layer passed +-65504 and was saturated (error word 0x%x)", h);
  }
  return ok();
}

moe_status_t moe_layer_forward_host(moe_layer_t* L, const void* hidden_host, void* out_host, int32_t T,
                                    void* stream, int32_t* topk_idx_host, float* topk_prob_host,
                                    int32_t* expert_counts_host) {
  if (!L) return fail(MOE_ERR_INVALID_ARG, "null layer");
  if (T < 0 || T > L->cfg.max_tokens) return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, %d]", T, L->cfg.max_tokens);
  if (T == 0) return ok();
  if (!hidden_host || !out_host) return fail(MOE_ERR_INVALID_ARG, "null host buffer");
  DeviceGuard g(L->device);
  if (!g.ok) return fail(MOE_ERR_CUDA, "cannot select device %d", L->device);
  const size_t d = (size_t)L->cfg.d_model, maxT = (size_t)L->cfg.max_tokens;
  const size_t x_bytes = align_up(maxT * d * 2, 1024), ip_bytes = align_up(maxT * 2 * 4, 1024);
  const size_t need = x_bytes + 2 * ip_bytes + 1024;
  if (!L->host_stage) {
    MOE_CUDA_TRY(cudaMalloc(&L->host_stage, need));
    L->host_stage_bytes = need;
  }
  char* b = static_cast<char*>(L->host_stage);
  void* xs = b;
  int32_t* is = reinterpret_cast<int32_t*>(b + x_bytes);
  float* ps = reinterpret_cast<float*>(b + x_bytes + ip_bytes);
  int32_t* cs = reinterpret_cast<int32_t*>(b + x_bytes + 2 * ip_bytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t nb = (size_t)T * d * 2;
  MOE_CUDA_TRY(cudaMemcpyAsync(xs, hidden_host, nb, cudaMemcpyHostToDevice, st));
  moe_status_t s = enqueue_forward(L, xs, xs, T, st, topk_idx_host ? is : nullptr, topk_prob_host ? ps : nullptr,
                                   expert_counts_host ? cs : nullptr);
  if (s != MOE_OK) return s;
  MOE_CUDA_TRY(cudaMemcpyAsync(out_host, xs, nb, cudaMemcpyDeviceToHost, st));
  if (topk_idx_host)
    MOE_CUDA_TRY(cudaMemcpyAsync(topk_idx_host, is, (size_t)T * 8, cudaMemcpyDeviceToHost, st));
  if (topk_prob_host)
    MOE_CUDA_TRY(cudaMemcpyAsync(topk_prob_host, ps, (size_t)T * 8, cudaMemcpyDeviceToHost, st));
  if (expert_counts_host)
    MOE_CUDA_TRY(cudaMemcpyAsync(expert_counts_host, cs, kNumExperts * 4, cudaMemcpyDeviceToHost, st));
  return moe_layer_sync_status(L, stream);
}

// Device staging of one asynchronous host call: x [max_T, d] bf16 (in place),
// topk_idx, topk_prob [max_T, 2], counts [E].
static size_t async_slot_bytes(const moe_layer* L, size_t* x_bytes, size_t* ip_bytes) {
  const size_t d = (size_t)L->cfg.d_model, maxT = (size_t)L->cfg.max_tokens;
  *x_bytes = align_up(maxT * d * 2, 1024);
  *ip_bytes = align_up(maxT * 2 * 4, 1024);
  return *x_bytes + 2 * *ip_bytes + 1024;
}

moe_status_t moe_layer_forward_host_async(moe_layer_t* L, const void* hidden_host, void* out_host, int32_t T,
                                          void* stream, int32_t* topk_idx_host, float* topk_prob_host,
                                          int32_t* expert_counts_host) {
  if (!L) return fail(MOE_ERR_INVALID_ARG, "null layer");
  if (T < 0 || T > L->cfg.max_tokens) return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, %d]", T, L->cfg.max_tokens);
  if (T == 0) return ok();
  if (!hidden_host || !out_host) return fail(MOE_ERR_INVALID_ARG, "null host buffer");
  DeviceGuard g(L->device);
  if (!g.ok) return fail(MOE_ERR_CUDA, "cannot select device %d", L->device);
  size_t x_bytes = 0, ip_bytes = 0;
  const size_t need = async_slot_bytes(L, &x_bytes, &ip_bytes);
  if (!L->copy_in) {  // first call: two staging slots, two copy streams, events
    for (int i = 0; i < 2; ++i) {
      MOE_CUDA_TRY(cudaMalloc(&L->async_stage[i], need));
      MOE_CUDA_TRY(cudaEventCreateWithFlags(&L->in_ready[i], cudaEventDisableTiming));
      MOE_CUDA_TRY(cudaEventCreateWithFlags(&L->fwd_done[i], cudaEventDisableTiming));
      MOE_CUDA_TRY(cudaEventCreateWithFlags(&L->slot_free[i], cudaEventDisableTiming));
    }
    MOE_CUDA_TRY(cudaStreamCreateWithFlags(&L->copy_out, cudaStreamNonBlocking));
    MOE_CUDA_TRY(cudaStreamCreateWithFlags(&L->copy_in, cudaStreamNonBlocking));
  }
  const int slot = L->async_slot;
  L->async_slot ^= 1;
  char* b = static_cast<char*>(L->async_stage[slot]);
  void* xs = b;
  int32_t* is = reinterpret_cast<int32_t*>(b + x_bytes);
  float* ps = reinterpret_cast<float*>(b + x_bytes + ip_bytes);
  int32_t* cs = reinterpret_cast<int32_t*>(b + x_bytes + 2 * ip_bytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t nb = (size_t)T * L->cfg.d_model * 2;
  // input copy once this slot's previous output copy is done (slot_free), the
  // forward on the caller's stream once the input landed, the output copy once
  // the forward is done; consecutive calls overlap one's copies with the
  // other's forward
  if (L->async_pending) MOE_CUDA_TRY(cudaStreamWaitEvent(L->copy_in, L->slot_free[slot], 0));
  MOE_CUDA_TRY(cudaMemcpyAsync(xs, hidden_host, nb, cudaMemcpyHostToDevice, L->copy_in));
  MOE_CUDA_TRY(cudaEventRecord(L->in_ready[slot], L->copy_in));
  MOE_CUDA_TRY(cudaStreamWaitEvent(st, L->in_ready[slot], 0));
  moe_status_t s = enqueue_forward(L, xs, xs, T, st, topk_idx_host ? is : nullptr, topk_prob_host ? ps : nullptr,
                                   expert_counts_host ? cs : nullptr);
  if (s != MOE_OK) return s;
  MOE_CUDA_TRY(cudaEventRecord(L->fwd_done[slot], st));
  MOE_CUDA_TRY(cudaStreamWaitEvent(L->copy_out, L->fwd_done[slot], 0));
  MOE_CUDA_TRY(cudaMemcpyAsync(out_host, xs, nb, cudaMemcpyDeviceToHost, L->copy_out));
  if (topk_idx_host)
    MOE_CUDA_TRY(cudaMemcpyAsync(topk_idx_host, is, (size_t)T * 8, cudaMemcpyDeviceToHost, L->copy_out));
  if (topk_prob_host)
    MOE_CUDA_TRY(cudaMemcpyAsync(topk_prob_host, ps, (size_t)T * 8, cudaMemcpyDeviceToHost, L->copy_out));
  if (expert_counts_host)
    MOE_CUDA_TRY(cudaMemcpyAsync(expert_counts_host, cs, kNumExperts * 4, cudaMemcpyDeviceToHost, L->copy_out));
  MOE_CUDA_TRY(cudaEventRecord(L->slot_free[slot], L->copy_out));
  L->async_pending = true;
  return ok();
}

moe_status_t moe_layer_host_wait(moe_layer_t* L, void* stream) {
  if (!L) return fail(MOE_ERR_INVALID_ARG, "null layer");
  DeviceGuard g(L->device);
  if (L->copy_out) MOE_CUDA_TRY(cudaStreamSynchronize(L->copy_out));
  return moe_layer_sync_status(L, stream);
}

moe_status_t moe_layer_set_profiling(moe_layer_t* L, int32_t enable) {
  if (!L) return fail(MOE_ERR_INVALID_ARG, "null layer");
  L->profiling = enable != 0;
  return ok();
}

moe_status_t moe_layer_profile_read(moe_layer_t* L, double* ms_total, int64_t* launches, int32_t reset) {
  if (!L) return fail(MOE_ERR_INVALID_ARG, "null layer");
  DeviceGuard g(L->device);
  for (int s = 0; s < kProfRing; ++s) harvest(L, s);
  for (int k = 0; k < MOE_K_COUNT; ++k) {
    if (ms_total) ms_total[k] = L->prof_ms[k];
    if (launches) launches[k] = L->prof_n[k];
  }
  if (reset)
    for (int k = 0; k < MOE_K_COUNT; ++k) {
      L->prof_ms[k] = 0.0;
      L->prof_n[k] = 0;
    }
  return ok();
}

moe_status_t moe_layer_router_stats(moe_layer_t* L, float* stats, void* stream) {
  if (!L || !stats) return fail(MOE_ERR_INVALID_ARG, "null argument");
  if (!aligned4(stats)) return fail(MOE_ERR_INVALID_ARG, "stats not 4-byte aligned");
  if (L->last_T < 1) return fail(MOE_ERR_INVALID_ARG, "no forward with T > 0 has been enqueued on this handle");
  DeviceGuard g(L->device);
  if (!g.ok) return fail(MOE_ERR_CUDA, "cannot select device %d", L->device);
  router_stats_kernel<<<1, 32 * kNumExperts, 0, static_cast<cudaStream_t>(stream)>>>(L->p_part, L->last_T, L->last_T,
                                                                                      stats);
  L->launches += 1;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return ok();
}

moe_status_t moe_layer_gemm_grid(const moe_layer_t* L, int32_t grid[4]) {
  if (!L || !grid) return fail(MOE_ERR_INVALID_ARG, "null argument");
  const int pr = L->pair_mblocks ? 1 : 0;  // the kernels a forward with T >= kPairMinT launches
  grid[0] = L->gemm_grid[kEpiGeglu][0][pr];
  grid[1] = L->gemm_grid[kEpiDown][0][pr];
  grid[2] = L->gemm_grid[kEpiGeglu][1][pr];
  grid[3] = L->gemm_grid[kEpiDown][1][pr];
  return ok();
}

int64_t moe_layer_launch_count(const moe_layer_t* L) { return L ? L->launches.load() : 0; }

moe_status_t moe_layer_workspace(const moe_layer_t* L, moe_workspace_view_t* v) {
  if (!L || !v) return fail(MOE_ERR_INVALID_ARG, "null argument");
  v->rnorm = L->rnorm;
  v->counts = L->sched;
  v->row_offset = L->sched + kNumExperts;
  v->row_of_slot = L->row_of_slot;
  v->xn_perm = L->xn_perm;
  v->act = L->act;
  v->y_rows = L->y_rows;
  v->rows_cap = L->rows_cap;
  return ok();
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Allocation-free grouping of routed slots (moe_group_slots_noalloc).
//
// Some callers cannot call cudaMalloc: a serving runtime that reserved all free
// device memory for its own pool at start-up, or a plugin host that hands an op
// only its input and output buffers.  There cudaMalloc either fails or stalls the
// device in the middle of a latency-critical step.  This entry point runs the
// grouping kernel with its scratch (schedule block, row -> token map, row
// weights) in the file-scope array below instead of a handle's workspace.
//
// The array is modest (see kNoAllocScratchBytes) and every GPU that loads this
// library holds it until the process exits.  Host code cannot use the array's
// name as a device address: the first call on each device asks the runtime for
// the address (cudaGetSymbolAddress, with that device current) and caches it.
namespace {
constexpr int kNoAllocMaxTokens = 16384;
constexpr int kNoAllocRows = 2 * kNoAllocMaxTokens + kNumExperts * kRowPad;
constexpr size_t kNoAllocSchedBytes = 256;  // kSchedInts int32, padded
// schedule block, then token_of_row and prob_of_row of every permuted row
constexpr size_t kNoAllocScratchBytes = kNoAllocSchedBytes + 2 * (size_t)kNoAllocRows * 4;
static_assert(kNoAllocScratchBytes == 270592, "the size stated in moe_layer.h");
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

extern "C" moe_status_t moe_group_slots_noalloc(const int32_t* topk_idx, const float* topk_prob, int32_t T,
                                                int32_t* expert_counts, int32_t* row_of_slot, void* stream) {
  if (T < 0 || T > kNoAllocMaxTokens)
    return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, %d], the limit of the static scratch array", T,
                kNoAllocMaxTokens);
  if (T == 0) return ok();
  if (!topk_idx || !topk_prob || !expert_counts || !row_of_slot)
    return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned4(topk_idx) || !aligned4(topk_prob) || !aligned4(expert_counts) || !aligned4(row_of_slot))
    return fail(MOE_ERR_INVALID_ARG, "pointer argument not 4-byte aligned");
  int dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p)
        return fail(MOE_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s", cudaGetErrorString(e));
      g_noalloc_addr[dev] = p;
    }
    base = g_noalloc_addr[dev];
  }
  char* b = static_cast<char*>(base);
  int32_t* sched = reinterpret_cast<int32_t*>(b);
  int32_t* token_of_row = reinterpret_cast<int32_t*>(b + kNoAllocSchedBytes);
  float* prob_of_row = reinterpret_cast<float*>(b + kNoAllocSchedBytes + (size_t)kNoAllocRows * 4);
  // Index checks on: the indices come from the caller, and an out-of-range one
  // is counted as expert 0 instead of indexing past the arrays.  No error word
  // is passed, so such an index is not reported (the header says so).  The
  // kernel writes every scratch word it later reads, so nothing needs clearing.
  permute_kernel<<<1, kPermuteThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      topk_idx, topk_prob, T, sched, row_of_slot, token_of_row, prob_of_row, expert_counts, kNoAllocRows, 1,
      nullptr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return ok();
}
