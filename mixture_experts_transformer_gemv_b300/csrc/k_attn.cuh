// Kernels of the attention half of a Grok-1 decoder layer (sm_103a).
//
// Per causal sequence x [T, d] ("Jah-yee/grok" README, architecture diagram:
// grouped-query attention, 48 query and 8 key/value heads, rotary embeddings,
// RMSNorm; "TevunahAi/Grok-1-BF16", "Grok-1 Specific Behaviors": logits
// hard-clamped to [-30, 30] before the softmax, pre- and post-attention norms;
// "Weight Verification": q_proj [6144, 6144], k_proj / v_proj [1024, 6144],
// o_proj [6144, 6144], so heads of 128):
//
//   A1 attn_prenorm_kernel   xn = fp16(RMSNorm_pre(x)) and the one-group GEMM schedule
//   A2 grouped_gemm<down>    qkv = xn [Wq; Wk; Wv]^T, fp16 operands, fp32 out (tcgen05, CTA pairs)
//   A3 rope_layout_kernel    Q, K rotated (RoFormer pairs (2i, 2i + 1)) in fp16, V transposed in bf16
//   A4 attn_kernel           ctx = softmax(clamp(Q K^T / sqrt(128))) V, causal (tcgen05)
//   A5 grouped_gemm<down>    o = ctx Wo^T, fp32                           (tcgen05, CTA pairs)
//   A6 attn_post_kernel      y = x + RMSNorm_post(o)
//
// A4 needs no running maximum: every clamped logit lies in [-c, c], so
// exp(s - c) lies in [exp(-2c), 1] (normal in fp32 and bf16 for c <= 40) and
// the softmax is sum_j exp(s_j - c) v_j / sum_j exp(s_j - c) exactly, without
// the rescaling of the accumulator a flash-attention kernel does when the
// maximum grows.
//
// Precision: the logits are the sensitive part (their error scales with |q||k|),
// so the path that feeds them (xn, Wq, Wk, q, k) is carried in fp16, 3 mantissa
// bits more than bf16 at the same tensor-core rate, with saturation at +-65504.
// The softmax weights, V and ctx stay bf16: the weights go down to exp(-2c) =
// 8.8e-27, below fp16's range, and both operands of one MMA share a type.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"
#include "ptx_pair.cuh"
#include "ptx_tmem.cuh"

namespace moe {

constexpr int kAttnDh = 128;                         // head dimension
constexpr int kAttnBM = 128;                         // queries of one tile (TMEM lanes)
constexpr int kAttnBN = 128;                         // keys of one block
constexpr int kAttnKStages = 3;                      // K ring stages
constexpr int kAttnVStages = 2;                      // V^T ring stages
constexpr int kAttnTile = kAttnBM * kAttnDh * 2;     // 32 KB: 128 rows x 128 16-bit values, two 64-column boxes
constexpr int kAttnHalf = kAttnTile / 2;             // one box of 128 rows x 64 values, 128-byte swizzle
constexpr int kAttnSoftmaxWarps = 16;                // eight per query tile: two per TMEM lane quarter, 64 keys each
constexpr int kAttnSoftmaxThreads = 32 * kAttnSoftmaxWarps;
constexpr int kAttnThreads = 64 + kAttnSoftmaxThreads;  // warp 0 TMA, warp 1 MMA, warps 2-9 softmax + epilogue
// q_full, q_empty, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2], p_full[2], o_full, o_empty, drain
constexpr int kAttnNumBars = 2 + 2 * kAttnKStages + 2 * kAttnVStages + 4 + 3;
constexpr size_t kAttnBarBytes = 256;                // barriers, TMEM address, abort flag
constexpr size_t kAttnSmemBytes =
    1024 + (size_t)kAttnTile * (2 + kAttnKStages + kAttnVStages) + kAttnBarBytes + 2 * kAttnBM * sizeof(float);
static_assert(8 * kAttnNumBars + 8 <= kAttnBarBytes, "barrier block");
constexpr uint32_t kAttnTmemCols = 512;              // O_A | O_B | S_A | S_B (P_t over columns [0,32) and [64,96) of S_t)
constexpr uint32_t kAttnColO = 0, kAttnColS = 256;
constexpr uint32_t kAttnIdesc = idesc_bf16_f32(kAttnBM, kAttnBN);  // P V: bf16 x bf16
// Q K^T: fp16 x fp16 (format 0 in bits 7-9 and 10-12), fp32 accumulator
constexpr uint32_t kAttnIdescF16 = (1u << 4) | (static_cast<uint32_t>(kAttnBN >> 3) << 17) |
                                   (static_cast<uint32_t>(kAttnBM >> 4) << 24);
static_assert(kAttnBN == kAttnDh, "S and O share the instruction shape");
static_assert(kAttnSmemBytes <= 232448, "fits one CTA per SM");

struct AttnParams {
  int T;               // sequence length
  int t_stride;        // rows per head of Q and K, columns of Vt (multiple of 256)
  int n_q_heads;       // query heads
  int group;           // query heads per key/value head
  int n_qpairs;        // ceil(T / 256): pairs of query tiles
  float sat_scale;     // log2(e) / (sqrt(128) 2 c log2(e)) = 1 / (2 c sqrt(128))
  float clamp2_log2;   // 2 c log2(e)
  __nv_bfloat16* ctx;  // [rows, n_q_heads * 128]
  int ctx_ld;
  uint32_t* err;
  uint64_t timeout_ns;
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Bounded wait that lets the warp sleep: each try_wait may suspend the thread
// until the phase completes or about 0.5 ms pass, so waiting warps take no
// issue slots from the working ones.  Gives up (false) after limit_ns or when
// *abort becomes non-zero, like wait_bounded.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(500000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool wait_sleep(uint32_t bar, uint32_t parity, const volatile uint32_t* abort,
                                           uint64_t limit_ns) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Named barrier over `count` threads (whole warps) of this CTA.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// a * b + c clamped to [0, 1]
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float r;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// two fp32 in one 64-bit register (lo in the low half) and packed arithmetic on them
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Work item i (heaviest first): the query tiles qa = 2 (n_qpairs - 1 - i / Hq)
// and qb = qa + 1 of head h = i % Hq, i.e. 256 queries against the key blocks
// 0..qb.  The kernel is persistent: CTA c takes items c, 2G - 1 - c, 2G + c,
// 4G - 1 - c, ... (G CTAs, alternating direction so long and short items even out).
__device__ __forceinline__ int attn_item_of(int c, int k, int G) {
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Per CTA, one item after another, two query tiles A and B sharing every K and
// V^T block (half the key traffic per flop of one tile per CTA):
//  - warp 0 (TMA): Q_A and Q_B (reloaded as soon as the item's last Q K^T
//    product is done), K blocks through a 3-stage ring and V^T blocks through a
//    2-stage ring, each V^T issued after the next block's K so a wait for a V^T
//    stage never holds back keys;
//  - warp 1 (MMA): S_A(0), S_B(0), then per block j: P V_A(j), S_A(j+1),
//    P V_B(j), S_B(j+1).  The tensor cores work on one tile while the softmax
//    of the other runs.  P_t (bf16) is written over S_t (see below) and read
//    from TMEM as the A operand of P V_t; the tensor core runs one
//    CTA's MMAs in issue order, so S_t(j+1), issued after P V_t(j), overwrites
//    P_t(j) only after it was read;
//  - warps 2-9 (tile A) and 10-17 (tile B): two threads per query row (keys
//    0-63 and 64-127 of a block) turn S_t(j) into P_t(j); each writes its 32
//    columns of P over S columns it read itself ([0,32) and [64,96)), so no
//    thread overwrites S another has not read; at the end of the item the two
//    row sums meet in shared memory and ctx = O_t / l is written.
// Ring, buffer and phase counters run across items.
//
// Softmax weight of a logit s (c' = c log2(e)):
//   2^(clamp(s log2(e) / sqrt(128), -c', c') - c') = 2^(2c' (u - 1)),
//   u = saturate(s / (2 c sqrt(128)) + 1/2)
// one saturating FMA per value, one packed FMA per pair, then ex2.
__global__ void __maxnreg__(96)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_vt, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                   // Q_A, Q_B (fp16)
  uint8_t* sK = smem + 2 * (size_t)kAttnTile;           // K ring (fp16)
  uint8_t* sV = sK + (size_t)kAttnKStages * kAttnTile;  // V^T ring (bf16)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kAttnTile * (2 + kAttnKStages + kAttnVStages));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kAttnNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  float* l_row = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + kAttnBarBytes);  // [tile][128]
  const uint32_t b0 = smem_addr(bars);
  const uint32_t q_full = b0, q_empty = b0 + 8u;
  auto k_full = [&](int s) { return b0 + 8u * (2 + s); };
  auto k_empty = [&](int s) { return b0 + 8u * (2 + kAttnKStages + s); };
  auto v_full = [&](int s) { return b0 + 8u * (2 + 2 * kAttnKStages + s); };
  auto v_empty = [&](int s) { return b0 + 8u * (2 + 2 * kAttnKStages + kAttnVStages + s); };
  auto s_full = [&](int t) { return b0 + 8u * (2 + 2 * kAttnKStages + 2 * kAttnVStages + t); };
  auto p_full = [&](int t) { return b0 + 8u * (4 + 2 * kAttnKStages + 2 * kAttnVStages + t); };
  const uint32_t o_full = b0 + 8u * (6 + 2 * kAttnKStages + 2 * kAttnVStages);
  const uint32_t o_empty = o_full + 8u;
  const uint32_t drain = o_full + 16u;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = (int)gridDim.x, n_items = p.n_qpairs * p.n_q_heads;
  auto item_qa = [&](int i) { return 2 * (p.n_qpairs - 1 - i / p.n_q_heads); };
  auto item_h = [&](int i) { return i % p.n_q_heads; };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kAttnKStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < kAttnVStages; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), kAttnSoftmaxThreads / 2);  // every thread of the tile's group
    }
    mbar_init(o_full, 1);
    mbar_init(o_empty, kAttnSoftmaxWarps);  // one arrival per softmax warp
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_vt);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kAttnTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      bool ok = true;
      int n_k = 0, n_v = 0, n_q = 0;  // K and V^T blocks issued (across items), Q pairs issued
      int pend_g = -1, pend_j = 0;    // the V^T block issued after the next K
      auto load_v = [&]() -> bool {
        const int s = n_v % kAttnVStages;
        if (n_v >= kAttnVStages &&
            !wait_sleep(v_empty(s), (uint32_t)((n_v / kAttnVStages) - 1) & 1u, abort_flag, p.timeout_ns))
          return false;
        mbar_arrive_expect_tx(v_full(s), kAttnTile);
        uint8_t* dst = sV + (size_t)s * kAttnTile;
        tma_load_2d(smem_addr(dst), &tm_vt, v_full(s), pend_j * kAttnBN, pend_g * kAttnDh);
        tma_load_2d(smem_addr(dst + kAttnHalf), &tm_vt, v_full(s), pend_j * kAttnBN + 64, pend_g * kAttnDh);
        ++n_v;
        pend_g = -1;
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int i = attn_item_of((int)blockIdx.x, k, G);
        if (i >= n_items) break;
        const int qa = item_qa(i), h = item_h(i), g = h / p.group;
        if (pend_g >= 0 && !load_v()) {  // the previous item's last V^T
          ok = false;
          break;
        }
        // the previous item's Q K^T products are done with the Q buffers
        if (k > 0 && !wait_sleep(q_empty, (uint32_t)(k - 1) & 1u, abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * kAttnTile);
        const int qrow0 = h * p.t_stride + qa * kAttnBM;
        tma_load_2d(smem_addr(sQ), &tm_q, q_full, 0, qrow0);
        tma_load_2d(smem_addr(sQ + kAttnHalf), &tm_q, q_full, 64, qrow0);
        tma_load_2d(smem_addr(sQ + kAttnTile), &tm_q, q_full, 0, qrow0 + kAttnBM);
        tma_load_2d(smem_addr(sQ + kAttnTile + kAttnHalf), &tm_q, q_full, 64, qrow0 + kAttnBM);
        n_q = k + 1;
        for (int j = 0; j <= qa + 1; ++j) {
          const int s = n_k % kAttnKStages;
          if (n_k >= kAttnKStages &&
              !wait_sleep(k_empty(s), (uint32_t)((n_k / kAttnKStages) - 1) & 1u, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(k_full(s), kAttnTile);
          const int krow = g * p.t_stride + j * kAttnBN;
          tma_load_2d(smem_addr(sK + (size_t)s * kAttnTile), &tm_k, k_full(s), 0, krow);
          tma_load_2d(smem_addr(sK + (size_t)s * kAttnTile + kAttnHalf), &tm_k, k_full(s), 64, krow);
          ++n_k;
          if (pend_g >= 0 && !load_v()) {
            ok = false;
            break;
          }
          pend_g = g;
          pend_j = j;
        }
      }
      if (ok && pend_g >= 0) ok = load_v();
      // every release of a stage by the MMA issuer has landed before exit
      for (int b = (n_k > kAttnKStages ? n_k - kAttnKStages : 0); b < n_k && ok; ++b)
        if (!wait_sleep(k_empty(b % kAttnKStages), (uint32_t)(b / kAttnKStages) & 1u, abort_flag, p.timeout_ns))
          ok = false;
      for (int b = (n_v > kAttnVStages ? n_v - kAttnVStages : 0); b < n_v && ok; ++b)
        if (!wait_sleep(v_empty(b % kAttnVStages), (uint32_t)(b / kAttnVStages) & 1u, abort_flag, p.timeout_ns))
          ok = false;
      if (!ok) {
        raise_abort(abort_flag, p.err);
        // this role's copies still in flight land before the CTA exits
        if (n_q > 0) wait_sleep(q_full, (uint32_t)(n_q - 1) & 1u, nullptr, p.timeout_ns);
        for (int b = (n_k > kAttnKStages ? n_k - kAttnKStages : 0); b < n_k; ++b)
          wait_sleep(k_full(b % kAttnKStages), (uint32_t)(b / kAttnKStages) & 1u, nullptr, p.timeout_ns);
        for (int b = (n_v > kAttnVStages ? n_v - kAttnVStages : 0); b < n_v; ++b)
          wait_sleep(v_full(b % kAttnVStages), (uint32_t)(b / kAttnVStages) & 1u, nullptr, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      bool ok = true;
      int gb = 0;           // first K/V block of the current item (across items)
      int na_tot = 0;       // tile-A blocks before this item (phases of s_full(0), p_full(0))
      int nb_tot = 0;       // tile-B blocks before this item (phases of s_full(1), p_full(1))
      // S_t = Q_t K_b^T into tile t's S buffer
      auto issue_s = [&](int t, int b) {
        const uint32_t qa = smem_addr(sQ + (size_t)t * kAttnTile);
        const uint32_t kb = smem_addr(sK + (size_t)(b % kAttnKStages) * kAttnTile);
        const uint32_t d = tmem_base + kAttnColS + (uint32_t)t * kAttnBN;
#pragma unroll
        for (int kk = 0; kk < kAttnDh / 16; ++kk)  // K = 16 along the head dimension
          umma_bf16(d, smem_desc_k_sw128(qa + (kk >> 2) * kAttnHalf) + 2 * (kk & 3),
                    smem_desc_k_sw128(kb + (kk >> 2) * kAttnHalf) + 2 * (kk & 3), kAttnIdescF16, kk != 0);
        umma_commit(s_full(t));
      };
      // O_t += P_t V_b
      auto issue_pv = [&](int t, int b, bool acc) {
        const uint32_t vb = smem_addr(sV + (size_t)(b % kAttnVStages) * kAttnTile);
        // P_t: keys 0-63 in S_t columns [0,32), keys 64-127 in [64,96)
        const uint32_t pa = tmem_base + kAttnColS + (uint32_t)t * kAttnBN;
        const uint32_t d = tmem_base + kAttnColO + (uint32_t)t * kAttnBN;
#pragma unroll
        for (int kk = 0; kk < kAttnBN / 16; ++kk)  // K = 16 keys: 8 TMEM columns of P
          umma_bf16_tmem_a(d, pa + (kk >> 2) * 64 + 8 * (kk & 3),
                           smem_desc_k_sw128(vb + (kk >> 2) * kAttnHalf) + 2 * (kk & 3), kAttnIdesc,
                           (acc || kk != 0) ? 1u : 0u);
      };
      auto wait_k = [&](int b) {
        const bool got = wait_sleep(k_full(b % kAttnKStages), (uint32_t)(b / kAttnKStages) & 1u, abort_flag,
                                    p.timeout_ns);
        tc_fence_after_sync();
        return got;
      };
      for (int k = 0; ok; ++k) {
        const int i = attn_item_of((int)blockIdx.x, k, G);
        if (i >= n_items) break;
        const int na = item_qa(i) + 1, nb = na + 1;  // key blocks of tile A (0..qa) and tile B (0..qa+1)
        if (!wait_sleep(q_full, (uint32_t)k & 1u, abort_flag, p.timeout_ns) || !wait_k(gb)) {
          ok = false;
          break;
        }
        issue_s(0, gb);
        issue_s(1, gb);
        umma_commit(k_empty(gb % kAttnKStages));
        for (int j = 0; j < nb && ok; ++j) {
          const int b = gb + j;
          // the V^T block of j (both tiles' P V read it)
          if (!wait_sleep(v_full(b % kAttnVStages), (uint32_t)(b / kAttnVStages) & 1u, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          if (j < na) {
            // tile A: P V_A(j), then S_A(j+1) over the buffer P V_A(j) just read
            if (!wait_sleep(p_full(0), (uint32_t)(na_tot + j) & 1u, abort_flag, p.timeout_ns) ||
                (j == 0 && k > 0 && !wait_sleep(o_empty, (uint32_t)(k - 1) & 1u, abort_flag, p.timeout_ns))) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            issue_pv(0, b, j > 0);
          }
          const bool more = j + 1 < nb;
          if (more) {
            if (!wait_k(b + 1)) {
              ok = false;
              break;
            }
            if (j + 1 < na) issue_s(0, b + 1);
          }
          // tile B: P V_B(j), then S_B(j+1)
          // (O_B is free too: every softmax warp arrived on o_empty, which P V_A(0) waited for)
          if (!wait_sleep(p_full(1), (uint32_t)(nb_tot + j) & 1u, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_pv(1, b, j > 0);
          umma_commit(v_empty(b % kAttnVStages));  // both tiles' products of block j are issued
          if (more) {
            issue_s(1, b + 1);
            umma_commit(k_empty((b + 1) % kAttnKStages));
            if (j + 2 == nb) umma_commit(q_empty);  // the item's last Q K^T product is issued
          }
        }
        if (!ok) break;
        umma_commit(o_full);
        gb += nb;
        na_tot += na;
        nb_tot += nb;
      }
      // all MMAs issued by this thread are complete before TMEM is freed
      umma_commit(drain);
      if (!wait_sleep(drain, 0, nullptr, p.timeout_ns)) ok = false;
      if (!ok) raise_abort(abort_flag, p.err);
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    const int q4 = warp & 3;             // TMEM lanes [32 q4, 32 q4 + 32) are reachable from this warp
    const int t = (warp - 2) >> 3;       // query tile: 0 = A, 1 = B
    const int half = ((warp - 2) >> 2) & 1;  // keys [64 half, 64 half + 64) of each block; O columns likewise
    const int r = q4 * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t sb = tmem_base + lane_off + kAttnColS + (uint32_t)t * kAttnBN + half * 64;  // this half of S_t
    const uint32_t ob = tmem_base + lane_off + kAttnColO + (uint32_t)t * kAttnBN + half * 64;  // this half of O_t
    const float ss = p.sat_scale;
    const uint64_t w2 = f32x2(p.clamp2_log2, p.clamp2_log2), mw2 = f32x2(-p.clamp2_log2, -p.clamp2_log2);
    bool ok = true;
    int n_tot = 0;  // this tile's blocks before the current item
    for (int k = 0;; ++k) {
      const int i = attn_item_of((int)blockIdx.x, k, G);
      if (i >= n_items) break;
      const int qt = item_qa(i) + t, h = item_h(i), nblk = qt + 1;
      uint64_t l2 = f32x2(0.f, 0.f);
      for (int j = 0; j < nblk && ok; ++j) {
        if (!__all_sync(0xffffffffu, wait_sleep(s_full(t), (uint32_t)(n_tot + j) & 1u, abort_flag, p.timeout_ns))) {
          ok = false;
          if (lane == 0) raise_abort(abort_flag, p.err);
          break;
        }
        tc_fence_after_sync();
        const bool diag = (j == qt);  // the only block with keys after some queries
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {  // 32 keys at a time
          uint32_t sv[32];
          tmem_ld_32x32b_x32(sb + cc * 32, sv);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const uint64_t t2 = fma_f32x2(f32x2(fma_sat(__uint_as_float(sv[2 * c]), ss, 0.5f),
                                                fma_sat(__uint_as_float(sv[2 * c + 1]), ss, 0.5f)),
                                          w2, mw2);
            float t0, t1;
            f32x2_split(t2, t0, t1);
            float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
            if (diag) {
              const int key = half * 64 + cc * 32 + 2 * c;
              if (key > r) p0 = 0.f;
              if (key + 1 > r) p1 = 0.f;
            }
            l2 = add_f32x2(l2, f32x2(p0, p1));
            pk[c] = pack_bf16x2(p0, p1);
          }
          // 16 P columns over S columns this thread has already read
          tmem_st_32x32b_x16(sb + cc * 16, pk);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(p_full(t));
      }
      n_tot += nblk;
      const bool got = ok && __all_sync(0xffffffffu, wait_sleep(o_full, (uint32_t)k & 1u, abort_flag, p.timeout_ns));
      float la, lb;
      f32x2_split(l2, la, lb);
      const float l_mine = la + lb;
      if (half == 1) l_row[t * kAttnBM + r] = l_mine;
      // every softmax thread reaches this barrier once per item (a thread that
      // gave up takes all of them out together); it also publishes the second
      // halves' row sums
      ok = named_bar_and(1, kAttnSoftmaxThreads, got);
      if (!ok) break;
      if (half == 0) l_row[t * kAttnBM + r] += l_mine;
      named_bar_sync(1, kAttnSoftmaxThreads);  // the whole row sums are in place
      tc_fence_after_sync();
      const float inv = 1.f / l_row[t * kAttnBM + r];
      const int qrow = qt * kAttnBM + r;
      __nv_bfloat16* dst = p.ctx + (size_t)qrow * p.ctx_ld + (size_t)h * kAttnDh + half * 64;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(ob + cc * 32, o);
        tmem_ld_wait();
        if (cc == 1) {
          // this warp's reads of O and of the row sums are done: the next item may overwrite them
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_empty);
        }
        if (qrow < p.T) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
          uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
    }
    if (!ok && lane == 0) raise_abort(abort_flag, p.err);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kAttnTmemCols);
  }
}

// A1: xn[t] = fp16(x[t] / sqrt(mean(x[t]^2) + eps) * s) for t < T, zero rows for
// T <= t < rows_pad; block 0 also writes the schedule that makes the grouped
// GEMM one dense GEMM (group 0 holds rows [0, rows_pad), the others none).
// One block of 256 threads per row; d a multiple of 8.
__global__ void __launch_bounds__(256) attn_prenorm_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const float* __restrict__ s, float eps, int T,
                                                           int rows_pad, int d, __half* __restrict__ xn,
                                                           int32_t* __restrict__ sched) {
  const int t = blockIdx.x;
  if (t == 0 && threadIdx.x < kSchedInts)
    sched[threadIdx.x] = threadIdx.x == 0 ? T : (threadIdx.x < kNumExperts ? 0 : (threadIdx.x == kNumExperts ? 0 : rows_pad));
  uint4* dst = reinterpret_cast<uint4*>(xn + (size_t)t * d);
  const int nv = d / 8;
  if (t >= T) {
    for (int i = threadIdx.x; i < nv; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
  float ss = 0.f;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = bf16_lo(w[k]), b = bf16_hi(w[k]);
      ss = fmaf(a, a, fmaf(b, b, ss));
    }
  }
  __shared__ float red[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float rr = rsqrtf(tot / (float)d + eps);
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const float4 s0 = reinterpret_cast<const float4*>(s)[2 * i];
    const float4 s1 = reinterpret_cast<const float4*>(s)[2 * i + 1];
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      o[k] = pack_f16x2_sat(bf16_lo(w[k]) * rr * sv[2 * k], bf16_hi(w[k]) * rr * sv[2 * k + 1]);
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// In-place bf16 -> fp16 of n values (round to nearest, saturating; values
// below 2^-14 in magnitude become fp16 subnormals).
__global__ void bf16_to_f16_kernel(uint32_t* p, int64_t n_pairs) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_pairs; i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t u = p[i];
    p[i] = pack_f16x2_sat(bf16_lo(u), bf16_hi(u));
  }
}

// Rotation table: cs[t * 64 + i] = (cos, sin)(t * base^(-2i / 128)), angles in fp64.
__global__ void rope_table_kernel(float2* cs, int n_pos, double base) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_pos * (kAttnDh / 2)) return;
  const int t = idx / (kAttnDh / 2), i = idx % (kAttnDh / 2);
  const double a = (double)t * pow(base, -2.0 * (double)i / (double)kAttnDh);
  double sn, cn;
  sincos(a, &sn, &cn);
  cs[idx] = make_float2((float)cn, (float)sn);
}

__global__ void fill_f32_kernel(float* p, float v, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = v;
}

// A3: from qkv fp32 [T, ld] (query heads, then key heads, then value heads, 128
// columns each) write Q [Hq][t_stride][128] and K [Hkv][t_stride][128] rotated
// (pair (2i, 2i + 1) of each head turned by t * base^(-2i/128)) in fp16
// (saturating) and Vt [Hkv][128][t_stride] (V transposed: keys along rows) in bf16; token rows
// T <= t < gridDim.x * 32 are written as zeros.  Grid (ceil(T / 256) * 8,
// Hq + 2 Hkv), 256 threads: 32 tokens x one head per block.
__global__ void __launch_bounds__(256) rope_layout_kernel(const float* __restrict__ qkv, int ld,
                                                          const float2* __restrict__ cs, int T, int t_stride, int Hq,
                                                          int Hkv, __half* __restrict__ Q,
                                                          __half* __restrict__ K,
                                                          __nv_bfloat16* __restrict__ Vt) {
  __shared__ float vt[kAttnDh][33];
  const int t0 = blockIdx.x * 32, col = blockIdx.y;
  const int tl = threadIdx.x >> 3, part = threadIdx.x & 7;  // token of the block, 16 columns of the head
  const int t = t0 + tl;
  float v[16];
  if (t < T) {
    const float4* src = reinterpret_cast<const float4*>(qkv + (size_t)t * ld + (size_t)col * kAttnDh + part * 16);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 a = src[k];
      v[4 * k] = a.x;
      v[4 * k + 1] = a.y;
      v[4 * k + 2] = a.z;
      v[4 * k + 3] = a.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = 0.f;
  }
  if (col < Hq + Hkv) {
    if (t < T) {
      const float2* c = cs + (size_t)t * (kAttnDh / 2) + part * 8;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 e = c[k];
        const float x0 = v[2 * k], x1 = v[2 * k + 1];
        v[2 * k] = x0 * e.x - x1 * e.y;
        v[2 * k + 1] = x0 * e.y + x1 * e.x;
      }
    }
    __half* dst = col < Hq ? Q + ((size_t)col * t_stride + t) * kAttnDh
                           : K + ((size_t)(col - Hq) * t_stride + t) * kAttnDh;
    uint32_t pk[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) pk[k] = pack_f16x2_sat(v[2 * k], v[2 * k + 1]);
    uint4* d4 = reinterpret_cast<uint4*>(dst + part * 16);
    d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  } else {
    const int gv = col - Hq - Hkv;
#pragma unroll
    for (int k = 0; k < 16; ++k) vt[part * 16 + k][tl] = v[k];
    __syncthreads();
    const int c = threadIdx.x >> 1, hh = threadIdx.x & 1;  // row of Vt, 16 of the block's 32 tokens
    uint32_t pk[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) pk[k] = pack_bf16x2(vt[c][hh * 16 + 2 * k], vt[c][hh * 16 + 2 * k + 1]);
    uint4* d4 = reinterpret_cast<uint4*>(Vt + ((size_t)gv * kAttnDh + c) * t_stride + t0 + hh * 16);
    d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  }
}

// A6: y[t] = bf16(x[t] + o[t] / sqrt(mean(o[t]^2) + eps) * s), o fp32 [T, ld].
// One block of 256 threads per row; d a multiple of 8.
__global__ void __launch_bounds__(256) attn_post_kernel(const __nv_bfloat16* __restrict__ x,
                                                        const float* __restrict__ o, int ld,
                                                        const float* __restrict__ s, float eps, int d,
                                                        __nv_bfloat16* __restrict__ y) {
  const int t = blockIdx.x;
  const float4* orow = reinterpret_cast<const float4*>(o + (size_t)t * ld);
  const int nv = d / 8;
  float ss = 0.f;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    const float4 a = orow[2 * i], b = orow[2 * i + 1];
    ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w;
  }
  __shared__ float red[8];
#pragma unroll
  for (int k = 16; k > 0; k >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, k);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float rr = rsqrtf(tot / (float)d + eps);
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
  uint4* yr = reinterpret_cast<uint4*>(y + (size_t)t * d);
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    const float4 a = orow[2 * i], b = orow[2 * i + 1];
    const float4 s0 = reinterpret_cast<const float4*>(s)[2 * i];
    const float4 s1 = reinterpret_cast<const float4*>(s)[2 * i + 1];
    const uint4 xv = xr[i];
    uint4 out;
    out.x = pack_bf16x2(bf16_lo(xv.x) + a.x * rr * s0.x, bf16_hi(xv.x) + a.y * rr * s0.y);
    out.y = pack_bf16x2(bf16_lo(xv.y) + a.z * rr * s0.z, bf16_hi(xv.y) + a.w * rr * s0.w);
    out.z = pack_bf16x2(bf16_lo(xv.z) + b.x * rr * s1.x, bf16_hi(xv.z) + b.y * rr * s1.y);
    out.w = pack_bf16x2(bf16_lo(xv.w) + b.z * rr * s1.z, bf16_hi(xv.w) + b.w * rr * s1.w);
    yr[i] = out;
  }
}

}  // namespace moe
