// Decode path (T <= 16): weight-streaming expert GEMMs with the operands swapped.
//
// With at most 16 tokens no expert receives more than 16 slots, so the expert
// FFN is a matrix-vector product per slot: the cost is reading the chosen
// experts' weights once from HBM (up to 9.66 GB per layer).  The tensor core
// still does the arithmetic, with the weights as the 128-row M operand and the
// expert's slots as the N = 16 operand:
//
//   K3d  unit (e, n-block):       Dh[n, s] = sum_k W[e,n,k] xn_e[s,k],  Dv likewise with Wv
//                                 act[row(e,s), n] = GELU(Dh) * Dv            (s < counts[e])
//   K4d  unit (e, j-block, kc):   D[j, s] = sum_{f in chunk kc} W1[e,j,f] act[row(e,s), f]
//                                 part[kc][e][s][j] = p(row(e,s)) * D[j, s]
//
// K4d splits the reduction over F into `ksplit` chunks so that the few active
// experts still give every SM several units; the combine kernel sums the
// partials in a fixed order (deterministic).  Units are spread round-robin over
// one CTA per SM.  The pipeline is the one of the grouped GEMM (TMA producer
// warp, MMA warp, four epilogue warps, double-buffered TMEM), with deeper
// rings since each stage is small: 6 stages of 34 KB (K3d), 11 of 18 KB (K4d).
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kDecNS = 16;    // slot columns (MMA N)
constexpr int kDecBM = 128;   // weight rows per unit (MMA M)
constexpr int kDecBK = 64;
constexpr int kDecThreads = 192;
constexpr int kDecATile = kDecBM * kDecBK * 2;  // 16 KB
constexpr int kDecBTile = kDecNS * kDecBK * 2;  // 2 KB
constexpr uint32_t kDecIdesc = idesc_bf16_f32(kDecBM, kDecNS);
constexpr int kDecMaxSplit = 8;

template <int EPI>
struct DecCfg {
  static constexpr int kATiles = (EPI == kEpiGeglu) ? 2 : 1;
  static constexpr int kStageBytes = kATiles * kDecATile + kDecBTile;
  static constexpr int kStages = (EPI == kEpiGeglu) ? 6 : 11;
  static constexpr uint32_t kAccCols = (EPI == kEpiGeglu) ? 64 : 32;  // one accumulator buffer
  static constexpr uint32_t kTmemCols = 2 * kAccCols;
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kNumBars * 8 + 16;
};

struct DecParams {
  const int32_t* sched;       // counts[E], row_offset[E + 1]
  int K;                      // reduction length: d (K3d) or F (K4d)
  int rows_per_expert;        // rows of the weight per expert: F (W, Wv) or d (W1)
  int n_out;                  // leading dimension of the output: F (act) or d (partials)
  int ksplit;                 // K4d: chunks of the reduction (1 for K3d)
  void* out;                  // act [rows_cap, F] bf16 or part [ksplit][E][16][d] fp32
  const float* row_scale;     // K4d: combine weight of each permuted row
  uint32_t* err;
  uint64_t timeout_ns;
};

struct DecUnit {
  int e, row0, cnt, blk, kc;
};

template <int EPI>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                       const __grid_constant__ CUtensorMap tm_x, const DecParams p) {
  using C = DecCfg<EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)C::kStages * C::kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (C::kStages + s); };
  auto tfull_bar = [&](uint32_t a) { return bar0 + 8u * (2 * C::kStages + a); };
  auto tempty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * C::kStages + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C::kStages + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // active experts (counts > 0), in expert order
  int act_e[kNumExperts], n_act = 0;
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e) act_e[e] = 0;
  for (int e = 0; e < kNumExperts; ++e)
    if (p.sched[e] > 0) act_e[n_act++] = e;
  const int blocks = p.rows_per_expert / kDecBM;
  const int num_units = n_act * blocks * p.ksplit;
  const int kb_per_unit = p.K / kDecBK / p.ksplit;
  auto unit_of = [&](int u) {
    DecUnit d;
    const int kc = u % p.ksplit;
    const int rest = u / p.ksplit;
    d.blk = rest % blocks;
    int ai = rest / blocks, e = 0;
    for (int q = 0; q < kNumExperts; ++q)
      if (q == ai) e = act_e[q];
    d.e = e;
    d.kc = kc;
    d.row0 = p.sched[kNumExperts + e];
    d.cnt = min(p.sched[e], kDecNS);
    return d;
  };

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < (uint32_t)C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (uint32_t a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w0);
    if (EPI == kEpiGeglu) tma_prefetch_desc(&tm_w1);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------------ TMA
      const uint64_t stream_policy = l2_policy_evict_first();  // weights are read once
      uint32_t stage = 0, phase = 0;
      int issued[C::kStages];
      for (int s = 0; s < C::kStages; ++s) issued[s] = -1;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const DecUnit d = unit_of(u);
        const int wrow = d.e * p.rows_per_expert + d.blk * kDecBM;
        for (int i = 0; i < kb_per_unit; ++i) {
          const int kx = (d.kc * kb_per_unit + i) * kDecBK;
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          uint8_t* sb = smem + (size_t)stage * C::kStageBytes;
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          tma_load_2d_hint(smem_addr(sb), &tm_w0, fb, kx, wrow, stream_policy);
          if (EPI == kEpiGeglu) tma_load_2d_hint(smem_addr(sb + kDecATile), &tm_w1, fb, kx, wrow, stream_policy);
          tma_load_2d(smem_addr(sb + C::kATiles * kDecATile), &tm_x, fb, kx, d.row0);
          for (int s = 0; s < C::kStages; ++s)
            if (s == (int)stage) issued[s] = (int)phase;
          if (++stage == (uint32_t)C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int i = 0; i < C::kStages && ok; ++i) {
        if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) ok = false;
        if (++stage == (uint32_t)C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        raise_abort(abort_flag, p.err);
        for (int s = 0; s < C::kStages; ++s)
          if (issued[s] >= 0) wait_bounded(full_bar(s), (uint32_t)issued[s], nullptr, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------ MMA
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + acc * C::kAccCols;
        for (int i = 0; i < kb_per_unit; ++i) {
          if (!wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sb = smem_addr(smem + (size_t)stage * C::kStageBytes);
          const uint64_t a0 = smem_desc_k_sw128(sb);
          const uint64_t bx = smem_desc_k_sw128(sb + C::kATiles * kDecATile);
#pragma unroll
          for (int kk = 0; kk < kDecBK / 16; ++kk) {
            umma_bf16(d0, a0 + 2 * kk, bx + 2 * kk, kDecIdesc, (i | kk) != 0);
            if (EPI == kEpiGeglu) {
              const uint64_t a1 = smem_desc_k_sw128(sb + kDecATile);
              umma_bf16(d0 + 32, a1 + 2 * kk, bx + 2 * kk, kDecIdesc, (i | kk) != 0);
            }
          }
          umma_commit(empty_bar(stage));
          if (++stage == (uint32_t)C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit(drain_bar);
      if (!wait_bounded(drain_bar, 0, nullptr, p.timeout_ns)) ok = false;
      if (!ok) raise_abort(abort_flag, p.err);
    }
  } else {  // -------------------------------------------------------- epilogue
    const int q = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      const DecUnit d = unit_of(u);
      bool ok = wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) raise_abort(abort_flag, p.err);
        break;
      }
      tc_fence_after_sync();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::kAccCols;
      const int n = d.blk * kDecBM + q * 32 + lane;  // weight row = output column
      if (EPI == kEpiGeglu) {
        uint32_t h[16], v[16];
        tmem_ld_32x32b_x16(tb, h);       // columns [0, 16): W branch
        tmem_ld_32x32b_x16(tb + 32, v);  // columns [32, 48): Wv branch
        tmem_ld_wait();
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
        for (int s = 0; s < kDecNS; ++s)
          if (s < d.cnt)
            out[(size_t)(d.row0 + s) * p.n_out + n] =
                __float2bfloat16_rn(gelu_tanh(__uint_as_float(h[s])) * __uint_as_float(v[s]));
      } else {
        uint32_t y[16];
        tmem_ld_32x32b_x16(tb, y);
        tmem_ld_wait();
        float* out = static_cast<float*>(p.out) + ((size_t)(d.kc * kNumExperts + d.e) * kDecNS) * p.n_out;
#pragma unroll
        for (int s = 0; s < kDecNS; ++s)
          if (s < d.cnt) out[(size_t)s * p.n_out + n] = p.row_scale[d.row0 + s] * __uint_as_float(y[s]);
      }
      tc_fence_before_sync();
      mbar_arrive(tempty_bar(acc));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace moe
