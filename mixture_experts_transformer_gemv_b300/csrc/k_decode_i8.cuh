// Decode path with int8 weights (T <= 16): weight-streaming expert GEMMs that
// read each chosen expert's int8 weights once, half the bytes of bf16.
//
// int8 weights with bf16 scales, one per expert and output channel
// ("TevunahAi/Grok-1-BF16", "Conversion Details"; the (8, 1, N) scale shape).
// As in the bf16 decode kernels the weights are the MMA's M = 128 operand and
// the expert's slots the N = 16 operand:
//
//   K3q  unit (e, n-block):      Dh[n, s] = sum_k q_W[e,n,k] xn_e[s,k],  Dv likewise with Wv
//                                act[row(e,s), n] = GELU(s_W[e,n] Dh) * (s_Wv[e,n] Dv)
//   K4q  unit (e, j-block, kc):  D[j, s] = sum_{f in chunk kc} q_W1[e,j,f] act[row(e,s), f]
//                                part[kc][e][s][j] = p(row(e,s)) * s_W1[e,j] * D[j, s]
//
// Data path per k-block of 128: TMA brings the int8 weight tile(s) (128 x 128,
// 128-byte swizzle: whole 128-byte rows, the granule the bf16 kernels stream at
// full HBM speed; 64-byte rows measured at two thirds of it) and the slot rows
// (16 x 128, two 128-byte-swizzled boxes) into a deep shared-memory ring;
// sixteen converter warps turn each weight row into fp16 and store it straight
// into Tensor Memory with tcgen05.st, where the MMA reads its A operand
// (tcgen05.mma with A in TMEM).  The converted weights never
// go back through shared memory, so shared memory carries only the int8 bytes
// and the slot rows.
//
// This path multiplies in fp16, not bf16: an int8 value converts exactly to
// fp16 with one byte shuffle and one subtraction per pair (fp16's 10-bit
// mantissa holds a whole byte: the pattern 0x64uu is 1024 + u), half the
// integer work of the bf16 conversion, which bounded the rate at the HBM speed
// this path runs at.  Its activation rows are therefore fp16 too: the gather
// kernel writes the normed rows as fp16 (exact but below 2^-14) and the up
// projection's epilogue writes the GeGLU activations as fp16, saturating at
// +-65504; fp16 carries 3 more mantissa bits than bf16 within that range.
// The per-channel scales factor out of the reduction and are applied in fp32 in
// the epilogue (one scale per thread: its TMEM lane is one weight row); scales
// that also vary along k (G > 1 groups) multiply the converted weights instead
// (f16x2, one rounding).
//
// Warps: 0 TMA producer; 1 TMEM allocation + MMA issuer; 2-5 epilogue;
// 6-21 converters, each converting a quarter of every k-block.  Every wait is
// bounded, as in the other kernels.
#pragma once
#include "common.cuh"
#include "k_decode.cuh"
#include "k_gemm.cuh"
#include "ptx.cuh"
#include "ptx_tmem.cuh"

namespace moe {

constexpr int kDq8BK = 128;                  // K per stage: one 128-byte int8 row per weight row
constexpr int kDq8Tile = kDecBM * kDq8BK;     // 16 KB: one int8 weight tile, 128 rows x 128
constexpr int kDq8XTile = kDecNS * kDq8BK * 2;  // 4 KB: 16 slot rows x 128 fp16, as two 64-wide boxes
constexpr int kDq8ConvWarp0 = 6;
constexpr int kDq8ConvWarps = 16;

template <int EPI>
struct DecI8Cfg {
  static constexpr int kATiles = (EPI == kEpiGeglu) ? 2 : 1;
  static constexpr int kStageBytes = kATiles * kDq8Tile + kDq8XTile;  // int8 weights + fp16 slot rows
  static constexpr int kStages = (EPI == kEpiGeglu) ? 6 : 10;         // ~200 KB in flight per SM
  static constexpr uint32_t kAccCols = (EPI == kEpiGeglu) ? 64 : 32;  // one accumulator buffer
  static constexpr uint32_t kACols = kATiles * kDq8BK / 2;            // fp16 A of one k-block
  static constexpr int kAStages = (EPI == kEpiGeglu) ? 3 : 7;         // converted A ring in TMEM
  static constexpr uint32_t kAColBase = 2 * kAccCols;
  static constexpr uint32_t kTmemUsed = kAColBase + kAStages * kACols;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 32 * (kDq8ConvWarp0 + kDq8ConvWarps);
  // full, empty (TMA ring), afull, aempty (TMEM A ring), tmem_full x2, tmem_empty x2, drain
  static constexpr int kNumBars = 2 * kStages + 2 * kAStages + 5;
  static constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kNumBars * 8 + 16;
  static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled tiles");
  static_assert(kTmemUsed <= 512, "TMEM columns");
};

// Instruction descriptor of tcgen05.mma kind::f16 with fp16 A and B (format 0 in
// bits 7-9 and 10-12), fp32 D, both K-major; M = 128, N = 16.
constexpr uint32_t kDq8Idesc = (1u << 4) | (static_cast<uint32_t>(kDecNS >> 3) << 17) |
                               (static_cast<uint32_t>(kDecBM >> 4) << 24);

__device__ __forceinline__ uint16_t f16_sat(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.f16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}

struct DecI8Params {
  const int32_t* sched;       // counts[E], row_offset[E + 1]
  int K;                      // reduction length: d (K3q) or F (K4q)
  int rows_per_expert;        // weight rows per expert: F (W, Wv) or d (W1)
  int n_out;                  // leading dimension of the output: F (act) or d (partials)
  int ksplit;                 // K4q: chunks of the reduction (1 for K3q)
  void* out;                  // act [rows_cap, F] fp16 or part [ksplit][E][16][d] fp32
  const float* row_scale;     // K4q: combine weight of each permuted row
  const uint16_t* scale0;     // bf16 bits [E_s, G, rows_per_expert]: scale of W (K3q) or W1 (K4q)
  const uint16_t* scale1;     // K3q: bf16 bits [E_s, G, F], scale of Wv
  int scale_experts;          // E_s: 8 (per expert) or 1 (shared)
  int scale_groups;           // G groups along the reduction; 1 = per output channel only
  int group_kb;               // G > 1: k-blocks of 128 per group
  int checks;                 // K3q: report activations past the fp16 range
  uint32_t* err;
  uint64_t timeout_ns;
};

template <int EPI>
__global__ void __launch_bounds__(DecI8Cfg<EPI>::kThreads, 1)
    decode_gemm_i8_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                          const __grid_constant__ CUtensorMap tm_x, const DecI8Params p) {
  using C = DecI8Cfg<EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // stage s: [int8 W tile | int8 Wv tile (up)] [16 slot rows x 128 fp16]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)C::kStages * C::kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (C::kStages + s); };
  auto afull_bar = [&](uint32_t j) { return bar0 + 8u * (2 * C::kStages + j); };
  auto aempty_bar = [&](uint32_t j) { return bar0 + 8u * (2 * C::kStages + C::kAStages + j); };
  const uint32_t bar_t = bar0 + 8u * (2 * C::kStages + 2 * C::kAStages);
  auto tfull_bar = [&](uint32_t a) { return bar_t + 8u * a; };
  auto tempty_bar = [&](uint32_t a) { return bar_t + 8u * (2 + a); };
  const uint32_t drain_bar = bar_t + 8u * 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // active experts (counts > 0), in expert order
  int act_e[kNumExperts], n_act = 0;
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e) act_e[e] = 0;
  for (int e = 0; e < kNumExperts; ++e)
    if (p.sched[e] > 0) act_e[n_act++] = e;
  const int blocks = p.rows_per_expert / kDecBM;
  const int num_units = n_act * blocks * p.ksplit;
  const int kb_per_unit = p.K / kDq8BK / p.ksplit;
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
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int j = 0; j < C::kAStages; ++j) {
      mbar_init(afull_bar(j), kDq8ConvWarps);  // one arrival per converter warp
      mbar_init(aempty_bar(j), 1);
    }
    for (int a = 0; a < 2; ++a) {
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
      int n_issued = 0;  // stages issued so far (no per-stage array: it would live in local memory)
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const DecUnit d = unit_of(u);
        const int wrow = d.e * p.rows_per_expert + d.blk * kDecBM;
        for (int i = 0; i < kb_per_unit; ++i) {
          const int kx = (d.kc * kb_per_unit + i) * kDq8BK;
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          uint8_t* sb = smem + (size_t)stage * C::kStageBytes;
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          tma_load_2d_hint(smem_addr(sb), &tm_w0, fb, kx, wrow, stream_policy);
          if (EPI == kEpiGeglu) tma_load_2d_hint(smem_addr(sb + kDq8Tile), &tm_w1, fb, kx, wrow, stream_policy);
          tma_load_2d(smem_addr(sb + C::kATiles * kDq8Tile), &tm_x, fb, kx, d.row0);
          tma_load_2d(smem_addr(sb + C::kATiles * kDq8Tile + kDq8XTile / 2), &tm_x, fb, kx + 64, d.row0);
          ++n_issued;
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
        // the copies of the last (up to kStages) issued stages complete before the CTA exits
        for (int j = max(0, n_issued - C::kStages); j < n_issued; ++j)
          wait_bounded(full_bar((uint32_t)(j % C::kStages)), (uint32_t)((j / C::kStages) & 1), nullptr, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------ MMA
      uint32_t stage = 0, phase = 0, astage = 0, aphase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + acc * C::kAccCols;
        for (int i = 0; i < kb_per_unit; ++i) {
          if (!wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns) ||
              !wait_bounded(afull_bar(astage), aphase, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = tmem_base + C::kAColBase + astage * C::kACols;
          const uint32_t xs = smem_addr(smem + (size_t)stage * C::kStageBytes + C::kATiles * kDq8Tile);
#pragma unroll
          for (int kk = 0; kk < kDq8BK / 16; ++kk) {  // K = 16: 8 TMEM columns of A, 32 bytes of a B row
            const uint64_t bx = smem_desc_k_sw128(xs + (kk >> 2) * (kDq8XTile / 2)) + 2 * (kk & 3);
            const uint32_t accum = (i | kk) != 0;
            umma_bf16_tmem_a(d0, a0 + 8 * kk, bx, kDq8Idesc, accum);
            if (EPI == kEpiGeglu) umma_bf16_tmem_a(d0 + 32, a0 + 64 + 8 * kk, bx, kDq8Idesc, accum);
          }
          umma_commit(empty_bar(stage));
          umma_commit(aempty_bar(astage));
          if (++stage == (uint32_t)C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (++astage == (uint32_t)C::kAStages) {
            astage = 0;
            aphase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit(drain_bar);
      if (!wait_bounded(drain_bar, 0, nullptr, p.timeout_ns)) ok = false;
      // every release of a TMEM A buffer has landed before exit
      for (int j = 0; j < C::kAStages && ok; ++j) {
        if (!wait_bounded(aempty_bar(astage), aphase ^ 1u, abort_flag, p.timeout_ns)) ok = false;
        if (++astage == (uint32_t)C::kAStages) {
          astage = 0;
          aphase ^= 1u;
        }
      }
      if (!ok) raise_abort(abort_flag, p.err);
    }
  } else if (warp < kDq8ConvWarp0) {  // ---------------------------------- epilogue
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
      // per-output-channel scales (G == 1); grouped scales were applied in conversion
      const size_t si = (size_t)(p.scale_experts > 1 ? d.e : 0) * p.rows_per_expert + n;
      const bool chan = p.scale_groups == 1;
      if (EPI == kEpiGeglu) {
        uint32_t h[16], v[16];
        tmem_ld_32x32b_x16(tb, h);       // columns [0, 16): W branch
        tmem_ld_32x32b_x16(tb + 32, v);  // columns [32, 48): Wv branch
        tmem_ld_wait();
        const float sw = chan ? __uint_as_float((uint32_t)p.scale0[si] << 16) : 1.0f;
        const float sv = chan ? __uint_as_float((uint32_t)p.scale1[si] << 16) : 1.0f;
        uint16_t* out = static_cast<uint16_t*>(p.out);
        bool sat = false;
#pragma unroll
        for (int s = 0; s < kDecNS; ++s)
          if (s < d.cnt) {
            const float a = gelu_tanh(sw * __uint_as_float(h[s])) * (sv * __uint_as_float(v[s]));
            sat |= fabsf(a) > kF16Max;
            out[(size_t)(d.row0 + s) * p.n_out + n] = f16_sat(a);
          }
        if (p.checks && __any_sync(0xffffffffu, sat) && lane == 0) atomicOr(p.err, kErrSaturate);
      } else {
        uint32_t y[16];
        tmem_ld_32x32b_x16(tb, y);
        tmem_ld_wait();
        const float s1 = chan ? __uint_as_float((uint32_t)p.scale0[si] << 16) : 1.0f;
        float* out = static_cast<float*>(p.out) + ((size_t)(d.kc * kNumExperts + d.e) * kDecNS) * p.n_out;
#pragma unroll
        for (int s = 0; s < kDecNS; ++s)
          if (s < d.cnt) out[(size_t)s * p.n_out + n] = p.row_scale[d.row0 + s] * (s1 * __uint_as_float(y[s]));
      }
      tc_fence_before_sync();
      mbar_arrive(tempty_bar(acc));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  } else {  // ------------------------------------------ int8 -> fp16 into TMEM
    // All 16 converter warps work on every k-block, in order (a waiter that ran
    // ahead by two phases of a barrier would read its parity as complete).  The
    // four warps on the same TMEM lanes (warp w reaches lanes [32 (w % 4), +32))
    // split the k-block: up projection W or Wv times K [0,64) or [64,128); down
    // projection K [32 part, 32 part + 32).
    // Staging tile (128-byte swizzle): the 16-byte chunk c of weight row r sits at
    // r * 128 + 16 * (c ^ (r % 8)), so a warp's 32 rows read conflict-free.
    // TMEM A: lane r, column 8 c + i holds K elements 16 c + 2 i and
    // 16 c + 2 i + 1 of the k-block (fp16).
    const int q = warp & 3;                                 // TMEM lanes [32q, 32q + 32)
    const int part = (warp - kDq8ConvWarp0) >> 2;           // 0..3
    const int r = q * 32 + lane;                            // weight row of this thread
    const int rsw = r & 7;
    const uint32_t lane_bits = static_cast<uint32_t>(q * 32) << 16;
    uint32_t stage = 0, phase = 0, astage = 0, aphase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const DecUnit du = unit_of(u);
      const int n = du.blk * kDecBM + r;  // this thread's weight row
      const size_t gsc_e = (size_t)(p.scale_experts > 1 ? du.e : 0) * p.scale_groups;
      for (int i = 0; i < kb_per_unit; ++i) {
        // grouped scales (G > 1): this row's scale for the k-block's group, as fp16
        __half2 gs2 = __float2half2_rn(1.0f);
        if (p.scale_groups > 1) {
          const size_t gi = (gsc_e + (du.kc * kb_per_unit + i) / p.group_kb) * p.rows_per_expert + n;
          const float s0 = __uint_as_float((uint32_t)p.scale0[gi] << 16);
          gs2 = __float2half2_rn(s0);
          if (EPI == kEpiGeglu && (part >> 1) == 1) gs2 = __float2half2_rn(__uint_as_float((uint32_t)p.scale1[gi] << 16));
        }
        const uint32_t gsu = *reinterpret_cast<uint32_t*>(&gs2);
        ok = __all_sync(0xffffffffu, wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns) &&
                                         wait_bounded(aempty_bar(astage), aphase ^ 1u, abort_flag, p.timeout_ns));
        if (!ok) break;
        tc_fence_after_sync();
        const uint8_t* sb = smem + (size_t)stage * C::kStageBytes;
        const uint32_t acol = tmem_base + lane_bits + C::kAColBase + astage * C::kACols;
        if (EPI == kEpiGeglu) {  // matrix part / 2, K [64 (part % 2), +64) -> 32 columns
          const int mat = part >> 1, hh = part & 1;
          const uint8_t* row = sb + mat * kDq8Tile + r * 128;
          uint32_t a[32];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int c = 4 * hh + cc;
            const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * (c ^ rsw));
            i8x4_to_f16x4(v.x, a[8 * cc + 0], a[8 * cc + 1]);
            i8x4_to_f16x4(v.y, a[8 * cc + 2], a[8 * cc + 3]);
            i8x4_to_f16x4(v.z, a[8 * cc + 4], a[8 * cc + 5]);
            i8x4_to_f16x4(v.w, a[8 * cc + 6], a[8 * cc + 7]);
          }
          if (p.scale_groups > 1) {
#pragma unroll
            for (int j = 0; j < 32; ++j) a[j] = f16x2_mul(a[j], gsu);
          }
          tmem_st_32x32b_x32(acol + mat * 64 + hh * 32, a);
        } else {  // K [32 part, 32 part + 32) of the W1 row -> 16 columns
          const uint8_t* row = sb + r * 128;
          uint32_t a[16];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * part + cc;
            const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * (c ^ rsw));
            i8x4_to_f16x4(v.x, a[8 * cc + 0], a[8 * cc + 1]);
            i8x4_to_f16x4(v.y, a[8 * cc + 2], a[8 * cc + 3]);
            i8x4_to_f16x4(v.z, a[8 * cc + 4], a[8 * cc + 5]);
            i8x4_to_f16x4(v.w, a[8 * cc + 6], a[8 * cc + 7]);
          }
          if (p.scale_groups > 1) {
#pragma unroll
            for (int j = 0; j < 16; ++j) a[j] = f16x2_mul(a[j], gsu);
          }
          tmem_st_32x32b_x16(acol + part * 16, a);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(afull_bar(astage));
        if (++stage == (uint32_t)C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++astage == (uint32_t)C::kAStages) {
          astage = 0;
          aphase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) raise_abort(abort_flag, p.err);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace moe
