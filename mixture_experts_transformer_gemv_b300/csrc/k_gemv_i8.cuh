// Decode path with int8 weights for T <= 16: the expert GEMVs on the CUDA cores.
//
// int8 weights with bf16 scales, one per expert and output channel
// ("TevunahAi/Grok-1-BF16", "Conversion Details"; the (8, 1, N) scale shape).
// With T <= 16 an expert holds at most 16 slot rows, so every weight byte is
// used by at most 16 products.  The tensor-core form of this step (weights as
// the M = 128 operand, converted to fp16 in Tensor Memory, slots as N = 16)
// is bounded by its MMA rate: each MMA moves 4 KB of fp16 A for 2 K weights
// whatever N is.  Here each weight byte stays an int8 and is multiplied in the
// integer pipe: dp2a takes two 16-bit activations and two int8 weights and adds
// both products to a 32-bit accumulator, exactly.  The activation rows are put
// in 16-bit fixed point per 128-element block of each slot row:
//
//   sx[s, kb] = max_{k in kb} |x[s, k]| / 32767,   X[s, k] = rint(x[s, k] / sx[s, kb])
//
// so |x - sx X| <= sx / 2 (2^-16 of the block's largest value), and
//
//   K3g unit (e, n-block):      Dh[n, s] = sum_kb sx[s, kb] * sum_{k in kb} q_W[e,n,k] X[s,k], Dv likewise
//                               act[row(e,s), n] = GELU(s_W[e,n] Dh) * (s_Wv[e,n] Dv)
//   K4g unit (e, j-block, kc):  D[j, s] over the chunk kc of the F reduction
//                               part[kc][e][s][j] = p(row(e,s)) * s_W1[e,j] * D[j, s]
//
// The integer sum of one lane covers 16 k of one block (|sum| < 2^27), and is
// scaled into an fp32 accumulator once per block.  Scales that vary along k
// (G > 1 groups) multiply that block sum; per-channel scales (G == 1) multiply
// the fp32 result in the epilogue.  Outputs are the same as the tensor-core
// decode kernels': fp16 GeGLU activations (saturating at +-65504, reported
// under device checks) and fp32 split-K partials for the combine.
//
// The slot rows are quantised once per forward, before each GEMV, by
// quantize_slots_kernel (one warp per slot row and 128-element block), into a
// compact buffer of 16 rows per expert (row 16 e + j: the expert's j-th slot),
// each block stored in the order the compute lanes read it, and the block
// scales transposed ([block][row]).  A unit takes a group of up to 8 of an
// expert's slots (slots 0-7, and 8-15 when the expert has more than 8, which
// then reads its weights twice), so one TMA box brings the group's 8 rows of a
// block and another their 8 scales.
//
// Data path per k-block of 128: TMA brings two int8 weight tiles (128 x 128,
// 128-byte swizzle), the slot group's 8 quantised rows (8 x 256 bytes) and their
// 8 scales into a ring of shared-memory stages; sixteen compute warps read the
// weights once each.  Compute lanes: lane = 8 g + c, c the 16-byte chunk (k in
// [16 c, 16 c + 16)) and g a group of weight rows; the eight lanes of a group
// hold the eight chunks of the same rows, so a 16-byte load per lane is
// conflict-free under the swizzle and the sum over k finishes in the group with
// shuffles.
//
// Warps: 0 TMA producer; 1-16 compute.  Every wait is bounded.
#pragma once
#include "common.cuh"
#include "k_decode.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kGv8NS = 8;                        // slot rows per unit (a group of an expert's slots)
constexpr int kGv8SlotsPerExpert = 16;           // T <= 16: at most 16 slots on one expert
constexpr int kGv8BK = 128;                      // K per stage: one 128-byte int8 row per weight row
constexpr int kGv8Tile = 128 * kGv8BK;           // 16 KB: one int8 weight tile, 128 rows x 128
constexpr int kGv8QRow = kGv8BK * 2;             // 256 B: one quantised block of a slot row, int16
constexpr int kGv8QTile = kGv8NS * kGv8QRow;     // 2 KB: a slot group's 8 rows
constexpr int kGv8QRows = kNumExperts * kGv8SlotsPerExpert;  // rows of the quantised buffer
constexpr int kGv8CompWarp0 = 1;
constexpr int kGv8CompWarps = 16;
constexpr int kGv8MaxT = kGv8SlotsPerExpert;
constexpr int kGv8R = 4;  // weight rows per compute lane: two adjacent rows of each of the stage's two tiles

// A unit's two 128-row weight tiles per k-block: up W and Wv rows [128 blk, +128)
// (one n-block, both GeGLU branches); down W1 rows [256 blk, +128) and
// [256 blk + 128, +128) (a 256-row j-block; the second tile of an odd last block
// reads rows past the expert's, whose results are dropped).
template <int EPI>
struct GvI8Cfg {
  static constexpr int kUnitRows = (EPI == kEpiGeglu) ? 128 : 256;
  // [two weight tiles][quantised rows][8 scales], padded to keep the swizzled tiles 1024-byte aligned
  static constexpr int kStageBytes = 2 * kGv8Tile + 3 * 1024;
  static constexpr int kStages = 6;  // 192 KB of weights in flight per SM
  static constexpr int kThreads = 32 * (kGv8CompWarp0 + kGv8CompWarps);
  static constexpr int kNumBars = 2 * kStages;  // full, empty
  static constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kNumBars * 8 + 16;
  static_assert(kGv8QTile + kGv8NS * 4 <= 3 * 1024, "stage padding holds the rows and scales");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kGv8CompWarps * 4 * 2 == 128, "16 warps x 4 row groups x 2 rows cover a 128-row tile");
};

// One warp per (slot s, 128-block kb) of the fp16 rows [R, K]: the block's
// largest |x| sets sx = max / 32767 and X = rint(x / sx) (0 for an all-zero
// block).  Lane l holds k = 4 l .. 4 l + 3; X is stored at element
// 64 ((l / 2) % 2) + 8 (l / 4) + 4 (l % 2) of the block, i.e. k = 16 c + 8 h + i
// at 64 h + 8 c + i: the two 16-byte halves of chunk c 128 bytes apart.
__global__ void __launch_bounds__(256) quantize_slots_kernel(const uint16_t* __restrict__ rows, int K,
                                                             const int32_t* __restrict__ row_of_slot,
                                                             const int32_t* __restrict__ idx,
                                                             const int32_t* __restrict__ sched, int S,
                                                             int16_t* __restrict__ xq, float* __restrict__ xs) {
  const int nkb = K / kGv8BK;
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= S * nkb) return;
  const int s = w / nkb, kb = w - s * nkb;
  const int row = row_of_slot[s], e = idx[s];
  if (e < 0 || e >= kNumExperts) return;  // (a routing index the grouping rejected)
  const int j = row - sched[kNumExperts + e];
  if (j < 0 || j >= kGv8SlotsPerExpert) return;
  const int qrow = e * kGv8SlotsPerExpert + j;
  const uint2 raw = *reinterpret_cast<const uint2*>(rows + (size_t)row * K + kb * kGv8BK + 4 * lane);
  const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
  const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
  float m = fmaxf(fmaxf(fabsf(f01.x), fabsf(f01.y)), fmaxf(fabsf(f23.x), fabsf(f23.y)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float inv = m > 0.f ? 32767.0f / m : 0.f;
  const int q0 = __float2int_rn(f01.x * inv), q1 = __float2int_rn(f01.y * inv);
  const int q2 = __float2int_rn(f23.x * inv), q3 = __float2int_rn(f23.y * inv);
  uint2 packed;
  packed.x = (static_cast<uint32_t>(q0) & 0xFFFFu) | (static_cast<uint32_t>(q1) << 16);
  packed.y = (static_cast<uint32_t>(q2) & 0xFFFFu) | (static_cast<uint32_t>(q3) << 16);
  const int pos = 64 * ((lane >> 1) & 1) + 8 * (lane >> 2) + 4 * (lane & 1);
  *reinterpret_cast<uint2*>(xq + (size_t)qrow * K + kb * kGv8BK + pos) = packed;
  if (lane == 0) xs[(size_t)kb * kGv8QRows + qrow] = m / 32767.0f;
}

__device__ __forceinline__ int dp2a_lo(uint32_t a16x2, uint32_t b8x4, int c) {
  int d;
  asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a16x2), "r"(b8x4), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a16x2, uint32_t b8x4, int c) {
  int d;
  asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a16x2), "r"(b8x4), "r"(c));
  return d;
}
// 16 products of one weight chunk (16 int8 in w) with 16 quantised activations
// (x0: k 0..7, x1: k 8..15, two int16 per register, lower k in the low half),
// as two independent chains of four
__device__ __forceinline__ int dot16_i8_i16(const uint4& w, const uint4& x0, const uint4& x1) {
  int s0 = dp2a_lo(x0.x, w.x, 0);
  int s1 = dp2a_lo(x1.x, w.z, 0);
  s0 = dp2a_hi(x0.y, w.x, s0);
  s1 = dp2a_hi(x1.y, w.z, s1);
  s0 = dp2a_lo(x0.z, w.y, s0);
  s1 = dp2a_lo(x1.z, w.w, s1);
  s0 = dp2a_hi(x0.w, w.y, s0);
  s1 = dp2a_hi(x1.w, w.w, s1);
  return s0 + s1;
}

// One stage of a compute lane with NT slot rows (the expert's count, a
// template argument so every slot's products can be interleaved): a[t * 4 + r]
// += sx[t] * (row r of the lane . X[t]) over the lane's 16 k, each block sum
// times gs[r] (grouped scales; 1 otherwise).
template <int NT>
__device__ __forceinline__ void gemv_stage(const uint8_t* sb, int col0, int c, const float (&gs)[kGv8R],
                                           float (&a)[kGv8NS * kGv8R]) {
  uint4 w[kGv8R];
#pragma unroll
  for (int r = 0; r < kGv8R; ++r) {  // r = 2 (row - col0) + tile
    const int row = col0 + (r >> 1);
    w[r] = *reinterpret_cast<const uint4*>(sb + (r & 1) * kGv8Tile + row * 128 + 16 * (c ^ (row & 7)));
  }
  const uint8_t* qt = sb + 2 * kGv8Tile + c * 16;
  const float* xsc = reinterpret_cast<const float*>(sb + 2 * kGv8Tile + kGv8QTile);
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const uint4 x0 = *reinterpret_cast<const uint4*>(qt + t * kGv8QRow);
    const uint4 x1 = *reinterpret_cast<const uint4*>(qt + t * kGv8QRow + 128);
    const float sx = xsc[t];
#pragma unroll
    for (int r = 0; r < kGv8R; ++r)
      a[t * kGv8R + r] = fmaf(static_cast<float>(dot16_i8_i16(w[r], x0, x1)), sx * gs[r], a[t * kGv8R + r]);
  }
}

template <int EPI, bool GROUPED>
__global__ void __launch_bounds__(GvI8Cfg<EPI>::kThreads, 1)
    gemv_i8_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                   const __grid_constant__ CUtensorMap tm_xq, const __grid_constant__ CUtensorMap tm_xs,
                   const DecI8Params p) {
  using C = GvI8Cfg<EPI>;
  constexpr int kV = kGv8NS * kGv8R;  // accumulators per lane: value t * 4 + r
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // stage s: [int8 weight tile 0 | tile 1] [8 quantised rows x 256 B] [8 scales]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)C::kStages * C::kStageBytes);
  volatile uint32_t* abort_flag = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (C::kStages + s); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // active slot groups 2 e + h (expert e has more than 8 h slots), in order
  int grp[2 * kNumExperts], n_grp = 0;
#pragma unroll
  for (int q = 0; q < 2 * kNumExperts; ++q) grp[q] = 0;
  for (int q = 0; q < 2 * kNumExperts; ++q)
    if (p.sched[q >> 1] > kGv8NS * (q & 1)) grp[n_grp++] = q;
  const int blocks = (p.rows_per_expert + C::kUnitRows - 1) / C::kUnitRows;
  const int num_units = n_grp * blocks * p.ksplit;
  const int kb_per_unit = p.K / kGv8BK / p.ksplit;
  // unit: expert e, its slots [s0, s0 + cnt) (s0 = 0 or 8), rows row0 = row_offset[e] + s0
  auto unit_of = [&](int u, int& s0) {
    DecUnit d;
    const int kc = u % p.ksplit;
    const int rest = u / p.ksplit;
    d.blk = rest % blocks;
    int ai = rest / blocks, g = 0;
    for (int q = 0; q < 2 * kNumExperts; ++q)
      if (q == ai) g = grp[q];
    d.e = g >> 1;
    s0 = kGv8NS * (g & 1);
    d.kc = kc;
    d.row0 = p.sched[kNumExperts + d.e] + s0;
    d.cnt = min(p.sched[d.e] - s0, kGv8NS);
    return d;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kGv8CompWarps);  // one arrival per compute warp
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w0);
    if (EPI == kEpiGeglu) tma_prefetch_desc(&tm_w1);
    tma_prefetch_desc(&tm_xq);
    tma_prefetch_desc(&tm_xs);
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------------ TMA
      const uint64_t stream_policy = l2_policy_evict_first();  // weights are read once
      constexpr uint32_t kTx = 2 * kGv8Tile + kGv8QTile + kGv8NS * 4;
      uint32_t stage = 0, phase = 0;
      int n_issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        int s0;
        const DecUnit d = unit_of(u, s0);
        const int wrow = d.e * p.rows_per_expert + d.blk * C::kUnitRows;
        const int qrow = d.e * kGv8SlotsPerExpert + s0;
        for (int i = 0; i < kb_per_unit; ++i) {
          const int kb = d.kc * kb_per_unit + i;
          const int kx = kb * kGv8BK;
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          uint8_t* sb = smem + (size_t)stage * C::kStageBytes;
          mbar_arrive_expect_tx(fb, kTx);
          tma_load_2d_hint(smem_addr(sb), &tm_w0, fb, kx, wrow, stream_policy);
          if (EPI == kEpiGeglu)
            tma_load_2d_hint(smem_addr(sb + kGv8Tile), &tm_w1, fb, kx, wrow, stream_policy);
          else
            tma_load_2d_hint(smem_addr(sb + kGv8Tile), &tm_w0, fb, kx, wrow + 128, stream_policy);
          uint8_t* qs = sb + 2 * kGv8Tile;
          tma_load_2d(smem_addr(qs), &tm_xq, fb, kx, qrow);
          tma_load_2d(smem_addr(qs + kGv8QTile), &tm_xs, fb, qrow, kb);
          ++n_issued;
          if (++stage == (uint32_t)C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every stage consumed before the CTA may exit
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
  } else {  // ------------------------------------------------------- compute
    const int cw = warp - kGv8CompWarp0;  // 0..15
    const int g = lane >> 3, c = lane & 7;
    const int col0 = cw * 8 + g * 2;      // first of this lane group's two rows in each tile
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    bool sat = false;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      int s0;
      const DecUnit d = unit_of(u, s0);
      // weight row (within the expert) of lane row r = 2 cb + tile, and whether it exists
      auto wrow_of = [&](int r) {
        return (EPI == kEpiGeglu) ? d.blk * 128 + col0 + (r >> 1) : d.blk * 256 + (r & 1) * 128 + col0 + (r >> 1);
      };
      float a[kV];
#pragma unroll
      for (int v = 0; v < kV; ++v) a[v] = 0.f;
      const size_t gsc_e = (size_t)(p.scale_experts > 1 ? d.e : 0) * p.scale_groups;
      for (int i = 0; i < kb_per_unit; ++i) {
        float gs[kGv8R];
#pragma unroll
        for (int r = 0; r < kGv8R; ++r) gs[r] = 1.f;
        if (GROUPED) {  // this block's group scale of each of the lane's rows
          const size_t gi = (gsc_e + (d.kc * kb_per_unit + i) / p.group_kb) * p.rows_per_expert;
#pragma unroll
          for (int r = 0; r < kGv8R; ++r) {
            const int j = wrow_of(r);
            const uint16_t* sc = (EPI == kEpiGeglu && (r & 1)) ? p.scale1 : p.scale0;
            gs[r] = j < p.rows_per_expert ? __uint_as_float((uint32_t)sc[gi + j] << 16) : 0.f;
          }
        }
        ok = __all_sync(0xffffffffu, wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns));
        if (!ok) break;
        const uint8_t* sb = smem + (size_t)stage * C::kStageBytes;
        switch (d.cnt) {
          case 1: gemv_stage<1>(sb, col0, c, gs, a); break;
          case 2: gemv_stage<2>(sb, col0, c, gs, a); break;
          case 3: gemv_stage<3>(sb, col0, c, gs, a); break;
          case 4: gemv_stage<4>(sb, col0, c, gs, a); break;
          case 5: gemv_stage<5>(sb, col0, c, gs, a); break;
          case 6: gemv_stage<6>(sb, col0, c, gs, a); break;
          case 7: gemv_stage<7>(sb, col0, c, gs, a); break;
          default: gemv_stage<8>(sb, col0, c, gs, a); break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(stage));
        if (++stage == (uint32_t)C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      // Sum over the eight chunks of each lane group, scattered so that lane c
      // ends with slot t = c: three butterfly steps on the slot bits.
      float b[kV / 2];
#pragma unroll
      for (int v = 0; v < kV / 2; ++v) {
        const bool hi = lane & 4;
        const float keep = hi ? a[v + kV / 2] : a[v], send = hi ? a[v] : a[v + kV / 2];
        b[v] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
      }
      float b2[kV / 4];
#pragma unroll
      for (int v = 0; v < kV / 4; ++v) {
        const bool hi = lane & 2;
        const float keep = hi ? b[v + kV / 4] : b[v], send = hi ? b[v] : b[v + kV / 4];
        b2[v] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
      }
      float y[kGv8R];  // y[2 cb + tile]
#pragma unroll
      for (int v = 0; v < kGv8R; ++v) {
        const bool hi = lane & 1;
        const float keep = hi ? b2[v + kGv8R] : b2[v], send = hi ? b2[v] : b2[v + kGv8R];
        y[v] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
      }
      const int t = c;  // this lane's slot in the group
      const size_t se = (size_t)(p.scale_experts > 1 ? d.e : 0) * p.rows_per_expert;
      if (t < d.cnt) {
        if (EPI == kEpiGeglu) {  // columns n, n + 1: GELU(s_W h) * (s_Wv v)
          const int n = wrow_of(0);
          float o[2];
#pragma unroll
          for (int cb = 0; cb < 2; ++cb) {
            const float sw = GROUPED ? 1.f : __uint_as_float((uint32_t)p.scale0[se + n + cb] << 16);
            const float sv = GROUPED ? 1.f : __uint_as_float((uint32_t)p.scale1[se + n + cb] << 16);
            o[cb] = gelu_tanh(sw * y[2 * cb]) * (sv * y[2 * cb + 1]);
            sat |= fabsf(o[cb]) > kF16Max;
          }
          uint16_t* out = static_cast<uint16_t*>(p.out);
          *reinterpret_cast<uint32_t*>(out + (size_t)(d.row0 + t) * p.n_out + n) = pack_f16x2_sat(o[0], o[1]);
        } else {  // rows j, j + 1 of each tile: p * s_W1 * y
          const float ps = p.row_scale[d.row0 + t];
          float* out = static_cast<float*>(p.out) + ((size_t)(d.kc * kNumExperts + d.e) * kDecNS + s0 + t) * p.n_out;
#pragma unroll
          for (int tile = 0; tile < 2; ++tile) {
            const int j = wrow_of(tile);
            if (j < p.rows_per_expert) {
              const float s0 = GROUPED ? 1.f : __uint_as_float((uint32_t)p.scale0[se + j] << 16);
              const float s1 = GROUPED ? 1.f : __uint_as_float((uint32_t)p.scale0[se + j + 1] << 16);
              *reinterpret_cast<float2*>(out + j) = make_float2(ps * (s0 * y[tile]), ps * (s1 * y[2 + tile]));
            }
          }
        }
      }
    }
    if (EPI == kEpiGeglu && p.checks && __any_sync(0xffffffffu, sat) && lane == 0) atomicOr(p.err, kErrSaturate);
    if (!ok && lane == 0) raise_abort(abort_flag, p.err);
  }
  __syncthreads();
}

}  // namespace moe
