// K3 / K4: expert-grouped GEMMs on the 5th-generation tensor cores.
//
//   K3 (up, GeGLU):  act[r, n] = GELU(sum_k A[r,k] W[e,n,k]) * (sum_k A[r,k] Wv[e,n,k])
//   K4 (down):       Y[r, j]   = p[r] * sum_n act[r,n] W1[e,j,n]
// for every permuted row r of expert e ("Jah-yee/grok" README, architecture
// diagram: GELU(x W) (*) (x Wv), then the output projection; weights in PyTorch
// [out, in] order per "TevunahAi/Grok-1-BF16", "Weight Verification").
//
// Structure (one CTA per SM, persistent, static round-robin over tiles):
//   warp 0      TMA producer: A tile [128 x 64] and B tile [256 x 64] per stage,
//               128-byte swizzle, into a 4-stage shared-memory ring
//   warp 1      allocates 512 TMEM columns; lane 0 issues tcgen05.mma
//               (M=128, N=256, K=16, bf16 -> fp32) and tcgen05.commit
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, GeGLU or scale, stores
//   warps 6-13  int8 weights only: int8 -> bf16 conversion of the B tile
// Two TMEM accumulators (2 x 256 columns) let the epilogue of tile i overlap the
// mainloop of tile i+1.  In K3 the B tile stacks 128 rows of W over the same 128
// rows of Wv, so one N=256 MMA produces both branches of 128 output columns.
//
// Tiles never mix experts: expert e owns permuted rows [row_offset[e],
// row_offset[e+1]), a multiple of 128.  Tile t maps to (expert, n-block,
// m-block) with the m-block fastest, so CTAs working at the same time share the
// same weight tile through L2.
//
// int8 weights ("TevunahAi/Grok-1-BF16", "Conversion Details": int8 values
// with bf16 scales, one per expert and output channel for the (8, 1, N) scale
// shape): TMA brings the raw int8 B tile into a staging buffer; eight converter
// warps (6-13) rewrite it as bf16 in the 128-byte-swizzled K-major layout the MMA
// reads (|q| <= 127 is exact in bf16), make it visible to the tensor core's
// async proxy and release the stage to the MMA warp.  Because the scale belongs
// to an output channel it factors out of the reduction and is applied in fp32
// in the epilogue: sum_k a_k (q_nk s_n) = s_n sum_k a_k q_nk.
//
// Every wait is bounded (wait_bounded).  A role that times out raises the CTA's
// abort flag and the device error word; the others stop at their next wait; the
// producer then waits (bounded) for its own TMA copies in flight, the MMA issuer
// for its own MMAs, and TMEM is freed before the CTA exits.
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kGemmBM = 128;   // MMA M: permuted rows per tile
constexpr int kGemmBN = 256;   // MMA N
constexpr int kGemmBK = 64;    // K per stage (64 bf16 = one 128-byte swizzle row)
constexpr int kEpiWarp0 = 2;   // first epilogue warp (warps 2-5)
constexpr int kConvWarp0 = 6;  // first converter warp (warps 6-13, int8 weights only)
constexpr int kEpiThreads = 128;
constexpr int kConvThreads = 256;
constexpr int kATileBytes = kGemmBM * kGemmBK * 2;  // 16 KB
constexpr int kBTileBytes = kGemmBN * kGemmBK * 2;  // 32 KB (bf16, swizzled)
constexpr int kB8TileBytes = kGemmBN * kGemmBK;     // 16 KB (int8 staging, dense rows of 64 B)
constexpr uint32_t kTmemCols = 2 * kGemmBN;  // two fp32 accumulators of 128 x 256
constexpr uint32_t kGemmIdesc = idesc_bf16_f32(kGemmBM, kGemmBN);

// Per weight type:
//   bf16: one TMA ring of 4 stages, A 16 KB + B 32 KB each; 6 warps.
//   int8: a TMA ring of 5 stages, A 16 KB + int8 B 16 KB each, and a ring of 2
//         converted bf16 B tiles (32 KB each) between the converter warps and
//         the MMA warp; 14 warps.  The TMA ring stays deep (5 k-blocks of MMA
//         work in flight) while conversion runs one k-block ahead of the MMA.
template <bool WQ>
struct GemmCfg {
  static constexpr int kStages = WQ ? 5 : 4;   // TMA ring
  static constexpr int kBStages = WQ ? 2 : 0;  // converted-B ring
  static constexpr int kStageBytes = kATileBytes + (WQ ? kB8TileBytes : kBTileBytes);  // TMA bytes per stage
  static constexpr int kThreads = WQ ? 32 * kConvWarp0 + kConvThreads : 192;
  // full, empty (TMA ring), bfull, bempty (converted ring), tmem_full x2, tmem_empty x2, drain
  static constexpr int kNumBars = 2 * kStages + 2 * kBStages + 5;
  static constexpr size_t kSmemBytes =
      1024 + (size_t)kStages * kStageBytes + (size_t)kBStages * kBTileBytes + kNumBars * 8 + 16;
};
constexpr int kGemmThreads = GemmCfg<false>::kThreads;
constexpr size_t kGemmSmemBytes = GemmCfg<false>::kSmemBytes;

struct GemmParams {
  const int32_t* sched;          // counts[E], row_offset[E + 1] (written by K2)
  int K;                         // reduction length: d (up) or F (down); multiple of 64
  int n_tiles;                   // tiles per expert along the output columns
  int b_rows_per_expert;         // rows of B per expert: F (W, Wv) or d (W1)
  int n_out;                     // output columns / leading dimension: F (act) or d (Y)
  void* out;                     // act [rows_cap, F] bf16 or Y [rows_cap, d] fp32
  const float* row_scale;        // down: combine weight of each permuted row
  const uint16_t* scale0;        // int8: bf16 bits [E, n_out], scale of W (up) or W1 (down)
  const uint16_t* scale1;        // int8 up: bf16 bits [E, F], scale of Wv
  uint32_t* err;                 // device error word
  uint64_t timeout_ns;           // limit of every wait
};

struct TileCoord {
  int e, row0, n_blk;
};

// Tile t -> (expert, first row, n-block); tiles of expert e are
// [ (off[e]/128) * n_tiles, (off[e+1]/128) * n_tiles ), m-block fastest.
__device__ __forceinline__ TileCoord decode_tile(int t, const int (&off)[kNumExperts + 1], int n_tiles) {
  int e = 0;
#pragma unroll
  for (int q = 1; q < kNumExperts; ++q)
    if (t >= (off[q] / kRowTile) * n_tiles) e = q;
  const int mt = off[e + 1] / kRowTile - off[e] / kRowTile;
  const int local = t - (off[e] / kRowTile) * n_tiles;
  TileCoord c;
  c.e = e;
  c.n_blk = local / mt;
  c.row0 = off[e] + (local % mt) * kRowTile;
  return c;
}

// 4 int8 (one 32-bit word, element i in byte i) -> 4 bf16 in two words, exact,
// with integer byte shuffles and one bf16x2 subtraction per pair.  For the
// two's-complement byte q = m - 128 s (m = low 7 bits, s = sign bit), the bf16
// with high byte 0x43 and low byte m is 128 + m, and with low byte 0x80 s it is
// 128 + 128 s; their difference is q, exactly representable, so the
// subtraction is exact.
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void i8x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t m = w & 0x7F7F7F7Fu;
  const uint32_t s = w & 0x80808080u;
  lo = bf16x2_sub(__byte_perm(m, 0x43u, 0x4140), __byte_perm(s, 0x43u, 0x4140));
  hi = bf16x2_sub(__byte_perm(m, 0x43u, 0x4342), __byte_perm(s, 0x43u, 0x4342));
}

// 8 bf16 scales (16 bytes of bf16 bits) -> fp32.
__device__ __forceinline__ void load_scales8(const uint16_t* p, float (&s)[8]) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  s[0] = bf16_lo(v.x); s[1] = bf16_hi(v.x); s[2] = bf16_lo(v.y); s[3] = bf16_hi(v.y);
  s[4] = bf16_lo(v.z); s[5] = bf16_hi(v.z); s[6] = bf16_lo(v.w); s[7] = bf16_hi(v.w);
}

template <int EPI, bool WQ>
__global__ void __launch_bounds__(GemmCfg<WQ>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b0,
                        const __grid_constant__ CUtensorMap tm_b1, const GemmParams p) {
  using C = GemmCfg<WQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // bf16: sA [4][128 x 64] | sB [4][256 x 64]                (bf16, 128-byte swizzle)
  // int8: sA [5][128 x 64] | sB8 [5][256 x 64] int8 staging | sB [2][256 x 64] bf16
  uint8_t* sA = smem;
  uint8_t* sB8 = sA + C::kStages * kATileBytes;
  uint8_t* sB = WQ ? sB8 + C::kStages * kB8TileBytes : sA + C::kStages * kATileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + (WQ ? C::kBStages : C::kStages) * kBTileBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (C::kStages + s); };
  auto bfull_bar = [&](uint32_t j) { return bar0 + 8u * (2 * C::kStages + j); };
  auto bempty_bar = [&](uint32_t j) { return bar0 + 8u * (2 * C::kStages + C::kBStages + j); };
  const uint32_t bar_t = bar0 + 8u * (2 * C::kStages + 2 * C::kBStages);
  auto tfull_bar = [&](uint32_t a) { return bar_t + 8u * a; };
  auto tempty_bar = [&](uint32_t a) { return bar_t + 8u * (2 + a); };
  const uint32_t drain_bar = bar_t + 8u * 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int off[kNumExperts + 1];
#pragma unroll
  for (int q = 0; q <= kNumExperts; ++q) off[q] = p.sched[kNumExperts + q];
  const int num_tiles = (off[kNumExperts] / kRowTile) * p.n_tiles;
  const int kb_count = p.K / kGemmBK;

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < (uint32_t)C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int j = 0; j < C::kBStages; ++j) {
      mbar_init(bfull_bar(j), kConvThreads);
      mbar_init(bempty_bar(j), 1);
    }
    for (uint32_t a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kEpiThreads);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b0);
    if (EPI == kEpiGeglu) tma_prefetch_desc(&tm_b1);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued[C::kStages];
#pragma unroll
      for (int s = 0; s < C::kStages; ++s) issued[s] = -1;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        const TileCoord tc = decode_tile(t, off, p.n_tiles);
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          const uint32_t a_dst = smem_addr(sA + stage * kATileBytes);
          // bf16 weights land in the MMA's B buffer; int8 weights in the staging buffer
          const uint32_t b_dst = smem_addr(WQ ? sB8 + stage * kB8TileBytes : sB + stage * kBTileBytes);
          const int b_half = WQ ? kB8TileBytes / 2 : kBTileBytes / 2;
          tma_load_2d(a_dst, &tm_a, fb, kb * kGemmBK, tc.row0);
          if (EPI == kEpiGeglu) {
            const int brow = tc.e * p.b_rows_per_expert + tc.n_blk * (kGemmBN / 2);
            tma_load_2d(b_dst, &tm_b0, fb, kb * kGemmBK, brow);
            tma_load_2d(b_dst + b_half, &tm_b1, fb, kb * kGemmBK, brow);
          } else {
            const int brow = tc.e * p.b_rows_per_expert + tc.n_blk * kGemmBN;
            tma_load_2d(b_dst, &tm_b0, fb, kb * kGemmBK, brow);
          }
          for (int s = 0; s < C::kStages; ++s)
            if (s == (int)stage) issued[s] = (int)phase;
          if (++stage == (uint32_t)C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every release of a stage by the MMA issuer has landed before exit
      for (int i = 0; i < C::kStages && ok; ++i) {
        if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) ok = false;
        if (++stage == (uint32_t)C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        raise_abort(abort_flag, p.err);
        // this role's copies still in flight complete before the CTA exits
        for (int s = 0; s < C::kStages; ++s)
          if (issued[s] >= 0) wait_bounded(full_bar(s), (uint32_t)issued[s], nullptr, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, bstage = 0, bphase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * kGemmBN;
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns) ||
              (WQ && !wait_bounded(bfull_bar(bstage), bphase, abort_flag, p.timeout_ns))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t adesc = smem_desc_k_sw128(smem_addr(sA + stage * kATileBytes));
          const uint64_t bdesc = smem_desc_k_sw128(smem_addr(sB + (WQ ? bstage : stage) * kBTileBytes));
#pragma unroll
          for (int kk = 0; kk < kGemmBK / 16; ++kk)  // +32 bytes along K inside the swizzle row
            umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, kGemmIdesc, (kb | kk) != 0);
          umma_commit(empty_bar(stage));
          if (++stage == (uint32_t)C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (WQ) {
            umma_commit(bempty_bar(bstage));
            if (++bstage == (uint32_t)C::kBStages) {
              bstage = 0;
              bphase ^= 1u;
            }
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // all MMAs issued by this thread are complete before TMEM is freed
      umma_commit(drain_bar);
      if (!wait_bounded(drain_bar, 0, nullptr, p.timeout_ns)) ok = false;
      if (!ok) raise_abort(abort_flag, p.err);
    }
  } else if (warp < kConvWarp0) {
    // --------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lanes [32q, 32q + 32) are reachable from this warp
    uint32_t acc = 0, acc_phase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const TileCoord tc = decode_tile(t, off, p.n_tiles);
      bool ok = wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) raise_abort(abort_flag, p.err);
        break;
      }
      tc_fence_after_sync();
      const int row = tc.row0 + q * 32 + lane;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kGemmBN;
      if (EPI == kEpiGeglu) {
        const int n0 = tc.n_blk * (kGemmBN / 2);
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + (size_t)row * p.n_out + n0;
#pragma unroll 1
        for (int c = 0; c < kGemmBN / 2 / 32; ++c) {
          uint32_t h[32], v[32];
          tmem_ld_32x32b_x32(tbase + c * 32, h);
          tmem_ld_32x32b_x32(tbase + kGemmBN / 2 + c * 32, v);
          tmem_ld_wait();
          if (WQ) {  // per-output-channel scales of W and Wv (same for every row)
            const size_t so = (size_t)tc.e * p.n_out + n0 + c * 32;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              float sw[8], sv[8];
              load_scales8(p.scale0 + so + 8 * g, sw);
              load_scales8(p.scale1 + so + 8 * g, sv);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                h[8 * g + j] = __float_as_uint(__uint_as_float(h[8 * g + j]) * sw[j]);
                v[8 * g + j] = __float_as_uint(__uint_as_float(v[8 * g + j]) * sv[j]);
              }
            }
          }
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float a0 = gelu_tanh(__uint_as_float(h[2 * j])) * __uint_as_float(v[2 * j]);
            const float a1 = gelu_tanh(__uint_as_float(h[2 * j + 1])) * __uint_as_float(v[2 * j + 1]);
            pk[j] = pack_bf16x2(a0, a1);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      } else {
        float* orow = static_cast<float*>(p.out) + (size_t)row * p.n_out;
        const float ps = p.row_scale[row];
#pragma unroll 1
        for (int c = 0; c < kGemmBN / 32; ++c) {
          const int col0 = tc.n_blk * kGemmBN + c * 32;
          if (col0 >= p.n_out) break;  // ragged last block along d (warp-uniform)
          uint32_t y[32];
          tmem_ld_32x32b_x32(tbase + c * 32, y);
          tmem_ld_wait();
          float sc[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) sc[j] = ps;
          if (WQ) {  // per-output-channel scale of W1
            const size_t so = (size_t)tc.e * p.n_out + col0;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              float s8[8];
              load_scales8(p.scale0 + so + 8 * g, s8);
#pragma unroll
              for (int j = 0; j < 8; ++j) sc[8 * g + j] = s8[j] * ps;
            }
          }
          float4* dst = reinterpret_cast<float4*>(orow + col0);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(y[4 * k]) * sc[4 * k], __uint_as_float(y[4 * k + 1]) * sc[4 * k + 1],
                                 __uint_as_float(y[4 * k + 2]) * sc[4 * k + 2],
                                 __uint_as_float(y[4 * k + 3]) * sc[4 * k + 3]);
        }
      }
      tc_fence_before_sync();
      mbar_arrive(tempty_bar(acc));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  } else if (WQ) {
    // -------------------------------------------------- int8 -> bf16 converter
    // Staging tile: 256 rows x 64 int8, row r at byte 64 r.  MMA tile: 256 rows x
    // 64 bf16 in 128-byte swizzle atoms of 8 rows: element (r, k) at
    // (r / 8) * 1024 + (r % 8) * 128 + ((k / 8) ^ (r % 8)) * 16 + (k % 8) * 2.
    const int ct = threadIdx.x - kConvWarp0 * 32;
    uint32_t stage = 0, phase = 0, bstage = 0, bphase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      for (int kb = 0; kb < kb_count; ++kb) {
        ok = __all_sync(0xffffffffu, wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns) &&
                                         wait_bounded(bempty_bar(bstage), bphase ^ 1u, abort_flag, p.timeout_ns));
        if (!ok) break;
        const uint8_t* src = sB8 + stage * kB8TileBytes;
        uint8_t* dst = sB + bstage * kBTileBytes;
#pragma unroll
        for (int i = 0; i < kB8TileBytes / 16 / kConvThreads; ++i) {
          const int u = ct + i * kConvThreads;  // 16-byte unit: row u / 4, int8 columns [16 (u % 4), +16)
          const int r = u >> 2, c = u & 3;
          const uint4 qv = *reinterpret_cast<const uint4*>(src + r * 64 + c * 16);
          uint4 o0, o1;
          i8x4_to_bf16x4(qv.x, o0.x, o0.y);
          i8x4_to_bf16x4(qv.y, o0.z, o0.w);
          i8x4_to_bf16x4(qv.z, o1.x, o1.y);
          i8x4_to_bf16x4(qv.w, o1.z, o1.w);
          uint8_t* rowp = dst + (r >> 3) * 1024 + (r & 7) * 128;
          *reinterpret_cast<uint4*>(rowp + (((2 * c) ^ (r & 7)) << 4)) = o0;
          *reinterpret_cast<uint4*>(rowp + (((2 * c + 1) ^ (r & 7)) << 4)) = o1;
        }
        fence_proxy_async_smem();  // generic-proxy writes -> visible to tcgen05.mma
        mbar_arrive(bfull_bar(bstage));
        if (++stage == (uint32_t)C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++bstage == (uint32_t)C::kBStages) {
          bstage = 0;
          bphase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) raise_abort(abort_flag, p.err);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace moe
