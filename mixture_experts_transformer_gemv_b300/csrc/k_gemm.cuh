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
//               128-byte swizzle, into a kGemmStages-deep shared-memory ring
//   warp 1      allocates 512 TMEM columns; lane 0 issues tcgen05.mma
//               (M=128, N=256, K=16, bf16 -> fp32) and tcgen05.commit
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, GeGLU or scale, stores
// Two TMEM accumulators (2 x 256 columns) let the epilogue of tile i overlap the
// mainloop of tile i+1.  In K3 the B tile stacks 128 rows of W over the same 128
// rows of Wv, so one N=256 MMA produces both branches of 128 output columns.
//
// Tiles never mix experts: expert e owns permuted rows [row_offset[e],
// row_offset[e+1]), a multiple of 128.  Tile t maps to (expert, n-block,
// m-block) with the m-block fastest, so CTAs working at the same time share the
// same weight tile through L2.
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
constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192;
constexpr int kEpiWarp0 = 2;   // first epilogue warp
constexpr int kATileBytes = kGemmBM * kGemmBK * 2;  // 16 KB
constexpr int kBTileBytes = kGemmBN * kGemmBK * 2;  // 32 KB
constexpr int kStageBytes = kATileBytes + kBTileBytes;
constexpr uint32_t kTmemCols = 2 * kGemmBN;  // two fp32 accumulators of 128 x 256
constexpr int kNumBars = 2 * kGemmStages + 5;   // full, empty, tmem_full x2, tmem_empty x2, drain
constexpr size_t kGemmSmemBytes = 1024 + (size_t)kGemmStages * kStageBytes + kNumBars * 8 + 16;
constexpr uint32_t kGemmIdesc = idesc_bf16_f32(kGemmBM, kGemmBN);

enum : int { kEpiGeglu = 0, kEpiDown = 1 };

struct GemmParams {
  const int32_t* sched;          // counts[E], row_offset[E + 1] (written by K2)
  int K;                         // reduction length: d (up) or F (down); multiple of 64
  int n_tiles;                   // tiles per expert along the output columns
  int b_rows_per_expert;         // rows of B per expert: F (W, Wv) or d (W1)
  int n_out;                     // output columns / leading dimension: F (act) or d (Y)
  void* out;                     // act [rows_cap, F] bf16 or Y [rows_cap, d] fp32
  const float* row_scale;        // down: combine weight of each permuted row
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

__device__ __forceinline__ void raise_abort(volatile uint32_t* abort_flag, uint32_t* err) {
  *abort_flag = 1u;
  atomicOr(err, kErrTimeout);
}

template <int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b0,
                        const __grid_constant__ CUtensorMap tm_b1, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kGemmStages * kATileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kGemmStages * kBTileBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (kGemmStages + s); };
  auto tfull_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kGemmStages + a); };
  auto tempty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kGemmStages + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kGemmStages + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int off[kNumExperts + 1];
#pragma unroll
  for (int q = 0; q <= kNumExperts; ++q) off[q] = p.sched[kNumExperts + q];
  const int num_tiles = (off[kNumExperts] / kRowTile) * p.n_tiles;
  const int kb_count = p.K / kGemmBK;

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < kGemmStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (uint32_t a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 32 * (kGemmThreads / 32 - kEpiWarp0));
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
      int issued[kGemmStages];
#pragma unroll
      for (int s = 0; s < kGemmStages; ++s) issued[s] = -1;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        const TileCoord tc = decode_tile(t, off, p.n_tiles);
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, kStageBytes);
          const uint32_t a_dst = smem_addr(sA + stage * kATileBytes);
          const uint32_t b_dst = smem_addr(sB + stage * kBTileBytes);
          tma_load_2d(a_dst, &tm_a, fb, kb * kGemmBK, tc.row0);
          if (EPI == kEpiGeglu) {
            const int brow = tc.e * p.b_rows_per_expert + tc.n_blk * (kGemmBN / 2);
            tma_load_2d(b_dst, &tm_b0, fb, kb * kGemmBK, brow);
            tma_load_2d(b_dst + kBTileBytes / 2, &tm_b1, fb, kb * kGemmBK, brow);
          } else {
            const int brow = tc.e * p.b_rows_per_expert + tc.n_blk * kGemmBN;
            tma_load_2d(b_dst, &tm_b0, fb, kb * kGemmBK, brow);
          }
          for (int s = 0; s < kGemmStages; ++s)
            if (s == (int)stage) issued[s] = (int)phase;
          if (++stage == kGemmStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every release of a stage by the MMA issuer has landed before exit
      for (int i = 0; i < kGemmStages && ok; ++i) {
        if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) ok = false;
        if (++stage == kGemmStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        raise_abort(abort_flag, p.err);
        // this role's copies still in flight complete before the CTA exits
        for (int s = 0; s < kGemmStages; ++s)
          if (issued[s] >= 0) wait_bounded(full_bar(s), (uint32_t)issued[s], nullptr, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * kGemmBN;
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t adesc = smem_desc_k_sw128(smem_addr(sA + stage * kATileBytes));
          const uint64_t bdesc = smem_desc_k_sw128(smem_addr(sB + stage * kBTileBytes));
#pragma unroll
          for (int kk = 0; kk < kGemmBK / 16; ++kk)  // +32 bytes along K inside the swizzle row
            umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, kGemmIdesc, (kb | kk) != 0);
          umma_commit(empty_bar(stage));
          if (++stage == kGemmStages) {
            stage = 0;
            phase ^= 1u;
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
  } else {
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
        __nv_bfloat16* orow =
            static_cast<__nv_bfloat16*>(p.out) + (size_t)row * p.n_out + tc.n_blk * (kGemmBN / 2);
#pragma unroll 1
        for (int c = 0; c < kGemmBN / 2 / 32; ++c) {
          uint32_t h[32], v[32];
          tmem_ld_32x32b_x32(tbase + c * 32, h);
          tmem_ld_32x32b_x32(tbase + kGemmBN / 2 + c * 32, v);
          tmem_ld_wait();
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
          float4* dst = reinterpret_cast<float4*>(orow + col0);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(y[4 * k]) * ps, __uint_as_float(y[4 * k + 1]) * ps,
                                 __uint_as_float(y[4 * k + 2]) * ps, __uint_as_float(y[4 * k + 3]) * ps);
        }
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
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace moe
