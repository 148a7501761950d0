// K3 / K4: expert-grouped GEMMs on the 5th-generation tensor cores, one CTA pair
// (a cluster of two CTAs on neighbouring SMs) per 256-row tile.
//
//   K3 (up, GeGLU):  act[r, n] = GELU(sum_k A[r,k] W[e,n,k]) * (sum_k A[r,k] Wv[e,n,k])
//   K4 (down):       Y[r, j]   = p[r] * sum_n act[r,n] W1[e,j,n]
// for every permuted row r of expert e ("Jah-yee/grok" README, architecture
// diagram: GELU(x W) (*) (x Wv), then the output projection; weights in PyTorch
// [out, in] order per "TevunahAi/Grok-1-BF16", "Weight Verification").
//
// A full tile is M = 256 permuted rows x N = 256 accumulator columns.  One thread of
// the even CTA issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16): A rows
// [0,128) and B rows [0,128) come from the even CTA's shared memory, A rows
// [128,256) and B rows [128,256) from the odd CTA's, and each CTA's Tensor Memory
// receives the accumulator of its own 128 rows.  Each CTA therefore stages only
// half of the weight tile: per k-block of 64 it loads A 128 x 64 and B 128 x 64
// (32 KB in bf16) for 128 x 256 x 64 MMA work, against 48 KB when a CTA works
// alone.  In K3 the even CTA's B half is 128 rows of W and the odd CTA's the
// same 128 rows of Wv, so accumulator columns [0,128) hold x W and [128,256)
// hold x Wv for the same 128 output channels; in K4 the halves are 2 x 128 rows
// of W1 (256 output columns of d).
//
// Warp roles in each CTA (one CTA per SM, persistent, static round-robin of
// tiles over pairs):
//   warp 0      TMA producer: the CTA's A and B halves per k-block into a
//               6-stage shared-memory ring, 128-byte swizzle
//   warp 1      allocates 512 TMEM columns (both CTAs, cta_group::2).  Even CTA:
//               issues the MMAs and tcgen05.commit, multicast to both CTAs'
//               barriers.  Odd CTA, bf16 weights: forwards the completion of each
//               of its own TMA stages to the even CTA's barrier.
//   warps 2-5   epilogue of the CTA's 128 rows: tcgen05.ld, GeGLU or scaling,
//               stores; then tell the even CTA's MMA warp the accumulator is free
//   warps 6-13  int8 weights only: int8 -> fp16 conversion of the CTA's B half,
//               two groups of four warps on alternate k-blocks
// Two TMEM accumulators (2 x 256 columns) let the epilogue of tile i overlap the
// mainloop of tile i+1 (one m-block per tile); with two m-blocks per tile (MB = 2,
// below) the two accumulators belong to one tile.
//
// Tiles never mix experts: expert e owns permuted rows [row_offset[e],
// row_offset[e+1]), a multiple of 128.  Its rows are cut into full tiles of 256
// and, when 128 rows are left, one half tile: there the pair issues M = 128
// MMAs (half the tensor-core work of a full tile), each CTA staging 64 A rows.
// With M = 128 the pair's Tensor Memory layout differs: each CTA's TMEM lanes
// 0-63 hold its 64 rows against accumulator columns [0, 128) and lanes 64-127
// the same rows against columns [128, 256), in TMEM columns [0, 128).  So in
// the up projection's half tile each CTA stages 64 rows of W and the same 64
// rows of Wv (the even CTA channels [0, 64) of the n-block, the odd CTA [64,
// 128)): every TMEM lane then holds h and v of the same 64 channels of one row.
// Tile t maps to (expert, n-block, m-block) with the m-block fastest, so pairs
// working at the same time share the same weight tile through L2.
//
// A full tile's operands arrive as one 128-row TMA box per CTA and operand; a
// half tile's A and its up-projection B halves (64 rows of W, 64 of Wv) as
// 64-row boxes (a second set of tensor maps).
//
// int8 weights ("TevunahAi/Grok-1-BF16", "Conversion Details": int8 values
// with bf16 scales, one per expert and output channel for the (8, 1, N) scale
// shape): TMA brings the CTA's raw int8 B half into a staging buffer; the
// converter warps rewrite it as fp16 in the 128-byte-swizzled K-major layout
// the MMA reads (exact: one byte shuffle and one subtraction per pair), make it
// visible to the tensor core's async proxy and tell the even CTA's MMA warp.
// The MMA then runs on fp16 operands, so an int8 layer carries its activation
// rows in fp16 (the gather writes them, the up projection's epilogue writes the
// GeGLU activations, saturating at +-65504); fp16 has 3 more mantissa bits than
// bf16, and its conversion takes half the integer work, which set the rate.  Because the scale
// belongs to an output channel it factors out of the reduction and is applied
// in fp32 in the epilogue: sum_k a_k (q_nk s_n) = s_n sum_k a_k q_nk.  Scales that
// also vary along k (G > 1 groups) do not factor out; the converters then
// multiply each converted weight by its group's scale (f16x2, one rounding).
//
// Every wait is bounded (wait_bounded).  A role that times out raises its CTA's
// abort flag and the device error word; the others stop at their next wait
// (the other CTA's roles run out of time on theirs); the producer then waits
// (bounded) for its own TMA copies in flight, the MMA issuer for its own MMAs,
// and both CTAs meet at a cluster barrier before TMEM is freed and they exit.
#pragma once
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"
#include "ptx_pair.cuh"

namespace moe {

constexpr int kGemmBM = 256;     // rows per full tile (pair)
constexpr int kGemmHalfM = 128;  // rows per CTA of a full tile; rows of a half tile
constexpr int kGemmBoxRows = 64; // rows of the half tiles' TMA boxes
constexpr int kGemmBN = 256;     // MMA N (accumulator columns)
constexpr int kGemmHalfN = 128;  // B rows per CTA
constexpr int kGemmBK = 64;      // K per stage (64 bf16 = one 128-byte swizzle row)
constexpr int kEpiWarp0 = 2;     // first epilogue warp (warps 2-5)
constexpr int kConvWarp0 = 6;    // first converter warp (warps 6-13, int8 weights only)
constexpr int kEpiWarps = 4;
constexpr int kConvWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kConvGroups = 2;                              // converter groups, alternate k-blocks
constexpr int kConvGroupThreads = kConvThreads / kConvGroups;
constexpr int kATileBytes = kGemmHalfM * kGemmBK * 2;   // 16 KB
constexpr int kBTileBytes = kGemmHalfN * kGemmBK * 2;   // 16 KB (bf16, swizzled)
constexpr int kB8TileBytes = kGemmHalfN * kGemmBK;      // 8 KB (int8 staging, dense rows of 64 B)
constexpr uint32_t kTmemCols = 2 * kGemmBN;              // two fp32 accumulators of 128 x 256 per CTA
constexpr uint32_t kGemmIdesc = idesc_bf16_f32(kGemmBM, kGemmBN);
constexpr uint32_t kGemmIdescHalf = idesc_bf16_f32(kGemmHalfM, kGemmBN);
// fp16 A and B (format 0 in bits 7-9 and 10-12): int8 weights converted to fp16,
// or fp16 operands on the bf16 path (f16_operands)
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t kGemmIdescF16 = idesc_f16_f32(kGemmBM, kGemmBN);
constexpr uint32_t kGemmIdescF16Half = idesc_f16_f32(kGemmHalfM, kGemmBN);
static_assert(kGemmBM == 2 * kRowPad, "an expert's row block is full tiles and at most one half tile");

// Per weight type:
//   bf16: a TMA ring of 6 stages, A 16 KB + B 16 KB each; 6 warps.
//   int8: a TMA ring of 5 stages, A 16 KB + int8 B 8 KB each, and a ring of 5
//         converted fp16 B halves (16 KB each) between the converter warps and
//         the MMA warp; 14 warps.  Both rings have the same depth, so k-block g
//         uses TMA stage g % 5 and converted buffer g % 5, and one commit of the
//         MMA issuer per k-block (to the stage's empty barrier, which the
//         converters also wait on) frees both; a second commit per k-block cost
//         8 %.  (Measured at the int8 workload, TMA + converted stages with two
//         commits: 6 + 3 1030-1040 TFLOP/s, 5 + 6 1059-1072, 5 + 5 1064, 4 + 6
//         1009, 3 + 6 883; 5 + 5 with one commit 1126-1144.  Loading the int8
//         weights into the converters' registers straight from global memory,
//         two k-blocks ahead, instead of staging them by TMA: 660.)
//   MB = 2 (paired m-blocks, taken by the layer for F >= 16384): every tile is
//         two m-blocks of one expert against one n-block, accumulated in TMEM
//         columns [0, 256) and [256, 512), so each B k-block (converted once for
//         int8) feeds twice the MMA work and B crosses L2 half as often; the
//         epilogue no longer overlaps the next tile.  In the up projection a half
//         block stays a tile of its own (its B is staged differently); in the
//         down projection it pairs with the full block before it.  Rings of 4
//         stages (A 2 x 16 KB + B).
// Dynamic tile schedule: slots of the ring through which the even CTA's
// producer thread hands each tile index to every other role of the pair.
constexpr int kTileRing = 8;

template <bool WQ, int MB = 1>
struct GemmCfg {
  static constexpr int kStages = MB == 2 ? 4 : (WQ ? 5 : 6);  // TMA ring
  static constexpr int kBStages = WQ ? kStages : 0;           // converted-B ring (same depth: one release for both)
  static constexpr int kStageBytes = MB * kATileBytes + (WQ ? kB8TileBytes : kBTileBytes);  // smem per stage
  static constexpr int kThreads = 32 * (kConvWarp0 + (WQ ? kConvWarps : 0));
  // full, empty (TMA ring; empty also frees the converted buffer of the same index),
  // bfull (converted ring), tmem_full x2, tmem_empty x2, drain, tile ring fill / free
  static constexpr int kNumBars = 2 * kStages + kBStages + 5 + 2 * kTileRing;
  // readers of each tile-ring slot: even CTA MMA thread, epilogue warps,
  // converter warps; odd CTA producer thread, forwarding thread (bf16),
  // epilogue warps, converter warps
  static constexpr int kTileReaders = 1 + kEpiWarps + (WQ ? kConvWarps : 0) + 1 + (WQ ? 0 : 1) + kEpiWarps +
                                      (WQ ? kConvWarps : 0);
  static_assert(!WQ || kBStages == kStages, "one release frees a TMA stage and its converted buffer");
  static constexpr size_t kSmemBytes =
      1024 + (size_t)kStages * kStageBytes + (size_t)kBStages * kBTileBytes + kNumBars * 8 + 16 + kTileRing * 4;
};
constexpr int kGemmThreads = GemmCfg<false>::kThreads;
constexpr int kGemmMBPair = 2;  // m-blocks per tile of the layer's GEMMs when they pair m-blocks
constexpr size_t kGemmSmemBytes = GemmCfg<false>::kSmemBytes;

struct GemmParams {
  const int32_t* sched;          // counts[E], row_offset[E + 1] (written by K2)
  int K;                         // reduction length: d (up) or F (down); multiple of 64
  int n_tiles;                   // tiles per expert along the output columns
  int b_rows_per_expert;         // rows of B per expert: F (W, Wv) or d (W1)
  int n_out;                     // output columns / leading dimension: F (act) or d (Y)
  void* out;                     // act [rows_cap, F] bf16 or Y [rows_cap, d] fp32
  const float* row_scale;        // down: combine weight of each permuted row
  const uint16_t* scale0;        // int8: bf16 bits [E_s, G, n_out], scale of W (up) or W1 (down)
  const uint16_t* scale1;        // int8 up: bf16 bits [E_s, G, F], scale of Wv
  int scale_experts;             // int8: E_s, 8 (per expert) or 1 (shared)
  int scale_groups;              // int8: G groups along the reduction; 1 = per output channel only
  int group_kb;                  // int8, G > 1: k-blocks of 64 per group
  int f16_operands;              // bf16 path: A and B hold fp16 instead of bf16 (both the same type)
  int checks;                    // int8 up projection: report activations past the fp16 range
  int* tile_counter;             // dynamic tile schedule: a counter that is 0 at launch; nullptr: static
  uint32_t* err;                 // device error word
  uint64_t timeout_ns;           // limit of every wait
};

// A tile: MB consecutive m-blocks of one expert (the last tile of an expert
// may hold fewer) against one n-block.  An m-block is 256 rows, or 128 (a half
// tile) at the end of the expert's block.
template <int MB>
struct TileCoord {
  int e, n_blk, nm;  // nm: m-blocks in this tile
  int row0[MB];
  bool half[MB];     // 128 rows (M = 128 MMAs) instead of 256
};

// Tiles along m of one expert with `rows` padded rows (a multiple of 128): its
// m-blocks are rows / 256 full ones and, when rows % 256 = 128, one half block.
// MB = 1: one m-block per tile.  MB = 2 with PH (down projection): consecutive
// m-blocks in pairs, the half block included (ordered in two phases, see
// mblock_prefix).  MB = 2 without PH (up projection, whose half tiles stage B
// differently): the full blocks in pairs, the half block a tile of its own.
template <int MB, bool PH>
__device__ __forceinline__ int mtiles(int rows) {
  const int nblk = (rows + kGemmBM - 1) / kGemmBM;
  if (MB == 1) return nblk;
  if (PH) return (nblk + 1) / 2;
  const int nfull = rows / kGemmBM;
  return (nfull + 1) / 2 + (nblk - nfull);
}

// Tiles along m of the experts before e: mb[e] = sum_{q < e} mtiles(rows of q).
// Paired down projection (MB = 2, PH): two phases.  mb[] counts each expert's
// uniform tiles (two full m-blocks), pb[] its last tile when that holds less
// (a full block with a half one, or one block alone): every uniform tile of every
// expert first, so the long tiles in flight have the same length and stay in step,
// then the shorter ones.
template <int MB, bool PH>
__device__ __forceinline__ void mblock_prefix(const int (&off)[kNumExperts + 1], int (&mb)[kNumExperts + 1],
                                              int (&pb)[kNumExperts + 1]) {
  mb[0] = 0;
  pb[0] = 0;
#pragma unroll
  for (int q = 0; q < kNumExperts; ++q) {
    const int rows = off[q + 1] - off[q];
    if (MB == 2 && PH) {
      const int nblk = (rows + kGemmBM - 1) / kGemmBM, u = (rows / kGemmBM) / 2;
      mb[q + 1] = mb[q] + u;
      pb[q + 1] = pb[q] + (nblk > 2 * u ? 1 : 0);
    } else {
      mb[q + 1] = mb[q] + mtiles<MB, PH>(rows);
      pb[q + 1] = 0;
    }
  }
}

// Tile t -> (expert, n-block, its m-blocks); tiles of expert e are
// [mb[e] * n_tiles, mb[e + 1] * n_tiles), the m position fastest.
template <int MB, bool PH>
__device__ __forceinline__ TileCoord<MB> decode_tile(int t, const int (&off)[kNumExperts + 1],
                                                     const int (&mb)[kNumExperts + 1],
                                                     const int (&pb)[kNumExperts + 1], int n_tiles) {
  if (MB == 2 && PH && t >= mb[kNumExperts] * n_tiles) {  // phase 2: the experts' last, shorter tiles
    const int t2 = t - mb[kNumExperts] * n_tiles;
    int e = 0;
#pragma unroll
    for (int q = 1; q < kNumExperts; ++q)
      if (t2 >= pb[q] * n_tiles) e = q;
    const int rows = off[e + 1] - off[e];
    const int nblk = (rows + kGemmBM - 1) / kGemmBM;
    const int first = ((rows / kGemmBM) / 2) * 2;
    TileCoord<MB> c;
    c.e = e;
    c.n_blk = t2 - pb[e] * n_tiles;
    c.nm = nblk - first;
#pragma unroll
    for (int j = 0; j < MB; ++j) {
      c.row0[j] = off[e] + (first + j) * kGemmBM;
      c.half[j] = off[e + 1] - c.row0[j] < kGemmBM;
    }
    return c;
  }
  int e = 0;
#pragma unroll
  for (int q = 1; q < kNumExperts; ++q)
    if (t >= mb[q] * n_tiles) e = q;
  const int mt = mb[e + 1] - mb[e];
  const int local = t - mb[e] * n_tiles;
  const int nfull = (off[e + 1] - off[e]) / kGemmBM;
  const int i = local % mt;
  // first m-block of the tile and how many it holds
  int first = i * MB, nm = 1;
  if (MB == 2 && PH) nm = 2;  // phase 1: two full m-blocks
  if (MB == 2 && !PH) {
    const int npair = (nfull + 1) / 2;
    nm = i < npair ? min(2, nfull - first) : 1;
    if (i >= npair) first = nfull;
  }
  TileCoord<MB> c;
  c.e = e;
  c.n_blk = local / mt;
  c.nm = nm;
#pragma unroll
  for (int j = 0; j < MB; ++j) {
    c.row0[j] = off[e] + (first + j) * kGemmBM;
    c.half[j] = off[e + 1] - c.row0[j] < kGemmBM;
  }
  return c;
}

// 4 int8 (one 32-bit word, element i in byte i) -> 4 fp16 in two words, exact:
// u = q + 128 (sign bit flipped) in the low byte of the fp16 pattern 0x64uu is
// 1024 + u, and subtracting 1152 leaves q.
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = f16x2_sub(__byte_perm(u, 0x64u, 0x4140), 0x64806480u);
  hi = f16x2_sub(__byte_perm(u, 0x64u, 0x4342), 0x64806480u);
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 8 bf16 scales (16 bytes of bf16 bits) -> fp32.
__device__ __forceinline__ void load_scales8(const uint16_t* p, float (&s)[8]) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  s[0] = bf16_lo(v.x); s[1] = bf16_hi(v.x); s[2] = bf16_lo(v.y); s[3] = bf16_hi(v.y);
  s[4] = bf16_lo(v.z); s[5] = bf16_hi(v.z); s[6] = bf16_lo(v.w); s[7] = bf16_hi(v.w);
}

template <int EPI, bool WQ, int MB = 1>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GemmCfg<WQ, MB>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b0,
                        const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_ah,
                        const __grid_constant__ CUtensorMap tm_b0h, const __grid_constant__ CUtensorMap tm_b1h,
                        const GemmParams p) {
  using C = GemmCfg<WQ, MB>;
  // Paired m-blocks: a half block pairs with a full one only in the down
  // projection (its half-tile B is staged like a full tile's).
  constexpr bool PH = EPI == kEpiDown;
  extern __shared__ uint8_t smem_raw[];
  // The layout depends only on compile-time sizes, so the offsets are the same
  // in both CTAs of the pair (the MMA relies on that).
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // sA [stages][MB][128 x 64] | sB [stages][128 x 64]                (bf16 weights)
  // sA [stages][MB][128 x 64] | sB8 [stages][128 x 64] int8 | sB [stages][128 x 64] fp16  (int8 weights)
  uint8_t* sA = smem;
  uint8_t* sB8 = sA + C::kStages * MB * kATileBytes;
  uint8_t* sB = WQ ? sB8 + C::kStages * kB8TileBytes : sA + C::kStages * MB * kATileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + (WQ ? C::kBStages : C::kStages) * kBTileBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile int* tile_ring = reinterpret_cast<volatile int*>(tmem_slot + 4);  // [kTileRing]
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (C::kStages + s); };
  auto bfull_bar = [&](uint32_t j) { return bar0 + 8u * (2 * C::kStages + j); };
  const uint32_t bar_t = bar0 + 8u * (2 * C::kStages + C::kBStages);
  auto tfull_bar = [&](uint32_t a) { return bar_t + 8u * a; };
  auto tempty_bar = [&](uint32_t a) { return bar_t + 8u * (2 + a); };
  const uint32_t drain_bar = bar_t + 8u * 4;
  auto tfill_bar = [&](uint32_t i) { return bar_t + 8u * (5 + i); };
  auto tfree_bar = [&](uint32_t i) { return bar_t + 8u * (5 + kTileRing + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its partner
  const bool leader = rank == 0;
  const int pair = (int)cluster_id_x(), num_pairs = (int)num_clusters_x();

  int off[kNumExperts + 1], mb[kNumExperts + 1], pb[kNumExperts + 1];
#pragma unroll
  for (int q = 0; q <= kNumExperts; ++q) off[q] = p.sched[kNumExperts + q];
  mblock_prefix<MB, PH>(off, mb, pb);
  const int num_tiles = (mb[kNumExperts] + pb[kNumExperts]) * p.n_tiles;
  const int kb_count = p.K / kGemmBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      // bf16: the even CTA's stage is full when its own copies landed and the
      // odd CTA forwarded the completion of its copies
      mbar_init(full_bar(s), (!WQ && leader) ? 2 : 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int j = 0; j < C::kBStages; ++j) {
      mbar_init(bfull_bar(j), 2);  // one arrival per CTA (after all its converter warps)
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * kEpiWarps);  // one arrival per epilogue warp of either CTA
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < kTileRing; ++i) {
      mbar_init(tfill_bar(i), 1);                  // the even CTA's scheduler
      mbar_init(tfree_bar(i), C::kTileReaders);    // used in the even CTA only
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b0);
    tma_prefetch_desc(&tm_ah);
    if (EPI == kEpiGeglu) {
      tma_prefetch_desc(&tm_b1);
      tma_prefetch_desc(&tm_b0h);
      tma_prefetch_desc(&tm_b1h);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // ---- the pair's tile sequence
  // Static (p.tile_counter == nullptr): tiles pair, pair + num_pairs, ...
  // Dynamic: the pair's first tile is `pair`, every later one num_pairs +
  // atomicAdd(counter, 1), taken by the even CTA's producer thread when it
  // starts the tile and published in slot i % kTileRing of both CTAs' tile
  // rings; every other role of both CTAs reads the same sequence from its own
  // CTA's ring and frees the slot on the even CTA's tfree barrier.  A pair that
  // finishes early takes the next tile, so the tiles in flight stay a window of
  // consecutive indices (m-block fastest) whose weight tiles and A rows are
  // shared through L2; under the static order pairs drift apart over a long
  // launch and re-read both from DRAM.
  const bool dyn = p.tile_counter != nullptr;
  // the even CTA's producer thread: tile i of the pair, or -1 when none is left
  auto sched_tile = [&](int i, bool& ok) -> int {
    if (!dyn) {
      const int t = pair + i * num_pairs;
      return t < num_tiles ? t : -1;
    }
    const uint32_t slot = (uint32_t)(i % kTileRing), ph = (uint32_t)(i / kTileRing) & 1u;
    if (!wait_bounded_cluster(tfree_bar(slot), ph ^ 1u, abort_flag, p.timeout_ns)) {
      ok = false;
      return -1;
    }
    int t = i == 0 ? pair : num_pairs + atomicAdd(p.tile_counter, 1);
    if (t >= num_tiles) t = -1;
    tile_ring[slot] = t;
    st_cluster_u32(map_to_cta(smem_addr(const_cast<int*>(&tile_ring[slot])), 1), (uint32_t)t);
    mbar_arrive(tfill_bar(slot));
    mbar_arrive_cluster(map_to_cta(tfill_bar(slot), 1));
    return t;
  };
  // every other role: tile i of the pair, or -1 (every lane of a warp role calls it)
  auto next_tile = [&](int i, bool warp_role, bool& ok) -> int {
    if (!dyn) {
      const int t = pair + i * num_pairs;
      return t < num_tiles ? t : -1;
    }
    const uint32_t slot = (uint32_t)(i % kTileRing), ph = (uint32_t)(i / kTileRing) & 1u;
    bool got = leader ? wait_bounded(tfill_bar(slot), ph, abort_flag, p.timeout_ns)
                      : wait_bounded_cluster(tfill_bar(slot), ph, abort_flag, p.timeout_ns);
    if (warp_role) got = __all_sync(0xffffffffu, got);
    if (!got) {
      ok = false;
      return -1;
    }
    const int t = tile_ring[slot];
    if (warp_role) __syncwarp();
    if (!warp_role || lane == 0) {
      if (leader)
        mbar_arrive(tfree_bar(slot));
      else
        mbar_arrive_cluster(map_to_cta(tfree_bar(slot), 0));
    }
    return t;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued[C::kStages];
#pragma unroll
      for (int s = 0; s < C::kStages; ++s) issued[s] = -1;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int t = leader ? sched_tile(i, ok) : next_tile(i, false, ok);
        if (t < 0) break;
        const TileCoord<MB> tc = decode_tile<MB, PH>(t, off, mb, pb, p.n_tiles);
        // this CTA's 128 rows of B.  Up projection, full tile: 128 rows of W
        // (even) or Wv (odd), one box; half tile: the CTA's 64 rows of the
        // n-block from W, then the same 64 rows from Wv (two 64-row boxes).
        // Down projection: the first or second 128 output rows of W1, one box.
        const int nrow = tc.e * p.b_rows_per_expert;
        const bool split_b = EPI == kEpiGeglu && tc.half[0];
        const int brow = (EPI == kEpiGeglu) ? nrow + tc.n_blk * kGemmHalfN + (tc.half[0] ? (int)rank * kGemmBoxRows : 0)
                                            : nrow + tc.n_blk * kGemmBN + (int)rank * kGemmHalfN;
        const CUtensorMap* bmap = (EPI == kEpiGeglu && !leader) ? &tm_b1 : &tm_b0;
        constexpr int kBBox = (WQ ? kB8TileBytes : kBTileBytes) / 2;
        // bytes per stage: each m-block's A rows (128 per CTA, 64 in a half tile) and B
        uint32_t tx = WQ ? kB8TileBytes : kBTileBytes;
#pragma unroll
        for (int j = 0; j < MB; ++j)
          if (j < tc.nm) tx += tc.half[j] ? kATileBytes / 2 : kATileBytes;
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, tx);
#pragma unroll
          for (int j = 0; j < MB; ++j)  // this CTA's A rows of each m-block: 128, or 64 of a half tile
            if (j < tc.nm)
              tma_load_2d(smem_addr(sA + (stage * MB + j) * kATileBytes), tc.half[j] ? &tm_ah : &tm_a, fb,
                          kb * kGemmBK, tc.row0[j] + (int)rank * (tc.half[j] ? kGemmBoxRows : kGemmHalfM));
          const uint32_t sb = smem_addr(WQ ? sB8 + stage * kB8TileBytes : sB + stage * kBTileBytes);
          if (split_b) {
            tma_load_2d(sb, &tm_b0h, fb, kb * kGemmBK, brow);
            tma_load_2d(sb + kBBox, &tm_b1h, fb, kb * kGemmBK, brow);
          } else {
            tma_load_2d(sb, bmap, fb, kb * kGemmBK, brow);
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
        // (each one completes the phase of this CTA's own full barrier it was
        // issued for; the even CTA's barrier also needs the odd CTA's arrival,
        // which the bounded wait gives up on)
        for (int s = 0; s < C::kStages; ++s)
          if (issued[s] >= 0) wait_bounded(full_bar(s), (uint32_t)issued[s], nullptr, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // --------------------------------------------------- MMA issuer (even CTA)
      uint32_t stage = 0, phase = 0, bstage = 0, bphase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int t = next_tile(i, false, ok);
        if (t < 0) break;
        const TileCoord<MB> tc = decode_tile<MB, PH>(t, off, mb, pb, p.n_tiles);
        if (!wait_bounded_cluster(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t idesc[MB];
#pragma unroll
        for (int j = 0; j < MB; ++j)
          idesc[j] = (WQ || p.f16_operands) ? (tc.half[j] ? kGemmIdescF16Half : kGemmIdescF16)
                                            : (tc.half[j] ? kGemmIdescHalf : kGemmIdesc);
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!wait_bounded_cluster(full_bar(stage), phase, abort_flag, p.timeout_ns) ||
              (WQ && !wait_bounded_cluster(bfull_bar(bstage), bphase, abort_flag, p.timeout_ns))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t bdesc = smem_desc_k_sw128(smem_addr(sB + (WQ ? bstage : stage) * kBTileBytes));
#pragma unroll
          for (int j = 0; j < MB; ++j) {
            if (j >= tc.nm) break;
            // MB = 1: accumulator acc (two, alternating per tile); MB = 2: m-block j in TMEM columns [256 j, +256)
            const uint32_t d_tmem = tmem_base + (MB == 2 ? (uint32_t)j : acc) * kGemmBN;
            const uint64_t adesc = smem_desc_k_sw128(smem_addr(sA + (stage * MB + j) * kATileBytes));
#pragma unroll
            for (int kk = 0; kk < kGemmBK / 16; ++kk)  // +32 bytes along K inside the swizzle row
              umma_bf16_pair(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc[j], (kb | kk) != 0);
          }
          umma_commit_pair(empty_bar(stage), 0x3);  // frees the stage in both CTAs
          if (++stage == (uint32_t)C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (WQ) {
            if (++bstage == (uint32_t)C::kBStages) {
              bstage = 0;
              bphase ^= 1u;
            }
          }
        }
        if (!ok) break;
        umma_commit_pair(tfull_bar(acc), 0x3);  // both CTAs' epilogues may read
        if (MB == 2) {  // one set of accumulators (all 512 columns) per tile
          acc_phase ^= 1u;
        } else {
          acc ^= 1u;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      // all MMAs issued by this thread are complete before TMEM is freed
      umma_commit_pair(drain_bar, 0x1);
      if (!wait_bounded(drain_bar, 0, nullptr, p.timeout_ns)) ok = false;
      if (!ok) raise_abort(abort_flag, p.err);
    } else if (!WQ && !leader && lane == 0) {
      // ------------------------- odd CTA, bf16: forward its stage completions
      // The MMA of the even CTA reads this CTA's A and B halves; it may start a
      // k-block once this CTA's copies of it have landed.
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        if (next_tile(i, false, ok) < 0) break;
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          // The copies were made by this CTA's TMA and are complete (the local
          // phase completed); this thread wrote nothing, so a relaxed arrival
          // is enough and avoids a cluster-scope release per k-block.
          mbar_arrive_cluster_relaxed(map_to_cta(full_bar(stage), 0));
          if (++stage == (uint32_t)C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) raise_abort(abort_flag, p.err);
    }
  } else if (warp < kEpiWarp0 + kEpiWarps) {
    // --------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lanes [32q, 32q + 32) are reachable from this warp
    uint32_t acc = 0, acc_phase = 0;
    for (int i = 0;; ++i) {
      bool ok = true;
      const int t = next_tile(i, true, ok);
      if (t < 0) {
        if (!ok && lane == 0) raise_abort(abort_flag, p.err);
        break;
      }
      const TileCoord<MB> tc = decode_tile<MB, PH>(t, off, mb, pb, p.n_tiles);
      ok = wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) raise_abort(abort_flag, p.err);
        break;
      }
      tc_fence_after_sync();
#pragma unroll
      for (int jm = 0; jm < MB; ++jm) {
      if (jm >= tc.nm) break;
      // Full tile: lane = row of the CTA's 128, all 256 accumulator columns.
      // Half tile: lane % 64 = row of the CTA's 64, lanes >= 64 hold accumulator
      // columns [128, 256) in TMEM columns [0, 128).
      const bool thalf = tc.half[jm];
      const int hsel = thalf ? (q >> 1) : 0;
      const int row = thalf ? tc.row0[jm] + (int)rank * kGemmBoxRows + (q & 1) * 32 + lane
                            : tc.row0[jm] + (int)rank * kGemmHalfM + q * 32 + lane;
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + (MB == 2 ? (uint32_t)jm : acc) * kGemmBN;
      if (EPI == kEpiGeglu) {
        // full tile: channels n0 + [0, 128), h in TMEM columns [0, 128), v in [128, 256);
        // half tile: channels n0 + 64 hsel + [0, 64), h in [0, 64), v in [64, 128)
        const int nch = thalf ? kGemmHalfN / 2 : kGemmHalfN;
        const int n0 = tc.n_blk * kGemmHalfN + hsel * (kGemmHalfN / 2);
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + (size_t)row * p.n_out + n0;
        bool sat = false;  // int8 layers, device checks: an activation past the fp16 range
#pragma unroll 1
        for (int c = 0; c < nch / 32; ++c) {
          uint32_t h[32], v[32];
          tmem_ld_32x32b_x32(tbase + c * 32, h);
          tmem_ld_32x32b_x32(tbase + nch + c * 32, v);
          tmem_ld_wait();
          if (WQ && p.scale_groups == 1) {  // per-output-channel scales of W and Wv (same for every row)
            const size_t so = (size_t)(p.scale_experts > 1 ? tc.e : 0) * p.n_out + n0 + c * 32;
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
            pk[j] = WQ ? pack_f16x2_sat(a0, a1) : pack_bf16x2(a0, a1);  // int8 layers carry fp16 rows
            if (WQ) sat |= fmaxf(fabsf(a0), fabsf(a1)) > kF16Max;
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
        if (WQ && p.checks && __any_sync(0xffffffffu, sat) && lane == 0) atomicOr(p.err, kErrSaturate);
      } else {
        // full tile: output columns n_blk 256 + [0, 256); half tile: n_blk 256 + 128 hsel + [0, 128)
        float* orow = static_cast<float*>(p.out) + (size_t)row * p.n_out;
        const float ps = p.row_scale[row];
        const int ncol = thalf ? kGemmBN / 2 : kGemmBN;
#pragma unroll 1
        for (int c = 0; c < ncol / 32; ++c) {
          const int col0 = tc.n_blk * kGemmBN + hsel * (kGemmBN / 2) + c * 32;
          if (col0 >= p.n_out) break;  // ragged last block along d (warp-uniform)
          uint32_t y[32];
          tmem_ld_32x32b_x32(tbase + c * 32, y);
          tmem_ld_wait();
          float sc[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) sc[j] = ps;
          if (WQ && p.scale_groups == 1) {  // per-output-channel scale of W1
            const size_t so = (size_t)(p.scale_experts > 1 ? tc.e : 0) * p.n_out + col0;
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
      }  // m-blocks of the tile
      // this warp's TMEM reads are complete: free the accumulator for the MMA warp
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(tempty_bar(acc));
        else
          mbar_arrive_cluster(map_to_cta(tempty_bar(acc), 0));
      }
      if (MB == 2) {
        acc_phase ^= 1u;
      } else {
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
  } else if constexpr (WQ) {
    // -------------------------------------------------- int8 -> fp16 converter
    // Staging tile: 128 rows x 64 int8, row r at byte 64 r.  MMA tile: 128 rows x
    // 64 fp16 in 128-byte swizzle atoms of 8 rows: element (r, k) at
    // (r / 8) * 1024 + (r % 8) * 128 + ((k / 8) ^ (r % 8)) * 16 + (k % 8) * 2.
    // Two groups of four warps take alternate k-blocks (group g the k-blocks
    // with an even or odd running count), so two conversions are in flight at
    // once.  A wait on a ring barrier never sees a phase two ahead of the one
    // it expects: the next phase of any slot a group waits on (a TMA stage or
    // a converted buffer) needs that group's own conversion first.
    const int grp = (warp - kConvWarp0) / (kConvWarps / kConvGroups);
    const int ct = threadIdx.x - (kConvWarp0 + grp * (kConvWarps / kConvGroups)) * 32;
    int gk = 0;  // running k-block count over this CTA's tiles
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int t = next_tile(i, true, ok);
      if (t < 0) break;
      // grouped scales (G > 1): staged B row r is weight row nb + r of the matrix
      // whose scales are gsc; in an up-projection half tile rows [64, 128) are
      // the same channels of Wv as rows [0, 64) of W
      const TileCoord<MB> tc = decode_tile<MB, PH>(t, off, mb, pb, p.n_tiles);
      const bool split_wv = EPI == kEpiGeglu && tc.half[0];
      const int nb = (EPI == kEpiGeglu) ? tc.n_blk * kGemmHalfN + (tc.half[0] ? (int)rank * kGemmBoxRows : 0)
                                        : tc.n_blk * kGemmBN + (int)rank * kGemmHalfN;
      const uint16_t* gsc = (EPI == kEpiGeglu && !leader && !tc.half[0]) ? p.scale1 : p.scale0;
      const size_t gsc_e = (size_t)(p.scale_experts > 1 ? tc.e : 0) * p.scale_groups;
      for (int kb = 0; kb < kb_count; ++kb) {
        const int my = gk++;
        if ((my & 1) != grp) continue;
        const uint32_t stage = (uint32_t)(my % C::kStages), phase = (uint32_t)(my / C::kStages) & 1u;
        const uint32_t bstage = (uint32_t)(my % C::kBStages), bphase = (uint32_t)(my / C::kBStages) & 1u;
        const bool got = __all_sync(0xffffffffu, wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns) &&
                                                     wait_bounded(empty_bar(bstage), bphase ^ 1u, abort_flag,
                                                                  p.timeout_ns));
        if (got) {
          const uint8_t* src = sB8 + stage * kB8TileBytes;
          uint8_t* dst = sB + bstage * kBTileBytes;
          // one 16-byte unit: row u / 4, int8 columns [16 (u % 4), +16), optionally times
          // this row's group scale (bf16 bits in both halves of s2)
          auto convert = [&](auto with_scale) {
#pragma unroll
            for (int i = 0; i < kB8TileBytes / 16 / kConvGroupThreads; ++i) {
              const int u = ct + i * kConvGroupThreads;
              const int r = u >> 2, c = u & 3;
              const uint4 qv = *reinterpret_cast<const uint4*>(src + r * 64 + c * 16);
              uint4 o0, o1;
              i8x4_to_f16x4(qv.x, o0.x, o0.y);
              i8x4_to_f16x4(qv.y, o0.z, o0.w);
              i8x4_to_f16x4(qv.z, o1.x, o1.y);
              i8x4_to_f16x4(qv.w, o1.z, o1.w);
              if constexpr (decltype(with_scale)::value) {
                const bool wv_row = split_wv && r >= kGemmBoxRows;
                const int n = nb + (wv_row ? r - kGemmBoxRows : r);
                const uint16_t* sarr = wv_row ? p.scale1 : gsc;
                const uint32_t sb = n < p.n_out ? sarr[(gsc_e + kb / p.group_kb) * p.n_out + n] : 0u;
                __half2 sh = __float2half2_rn(__uint_as_float(sb << 16));
                const uint32_t s2 = *reinterpret_cast<uint32_t*>(&sh);
                o0 = make_uint4(f16x2_mul(o0.x, s2), f16x2_mul(o0.y, s2), f16x2_mul(o0.z, s2), f16x2_mul(o0.w, s2));
                o1 = make_uint4(f16x2_mul(o1.x, s2), f16x2_mul(o1.y, s2), f16x2_mul(o1.z, s2), f16x2_mul(o1.w, s2));
              }
              uint8_t* rowp = dst + (r >> 3) * 1024 + (r & 7) * 128;
              *reinterpret_cast<uint4*>(rowp + (((2 * c) ^ (r & 7)) << 4)) = o0;
              *reinterpret_cast<uint4*>(rowp + (((2 * c + 1) ^ (r & 7)) << 4)) = o1;
            }
          };
          if (p.scale_groups > 1)
            convert(std::true_type{});
          else
            convert(std::false_type{});
          fence_proxy_async_smem();  // generic-proxy writes -> visible to tcgen05.mma
        }
        // Every warp of the group reaches this barrier each of its k-blocks and
        // they leave the loop together (a warp that gave up waiting makes the
        // group give up; the abort flag then stops the other group).  After it
        // every converted row of the buffer is written and fenced for the async
        // proxy; one thread tells the even CTA's MMA warp.  The odd CTA's
        // arrival is relaxed: a cluster-scope release costs about a microsecond
        // per k-block, and the barrier already ordered the writes.
        // (barrier ids 1 and 2 as constants: a computed id reserves all 16)
        ok = grp == 0 ? named_bar_and(1, kConvGroupThreads, got) : named_bar_and(2, kConvGroupThreads, got);
        if (!ok) break;
        if (ct == 0) {
          if (leader)
            mbar_arrive(bfull_bar(bstage));
          else
            mbar_arrive_cluster_relaxed(map_to_cta(bfull_bar(bstage), 0));
        }
      }
    }
    // every release of a converted buffer by the MMA issuer has landed before
    // exit: group 0 waits for the releases of the last uses of every buffer
    if (grp == 0)
      for (int j = max(0, gk - C::kBStages); j < gk && ok; ++j)
        ok = __all_sync(0xffffffffu, wait_bounded(empty_bar((uint32_t)(j % C::kBStages)),
                                                  (uint32_t)(j / C::kBStages) & 1u, abort_flag, p.timeout_ns));
    if (!ok && lane == 0) raise_abort(abort_flag, p.err);
  }

  // Both CTAs are done with each other's shared memory and barriers, and every
  // TMEM read of either epilogue is complete, before TMEM is freed and the CTAs exit.
  tc_fence_before_sync();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace moe
