// K2: per-expert grouping of the 2T (token, rank) slots, and the row gather.
//
// The sources route every token to two experts and sum the experts' outputs
// ("Grok-1: 314B Total Parameters, 25B Active Per Token (MoE Explained)",
// "How MoE Works in Practice"); they do not say how the
// work is grouped.  Here the slots are grouped so each expert's rows are
// contiguous and its expert FFN becomes a dense GEMM:
//   counts[e]      = #slots with expert e
//   row_offset[e]  = sum_{e' < e} ceil(counts[e'] / 128) * 128   (tiles never mix experts)
//   rows of expert e, in slot order s = 2t + r (stable: token, then rank);
//   padding rows (up to the next multiple of 128) get token -1 and weight 0.
// With checks != 0 an expert index outside [0, 8) is counted as expert 0 and a
// row past rows_cap is not written; each case also sets kErrCheck in *err
// unless err is null.
// A single CTA does the scan (it is a few microseconds even at T = 65536);
// the gather, which forms the normed rows and puts them in expert order, runs
// on all SMs.
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kPermuteThreads = 1024;

__global__ void __launch_bounds__(kPermuteThreads) permute_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ prob, int T, int32_t* __restrict__ sched,
    int32_t* __restrict__ row_of_slot, int32_t* __restrict__ token_of_row, float* __restrict__ prob_of_row,
    int32_t* __restrict__ user_counts, int rows_cap, int checks, uint32_t* __restrict__ err) {
  __shared__ int32_t warp_tot[kPermuteThreads / 32][kNumExperts];
  __shared__ int32_t s_counts[kNumExperts];
  __shared__ int32_t s_off[kNumExperts + 1];
  const int S = 2 * T;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (S + kPermuteThreads - 1) / kPermuteThreads;
  const int s0 = min(S, tid * per), s1 = min(S, s0 + per);

  int cnt[kNumExperts];
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e) cnt[e] = 0;
  for (int s = s0; s < s1; ++s) {
    int e = idx[s];
    if (checks && (e < 0 || e >= kNumExperts)) {
      if (err) atomicOr(err, kErrCheck);
      e = 0;
    }
#pragma unroll
    for (int q = 0; q < kNumExperts; ++q) cnt[q] += (q == e);
  }
  // exclusive scan over threads, per expert: warp scan then scan of warp totals
  int excl[kNumExperts];
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e) {
    int v = cnt[e];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    excl[e] = v - cnt[e];
    if (lane == 31) warp_tot[warp][e] = v;
  }
  __syncthreads();
  if (tid < kNumExperts) {
    int run = 0;
    for (int w = 0; w < kPermuteThreads / 32; ++w) {
      int v = warp_tot[w][tid];
      warp_tot[w][tid] = run;
      run += v;
    }
    s_counts[tid] = run;
  }
  __syncthreads();
  if (tid == 0) {
    int off = 0;
    for (int e = 0; e < kNumExperts; ++e) {
      s_off[e] = off;
      off += (s_counts[e] + kRowPad - 1) / kRowPad * kRowPad;
    }
    s_off[kNumExperts] = off;
    if (checks && off > rows_cap) if (err) atomicOr(err, kErrCheck);
  }
  __syncthreads();
  int pos[kNumExperts];
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e) pos[e] = s_off[e] + warp_tot[warp][e] + excl[e];
  for (int s = s0; s < s1; ++s) {
    int e = idx[s];
    if (checks && (e < 0 || e >= kNumExperts)) e = 0;
    int row = 0;
#pragma unroll
    for (int q = 0; q < kNumExperts; ++q)
      if (q == e) row = pos[q]++;
    if (checks && row >= rows_cap) {
      if (err) atomicOr(err, kErrCheck);
      row_of_slot[s] = 0;
      continue;
    }
    row_of_slot[s] = row;
    token_of_row[row] = s >> 1;
    prob_of_row[row] = prob[s];
  }
  // padding rows of every expert block
  for (int e = 0; e < kNumExperts; ++e) {
    const int r0 = s_off[e] + s_counts[e], r1 = min(s_off[e + 1], rows_cap);
    for (int row = r0 + tid; row < r1; row += kPermuteThreads) {
      token_of_row[row] = -1;
      prob_of_row[row] = 0.f;
    }
  }
  if (tid < kNumExperts) {
    sched[tid] = s_counts[tid];
    if (user_counts) user_counts[tid] = s_counts[tid];
  }
  if (tid <= kNumExperts) sched[kNumExperts + tid] = s_off[tid];
  if (tid < 2) sched[kSchedTileCtr + tid] = 0;  // the grouped GEMMs' tile counters
}

// xn_perm[row] = xn of token token_of_row[row], formed here from the hidden
// row x, the token's r = 1 / rms (written by the router) and s_pre: the fp32
// product (x_j r) s_pre_j rounded to bf16 ("TevunahAi/Grok-1-BF16", "Grok-1
// Specific Behaviors": the pre-MoE RMSNorm); zeros for padding rows.  Rows
// beyond row_offset[E] are left alone.  Grid-stride over rows, 16-byte
// accesses.  to_f16 != 0 (int8 weights) stores the rows as fp16 instead of
// bf16: every bf16 value converts exactly unless it is below the fp16 normal
// range (|v| < 2^-14), where the error is under 2^-24, or beyond its largest
// value (|v| > 65504, stored as infinity; with checks != 0 this sets
// kErrSaturate in *err).
__global__ void __launch_bounds__(256) gather_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const float* __restrict__ rnorm,
                                                          const float* __restrict__ s_pre,
                                                          const int32_t* __restrict__ token_of_row,
                                                          const int32_t* __restrict__ sched, int d, int to_f16,
                                                          __nv_bfloat16* __restrict__ xn_perm, int checks,
                                                          uint32_t* __restrict__ err) {
  const int rows = sched[2 * kNumExperts];
  const int nchunk = d >> 3;
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const int tok = token_of_row[row];
    uint4* dst = reinterpret_cast<uint4*>(xn_perm + (size_t)row * d);
    if (tok >= 0) {
      const float r = rnorm[tok];
      const __nv_bfloat16* src = x + (size_t)tok * d;
      for (int c = threadIdx.x; c < nchunk; c += blockDim.x) {
        const uint4 xv = ld_nc_v4(src + (size_t)c * 8);
        const float4 sa = __ldg(reinterpret_cast<const float4*>(s_pre + (size_t)c * 8));
        const float4 sb = __ldg(reinterpret_cast<const float4*>(s_pre + (size_t)c * 8 + 4));
        uint4 v;
        v.x = pack_bf16x2(bf16_lo(xv.x) * r * sa.x, bf16_hi(xv.x) * r * sa.y);
        v.y = pack_bf16x2(bf16_lo(xv.y) * r * sa.z, bf16_hi(xv.y) * r * sa.w);
        v.z = pack_bf16x2(bf16_lo(xv.z) * r * sb.x, bf16_hi(xv.z) * r * sb.y);
        v.w = pack_bf16x2(bf16_lo(xv.w) * r * sb.z, bf16_hi(xv.w) * r * sb.w);
        if (to_f16) {
          if (checks) {
            const float m = fmaxf(fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))),
                                        fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)))),
                                  fmaxf(fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))),
                                        fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w)))));
            if (m > kF16Max) atomicOr(err, kErrSaturate);
          }
          v.x = f16x2_from_bf16x2(v.x);
          v.y = f16x2_from_bf16x2(v.y);
          v.z = f16x2_from_bf16x2(v.z);
          v.w = f16x2_from_bf16x2(v.w);
        }
        dst[c] = v;
      }
    } else {
      for (int c = threadIdx.x; c < nchunk; c += blockDim.x) dst[c] = make_uint4(0, 0, 0, 0);
    }
  }
}

}  // namespace moe
