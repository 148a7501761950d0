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
#include <type_traits>
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

// The layer's grouping and row gather in one kernel (grid: G CTAs of
// kGroupThreads, any G >= 1).  CTA c owns tokens [c T / G, (c + 1) T / G) (none
// when G > T) and their
// slots s = 2t + r, and computes the same grouping as permute_kernel:
//  1. it counts the experts of all 2T slots (idx is 8 T bytes, read from L2):
//     the totals give counts[e] and row_offset[e], the slots before its own
//     range give where its own slots of each expert start;
//  2. its slots get rows in slot order (per expert: a ballot within each warp,
//     then the warps in order), written to row_of_slot, token_of_row and
//     prob_of_row;
//  3. each of its tokens' hidden rows is read once and its normed row, the
//     fp32 product (x_j r) s_pre_j rounded to bf16 ("TevunahAi/Grok-1-BF16",
//     "Grok-1 Specific Behaviors": the pre-MoE RMSNorm; r = 1 / rms from the
//     router), is written to both of its rows, one warp per token;
//  4. the padding rows (each expert's block up to the next multiple of 128)
//     are zeroed, with token -1 and weight 0, spread over the CTAs.
// CTA 0 writes the schedule block (counts, offsets, the GEMMs' zeroed tile
// counters) and the caller's counts.  With checks != 0 an expert index outside
// [0, 8) counts as expert 0 and a row past rows_cap is not written; each sets
// kErrCheck.  to_f16 != 0 (int8 weights) stores the normed rows as fp16: every
// bf16 value converts exactly unless it is below the fp16 normal range
// (|v| < 2^-14, error under 2^-24) or beyond 65504 (stored as infinity; with
// checks != 0 this sets kErrSaturate).
constexpr int kGroupThreads = 256;

__global__ void __launch_bounds__(kGroupThreads) group_rows_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ prob, int T, const __nv_bfloat16* __restrict__ x,
    const float* __restrict__ rnorm, const float* __restrict__ s_pre, int d, int to_f16,
    int32_t* __restrict__ sched, int32_t* __restrict__ row_of_slot, int32_t* __restrict__ token_of_row,
    float* __restrict__ prob_of_row, __nv_bfloat16* __restrict__ xn_perm, int32_t* __restrict__ user_counts,
    int rows_cap, int checks, uint32_t* __restrict__ err) {
  constexpr int kWarps = kGroupThreads / 32;
  __shared__ int32_t s_tot[kWarps][kNumExperts], s_pre_cnt[kWarps][kNumExperts];
  __shared__ int32_t s_off[kNumExperts + 1], s_base[kNumExperts], s_cnt[kNumExperts];
  __shared__ int32_t s_wsum[kWarps][kNumExperts];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, c = blockIdx.x;
  const int t0 = (int)((int64_t)c * T / G), t1 = (int)((int64_t)(c + 1) * T / G);
  const int S = 2 * T, s0 = 2 * t0, s1 = 2 * t1;
  auto expert_of = [](int e) { return (e < 0 || e >= kNumExperts) ? 0 : e; };

  // ---- 1. counts of all slots and of the slots before this CTA's range
  int tot[kNumExperts], before[kNumExperts];
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e) tot[e] = before[e] = 0;
  {
    bool bad = false;
    auto count = [&](int q, int e) {
      bad |= e < 0 || e >= kNumExperts;
      e = expert_of(e);
#pragma unroll
      for (int k = 0; k < kNumExperts; ++k) {
        tot[k] += (k == e);
        before[k] += (k == e && q < s0);
      }
    };
    // S = 2T is even; 16-byte loads of 4 slots, 4 of them in flight per thread
    const int nv = S >> 2;
#pragma unroll 4
    for (int v = tid; v < nv; v += kGroupThreads) {
      const int4 e4 = __ldg(reinterpret_cast<const int4*>(idx) + v);
      count(4 * v, e4.x);
      count(4 * v + 1, e4.y);
      count(4 * v + 2, e4.z);
      count(4 * v + 3, e4.w);
    }
    if (tid < S - 4 * nv) count(4 * nv + tid, idx[4 * nv + tid]);
    if (checks && bad && c == 0 && err) atomicOr(err, kErrCheck);
  }
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tot[e] += __shfl_xor_sync(0xffffffffu, tot[e], o);
      before[e] += __shfl_xor_sync(0xffffffffu, before[e], o);
    }
    if (lane == 0) {
      s_tot[warp][e] = tot[e];
      s_pre_cnt[warp][e] = before[e];
    }
  }
  __syncthreads();
  if (tid < kNumExperts) {
    int n = 0, m = 0;
    for (int w = 0; w < kWarps; ++w) {
      n += s_tot[w][tid];
      m += s_pre_cnt[w][tid];
    }
    s_cnt[tid] = n;
    s_base[tid] = m;  // this CTA's first slot of expert tid is its m-th
  }
  __syncthreads();
  if (tid == 0) {
    int off = 0;
    for (int e = 0; e < kNumExperts; ++e) {
      s_off[e] = off;
      off += (s_cnt[e] + kRowPad - 1) / kRowPad * kRowPad;
    }
    s_off[kNumExperts] = off;
    if (checks && off > rows_cap && c == 0 && err) atomicOr(err, kErrCheck);
    for (int e = 0; e < kNumExperts; ++e) s_base[e] += s_off[e];
  }
  __syncthreads();
  if (c == 0) {
    if (tid < kNumExperts) {
      sched[tid] = s_cnt[tid];
      if (user_counts) user_counts[tid] = s_cnt[tid];
    }
    if (tid <= kNumExperts) sched[kNumExperts + tid] = s_off[tid];
    if (tid < 2) sched[kSchedTileCtr + tid] = 0;  // the grouped GEMMs' tile counters
  }

  // ---- 2. rows of this CTA's slots, in slot order
  for (int q0 = s0; q0 < s1; q0 += kGroupThreads) {
    const int q = q0 + tid;
    const bool have = q < s1;
    const int e = have ? expert_of(idx[q]) : -1;  // (checks report a bad index in step 1)
    int rank = 0;
#pragma unroll
    for (int k = 0; k < kNumExperts; ++k) {
      const uint32_t m = __ballot_sync(0xffffffffu, e == k);
      if (e == k) rank = __popc(m & ((1u << lane) - 1u));
      if (lane == 0) s_wsum[warp][k] = __popc(m);
    }
    __syncthreads();
    if (have) {
      int row = s_base[e] + rank;
      for (int w = 0; w < warp; ++w) row += s_wsum[w][e];
      if (checks && row >= rows_cap) {
        if (err) atomicOr(err, kErrCheck);
        row_of_slot[q] = 0;
      } else {
        row_of_slot[q] = row;
        token_of_row[row] = q >> 1;
        prob_of_row[row] = prob[q];
      }
    }
    __syncthreads();
    if (tid < kNumExperts) {
      int n = 0;
      for (int w = 0; w < kWarps; ++w) n += s_wsum[w][tid];
      s_base[tid] += n;
    }
    __syncthreads();
  }

  // ---- 3. each token's normed row, written to both of its rows: one warp per
  // token, or, with fewer tokens than warps in the CTA (small batches), every
  // warp a share of each token's chunks (one warp's chunk loads were the
  // latency of the step: 17-20 us at T = 8, 9-10 us shared)
  const int nchunk = d >> 3;
  // one token's row: this lane's chunks c0, c0 + STEP, ... (STEP a compile-time
  // constant, so the loop unrolls and its loads issue together)
  auto row = [&](int t, int c0, auto step_tag) {
    constexpr int STEP = decltype(step_tag)::value;
    const int ra = row_of_slot[2 * t], rb = row_of_slot[2 * t + 1];
    const bool wa = !(checks && ra >= rows_cap), wb = !(checks && rb >= rows_cap);
    const float r = rnorm[t];
    const __nv_bfloat16* src = x + (size_t)t * d;
    bool sat = false;
#pragma unroll 8
    for (int ch = c0; ch < nchunk; ch += STEP) {
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(src) + ch);
      const float4 sa = __ldg(reinterpret_cast<const float4*>(s_pre + (size_t)ch * 8));
      const float4 sb = __ldg(reinterpret_cast<const float4*>(s_pre + (size_t)ch * 8 + 4));
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
          sat |= m > kF16Max;
        }
        v.x = f16x2_from_bf16x2(v.x);
        v.y = f16x2_from_bf16x2(v.y);
        v.z = f16x2_from_bf16x2(v.z);
        v.w = f16x2_from_bf16x2(v.w);
      }
      if (wa) reinterpret_cast<uint4*>(xn_perm + (size_t)ra * d)[ch] = v;
      if (wb) reinterpret_cast<uint4*>(xn_perm + (size_t)rb * d)[ch] = v;
    }
    if (sat && err) atomicOr(err, kErrSaturate);
  };
  if (t1 - t0 < kWarps) {  // few tokens (small batches): every warp a share of each token's chunks
    for (int t = t0; t < t1; ++t) row(t, lane + 32 * warp, std::integral_constant<int, 32 * kWarps>{});
  } else {  // one warp per token
    for (int t = t0 + warp; t < t1; t += kWarps) row(t, lane, std::integral_constant<int, 32>{});
  }

  // ---- 4. padding rows, row p of the padding handled by CTA p % G
  int pbase = 0;  // padding rows of the experts before e
  for (int e = 0; e < kNumExperts; ++e) {
    const int r0 = s_off[e] + s_cnt[e], r1 = min(s_off[e + 1], rows_cap);
    const int np = max(0, r1 - r0);
    // this CTA's padding rows of expert e: global padding index pbase + i with (pbase + i) % G == c
    int i = ((c - pbase) % G + G) % G;
    for (int k = i + warp * G; k < np; k += kWarps * G) {
      const int row = r0 + k;
      for (int ch = lane; ch < nchunk; ch += 32)
        reinterpret_cast<uint4*>(xn_perm + (size_t)row * d)[ch] = make_uint4(0, 0, 0, 0);
      if (lane == 0) {
        token_of_row[row] = -1;
        prob_of_row[row] = 0.f;
      }
    }
    pbase += np;
  }
}

}  // namespace moe
