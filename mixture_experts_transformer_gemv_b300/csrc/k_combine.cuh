// K5: combine of the two expert rows + post-MoE RMSNorm + residual add.
//
// Per token t ("Grok-1: 314B Total Parameters, 25B Active Per Token (MoE Explained)",
// "How MoE Works in Practice": gate-weighted
// sum of the chosen experts' outputs; "TevunahAi/Grok-1-BF16", "Grok-1 Specific
// Behaviors": post-MoE norm; "Why JAX Instead of PyTorch" block listing:
// x + sublayer output):
//   m   = Y[row(t,0)] + Y[row(t,1)]       (Y rows already hold p * o, fp32;
//                                          the decode path first sums o's split-K parts)
//   out = bf16(x + m / sqrt(mean(m^2) + eps) * s_post)
// One CTA of 256 threads per token; m stays in registers between the two
// passes (d <= 256 * 4 * kCombineVec), 16-byte loads and stores throughout.
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kCombineThreads = 256;  // per token for large T; 1024 for T below the SM count
constexpr int kCombineVec = 16;       // largest float4 count per thread kept in registers: d <= 16384
constexpr int kDecMaxSplitCombine = 8;  // largest split of the decode path's down projection

// kSplit = false: Y rows of the grouped GEMM path, Y[row] = p * o.
// kSplit = true:  decode path, o split over `ksplit` reduction chunks:
//                 part[kc][e][s][:], s = row - row_offset[e]; summed in kc order.
// THREADS per token (256, or 1024 when there are fewer tokens than SMs); VEC =
// ceil(d / (4 THREADS)) float4 of m per thread, sized to d so that registers (and
// so the number of CTAs per SM) follow the row length.
template <bool kSplit, int THREADS, int VEC>
__global__ void __launch_bounds__(THREADS) combine_kernel(
    const float* __restrict__ y_rows, const int32_t* __restrict__ row_of_slot, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ sched, int ksplit, const __nv_bfloat16* x, const float* __restrict__ s_post,
    float eps, int d, int rows_valid_cap, int checks, uint32_t* __restrict__ err, __nv_bfloat16* out) {
  __shared__ float red[THREADS / 32];
  const int t = blockIdx.x;
  int r0 = row_of_slot[2 * t], r1 = row_of_slot[2 * t + 1];
  if (checks && (r0 < 0 || r0 >= rows_valid_cap || r1 < 0 || r1 >= rows_valid_cap)) {
    if (threadIdx.x == 0) atomicOr(err, kErrCheck);
    r0 = r1 = 0;
  }
  const float4* y0;
  const float4* y1;
  size_t kc_stride = 0;  // in float4
  if (kSplit) {
    int e0 = idx[2 * t], e1 = idx[2 * t + 1];
    int s0 = r0 - sched[kNumExperts + e0], s1 = r1 - sched[kNumExperts + e1];
    if (checks && (e0 < 0 || e0 >= kNumExperts || e1 < 0 || e1 >= kNumExperts || s0 < 0 || s0 >= 16 || s1 < 0 ||
                   s1 >= 16)) {
      if (threadIdx.x == 0) atomicOr(err, kErrCheck);
      e0 = e1 = s0 = s1 = 0;
    }
    y0 = reinterpret_cast<const float4*>(y_rows + ((size_t)e0 * 16 + s0) * d);
    y1 = reinterpret_cast<const float4*>(y_rows + ((size_t)e1 * 16 + s1) * d);
    kc_stride = (size_t)kNumExperts * 16 * d / 4;
  } else {
    y0 = reinterpret_cast<const float4*>(y_rows + (size_t)r0 * d);
    y1 = reinterpret_cast<const float4*>(y_rows + (size_t)r1 * d);
  }
  const int nv = d >> 2;
  const uint2* xr = reinterpret_cast<const uint2*>(x + (size_t)t * d);
  float4 m[VEC];
  uint2 xv[VEC];  // the residual row, read before the reduction (and before any aliasing write)
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const int c = threadIdx.x + i * THREADS;
    if (c < nv) {
      xv[i] = xr[c];
      float4 a = y0[c], b = y1[c];
      if (kSplit) {  // unrolled to the largest split: every part's loads in flight at once
#pragma unroll
        for (int kc = 1; kc < kDecMaxSplitCombine; ++kc) {
          if (kc < ksplit) {
            const float4 a2 = y0[kc * kc_stride + c], b2 = y1[kc * kc_stride + c];
            a = make_float4(a.x + a2.x, a.y + a2.y, a.z + a2.z, a.w + a2.w);
            b = make_float4(b.x + b2.x, b.y + b2.y, b.z + b2.z, b.w + b2.w);
          }
        }
      }
      m[i] = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
      ss = fmaf(m[i].x, m[i].x, ss);
      ss = fmaf(m[i].y, m[i].y, ss);
      ss = fmaf(m[i].z, m[i].z, ss);
      ss = fmaf(m[i].w, m[i].w, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < THREADS / 32; ++w) tot += red[w];
  const float rr = 1.0f / sqrtf(tot / (float)d + eps);

  uint2* orow = reinterpret_cast<uint2*>(out + (size_t)t * d);
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const int c = threadIdx.x + i * THREADS;
    if (c < nv) {
      const float4 s = reinterpret_cast<const float4*>(s_post)[c];
      uint2 o;
      o.x = pack_bf16x2(bf16_lo(xv[i].x) + m[i].x * rr * s.x, bf16_hi(xv[i].x) + m[i].y * rr * s.y);
      o.y = pack_bf16x2(bf16_lo(xv[i].y) + m[i].z * rr * s.z, bf16_hi(xv[i].y) + m[i].w * rr * s.w);
      orow[c] = o;
    }
  }
}

// Launch of combine_kernel<kSplit, THREADS, VEC> for a row length d (multiple of
// 128, <= 16384): VEC is the smallest count of float4 per thread that covers d/4.
template <bool kSplit, int THREADS, int VEC = 1>
inline void launch_combine(int T, cudaStream_t st, const float* y_rows, const int32_t* row_of_slot,
                           const int32_t* idx, const int32_t* sched, int ksplit, const __nv_bfloat16* x,
                           const float* s_post, float eps, int d, int rows_valid_cap, int checks, uint32_t* err,
                           __nv_bfloat16* out) {
  if constexpr (VEC * THREADS * 4 < kCombineVec * kCombineThreads * 4) {
    if (d > VEC * THREADS * 4) {
      launch_combine<kSplit, THREADS, VEC + 1>(T, st, y_rows, row_of_slot, idx, sched, ksplit, x, s_post, eps, d,
                                               rows_valid_cap, checks, err, out);
      return;
    }
  }
  combine_kernel<kSplit, THREADS, VEC><<<T, THREADS, 0, st>>>(y_rows, row_of_slot, idx, sched, ksplit, x, s_post,
                                                              eps, d, rows_valid_cap, checks, err, out);
}

}  // namespace moe
