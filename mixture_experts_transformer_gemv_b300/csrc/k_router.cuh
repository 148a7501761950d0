// K1: pre-MoE RMSNorm + router logits + softmax + top-2, fused.
//
// Per token t ("TevunahAi/Grok-1-BF16" model card, "Grok-1 Specific Behaviors":
// pre-MoE norm; "Grok-1: 314B Total Parameters, 25B Active Per Token (MoE Explained)",
// "Expert Routing Details": softmax of the gate logits, then top_k(k=2) of the
// softmax outputs):
//   r      = 1 / sqrt(mean_j x_j^2 + eps)
//   xn_j   = x_j * r * s_pre_j               (fp32; written out rounded to bf16)
//   l_e    = sum_j xn_j G[e, j] + b_e        (from the fp32 xn, not the bf16 copy)
//   p      = softmax(l)                      (max-subtracted, fp32)
//   i0, i1 = two largest p, ties to the lower index; weights p_i0, p_i1
//
// Two kernels compute this.  For T >= 8 x SMs with a gate that fits shared
// memory (d <= 7136), router_persistent_kernel: one CTA per SM holds the gate
// and walks groups of 4 tokens.  Otherwise router_kernel: one CTA of 256
// threads handles kRouterTok tokens (8 for large T at d <= 7168, fewer for wider
// rows, 1 for small T, where more CTAs hide latency better).
// Its x rows are copied once into shared memory (cp.async, 16 bytes per copy)
// and both passes read them there, so every x byte crosses HBM once.  Every
// gate value the CTA loads feeds all of its tokens (the gate is [8, d] fp32
// and is read from L2 once per CTA, not once per token); the experts are taken
// four (at 8 tokens, two) at a time so the gate values, the normed chunk and the
// 8 x kRouterTok partial logits fit in registers at two CTAs per SM.
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kRouterThreads = 256;
constexpr int kRouterTokMax = 8;             // tokens per CTA for large T
constexpr int kRouterSmemMax = 112 * 1024;   // staged x rows per CTA (two CTAs per SM)

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// softmax + top-2 of one token's 8 logits (gate bias included in l): writes
// the routing outputs of token t and leaves the probabilities in p.
__device__ __forceinline__ void softmax_top2(const float (&l)[kNumExperts], int t, int32_t* __restrict__ idx_out,
                                             float* __restrict__ prob_out, int32_t* __restrict__ user_idx,
                                             float* __restrict__ user_prob, float (&p)[kNumExperts]) {
  float mx = l[0];
#pragma unroll
  for (int e = 1; e < kNumExperts; ++e) mx = fmaxf(mx, l[e]);
  float Z = 0.f;
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e) {
    p[e] = expf(l[e] - mx);
    Z += p[e];
  }
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e) p[e] = p[e] / Z;
  // strict '>' keeps the lower index on ties
  int i0 = 0;
  float b0 = p[0];
#pragma unroll
  for (int e = 1; e < kNumExperts; ++e)
    if (p[e] > b0) {
      b0 = p[e];
      i0 = e;
    }
  int i1 = -1;
  float b1 = -1.f;
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e)
    if (e != i0 && p[e] > b1) {
      b1 = p[e];
      i1 = e;
    }
  idx_out[2 * t] = i0;
  idx_out[2 * t + 1] = i1;
  prob_out[2 * t] = b0;
  prob_out[2 * t + 1] = b1;
  if (user_idx) {
    user_idx[2 * t] = i0;
    user_idx[2 * t + 1] = i1;
  }
  if (user_prob) {
    user_prob[2 * t] = b0;
    user_prob[2 * t + 1] = b1;
  }
}

template <int kRouterTok>
__global__ void __launch_bounds__(kRouterThreads, 2) router_kernel(
    const __nv_bfloat16* __restrict__ x, int T, int d, const float* __restrict__ gate,
    const float* __restrict__ gate_bias, const float* __restrict__ s_pre, float eps,
    __nv_bfloat16* __restrict__ xn_out, int32_t* __restrict__ idx_out, float* __restrict__ prob_out,
    int32_t* __restrict__ user_idx, float* __restrict__ user_prob, float* __restrict__ p_part) {
  extern __shared__ __align__(16) uint8_t router_smem[];  // x rows [kRouterTok][d] bf16
  __shared__ float red[kRouterThreads / 32][kRouterTok * kNumExperts];
  __shared__ float rnorm[kRouterTok];
  __shared__ float s_p[kRouterTok][kNumExperts];
  const int t0 = blockIdx.x * kRouterTok;
  const int ntok = min(kRouterTok, T - t0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = d >> 3;  // 8 bf16 per 16-byte chunk
  const uint32_t xs = smem_addr(router_smem);
  auto xchunk = [&](int i, int c) {
    return *reinterpret_cast<const uint4*>(router_smem + ((size_t)i * d + (size_t)c * 8) * 2);
  };

  // ---- the CTA's x rows into shared memory, one read of HBM
  for (int i = 0; i < ntok; ++i)
    for (int c = threadIdx.x; c < nchunk; c += kRouterThreads)
      cp_async16(xs + (uint32_t)(((size_t)i * d + (size_t)c * 8) * 2), x + (size_t)(t0 + i) * d + c * 8);
  cp_async_wait_all();
  __syncthreads();

  // ---- pass 1: sum of squares per token
  float ss[kRouterTok];
#pragma unroll
  for (int i = 0; i < kRouterTok; ++i) ss[i] = 0.f;
  for (int c = threadIdx.x; c < nchunk; c += kRouterThreads) {
#pragma unroll
    for (int i = 0; i < kRouterTok; ++i) {
      if (i < ntok) {
        const uint4 v = xchunk(i, c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float a = bf16_lo(w[q]), b = bf16_hi(w[q]);
          ss[i] = fmaf(a, a, ss[i]);
          ss[i] = fmaf(b, b, ss[i]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kRouterTok; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], o);
    if (lane == 0) red[warp][i] = ss[i];
  }
  __syncthreads();
  if (threadIdx.x < kRouterTok) {
    float s = 0.f;
    for (int w = 0; w < kRouterThreads / 32; ++w) s += red[w][threadIdx.x];
    rnorm[threadIdx.x] = 1.0f / sqrtf(s / (float)d + eps);
  }
  __syncthreads();
  float r[kRouterTok];
#pragma unroll
  for (int i = 0; i < kRouterTok; ++i) r[i] = rnorm[i];

  // ---- pass 2: xn (bf16 copy out) and the 8 logits of every token, experts
  // in groups of four (two at 8 tokens per CTA); the normed chunk is recomputed
  // from shared memory for every group: the same fp32 products
  constexpr int kEPer = kRouterTok >= 8 ? 2 : 4;
  float lg[kRouterTok][kNumExperts];
#pragma unroll
  for (int i = 0; i < kRouterTok; ++i)
#pragma unroll
    for (int e = 0; e < kNumExperts; ++e) lg[i][e] = 0.f;

  for (int c = threadIdx.x; c < nchunk; c += kRouterThreads) {
    const float4 sa = *reinterpret_cast<const float4*>(s_pre + c * 8);
    const float4 sb = *reinterpret_cast<const float4*>(s_pre + c * 8 + 4);
    const float s8[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
    for (int h = 0; h < kNumExperts / kEPer; ++h) {
      float g[kEPer][8];
#pragma unroll
      for (int e = 0; e < kEPer; ++e) {
        const float4 ga = *reinterpret_cast<const float4*>(gate + (size_t)(kEPer * h + e) * d + c * 8);
        const float4 gb = *reinterpret_cast<const float4*>(gate + (size_t)(kEPer * h + e) * d + c * 8 + 4);
        g[e][0] = ga.x; g[e][1] = ga.y; g[e][2] = ga.z; g[e][3] = ga.w;
        g[e][4] = gb.x; g[e][5] = gb.y; g[e][6] = gb.z; g[e][7] = gb.w;
      }
#pragma unroll
      for (int i = 0; i < kRouterTok; ++i) {
        if (i < ntok) {
          const uint4 v = xchunk(i, c);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          float xn[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            xn[2 * q] = bf16_lo(w[q]) * r[i] * s8[2 * q];
            xn[2 * q + 1] = bf16_hi(w[q]) * r[i] * s8[2 * q + 1];
          }
          if (h == 0) {
            uint4 o;
            o.x = pack_bf16x2(xn[0], xn[1]);
            o.y = pack_bf16x2(xn[2], xn[3]);
            o.z = pack_bf16x2(xn[4], xn[5]);
            o.w = pack_bf16x2(xn[6], xn[7]);
            *reinterpret_cast<uint4*>(xn_out + (size_t)(t0 + i) * d + c * 8) = o;
          }
#pragma unroll
          for (int e = 0; e < kEPer; ++e)
#pragma unroll
            for (int j = 0; j < 8; ++j) lg[i][kEPer * h + e] = fmaf(xn[j], g[e][j], lg[i][kEPer * h + e]);
        }
      }
    }
  }
  // block reduction of the kRouterTok x 8 partial logits
#pragma unroll
  for (int i = 0; i < kRouterTok; ++i)
#pragma unroll
    for (int e = 0; e < kNumExperts; ++e) {
      float v = lg[i][e];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      lg[i][e] = v;
    }
  __syncthreads();  // red[] is reused
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kRouterTok; ++i)
#pragma unroll
      for (int e = 0; e < kNumExperts; ++e) red[warp][i * kNumExperts + e] = lg[i][e];
  }
  __syncthreads();

  // ---- softmax + top-2, one thread per token
  if (threadIdx.x < ntok) {
    const int i = threadIdx.x, t = t0 + i;
    float l[kNumExperts], p[kNumExperts];
#pragma unroll
    for (int e = 0; e < kNumExperts; ++e) {
      float s = 0.f;
      for (int w = 0; w < kRouterThreads / 32; ++w) s += red[w][i * kNumExperts + e];
      l[e] = s + (gate_bias ? gate_bias[e] : 0.f);
    }
    softmax_top2(l, t, idx_out, prob_out, user_idx, user_prob, p);
#pragma unroll
    for (int e = 0; e < kNumExperts; ++e) s_p[i][e] = p[e];
  } else if (threadIdx.x < kRouterTok) {
#pragma unroll
    for (int e = 0; e < kNumExperts; ++e) s_p[threadIdx.x][e] = 0.f;
  }
  // this CTA's sum of the router probabilities, per expert, in token order
  // (the routing diagnostics reduce these partial sums in block order)
  __syncthreads();
  if (threadIdx.x < kNumExperts) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kRouterTok; ++i) s += s_p[i][threadIdx.x];
    p_part[blockIdx.x * kNumExperts + threadIdx.x] = s;
  }
}

// Persistent router for large T: one CTA per SM copies the gate [8, d] fp32 into
// shared memory once and walks groups of kRouterPTok tokens (group g =
// blockIdx.x, blockIdx.x + gridDim.x, ...), each token's x chunks read once
// into registers.  A thread owns the same 16-byte chunks of d (c = tid + 256 k)
// for every token, and every sum runs in the same order as in router_kernel
// (over the thread's chunks, then the lanes of the warp, then the warps), so
// xn, the logits and the routing are the same bit for bit; only the gate no
// longer streams from L2 once per CTA of 8 tokens, and the next group's rows
// are loaded while the current group is computed.
constexpr int kRouterPTok = 4;

template <int CH>  // 16-byte chunks of d per thread: d <= 2048 CH
__global__ void __launch_bounds__(kRouterThreads, 1) router_persistent_kernel(
    const __nv_bfloat16* __restrict__ x, int T, int d, const float* __restrict__ gate,
    const float* __restrict__ gate_bias, const float* __restrict__ s_pre, float eps,
    __nv_bfloat16* __restrict__ xn_out, int32_t* __restrict__ idx_out, float* __restrict__ prob_out,
    int32_t* __restrict__ user_idx, float* __restrict__ user_prob, float* __restrict__ p_part) {
  extern __shared__ __align__(16) uint8_t router_smem[];  // gate [8][d] fp32
  __shared__ float red[kRouterThreads / 32][kRouterPTok * kNumExperts];
  __shared__ float rnorm[kRouterPTok];
  __shared__ float s_p[kRouterPTok][kNumExperts];
  const float* gsm = reinterpret_cast<const float*>(router_smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = d >> 3;
  for (int i = threadIdx.x; i < 2 * d; i += kRouterThreads)  // 8 d floats = 2 d chunks of 16 bytes
    cp_async16(smem_addr(router_smem) + (uint32_t)i * 16u, gate + (size_t)i * 4);
  cp_async_wait_all();
  __syncthreads();

  const int ngroups = (T + kRouterPTok - 1) / kRouterPTok;
  // this thread's x chunks of group g (zeros past T or d)
  auto load_group = [&](int g, uint4 (&v)[kRouterPTok][CH]) {
    const int nt = min(kRouterPTok, T - g * kRouterPTok);
#pragma unroll
    for (int i = 0; i < kRouterPTok; ++i)
#pragma unroll
      for (int k = 0; k < CH; ++k) {
        const int c = threadIdx.x + k * kRouterThreads;
        v[i][k] = (i < nt && c < nchunk) ? ld_nc_v4(x + (size_t)(g * kRouterPTok + i) * d + c * 8)
                                         : make_uint4(0, 0, 0, 0);
      }
  };
  // the next group's rows are loaded while this group is computed
  uint4 xnext[kRouterPTok][CH];
  if (blockIdx.x < ngroups) load_group(blockIdx.x, xnext);
  for (int grp = blockIdx.x; grp < ngroups; grp += gridDim.x) {
    const int t0 = grp * kRouterPTok;
    const int ntok = min(kRouterPTok, T - t0);
    uint4 xv[kRouterPTok][CH];
#pragma unroll
    for (int i = 0; i < kRouterPTok; ++i)
#pragma unroll
      for (int k = 0; k < CH; ++k) xv[i][k] = xnext[i][k];
    if (grp + (int)gridDim.x < ngroups) load_group(grp + gridDim.x, xnext);
    // ---- sum of squares per token
    float ss[kRouterPTok];
#pragma unroll
    for (int i = 0; i < kRouterPTok; ++i) ss[i] = 0.f;
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      if (threadIdx.x + k * kRouterThreads < nchunk) {
#pragma unroll
        for (int i = 0; i < kRouterPTok; ++i) {
          if (i < ntok) {
            const uint32_t w[4] = {xv[i][k].x, xv[i][k].y, xv[i][k].z, xv[i][k].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float a = bf16_lo(w[q]), b = bf16_hi(w[q]);
              ss[i] = fmaf(a, a, ss[i]);
              ss[i] = fmaf(b, b, ss[i]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kRouterPTok; ++i) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], o);
      if (lane == 0) red[warp][i] = ss[i];
    }
    __syncthreads();
    if (threadIdx.x < kRouterPTok) {
      float sum = 0.f;
      for (int w = 0; w < kRouterThreads / 32; ++w) sum += red[w][threadIdx.x];
      rnorm[threadIdx.x] = 1.0f / sqrtf(sum / (float)d + eps);
    }
    __syncthreads();
    float r[kRouterPTok];
#pragma unroll
    for (int i = 0; i < kRouterPTok; ++i) r[i] = rnorm[i];

    // ---- xn (bf16 copy out) and the 8 logits of every token
    float lg[kRouterPTok][kNumExperts];
#pragma unroll
    for (int i = 0; i < kRouterPTok; ++i)
#pragma unroll
      for (int e = 0; e < kNumExperts; ++e) lg[i][e] = 0.f;
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int c = threadIdx.x + k * kRouterThreads;
      if (c < nchunk) {
        const float4 sa = *reinterpret_cast<const float4*>(s_pre + c * 8);
        const float4 sb = *reinterpret_cast<const float4*>(s_pre + c * 8 + 4);
        const float s8[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
        float xn[kRouterPTok][8];
#pragma unroll
        for (int i = 0; i < kRouterPTok; ++i) {
          const uint32_t w[4] = {xv[i][k].x, xv[i][k].y, xv[i][k].z, xv[i][k].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            xn[i][2 * q] = bf16_lo(w[q]) * r[i] * s8[2 * q];
            xn[i][2 * q + 1] = bf16_hi(w[q]) * r[i] * s8[2 * q + 1];
          }
          if (i < ntok) {
            uint4 o;
            o.x = pack_bf16x2(xn[i][0], xn[i][1]);
            o.y = pack_bf16x2(xn[i][2], xn[i][3]);
            o.z = pack_bf16x2(xn[i][4], xn[i][5]);
            o.w = pack_bf16x2(xn[i][6], xn[i][7]);
            *reinterpret_cast<uint4*>(xn_out + (size_t)(t0 + i) * d + c * 8) = o;
          }
        }
#pragma unroll
        for (int e = 0; e < kNumExperts; ++e) {
          const float4 ga = *reinterpret_cast<const float4*>(gsm + (size_t)e * d + c * 8);
          const float4 gb = *reinterpret_cast<const float4*>(gsm + (size_t)e * d + c * 8 + 4);
          const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
          for (int i = 0; i < kRouterPTok; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) lg[i][e] = fmaf(xn[i][j], g[j], lg[i][e]);
        }
      }
    }
    // ---- block reduction of the partial logits, then softmax + top-2 per token
#pragma unroll
    for (int i = 0; i < kRouterPTok; ++i)
#pragma unroll
      for (int e = 0; e < kNumExperts; ++e) {
        float v = lg[i][e];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        lg[i][e] = v;
      }
    __syncthreads();  // red[] is reused
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < kRouterPTok; ++i)
#pragma unroll
        for (int e = 0; e < kNumExperts; ++e) red[warp][i * kNumExperts + e] = lg[i][e];
    }
    __syncthreads();
    if (threadIdx.x < ntok) {
      const int i = threadIdx.x;
      float l[kNumExperts], pr[kNumExperts];
#pragma unroll
      for (int e = 0; e < kNumExperts; ++e) {
        float sum = 0.f;
        for (int w = 0; w < kRouterThreads / 32; ++w) sum += red[w][i * kNumExperts + e];
        l[e] = sum + (gate_bias ? gate_bias[e] : 0.f);
      }
      softmax_top2(l, t0 + i, idx_out, prob_out, user_idx, user_prob, pr);
#pragma unroll
      for (int e = 0; e < kNumExperts; ++e) s_p[i][e] = pr[e];
    } else if (threadIdx.x < kRouterPTok) {
#pragma unroll
      for (int e = 0; e < kNumExperts; ++e) s_p[threadIdx.x][e] = 0.f;
    }
    // this group's sum of the router probabilities, per expert, in token order
    __syncthreads();
    if (threadIdx.x < kNumExperts) {
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < kRouterPTok; ++i) sum += s_p[i][threadIdx.x];
      p_part[grp * kNumExperts + threadIdx.x] = sum;
    }
  }
}

// Routing diagnostics of the last forward ("Jah-yee/grok" README, list "New
// metrics track MoE-specific grokking signals" and the --demo block "[3] MoE
// routing (layer 0)"):
//   stats[e]  = (1/T) sum_t p_t,e                mean router probability of expert e
//   stats[8]  = -sum_e stats[e] ln stats[e]      routing entropy, nats (max ln 8 = 2.079)
//   stats[9]  = 1 - stats[8] / ln 8              collapse index (0 uniform, 1 one expert)
// One CTA; warp e sums the per-CTA partial sums of expert e in a fixed order.
__global__ void __launch_bounds__(32 * kNumExperts) router_stats_kernel(const float* __restrict__ p_part,
                                                                       int n_part, int T, float* __restrict__ stats) {
  __shared__ float mean[kNumExperts];
  const int e = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float s = 0.f;
  for (int b = lane; b < n_part; b += 32) s += p_part[b * kNumExperts + e];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) mean[e] = s / (float)T;
  __syncthreads();
  if (threadIdx.x == 0) {
    float h = 0.f;
#pragma unroll
    for (int q = 0; q < kNumExperts; ++q) {
      stats[q] = mean[q];
      if (mean[q] > 0.f) h -= mean[q] * logf(mean[q]);
    }
    stats[kNumExperts] = h;
    stats[kNumExperts + 1] = 1.0f - h / logf((float)kNumExperts);
  }
}

}  // namespace moe
