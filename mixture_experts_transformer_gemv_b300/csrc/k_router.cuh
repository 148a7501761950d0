// K1: pre-MoE RMSNorm statistics + router logits + softmax + top-2, fused, one
// read of x.
//
// Per token t ("TevunahAi/Grok-1-BF16" model card, "Grok-1 Specific Behaviors":
// pre-MoE norm; "Grok-1: 314B Total Parameters, 25B Active Per Token (MoE Explained)",
// "Expert Routing Details": softmax of the gate logits, then top_k(k=2) of the
// softmax outputs):
//   r      = 1 / sqrt(mean_j x_j^2 + eps)
//   xn_j   = x_j r s_pre_j                   (the normed row)
//   l_e    = sum_j xn_j G[e, j] + b_e  =  r sum_j x_j (s_pre_j G[e, j]) + b_e
//   p      = softmax(l)                      (max-subtracted, fp32)
//   i0, i1 = two largest p, ties to the lower index; weights p_i0, p_i1
//
// One pass over x takes both sums, fp32: sum_j x_j^2 and the 8 sums
// sum_j x_j gs[e, j] with gs = s_pre (.) G (each product rounded to fp32 once);
// r scales the finished sums.  The kernel writes r (rnorm[t]), not the normed
// row: the row gather forms xn from x, r and s_pre as it copies the rows into
// expert order, so x crosses HBM once here and once there.
//
// Work split: a warp owns a contiguous run of tokens (the grid's warps split T
// evenly) and takes them 4 at a time; lane l owns the 16-byte chunks
// c = l + 32 k of d (8 elements each) and keeps kRouterDepth chunks of all 4
// tokens in flight.  Only the warp reduces (shuffles over its lanes): no block
// barrier after the set-up.  gs lives in shared memory ([8, d] fp32, written
// once per CTA) when it fits (GSMEM); otherwise each use multiplies G and s_pre
// from global memory (L2), with the same products.  Every token's sums run in
// the same order whatever T, the grid or the token's position in the batch
// (chunks in order per lane, then the lanes' xor butterfly), so a token routes
// the same bit for bit in any batch.
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace moe {

// 8 warps per CTA: at T = 8192 on 148 CTAs, 6.9 tokens per warp fill two passes
// of 4 (12 warps measured 15 % slower: 4.6 tokens, the second pass mostly empty)
constexpr int kRouterThreads = 256;
constexpr int kRouterWarps = kRouterThreads / 32;
constexpr int kRouterWTok = 4;   // tokens a warp takes at a time
constexpr int kRouterDepth = 3;  // chunks of x per lane in flight

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

__device__ __forceinline__ void load4(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p + 4));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Outputs per token t: idx_out / prob_out [T, 2] (and the caller's copies when
// given), rnorm_out[t] = r, p_part[t, e] = p_t,e (for the routing diagnostics).
template <bool GSMEM>
__global__ void __launch_bounds__(kRouterThreads, 1) router_kernel(
    const __nv_bfloat16* __restrict__ x, int T, int d, const float* __restrict__ gate,
    const float* __restrict__ gate_bias, const float* __restrict__ s_pre, float eps, float* __restrict__ rnorm_out,
    int32_t* __restrict__ idx_out, float* __restrict__ prob_out, int32_t* __restrict__ user_idx,
    float* __restrict__ user_prob, float* __restrict__ p_part) {
  extern __shared__ __align__(16) uint8_t router_smem[];  // GSMEM: gs [8][d] fp32
  float* gsm = reinterpret_cast<float*>(router_smem);
  constexpr int kThreads = kRouterThreads, kWarps = kRouterWarps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = d >> 3;
  if (GSMEM) {
    // 8 d floats = 2 d float4, kRouterPre of them per thread in flight at once
    constexpr int kRouterPre = 8;
    for (int i0 = threadIdx.x; i0 < 2 * d; i0 += kRouterPre * kThreads) {
      float4 g[kRouterPre], sv[kRouterPre];
#pragma unroll
      for (int u = 0; u < kRouterPre; ++u) {
        const int i = i0 + u * kThreads;
        if (i < 2 * d) {
          g[u] = __ldg(reinterpret_cast<const float4*>(gate) + i);
          sv[u] = __ldg(reinterpret_cast<const float4*>(s_pre + (4 * i) % d));
        }
      }
#pragma unroll
      for (int u = 0; u < kRouterPre; ++u) {
        const int i = i0 + u * kThreads;
        if (i < 2 * d)
          reinterpret_cast<float4*>(gsm)[i] =
              make_float4(sv[u].x * g[u].x, sv[u].y * g[u].y, sv[u].z * g[u].z, sv[u].w * g[u].w);
      }
    }
    __syncthreads();
  }
  const int nwarps = gridDim.x * kWarps;
  const int gw = blockIdx.x * kWarps + warp;
  const int lo = (int)((int64_t)gw * T / nwarps), hi = (int)((int64_t)(gw + 1) * T / nwarps);
  const int nk = (nchunk + 31) / 32;  // chunk steps per lane
  for (int t0 = lo; t0 < hi; t0 += kRouterWTok) {
    const int nt = min(kRouterWTok, hi - t0);
    // chunk k of the 4 tokens (zeros past the run or past d)
    auto load = [&](int k, uint4 (&v)[kRouterWTok]) {
      const int c = lane + 32 * k;
#pragma unroll
      for (int i = 0; i < kRouterWTok; ++i)
        v[i] = (i < nt && c < nchunk) ? ld_nc_v4(x + (size_t)(t0 + i) * d + (size_t)c * 8) : make_uint4(0, 0, 0, 0);
    };
    float ss[kRouterWTok], lg[kRouterWTok][kNumExperts];
#pragma unroll
    for (int i = 0; i < kRouterWTok; ++i) {
      ss[i] = 0.f;
#pragma unroll
      for (int e = 0; e < kNumExperts; ++e) lg[i][e] = 0.f;
    }
    uint4 buf[kRouterDepth][kRouterWTok];
#pragma unroll
    for (int q = 0; q < kRouterDepth; ++q) load(q, buf[q]);
    for (int k0 = 0; k0 < nk; k0 += kRouterDepth) {
#pragma unroll
      for (int q = 0; q < kRouterDepth; ++q) {
        const int c = lane + 32 * (k0 + q);
        if (c < nchunk) {
          float xf[kRouterWTok][8];
#pragma unroll
          for (int i = 0; i < kRouterWTok; ++i) {
            const uint32_t w[4] = {buf[q][i].x, buf[q][i].y, buf[q][i].z, buf[q][i].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              xf[i][2 * h] = bf16_lo(w[h]);
              xf[i][2 * h + 1] = bf16_hi(w[h]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) ss[i] = fmaf(xf[i][j], xf[i][j], ss[i]);
          }
          float s8[8];
          if (!GSMEM) load4(s_pre + (size_t)c * 8, s8);
#pragma unroll
          for (int e = 0; e < kNumExperts; ++e) {
            float g[8];
            if (GSMEM) {
              const float4 a = *reinterpret_cast<const float4*>(gsm + (size_t)e * d + (size_t)c * 8);
              const float4 b = *reinterpret_cast<const float4*>(gsm + (size_t)e * d + (size_t)c * 8 + 4);
              g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
              g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
            } else {
              load4(gate + (size_t)e * d + (size_t)c * 8, g);
#pragma unroll
              for (int j = 0; j < 8; ++j) g[j] = s8[j] * g[j];
            }
            // element-major over the tokens: the 4 tokens' sums advance together
            // (each still takes the elements in order)
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
              for (int i = 0; i < kRouterWTok; ++i) lg[i][e] = fmaf(xf[i][j], g[j], lg[i][e]);
          }
        }
        load(k0 + q + kRouterDepth, buf[q]);
      }
    }
    // the warp's sums (every lane ends with all of them)
#pragma unroll
    for (int i = 0; i < kRouterWTok; ++i) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], o);
#pragma unroll
      for (int e = 0; e < kNumExperts; ++e)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lg[i][e] += __shfl_xor_sync(0xffffffffu, lg[i][e], o);
    }
    // lane i finishes token t0 + i
    float mss = ss[0], ml[kNumExperts];
#pragma unroll
    for (int e = 0; e < kNumExperts; ++e) ml[e] = lg[0][e];
#pragma unroll
    for (int i = 1; i < kRouterWTok; ++i)
      if (lane == i) {
        mss = ss[i];
#pragma unroll
        for (int e = 0; e < kNumExperts; ++e) ml[e] = lg[i][e];
      }
    if (lane < nt) {
      const int t = t0 + lane;
      const float r = 1.0f / sqrtf(mss / (float)d + eps);
      float l[kNumExperts], p[kNumExperts];
#pragma unroll
      for (int e = 0; e < kNumExperts; ++e) l[e] = r * ml[e] + (gate_bias ? gate_bias[e] : 0.f);
      softmax_top2(l, t, idx_out, prob_out, user_idx, user_prob, p);
      rnorm_out[t] = r;
      float4* pp = reinterpret_cast<float4*>(p_part + (size_t)t * kNumExperts);
      pp[0] = make_float4(p[0], p[1], p[2], p[3]);
      pp[1] = make_float4(p[4], p[5], p[6], p[7]);
    }
  }
}

// Small batches (T <= kRouterSmallT, d <= 32 * 8 * kRouterSmallK): each token
// is split over kRouterSlices CTAs, with exactly the arithmetic of
// router_kernel, so a token routes the same to the last bit in any batch.  In
// router_kernel lane l of a warp sums the chunks c = l + 32 k of the token in
// order (sum of squares and the 8 sums x_j (s_pre_j G[e, j])), then the warp's
// xor butterfly adds the 32 lanes' sums.  Here "virtual lane" l is computed by
// one thread of CTA (t, l / 4) over the same chunks in the same order, from
// shared memory that its CTA filled with those chunks' G, s_pre and x (28.5 KB
// instead of the whole 221 KB gate for one token on one SM); the 9 sums of
// every virtual lane go to part[t][l], and the token's last CTA to finish
// (a counter per token, reset by that CTA) loads the 32 sets into the lanes of
// one warp and runs the same butterfly, softmax and top-2.
constexpr int kRouterSmallT = 16;
constexpr int kRouterSlices = 8;                             // CTAs per token
constexpr int kRouterSliceLanes = 32 / kRouterSlices;        // virtual lanes per CTA
constexpr int kRouterSmallK = 24;                            // chunks per virtual lane (d <= 6144)
constexpr int kRouterSplitThreads = kRouterSliceLanes * kRouterSmallK;  // one (lane, chunk) each to stage
constexpr int kRouterPartFloats = 32 * (1 + kNumExperts);    // per token: 32 virtual lanes x 9 sums

__global__ void __launch_bounds__(kRouterSplitThreads) router_split_kernel(
    const __nv_bfloat16* __restrict__ x, int d, const float* __restrict__ gate, const float* __restrict__ gate_bias,
    const float* __restrict__ s_pre, float eps, float* __restrict__ rnorm_out, int32_t* __restrict__ idx_out,
    float* __restrict__ prob_out, int32_t* __restrict__ user_idx, float* __restrict__ user_prob,
    float* __restrict__ p_part, float* __restrict__ part, int32_t* __restrict__ done) {
  __shared__ __align__(16) float gsl[kRouterSliceLanes][kRouterSmallK][kNumExperts][8];
  __shared__ __align__(16) float ssl[kRouterSliceLanes][kRouterSmallK][8];
  __shared__ __align__(16) uint4 xsl[kRouterSliceLanes][kRouterSmallK];
  __shared__ int last;
  const int t = blockIdx.x, slice = blockIdx.y, tid = threadIdx.x;
  const int nchunk = d >> 3;
  {  // stage chunk k of virtual lane v: G (8 experts), s_pre and x
    const int v = tid / kRouterSmallK, k = tid % kRouterSmallK;
    const int c = slice * kRouterSliceLanes + v + 32 * k;
    if (c < nchunk) {
      float4 g[2 * kNumExperts];
#pragma unroll
      for (int e = 0; e < kNumExperts; ++e) {
        g[2 * e] = __ldg(reinterpret_cast<const float4*>(gate + (size_t)e * d + (size_t)c * 8));
        g[2 * e + 1] = __ldg(reinterpret_cast<const float4*>(gate + (size_t)e * d + (size_t)c * 8 + 4));
      }
      const float4 s0 = __ldg(reinterpret_cast<const float4*>(s_pre + (size_t)c * 8));
      const float4 s1 = __ldg(reinterpret_cast<const float4*>(s_pre + (size_t)c * 8 + 4));
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * d) + c);
#pragma unroll
      for (int e = 0; e < kNumExperts; ++e) {
        reinterpret_cast<float4*>(gsl[v][k][e])[0] = g[2 * e];
        reinterpret_cast<float4*>(gsl[v][k][e])[1] = g[2 * e + 1];
      }
      reinterpret_cast<float4*>(ssl[v][k])[0] = s0;
      reinterpret_cast<float4*>(ssl[v][k])[1] = s1;
      xsl[v][k] = xv;
    }
  }
  __syncthreads();
  if (tid < kRouterSliceLanes) {  // virtual lane l: its chunks in order, as a lane of router_kernel
    const int l = slice * kRouterSliceLanes + tid;
    float ss = 0.f, lg[kNumExperts];
#pragma unroll
    for (int e = 0; e < kNumExperts; ++e) lg[e] = 0.f;
    for (int k = 0; k < kRouterSmallK; ++k) {
      if (l + 32 * k >= nchunk) break;
      const uint4 xv = xsl[tid][k];
      const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
      float xf[8];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        xf[2 * h] = bf16_lo(w[h]);
        xf[2 * h + 1] = bf16_hi(w[h]);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(xf[j], xf[j], ss);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float sj = ssl[tid][k][j];
#pragma unroll
        for (int e = 0; e < kNumExperts; ++e) lg[e] = fmaf(xf[j], sj * gsl[tid][k][e][j], lg[e]);
      }
    }
    float* pl = part + (size_t)t * kRouterPartFloats + (size_t)l * (1 + kNumExperts);
    pl[0] = ss;
#pragma unroll
    for (int e = 0; e < kNumExperts; ++e) pl[1 + e] = lg[e];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(done + t, 1) == kRouterSlices - 1;
  __syncthreads();
  if (!last || tid >= 32) return;
  __threadfence();
  // the token's last CTA: virtual lane = lane, then router_kernel's butterfly
  const float* pl = part + (size_t)t * kRouterPartFloats + (size_t)tid * (1 + kNumExperts);
  float ss = __ldcg(pl), lg[kNumExperts];
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e) lg[e] = __ldcg(pl + 1 + e);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
#pragma unroll
  for (int e = 0; e < kNumExperts; ++e)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lg[e] += __shfl_xor_sync(0xffffffffu, lg[e], o);
  if (tid == 0) {
    done[t] = 0;  // for the next forward (stream order)
    const float r = 1.0f / sqrtf(ss / (float)d + eps);
    float l[kNumExperts], p[kNumExperts];
#pragma unroll
    for (int e = 0; e < kNumExperts; ++e) l[e] = r * lg[e] + (gate_bias ? gate_bias[e] : 0.f);
    softmax_top2(l, t, idx_out, prob_out, user_idx, user_prob, p);
    rnorm_out[t] = r;
    float4* pp = reinterpret_cast<float4*>(p_part + (size_t)t * kNumExperts);
    pp[0] = make_float4(p[0], p[1], p[2], p[3]);
    pp[1] = make_float4(p[4], p[5], p[6], p[7]);
  }
}

// Routing diagnostics of the last forward ("Jah-yee/grok" README, list "New
// metrics track MoE-specific grokking signals" and the --demo block "[3] MoE
// routing (layer 0)"):
//   stats[e]  = (1/T) sum_t p_t,e                mean router probability of expert e
//   stats[8]  = -sum_e stats[e] ln stats[e]      routing entropy, nats (max ln 8 = 2.079)
//   stats[9]  = 1 - stats[8] / ln 8              collapse index (0 uniform, 1 one expert)
// One CTA; warp e sums p_part[t, e] over the tokens in a fixed order.
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
