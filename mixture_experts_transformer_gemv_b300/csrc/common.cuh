// Shared constants and small helpers of the MoE layer kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace moe {

constexpr int kNumExperts = 8;   // Grok-1: 8 experts ("Jah-yee/grok" README, architecture diagram)
constexpr int kTopK = 2;         // top-2 routing
constexpr int kRowPad = 128;     // expert row blocks are padded to a multiple of this (half a CTA-pair tile)

// Device error word bits (latched in the handle, read by moe_layer_sync_status).
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrCheck = 2u;
// An int8 layer carries its normed rows and GeGLU activations in fp16; with
// device checks on, a value beyond the fp16 range (|v| > 65504, stored
// saturated or, for a normed row, as infinity) sets this bit.
constexpr uint32_t kErrSaturate = 4u;
constexpr float kF16Max = 65504.f;

// Layout of the small scheduling block K2 writes and the GEMMs read:
//   [0, E)        counts[e]       slots routed to expert e
//   [E, 2E + 1)   row_offset[e]   first permuted row of expert e (multiple of kRowPad);
//                                 row_offset[E] = total padded rows
//   [24, 26)      tile counters of the up and down grouped GEMMs (dynamic tile
//                 schedule), zeroed by K2 before the GEMMs run
constexpr int kSchedInts = 2 * kNumExperts + 1;
constexpr int kSchedTileCtr = 24;
static_assert(kSchedTileCtr >= kSchedInts && kSchedTileCtr + 2 <= 64, "the block is 256 bytes");

// Epilogues of the expert GEMMs: GeGLU of the up projections, or the
// combine-weight scaling of the down projection.
enum : int { kEpiGeglu = 0, kEpiDown = 1 };

// A role of a warp-specialised kernel gave up waiting: tell the CTA's other
// roles (shared abort flag) and the host (device error word).
__device__ __forceinline__ void raise_abort(volatile uint32_t* abort_flag, uint32_t* err) {
  *abort_flag = 1u;
  atomicOr(err, kErrTimeout);
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two bf16 (low, high halves) -> two fp16, round to nearest.
__device__ __forceinline__ uint32_t f16x2_from_bf16x2(uint32_t u) {
  __half2 h = __floats2half2_rn(bf16_lo(u), bf16_hi(u));
  return *reinterpret_cast<uint32_t*>(&h);
}

// Two fp32 -> two fp16 (lo in the low half), round to nearest, saturating to
// +-65504 instead of overflowing to infinity.
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// GELU, tanh approximation: 0.5 u (1 + tanh(z)), z = sqrt(2/pi) (u + 0.044715 u^3).
// Evaluated through the identity 0.5 (1 + tanh z) = 1 / (1 + e^(-2z)) as
// u / (1 + 2^(-2 z log2 e)): one ex2 and one reciprocal on the special-function
// unit instead of a tanh sequence, and no cancellation for negative u, where
// 1 + tanh z is small.  The limits are exact: for z << 0 the power overflows to
// +inf and the result is u * 0 = -0; for z >> 0 it underflows to 0 and the
// result is u.
__device__ __forceinline__ float gelu_tanh(float u) {
  constexpr float kNeg2CLog2e = -2.0f * 0.7978845608028654f * 1.4426950408889634f;  // -2 sqrt(2/pi) log2(e)
  const float t = kNeg2CLog2e * fmaf(0.044715f * u, u * u, u);
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(t));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return u * r;
}

}  // namespace moe
