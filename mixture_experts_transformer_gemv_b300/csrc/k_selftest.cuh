// Self-tests: the library's bounded waits (one thread waits on an mbarrier
// phase that nothing completes and must give up after its time limit, or at
// once when the abort flag is already raised, leaving the GPU context usable),
// and the device GELU of the GeGLU epilogues evaluated on a buffer.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "k_attn.cuh"
#include "ptx.cuh"

namespace moe {

// mode 0: the spinning wait of the GEMM, decode and grouping kernels
// mode 1: the sleeping wait of the attention kernel
// mode 2: the spinning wait with the abort flag raised before it starts (limit_ns large)
// out[0] = 1 if the wait returned true (it must not), out[1] = elapsed ns.
__global__ void selftest_wait_kernel(int mode, uint64_t limit_ns, uint32_t* err, uint64_t* out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_word;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);  // one arrival expected; nobody arrives
  fence_mbar_init();
  abort_word = (mode == 2) ? 1u : 0u;
  volatile uint32_t* abort_flag = &abort_word;
  const uint64_t t0 = global_timer_ns();
  bool got;
  if (mode == 1)
    got = wait_sleep(b, 0, abort_flag, limit_ns);
  else
    got = wait_bounded(b, 0, abort_flag, limit_ns);
  out[1] = global_timer_ns() - t0;
  out[0] = got ? 1u : 0u;
  if (!got) atomicOr(err, kErrTimeout);
}

// The GELU every GeGLU epilogue uses, elementwise: y[i] = gelu_tanh(x[i]).
__global__ void selftest_gelu_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    y[i] = gelu_tanh(x[i]);
}

}  // namespace moe
