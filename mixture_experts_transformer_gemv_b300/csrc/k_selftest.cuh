// Self-test of the library's bounded waits: one thread waits on an mbarrier
// phase that nothing completes and must give up after its time limit (or at
// once when the abort flag is already raised), leaving the GPU context usable.
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

}  // namespace moe
