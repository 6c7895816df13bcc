// Self-test of the bounded-wait failure path, without a GPU fault.
//
// Every wait in the library's kernels (on an mbarrier, a counter) is
// bounded: when its deadline passes it records the site in a device error
// word, sets the CTA's abort flag and returns, so the kernel ends and the
// context stays usable; ba_last_device_error() reads and clears the word.
// k_selftest_wait exercises exactly that path: one warp waits, with a short
// deadline, for phase 0 of a freshly initialised mbarrier on which nothing
// ever arrives.  The wait gives up, records kSiteSelfTest, and the kernel
// returns.  Nothing traps, faults or spins without a bound.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ba_common.cuh"
#include "ba_internal.h"

namespace ba {

__global__ void __launch_bounds__(32) k_selftest_wait(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    abort_flag = 0;
  }
  __syncwarp();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, kSiteSelfTest, &abort_flag, limit_ns);
  __syncwarp();
}

cudaError_t run_selftest_wait(uint64_t limit_ns, cudaStream_t st) {
  k_selftest_wait<<<1, 32, 0, st>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t take_selftest_error_word(uint32_t *word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(uint32_t));
}

}  // namespace ba
