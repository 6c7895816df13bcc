// Opt-in validation of a selection's outputs before they are used: the
// BA-Att paper's Algorithm 1 steps 1-2 make pi_q and pi_k permutations of
// each sequence, and steps 8-11 keep kappa distinct key blocks per query
// block (the library emits them ascending).  The attention kernels trust
// these inputs (an out-of-range entry is clamped or dropped, never a fault,
// but the result is then meaningless); this call checks them on the device
// and reports what is wrong.
//
//   k_check_perm  one CTA per (b,h) sequence: a shared-memory bitmap of the L
//                 positions; an entry outside [0, L) or a position seen twice
//                 fails (L in-range entries with no repeat form a permutation).
//   k_check_idx   one thread per query-block row: ids in [0, N), strictly
//                 ascending.
// Failures are or-ed into a device word the host reads (and clears) after
// the stream has finished.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/ba.h"
#include "ba_internal.h"

namespace ba {

static __device__ uint32_t g_validate_word = 0;

constexpr int kCheckThreads = 1024;

__global__ void __launch_bounds__(kCheckThreads) k_check_perm(const int32_t *__restrict__ perm, int L,
                                                              uint32_t fail_bit) {
  extern __shared__ uint32_t seen[];
  const int words = (L + 31) / 32;
  for (int i = threadIdx.x; i < words; i += blockDim.x) seen[i] = 0u;
  __syncthreads();
  const int32_t *p = perm + static_cast<int64_t>(blockIdx.x) * L;
  bool bad = false;
  for (int i = threadIdx.x; i < L; i += blockDim.x) {
    const int v = __ldg(p + i);
    if (v < 0 || v >= L) {
      bad = true;
      continue;
    }
    const uint32_t bit = 1u << (v & 31);
    if (atomicOr(&seen[v >> 5], bit) & bit) bad = true;  // this position came twice
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&g_validate_word, fail_bit);
}

__global__ void __launch_bounds__(256) k_check_idx(const int32_t *__restrict__ idx, int64_t rows, int kappa,
                                                   int N, uint32_t fail_bit) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  bool bad = false;
  if (row < rows) {
    const int32_t *r = idx + row * kappa;
    int prev = -1;
    for (int i = 0; i < kappa; ++i) {
      const int v = __ldg(r + i);
      if (v < 0 || v >= N || v <= prev) bad = true;
      prev = v;
    }
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&g_validate_word, fail_bit);
}

cudaError_t run_validate_selection(const int32_t *perm_q, const int32_t *perm_k, const int32_t *block_idx,
                                   int64_t bh, int L, int N, int kappa, uint32_t *word, cudaStream_t st) {
  static std::atomic<uint64_t> configured{0};
  const int smem = ((L + 31) / 32) * 4;
  cudaError_t e = once_per_device(configured, [] {
    // up to 4096 blocks of 128 tokens: a 64 KB bitmap
    return cudaFuncSetAttribute(k_check_perm, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
  });
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  if ((e = cudaMemcpyToSymbolAsync(g_validate_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st)) !=
      cudaSuccess)
    return e;
  if (perm_q) k_check_perm<<<static_cast<unsigned>(bh), kCheckThreads, smem, st>>>(perm_q, L, 1u);
  if (perm_k) k_check_perm<<<static_cast<unsigned>(bh), kCheckThreads, smem, st>>>(perm_k, L, 2u);
  const int64_t rows = bh * N;
  k_check_idx<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, st>>>(block_idx, rows, kappa, N, 4u);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return e;
  return cudaMemcpyFromSymbol(word, g_validate_word, sizeof(uint32_t));
}

}  // namespace ba
