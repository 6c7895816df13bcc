// LoSA locality pruning and result reuse, for sm_103a (the LoSA summary
// post: step 1 "locality pruning" and the cache update of "merge and
// update").  Between two denoising steps, per group of `group` consecutive
// tokens (the block denoised in parallel), the `top_k` tokens whose query
// vectors changed most -- mean squared error over the d features -- are
// active; the others are stable and keep the attention result (O and its
// log-normaliser) cached from the previous step.  Ties go to the lower token
// index.
//
//   k_active_tokens  one CTA per (group, b*h): per-token MSE (16-byte loads,
//                    a shuffle tree per row), then each token's rank inside
//                    its group from shared memory; active iff rank < top_k.
//   k_reuse_rows     active rows of the cached O / LSE take the new result.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ba_internal.h"

namespace ba {

constexpr int kLosaThreads = 256;

template <int D>
__global__ void __launch_bounds__(kLosaThreads) k_active_tokens(
    const __nv_bfloat16 *__restrict__ qn, const __nv_bfloat16 *__restrict__ qp, int L, int group,
    int top_k, uint8_t *__restrict__ active, float *__restrict__ mse_out) {
  constexpr int TPR = D / 8;                 // threads per row, 16 bytes each
  constexpr int RPP = kLosaThreads / TPR;    // rows per pass
  __shared__ float s_mse[kLosaMaxGroup];
  const int64_t bh = blockIdx.y;
  const int g0 = blockIdx.x * group;
  const int n = min(group, L - g0);
  const int64_t base = bh * L + g0;
  const int part = threadIdx.x % TPR, rsub = threadIdx.x / TPR;
  for (int r0 = 0; r0 < n; r0 += RPP) {
    const int r = r0 + rsub;
    float acc = 0.f;
    if (r < n) {
      const uint4 a = __ldg(reinterpret_cast<const uint4 *>(qn + (base + r) * D) + part);
      const uint4 b = __ldg(reinterpret_cast<const uint4 *>(qp + (base + r) * D) + part);
      const __nv_bfloat162 *ha = reinterpret_cast<const __nv_bfloat162 *>(&a);
      const __nv_bfloat162 *hb = reinterpret_cast<const __nv_bfloat162 *>(&b);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fa = __bfloat1622float2(ha[i]), fb = __bfloat1622float2(hb[i]);
        const float dx = fa.x - fb.x, dy = fa.y - fb.y;
        acc = fmaf(dx, dx, acc);
        acc = fmaf(dy, dy, acc);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (r < n && part == 0) s_mse[r] = acc / static_cast<float>(D);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kLosaThreads) {
    const float mi = s_mse[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const float mj = s_mse[j];
      rank += (mj > mi) || (mj == mi && j < i);
    }
    active[base + i] = rank < top_k ? 1 : 0;
    if (mse_out) mse_out[base + i] = mi;
  }
}

// grid-stride over (row, 16-byte piece); the first piece of a row also
// carries the LSE
template <int D>
__global__ void __launch_bounds__(256) k_reuse_rows(const __nv_bfloat16 *__restrict__ o_new,
                                                    const float *__restrict__ lse_new,
                                                    const uint8_t *__restrict__ active,
                                                    int64_t rows, __nv_bfloat16 *__restrict__ o_cache,
                                                    float *__restrict__ lse_cache) {
  constexpr int VPR = D / 8;
  const int64_t total = rows * VPR;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = t / VPR;
    const int c = static_cast<int>(t % VPR);
    if (!active[row]) continue;
    reinterpret_cast<uint4 *>(o_cache + row * D)[c] =
        __ldg(reinterpret_cast<const uint4 *>(o_new + row * D) + c);
    if (c == 0) lse_cache[row] = lse_new[row];
  }
}

cudaError_t run_active_tokens(const void *q_now, const void *q_prev, int64_t bh, int L, int D,
                              int group, int top_k, uint8_t *active, float *mse, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>((L + group - 1) / group), static_cast<unsigned>(bh));
  const __nv_bfloat16 *a = static_cast<const __nv_bfloat16 *>(q_now);
  const __nv_bfloat16 *b = static_cast<const __nv_bfloat16 *>(q_prev);
  if (D == 128)
    k_active_tokens<128><<<grid, kLosaThreads, 0, st>>>(a, b, L, group, top_k, active, mse);
  else
    k_active_tokens<64><<<grid, kLosaThreads, 0, st>>>(a, b, L, group, top_k, active, mse);
  return cudaGetLastError();
}

cudaError_t run_reuse_rows(const void *o_new, const float *lse_new, const uint8_t *active,
                           int64_t rows, int D, void *o_cache, float *lse_cache, cudaStream_t st) {
  const int64_t pieces = rows * (D / 8);
  const int64_t blocks = (pieces + 255) / 256;
  const unsigned grid = static_cast<unsigned>(blocks < 152 * 16 ? blocks : 152 * 16);
  const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(o_new);
  __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(o_cache);
  if (D == 128)
    k_reuse_rows<128><<<grid, 256, 0, st>>>(src, lse_new, active, rows, dst, lse_cache);
  else
    k_reuse_rows<64><<<grid, 256, 0, st>>>(src, lse_new, active, rows, dst, lse_cache);
  return cudaGetLastError();
}

}  // namespace ba
