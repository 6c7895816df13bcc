// Merge of two attention results over disjoint key sets of the same rows,
// the online-softmax combination the LoSA summary post ("merge and update")
// uses to join cached prefix attention with new results:
//     lse = ln(exp(lse1) + exp(lse2))
//     O   = exp(lse1 - lse) O1 + exp(lse2 - lse) O2
// One thread moves 16 bytes (8 bf16) of a row; HBM-bound.  A part whose LSE
// is -inf (an empty key set) has weight 0; if both are -inf, O = 0 and
// lse = -inf.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ba_internal.h"

namespace ba {

// In place (o may be o1 or o2, lse may be lse1 or lse2): each lane reads and
// writes only its own 16 bytes of O, but lane 0 of a row writes the row's LSE
// that the row's other lanes read, so every lane reads its inputs before the
// warp barrier and writes after it (the VPR lanes of a row lie in one warp).
// No __restrict__ or read-only loads on pointers that may alias.
template <int D>
__global__ void __launch_bounds__(256) k_merge_lse(const __nv_bfloat16 *o1, const float *lse1,
                                                   const __nv_bfloat16 *o2, const float *lse2,
                                                   int64_t rows, __nv_bfloat16 *o, float *lse) {
  constexpr int VPR = D / 8;
  static_assert(32 % VPR == 0, "a row's lanes lie in one warp");
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gid / VPR;
  const int c = static_cast<int>(gid % VPR);
  const bool valid = row < rows;
  float a = -INFINITY, b = -INFINITY;
  uint4 x = make_uint4(0, 0, 0, 0), y = make_uint4(0, 0, 0, 0);
  if (valid) {
    a = lse1[row];
    b = lse2[row];
    x = reinterpret_cast<const uint4 *>(o1 + row * D)[c];
    y = reinterpret_cast<const uint4 *>(o2 + row * D)[c];
  }
  __syncwarp();
  if (!valid) return;
  const float m = fmaxf(a, b);
  float w1 = 0.f, w2 = 0.f, l = -INFINITY;
  if (m != -INFINITY) {
    const float e1 = expf(a - m), e2 = expf(b - m);  // exp(-inf) = 0
    const float s = e1 + e2;
    w1 = e1 / s;
    w2 = e2 / s;
    l = m + logf(s);
  }
  const __nv_bfloat162 *hx = reinterpret_cast<const __nv_bfloat162 *>(&x);
  const __nv_bfloat162 *hy = reinterpret_cast<const __nv_bfloat162 *>(&y);
  uint4 r;
  __nv_bfloat162 *hr = reinterpret_cast<__nv_bfloat162 *>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fx = __bfloat1622float2(hx[i]), fy = __bfloat1622float2(hy[i]);
    // a weight of 0 contributes nothing, whatever the other result holds
    const float r0 = (w1 != 0.f ? w1 * fx.x : 0.f) + (w2 != 0.f ? w2 * fy.x : 0.f);
    const float r1 = (w1 != 0.f ? w1 * fx.y : 0.f) + (w2 != 0.f ? w2 * fy.y : 0.f);
    hr[i] = __floats2bfloat162_rn(r0, r1);
  }
  reinterpret_cast<uint4 *>(o + row * D)[c] = r;
  if (c == 0) lse[row] = l;
}

cudaError_t run_merge_lse(const void *o1, const float *lse1, const void *o2, const float *lse2,
                          int64_t rows, int head_dim, void *o, float *lse, cudaStream_t st) {
  const int64_t threads = rows * (head_dim / 8);
  const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
  if (head_dim == 128)
    k_merge_lse<128><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(o1), lse1,
                                           static_cast<const __nv_bfloat16 *>(o2), lse2, rows,
                                           static_cast<__nv_bfloat16 *>(o), lse);
  else
    k_merge_lse<64><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(o1), lse1,
                                          static_cast<const __nv_bfloat16 *>(o2), lse2, rows,
                                          static_cast<__nv_bfloat16 *>(o), lse);
  return cudaGetLastError();
}

}  // namespace ba
