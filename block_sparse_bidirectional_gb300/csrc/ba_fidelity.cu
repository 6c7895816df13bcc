// Fidelity diagnostics of a block selection, for sm_103a ("Efficient
// Long-Context Modeling in Diffusion Language Models via Block Approximate
// Sparse Attention"):
//   * the oracle block mass of §3.1 Eq. 3,
//       m_hat[gq, gk] = (1 / |I(gq)|) sum_{i in I(gq)} sum_{j in J(gk)} A_ij,
//     with A_ij = exp(scale q_i.k_j - lse_i) the dense attention map of Eq. 1
//     (lse the dense row log-sum-exp) and I, J the sorted blocks;
//   * the largest token-vs-block logit deviation of §3.2 (Eq. 5),
//       dev[gq, gk] = max_{i in I, j in J} |scale q_i.k_j - scale Qbar.Kbar|;
//   * its bound, Eq. 7-8: U = scale (R^Q M^K + M^Q R^K + R^Q R^K), R the
//     block radii and M the block max norms;
//   * the recall of a selected mask: the block mass its kept blocks hold.
//
// Kernels: k_fid_blocks (block means, radii, max norms and the permuted row
// copies), k_fid_logits (scale Qbar.Kbar per block pair), k_fid_mass (a
// tcgen05 pass over every (query tile, key block): S = Q K^T in tensor
// memory, then per row the sum of exp(scale s - lse) and the largest
// |scale s - l| over the block, added / max-ed into the block-pair outputs),
// k_fid_bound_recall (U and the recall).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ba_common.cuh"
#include "ba_internal.h"

namespace ba {

constexpr int kFidThreads = 256;
constexpr int kFidSlots = 4;
constexpr int kFidTile = 128;  // query rows per mass CTA (tensor-memory lanes)

static size_t align256f(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct FidBlocksArgs {
  const __nv_bfloat16 *x[2];     // q, k
  const int32_t *perm[2];        // nullable: identity
  __nv_bfloat16 *xp[2];          // permuted copies
  float *mean[2];                // [bh, N, D]
  float *radius[2];              // [bh, N]
  float *maxnorm[2];             // [bh, N]
  int L, N;
};

// One CTA per (sorted block, bh, tensor): gathers the block's rows through
// pi (and writes them to the permuted copy), then the fp32 mean per feature,
// the radius max_i ||x_i - mean|| and the max norm max_i ||x_i|| (Eq. 7).
template <int D, int BK>
__global__ void __launch_bounds__(kFidThreads) k_fid_blocks(const FidBlocksArgs a) {
  constexpr int VPR = D / 8;  // 16-byte pieces per row
  __shared__ __align__(16) __nv_bfloat16 s_rows[BK * D];
  __shared__ float s_mean[D];
  __shared__ float s_red[2][kFidThreads / 32];
  const int z = blockIdx.z;
  const int g = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int r0 = g * BK;
  const int n = min(BK, a.L - r0);
  const int64_t head = bh * a.L;
  const __nv_bfloat16 *x = a.x[z];
  const int32_t *perm = a.perm[z];
  for (int t = threadIdx.x; t < n * VPR; t += kFidThreads) {
    const int row = t / VPR, c = t % VPR;
    const int pos = r0 + row;
    const int src = perm ? min(max(__ldg(perm + head + pos), 0), a.L - 1) : pos;
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + (head + src) * D) + c);
    reinterpret_cast<uint4 *>(s_rows + row * D)[c] = v;
    reinterpret_cast<uint4 *>(a.xp[z] + (head + pos) * D)[c] = v;
  }
  __syncthreads();
  if (threadIdx.x < D) {
    float acc = 0.f;
    for (int r = 0; r < n; ++r) acc += __bfloat162float(s_rows[r * D + threadIdx.x]);
    const float m = acc / static_cast<float>(n);
    s_mean[threadIdx.x] = m;
    a.mean[z][(bh * a.N + g) * D + threadIdx.x] = m;
  }
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  float md = 0.f, mn = 0.f;
  for (int r = warp; r < n; r += kFidThreads / 32) {
    float dd = 0.f, nn = 0.f;
    for (int c = lane; c < D; c += 32) {
      const float v = __bfloat162float(s_rows[r * D + c]);
      const float e = v - s_mean[c];
      dd = fmaf(e, e, dd);
      nn = fmaf(v, v, nn);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      dd += __shfl_xor_sync(0xffffffffu, dd, off);
      nn += __shfl_xor_sync(0xffffffffu, nn, off);
    }
    md = fmaxf(md, dd);
    mn = fmaxf(mn, nn);
  }
  if (lane == 0) {
    s_red[0][warp] = md;
    s_red[1][warp] = mn;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a0 = 0.f, a1 = 0.f;
    for (int w = 0; w < kFidThreads / 32; ++w) {
      a0 = fmaxf(a0, s_red[0][w]);
      a1 = fmaxf(a1, s_red[1][w]);
    }
    a.radius[z][bh * a.N + g] = sqrtf(a0);
    a.maxnorm[z][bh * a.N + g] = sqrtf(a1);
  }
}

// l[gq, gk] = scale * Qbar_gq . Kbar_gk (Eq. 2 with the call's scale), fp32,
// 16 x 16 outputs per CTA.
template <int D>
__global__ void __launch_bounds__(256) k_fid_logits(const float *__restrict__ mq,
                                                    const float *__restrict__ mk, int N,
                                                    float scale, float *__restrict__ ell) {
  __shared__ float sa[16][33], sb[16][33];
  const int64_t bh = blockIdx.z;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int gq = blockIdx.y * 16 + ty, gk = blockIdx.x * 16 + tx;
  float acc = 0.f;
  for (int t0 = 0; t0 < D; t0 += 32) {
    for (int i = threadIdx.x; i < 16 * 32; i += 256) {
      const int r = i / 32, c = i % 32;
      const int ga = blockIdx.y * 16 + r, gb = blockIdx.x * 16 + r;
      sa[r][c] = ga < N ? mq[(bh * N + ga) * D + t0 + c] : 0.f;
      sb[r][c] = gb < N ? mk[(bh * N + gb) * D + t0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 32; ++c) acc = fmaf(sa[ty][c], sb[tx][c], acc);
    __syncthreads();
  }
  if (gq < N && gk < N) ell[(bh * N + gq) * N + gk] = scale * acc;
}

// 2^x with the hardware approximation (relative error about 2^-22; results
// below 2^-126 flush to zero, far under any block mass that matters).
__device__ __forceinline__ float fid_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr int fid_tmem_cols(int x) {
  int c = 32;
  while (c < x) c <<= 1;
  return c;
}

template <int D, int BK>
struct FidLayout {
  static constexpr int kQBytes = kFidTile * D * 2;
  static constexpr int kSlotBytes = BK * D * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffSlots = kQBytes;
  static constexpr int kOffBar = kOffSlots + kFidSlots * kSlotBytes;
  static constexpr int kBytes = kOffBar + 256;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr int kTmemCols = fid_tmem_cols(2 * BK);
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

struct FidMassParams {
  int L, N;
  const int32_t *perm_q;   // nullable
  const float *lse;        // [bh, L], original order, natural log
  const float *ell;        // [bh, N, N] or null (no deviation)
  float *mass;             // [bh, N, N], zeroed before the launch
  float *dev;              // [bh, N, N] or null, zeroed before the launch
  float scale, scale_log2;
};

// grid = (query tiles of 128 sorted rows, bh).  Warp 0: TMA producer (the Q'
// tile, then every K' block into a 4-slot ring); warp 1: tensor-memory
// allocation and the MMA thread (S_j = Q K_j^T into one of two tensor-memory
// buffers); warps 4-7: thread r owns row r (tensor-memory lane r).  Each
// warp adds its 32 rows' share to the block-pair outputs with one atomic
// per key block (the rows of a warp lie in one query block); no CTA-wide
// barrier inside the loop, so a role that gives up on a bounded wait cannot
// strand the others.
template <int D, int BK>
__global__ void __launch_bounds__(kFidThreads, 1)
    k_fid_mass(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const FidMassParams p) {
  using Lay = FidLayout<D, BK>;
  constexpr int S = kFidSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + Lay::kOffQ;
  uint8_t *sSlot = smem + Lay::kOffSlots;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kOffBar);
  uint64_t *q_full = bars;
  uint64_t *slot_full = bars + 1;
  uint64_t *slot_empty = slot_full + S;
  uint64_t *s_full = slot_empty + S;  // [2]
  uint64_t *s_free = s_full + 2;      // [2]
  uint64_t *drain = s_free + 2;
  uint32_t *misc = reinterpret_cast<uint32_t *>(drain + 1);  // tmem, abort
  volatile int *abort_flag = reinterpret_cast<volatile int *>(&misc[1]);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tile = blockIdx.x;
  const int bh = blockIdx.y;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&slot_full[s], 1);
      mbar_init(&slot_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], kFidTile);
    }
    mbar_init(drain, 1);
    misc[1] = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&misc[0], Lay::kTmemCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const int N = p.N;

  if (warp == 0 && lane == 0) {
    // ===================== TMA producer =====================================
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    mbar_arrive_expect_tx(q_full, Lay::kQBytes);
#pragma unroll
    for (int c = 0; c < D / 64; ++c)
      tma_load_3d(sQ + c * kFidTile * 128, &tmQ, q_full, c * 64, tile * kFidTile, bh);
    int issued = 0;
    for (int j = 0; j < N; ++j) {
      const int s = j % S;
      if (j >= S && !mbar_wait(&slot_empty[s], ((j / S) & 1) ^ 1u, kSiteKEmpty, abort_flag)) break;
      mbar_arrive_expect_tx(&slot_full[s], Lay::kSlotBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(sSlot + s * Lay::kSlotBytes + c * BK * 128, &tmK, &slot_full[s], c * 64, j * BK,
                    bh);
      issued = j + 1;
    }
    mbar_wait_drain(q_full, 0);
    for (int s = 0; s < S && s < issued; ++s) {
      const int last = s + S * ((issued - 1 - s) / S);
      mbar_wait_drain(&slot_full[s], (last / S) & 1);
    }
  } else if (warp == 1 && lane == 0) {
    // ===================== MMA issuer =======================================
    const uint32_t idS = idesc_bf16_f32(kFidTile, BK, 0, 0);
    const uint32_t q_addr = smem_u32(sQ), slot_addr = smem_u32(sSlot);
    bool ok = mbar_wait(q_full, 0, kSiteQFull, abort_flag);
    tc_fence_after();
    for (int j = 0; ok && j < N; ++j) {
      const int s = j % S, b = j & 1;
      if (!(ok = mbar_wait(&slot_full[s], (j / S) & 1, kSiteKFull, abort_flag))) break;
      if (j >= 2 && !(ok = mbar_wait(&s_free[b], ((j >> 1) - 1) & 1, kSitePFull, abort_flag))) break;
      tc_fence_after();
      const uint32_t ka = slot_addr + s * Lay::kSlotBytes;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t da = smem_desc_sw128(q_addr + (ks / 4) * kFidTile * 128 + (ks % 4) * 32, 16, 1024);
        const uint64_t db = smem_desc_sw128(ka + (ks / 4) * BK * 128 + (ks % 4) * 32, 16, 1024);
        mma_bf16_ss(tmem + b * BK, da, db, idS, ks > 0 ? 1u : 0u);
      }
      mma_commit(&s_full[b]);
      mma_commit(&slot_empty[s]);
    }
    mma_commit(drain);
    mbar_wait_drain(drain, 0);
  } else if (warp >= 4) {
    // ===================== rows =============================================
    const int r = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int64_t head = static_cast<int64_t>(bh) * p.L;
    const int row = tile * kFidTile + r;
    const bool valid = row < p.L;
    // the rows of a warp share one query block (32 divides B)
    const int gq = min(row, p.L - 1) / BK;
    const int cnt = min(BK, p.L - gq * BK);
    const float inv_cnt = 1.f / static_cast<float>(cnt);
    int orig = 0;
    if (valid) orig = p.perm_q ? min(max(p.perm_q[head + row], 0), p.L - 1) : row;
    const float lse2 = valid ? p.lse[head + orig] * 1.4426950408889634f : 0.f;
    const float *ell_row = p.ell ? p.ell + (static_cast<int64_t>(bh) * N + gq) * N : nullptr;
    float *mass_row = p.mass + (static_cast<int64_t>(bh) * N + gq) * N;
    float *dev_row = p.dev ? p.dev + (static_cast<int64_t>(bh) * N + gq) * N : nullptr;
    const float cl = p.scale_log2, sc = p.scale;
    bool ok = true;
    for (int j = 0; j < N; ++j) {
      const int b = j & 1;
      ok = mbar_wait(&s_full[b], (j >> 1) & 1, kSiteSFull, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      float sv[BK];
#pragma unroll
      for (int c = 0; c < BK / 32; ++c) tmem_ld32(tmem + lane_base + b * BK + c * 32, sv + c * 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&s_free[b]);
      const int valid_cols = min(BK, p.L - j * BK);
      const float lj = ell_row ? ell_row[j] : 0.f;
      const float nl = -lse2, nlj = -lj;
      float sum, dv;
      if (valid_cols == BK) {
        // every block but a ragged last one: no per-element predicate, four
        // independent partial sums and two max chains
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, d0 = 0.f, d1 = 0.f;
#pragma unroll
        for (int c = 0; c < BK; c += 4) {
          s0 += fid_exp2(fmaf(sv[c], cl, nl));
          s1 += fid_exp2(fmaf(sv[c + 1], cl, nl));
          s2 += fid_exp2(fmaf(sv[c + 2], cl, nl));
          s3 += fid_exp2(fmaf(sv[c + 3], cl, nl));
          d0 = fmaxf(d0, fmaxf(fabsf(fmaf(sv[c], sc, nlj)), fabsf(fmaf(sv[c + 1], sc, nlj))));
          d1 = fmaxf(d1, fmaxf(fabsf(fmaf(sv[c + 2], sc, nlj)), fabsf(fmaf(sv[c + 3], sc, nlj))));
        }
        sum = (s0 + s1) + (s2 + s3);
        dv = fmaxf(d0, d1);
      } else {
        sum = 0.f;
        dv = 0.f;
#pragma unroll
        for (int c = 0; c < BK; ++c) {
          const bool in = c < valid_cols;
          sum += in ? fid_exp2(fmaf(sv[c], cl, nl)) : 0.f;
          dv = fmaxf(dv, in ? fabsf(fmaf(sv[c], sc, nlj)) : 0.f);
        }
      }
      if (!valid) {
        sum = 0.f;
        dv = 0.f;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        sum += __shfl_xor_sync(0xffffffffu, sum, off);
        dv = fmaxf(dv, __shfl_xor_sync(0xffffffffu, dv, off));
      }
      if (lane == 0 && gq * BK < p.L && (warp & 3) * 32 + tile * kFidTile < p.L) {
        atomicAdd(mass_row + j, sum * inv_cnt);
        if (dev_row) atomicMax(reinterpret_cast<int *>(dev_row + j), __float_as_int(dv));
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

// U[gq, gk] (Eq. 8 with the call's scale) and the recall of each row's list.
__global__ void __launch_bounds__(128) k_fid_bound_recall(
    const float *__restrict__ rq, const float *__restrict__ mq, const float *__restrict__ rk,
    const float *__restrict__ mk, const float *__restrict__ mass, const int32_t *__restrict__ idx,
    int N, int kappa, float scale, float *__restrict__ bound, float *__restrict__ recall) {
  __shared__ float s_part[4];
  const int gq = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int64_t row = bh * N + gq;
  if (bound) {
    const float a = rq[row], m = mq[row];
    for (int gk = threadIdx.x; gk < N; gk += blockDim.x) {
      const float b = rk[bh * N + gk], n = mk[bh * N + gk];
      bound[row * N + gk] = scale * (a * n + m * b + a * b);
    }
  }
  if (recall) {
    float acc = 0.f;
    for (int t = threadIdx.x; t < kappa; t += blockDim.x) {
      const int gk = min(max(idx[row * kappa + t], 0), N - 1);
      acc += mass[row * N + gk];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (threadIdx.x % 32 == 0) s_part[threadIdx.x / 32] = acc;
    __syncthreads();
    if (threadIdx.x == 0) recall[row] = s_part[0] + s_part[1] + s_part[2] + s_part[3];
  }
}

struct FidPlan {
  size_t rows, means, vec, ell, total;
};

static FidPlan plan_fid(int64_t bh, int L, int D, int B) {
  FidPlan f;
  const int64_t N = (L + B - 1) / B;
  f.rows = align256f(static_cast<size_t>(bh) * L * D * 2);
  f.means = align256f(static_cast<size_t>(bh) * N * D * sizeof(float));
  f.vec = align256f(static_cast<size_t>(bh) * N * sizeof(float));
  f.ell = align256f(static_cast<size_t>(bh) * N * N * sizeof(float));
  f.total = 2 * f.rows + 2 * f.means + 4 * f.vec + f.ell;
  return f;
}

template <int D, int BK>
static cudaError_t launch_fid_mass(const CUtensorMap &mq, const CUtensorMap &mk, const FidMassParams &p,
                            int64_t bh, cudaStream_t st) {
  using Lay = FidLayout<D, BK>;
  static std::atomic<uint64_t> configured{0};
  const cudaError_t e = once_per_device(configured, [] {
    return cudaFuncSetAttribute(k_fid_mass<D, BK>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kAlloc);
  });
  if (e != cudaSuccess) return e;
  const dim3 grid((p.L + kFidTile - 1) / kFidTile, static_cast<unsigned>(bh));
  k_fid_mass<D, BK><<<grid, kFidThreads, Lay::kAlloc, st>>>(mq, mk, p);
  return cudaGetLastError();
}

template <int D, int BK>
static cudaError_t run_fid_typed(const FidArgs &a, cudaStream_t st) {
  const int64_t bh = static_cast<int64_t>(a.batch) * a.heads;
  const int L = a.seqlen, N = (L + BK - 1) / BK;
  const FidPlan f = plan_fid(bh, L, D, BK);
  unsigned char *ws = static_cast<unsigned char *>(a.workspace);
  __nv_bfloat16 *qp = reinterpret_cast<__nv_bfloat16 *>(ws);
  __nv_bfloat16 *kp = reinterpret_cast<__nv_bfloat16 *>(ws + f.rows);
  float *mean_q = reinterpret_cast<float *>(ws + 2 * f.rows);
  float *mean_k = reinterpret_cast<float *>(ws + 2 * f.rows + f.means);
  unsigned char *v0 = ws + 2 * f.rows + 2 * f.means;
  float *rq = reinterpret_cast<float *>(v0);
  float *mq = reinterpret_cast<float *>(v0 + f.vec);
  float *rk = reinterpret_cast<float *>(v0 + 2 * f.vec);
  float *mk = reinterpret_cast<float *>(v0 + 3 * f.vec);
  float *ell = reinterpret_cast<float *>(v0 + 4 * f.vec);
  const size_t pair_bytes = static_cast<size_t>(bh) * N * N * sizeof(float);
  cudaError_t e;
  if ((e = cudaMemsetAsync(a.mass, 0, pair_bytes, st)) != cudaSuccess) return e;
  if (a.dev_max && (e = cudaMemsetAsync(a.dev_max, 0, pair_bytes, st)) != cudaSuccess) return e;

  FidBlocksArgs ba;
  ba.x[0] = static_cast<const __nv_bfloat16 *>(a.q);
  ba.x[1] = static_cast<const __nv_bfloat16 *>(a.k);
  ba.perm[0] = a.perm_q;
  ba.perm[1] = a.perm_k;
  ba.xp[0] = qp;
  ba.xp[1] = kp;
  ba.mean[0] = mean_q;
  ba.mean[1] = mean_k;
  ba.radius[0] = rq;
  ba.radius[1] = rk;
  ba.maxnorm[0] = mq;
  ba.maxnorm[1] = mk;
  ba.L = L;
  ba.N = N;
  k_fid_blocks<D, BK><<<dim3(N, static_cast<unsigned>(bh), 2), kFidThreads, 0, st>>>(ba);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const float scale = (a.scale > 0.f) ? a.scale : 1.0f / sqrtf(static_cast<float>(D));
  if (a.dev_max) {
    const unsigned gt = static_cast<unsigned>((N + 15) / 16);
    k_fid_logits<D><<<dim3(gt, gt, static_cast<unsigned>(bh)), 256, 0, st>>>(mean_q, mean_k, N,
                                                                              scale, ell);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  alignas(64) CUtensorMap mapq, mapk;
  if ((e = encode_tensor_map_3d(&mapq, qp, D, L, bh, 64, kFidTile)) != cudaSuccess) return e;
  if ((e = encode_tensor_map_3d(&mapk, kp, D, L, bh, 64, BK)) != cudaSuccess) return e;
  FidMassParams p;
  p.L = L;
  p.N = N;
  p.perm_q = a.perm_q;
  p.lse = a.lse;
  p.ell = a.dev_max ? ell : nullptr;
  p.mass = a.mass;
  p.dev = a.dev_max;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  if ((e = launch_fid_mass<D, BK>(mapq, mapk, p, bh, st)) != cudaSuccess) return e;
  if (a.bound || a.recall) {
    k_fid_bound_recall<<<dim3(N, static_cast<unsigned>(bh)), 128, 0, st>>>(
        rq, mq, rk, mk, a.mass, a.block_idx, N, a.kappa, scale, a.bound, a.recall);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

size_t fidelity_workspace_bytes(int64_t bh, int L, int D, int B) { return plan_fid(bh, L, D, B).total; }

cudaError_t run_fidelity(const FidArgs &a, cudaStream_t st) {
  if (a.head_dim == 128 && a.block == 128) return run_fid_typed<128, 128>(a, st);
  if (a.head_dim == 128 && a.block == 64) return run_fid_typed<128, 64>(a, st);
  if (a.head_dim == 64 && a.block == 128) return run_fid_typed<64, 128>(a, st);
  if (a.head_dim == 64 && a.block == 64) return run_fid_typed<64, 64>(a, st);
  return cudaErrorInvalidValue;
}

cudaError_t take_fidelity_error_word(uint32_t *word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(uint32_t));
}

}  // namespace ba
