// Selection stage of BA-Att ("Efficient Long-Context Modeling in Diffusion
// Language Models via Block Approximate Sparse Attention", Algorithm 1
// steps 1-11) for sm_103a.
//
//   k_sqnorm_keys   Eq. 9: fp32 squared norm of every Q / K row, packed with
//                   the token index into a 64-bit sort key.  One streaming
//                   pass over Q and K (16-byte vector loads, coalesced).
//   k_chunk_sort    Eq. 10: bitonic sort of 4096-key chunks in shared memory.
//   k_merge_pass    merge-path merge of sorted runs (width doubles per pass);
//                   the last pass emits pi (sorted position -> token index).
//                   Keys are unique (index in the low word), so the result is
//                   the stable sort.
//   k_block_stats   Algorithm 1 step 4: gathers the rows of one sorted block
//                   through pi into shared memory; fp32 mean and population
//                   variance per feature; writes the augmented vectors
//                     a = [Qbar/sqrt(d), beta/d*VarQ, beta/d*Qbar^2]
//                     b = [Kbar, Kbar^2 + VarK, VarK]
//                   so that a.b = Eq. 2 + beta * Eq. 14 (Eq. 13).
//   k_scores        l'[gq,gk] = a_gq . b_gk: a batched fp32 SIMT GEMM
//                   (64x64 tiles, 4x4 register micro-tiles).  Kept on the
//                   fp32 ALUs so the top-kappa decision is taken in fp32.
//   k_topk          steps 8-11: one warp per query-block row; MSB-first radix
//                   select of the kappa-th largest score on order-preserving
//                   integer keys (warp reductions), ties to the lower block
//                   index; emits the ascending index list and the bitmask.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ba_common.cuh"
#include "ba_internal.h"

namespace ba {

constexpr int kChunk = 4096;          // keys sorted per CTA in shared memory
constexpr int kChunkThreads = 1024;
constexpr int kMergeThreads = 256;
constexpr int kMergeItems = 8;        // outputs per merge thread
constexpr int kStatsThreads = 256;
constexpr int kTopkWarps = 4;

// ---------------------------------------------------------------------------
// step 1-2a: squared norms -> sort keys
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) k_sqnorm_keys(const __nv_bfloat16 *__restrict__ x,
                                                     uint64_t *__restrict__ keys, int64_t rows,
                                                     int L) {
  constexpr int TPR = D / 8;  // threads per row, 8 bf16 (16 B) each
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gtid / TPR;
  const int part = static_cast<int>(gtid % TPR);
  float acc = 0.f;
  if (row < rows) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(x + row * D) + part);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      acc = fmaf(f.x, f.x, acc);
      acc = fmaf(f.y, f.y, acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) {
    const uint32_t tok = static_cast<uint32_t>(row % L);
    keys[row] = (static_cast<uint64_t>(__float_as_uint(acc)) << 32) | tok;
  }
}

// ---------------------------------------------------------------------------
// step 1-2b: chunk sort.  grid = (chunks per window, windows, sequences)
// ---------------------------------------------------------------------------
struct SortGeom {
  int L;        // tokens per sequence
  int win;      // window length (== L for a whole-sequence sort)
  int nwin;     // windows per sequence
};

__device__ __forceinline__ int window_len(const SortGeom &g, int w) {
  const int start = w * g.win;
  return min(g.win, g.L - start);
}

__global__ void __launch_bounds__(kChunkThreads) k_chunk_sort(const uint64_t *__restrict__ keys_in,
                                                              uint64_t *__restrict__ keys_out,
                                                              int32_t *__restrict__ perm_out,
                                                              SortGeom g, int final_pass) {
  __shared__ uint64_t s[kChunk];
  const int w = blockIdx.y;
  const int seq = blockIdx.z;
  const int wlen = window_len(g, w);
  const int c0 = blockIdx.x * kChunk;
  if (c0 >= wlen) return;  // uniform over the CTA
  const int n = min(kChunk, wlen - c0);
  const int64_t base = static_cast<int64_t>(seq) * g.L + static_cast<int64_t>(w) * g.win + c0;
  for (int i = threadIdx.x; i < kChunk; i += kChunkThreads)
    s[i] = (i < n) ? keys_in[base + i] : ~0ull;
  __syncthreads();
  for (int k = 2; k <= kChunk; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int p = threadIdx.x; p < kChunk / 2; p += kChunkThreads) {
        const int i = 2 * j * (p / j) + (p % j);
        const int q = i + j;
        const bool up = (i & k) == 0;
        const uint64_t a = s[i], b = s[q];
        if ((a > b) == up) {
          s[i] = b;
          s[q] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n; i += kChunkThreads) {
    if (final_pass)
      perm_out[base + i] = static_cast<int32_t>(s[i] & 0xffffffffu);
    else
      keys_out[base + i] = s[i];
  }
}

// ---------------------------------------------------------------------------
// step 1-2c: merge pass.  Runs of `width` inside each window are merged in
// pairs.  grid = (ceil(win / (threads*items)), windows, sequences)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kMergeThreads) k_merge_pass(const uint64_t *__restrict__ in,
                                                              uint64_t *__restrict__ out,
                                                              int32_t *__restrict__ perm_out,
                                                              SortGeom g, int width,
                                                              int final_pass) {
  const int w = blockIdx.y;
  const int seq = blockIdx.z;
  const int wlen = window_len(g, w);
  const int o0 = (blockIdx.x * kMergeThreads + threadIdx.x) * kMergeItems;
  if (o0 >= wlen) return;
  const int64_t base = static_cast<int64_t>(seq) * g.L + static_cast<int64_t>(w) * g.win;
  const int pair = o0 / (2 * width);
  const int p0 = pair * 2 * width;
  const int a0 = p0, a1 = min(p0 + width, wlen);
  const int b0 = a1, b1 = min(p0 + 2 * width, wlen);
  const int la = a1 - a0, lb = b1 - b0;
  const uint64_t *A = in + base + a0;
  const uint64_t *B = in + base + b0;
  const int diag = o0 - p0;
  int lo = max(0, diag - lb), hi = min(diag, la);
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (A[mid] < B[diag - 1 - mid])
      lo = mid + 1;
    else
      hi = mid;
  }
  int i = lo, j = diag - lo;
  const int n = min(kMergeItems, (la + lb) - diag);
  for (int t = 0; t < n; ++t) {
    uint64_t v;
    if (i < la && (j >= lb || A[i] < B[j]))
      v = A[i++];
    else
      v = B[j++];
    const int64_t dst = base + o0 + t;
    if (final_pass)
      perm_out[dst] = static_cast<int32_t>(v & 0xffffffffu);
    else
      out[dst] = v;
  }
}

__global__ void k_iota(int32_t *__restrict__ perm, int64_t total, int L) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < total) perm[i] = static_cast<int32_t>(i % L);
}

// ---------------------------------------------------------------------------
// step 3-4: block statistics -> augmented vectors.  grid = (N, b*h)
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kStatsThreads) k_block_stats(
    const __nv_bfloat16 *__restrict__ x, const int32_t *__restrict__ perm, int L, int B, int N,
    float *__restrict__ aug, int query_side, float beta) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16 *rows = reinterpret_cast<__nv_bfloat16 *>(smem_raw);          // [B][D]
  float *red = reinterpret_cast<float *>(smem_raw + static_cast<size_t>(B) * D * 2);  // [P][D]
  __shared__ float s_mean[D];

  constexpr int P = kStatsThreads / D;
  const int g = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int r0 = g * B;
  const int n = min(B, L - r0);
  const __nv_bfloat16 *xs = x + bh * static_cast<int64_t>(L) * D;
  const int32_t *ps = perm + bh * static_cast<int64_t>(L) + r0;

  constexpr int VPR = D / 8;  // 16-byte vectors per row
  for (int idx = threadIdx.x; idx < n * VPR; idx += kStatsThreads) {
    const int r = idx / VPR, c = idx % VPR;
    const int src = __ldg(ps + r);
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xs + static_cast<int64_t>(src) * D) + c);
    reinterpret_cast<uint4 *>(rows + r * D)[c] = v;
  }
  __syncthreads();

  const int dim = threadIdx.x % D;
  const int part = threadIdx.x / D;
  float acc = 0.f;
  for (int r = part; r < n; r += P) acc += __bfloat162float(rows[r * D + dim]);
  red[part * D + dim] = acc;
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll
    for (int p = 0; p < P; ++p) s += red[p * D + dim];
    s_mean[dim] = s / static_cast<float>(n);
  }
  __syncthreads();
  const float mean = s_mean[dim];
  acc = 0.f;
  for (int r = part; r < n; r += P) {
    const float dv = __bfloat162float(rows[r * D + dim]) - mean;
    acc = fmaf(dv, dv, acc);
  }
  __syncthreads();
  red[part * D + dim] = acc;
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll
    for (int p = 0; p < P; ++p) s += red[p * D + dim];
    const float var = s / static_cast<float>(n);
    float *o = aug + (bh * N + g) * static_cast<int64_t>(3 * D);
    if (query_side) {
      const float c = beta / static_cast<float>(D);
      o[dim] = mean * rsqrtf(static_cast<float>(D));
      o[D + dim] = c * var;
      o[2 * D + dim] = c * mean * mean;
    } else {
      o[dim] = mean;
      o[D + dim] = fmaf(mean, mean, var);
      o[2 * D + dim] = var;
    }
  }
}

// ---------------------------------------------------------------------------
// step 5-7: scores = A . B^T per (b,h); A, B are [N][KS] rows with stride 3D.
// grid = (ceil(N/64), ceil(N/64), b*h)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_scores(const float *__restrict__ A,
                                                const float *__restrict__ Bm,
                                                float *__restrict__ C, int N, int KS,
                                                int stride) {
  constexpr int BM = 64, BK = 16, PAD = 4;
  __shared__ __align__(16) float As[BK][BM + PAD];
  __shared__ __align__(16) float Bs[BK][BM + PAD];
  const int64_t bh = blockIdx.z;
  const float *Ab = A + bh * N * static_cast<int64_t>(stride);
  const float *Bb = Bm + bh * N * static_cast<int64_t>(stride);
  const int i0 = blockIdx.y * BM, j0 = blockIdx.x * BM;
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int lr = tid / 4, lk = (tid % 4) * 4;  // loader: row, k offset
  float acc[4][4] = {};
  for (int k0 = 0; k0 < KS; k0 += BK) {
    float4 va = make_float4(0.f, 0.f, 0.f, 0.f), vb = va;
    if (i0 + lr < N) va = *reinterpret_cast<const float4 *>(Ab + (i0 + lr) * static_cast<int64_t>(stride) + k0 + lk);
    if (j0 + lr < N) vb = *reinterpret_cast<const float4 *>(Bb + (j0 + lr) * static_cast<int64_t>(stride) + k0 + lk);
    As[lk + 0][lr] = va.x; As[lk + 1][lr] = va.y; As[lk + 2][lr] = va.z; As[lk + 3][lr] = va.w;
    Bs[lk + 0][lr] = vb.x; Bs[lk + 1][lr] = vb.y; Bs[lk + 2][lr] = vb.z; Bs[lk + 3][lr] = vb.w;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4 *>(&Bs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
    }
    __syncthreads();
  }
  float *Cb = C + bh * N * static_cast<int64_t>(N);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = i0 + ty * 4 + r;
    if (i >= N) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = j0 + tx * 4 + c;
      if (j < N) Cb[i * static_cast<int64_t>(N) + j] = acc[r][c];
    }
  }
}

// ---------------------------------------------------------------------------
// step 8-11: per-row top-kappa.  One warp per row.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) == 0u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kTopkWarps * 32) k_topk(const float *__restrict__ scores,
                                                          int64_t rows, int N, int kappa,
                                                          int32_t *__restrict__ idx,
                                                          uint32_t *__restrict__ mask) {
  extern __shared__ uint32_t skeys[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kTopkWarps + warp;
  if (row >= rows) return;  // warp-uniform; no block barrier below
  uint32_t *keys = skeys + warp * N;
  const float *src = scores + row * N;
  for (int e = lane; e < N; e += 32) keys[e] = order_key(src[e]);
  __syncwarp();
  uint32_t T = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    uint32_t cnt = 0;
    for (int e = lane; e < N; e += 32) cnt += keys[e] >= cand;
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if (cnt >= static_cast<uint32_t>(kappa)) T = cand;
  }
  uint32_t gt = 0;
  for (int e = lane; e < N; e += 32) gt += keys[e] > T;
  gt = __reduce_add_sync(0xffffffffu, gt);
  const int need = kappa - static_cast<int>(gt);  // >= 1 equal keys to take
  const int nwords = (N + 31) / 32;
  const uint32_t lt_mask = (1u << lane) - 1u;
  int taken = 0, base = 0;
  for (int wd = 0; wd < nwords; ++wd) {
    const int e = wd * 32 + lane;
    const bool valid = e < N;
    const uint32_t key = valid ? keys[e] : 0u;
    const uint32_t eqb = __ballot_sync(0xffffffffu, valid && key == T);
    const int rem = need - taken;
    const bool sel_eq = valid && key == T && __popc(eqb & lt_mask) < rem;
    taken += min(__popc(eqb), max(rem, 0));
    const uint32_t selb = __ballot_sync(0xffffffffu, (valid && key > T) || sel_eq);
    if (lane == 0) mask[row * nwords + wd] = selb;
    if ((selb >> lane) & 1u) idx[row * kappa + base + __popc(selb & lt_mask)] = e;
    base += __popc(selb);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct SelectPlan {
  size_t keys_bytes = 0;    // one ping-pong buffer (both tensors)
  size_t aug_bytes = 0;     // one augmented-vector array
  size_t scores_bytes = 0;  // scratch scores when the caller passes none
  size_t total = 0;
};

static SelectPlan plan_select(int64_t bh, int L, int D, int B, int sort_mode, bool need_scores) {
  SelectPlan p;
  const int64_t N = (L + B - 1) / B;
  const int nsorted = ((sort_mode & 1) ? 1 : 0) + ((sort_mode & 2) ? 1 : 0);
  p.keys_bytes = align256(static_cast<size_t>(nsorted) * bh * L * sizeof(uint64_t));
  p.aug_bytes = align256(static_cast<size_t>(bh) * N * 3 * D * sizeof(float));
  p.scores_bytes = need_scores ? align256(static_cast<size_t>(bh) * N * N * sizeof(float)) : 0;
  p.total = 2 * p.keys_bytes + 2 * p.aug_bytes + p.scores_bytes;
  return p;
}

size_t select_workspace_bytes(int64_t bh, int L, int D, int B, int sort_mode) {
  // scores scratch is always reserved so the size does not depend on whether
  // the caller asks for the score output
  return plan_select(bh, L, D, B, sort_mode, true).total;
}

static cudaError_t sort_sequences(const uint64_t *keys, uint64_t *buf0, uint64_t *buf1,
                                  int32_t *perm, int nseq, int L, int win, cudaStream_t st) {
  SortGeom g;
  g.L = L;
  g.win = (win <= 0 || win >= L) ? L : win;
  g.nwin = (L + g.win - 1) / g.win;
  int npasses = 0;
  for (int w = kChunk; w < g.win; w <<= 1) ++npasses;
  const int chunks = (g.win + kChunk - 1) / kChunk;
  // chunk sort: keys -> buf0 (or perm when no merge pass follows)
  k_chunk_sort<<<dim3(chunks, g.nwin, nseq), kChunkThreads, 0, st>>>(keys, buf0, perm, g,
                                                                     npasses == 0);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const uint64_t *src = buf0;
  uint64_t *dst = buf1;
  int width = kChunk;
  for (int p = 0; p < npasses; ++p) {
    const int per_cta = kMergeThreads * kMergeItems;
    const int gx = (g.win + per_cta - 1) / per_cta;
    k_merge_pass<<<dim3(gx, g.nwin, nseq), kMergeThreads, 0, st>>>(src, dst, perm, g, width,
                                                                   p == npasses - 1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const uint64_t *t = dst;
    dst = const_cast<uint64_t *>(src);
    src = t;
    width <<= 1;
  }
  return cudaSuccess;
}

template <int D>
static cudaError_t launch_stats(const void *x, const int32_t *perm, int64_t bh, int L, int B,
                                int N, float *aug, int query_side, float beta, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(B) * D * 2 + (kStatsThreads / D) * D * sizeof(float);
  static bool attr_set = false;  // smem <= 40 KB, below the default 48 KB limit
  (void)attr_set;
  k_block_stats<D><<<dim3(N, static_cast<unsigned>(bh)), kStatsThreads, smem, st>>>(
      static_cast<const __nv_bfloat16 *>(x), perm, L, B, N, aug, query_side, beta);
  return cudaGetLastError();
}

cudaError_t run_select(const SelectArgs &a, cudaStream_t st) {
  const int64_t bh = static_cast<int64_t>(a.batch) * a.heads;
  const int L = a.seqlen, D = a.head_dim, B = a.block;
  const int N = (L + B - 1) / B;
  const int64_t rows = bh * L;
  const bool sort_q = (a.sort_mode & 2) != 0, sort_k = (a.sort_mode & 1) != 0;
  const SelectPlan plan = plan_select(bh, L, D, B, a.sort_mode, true);
  unsigned char *ws = static_cast<unsigned char *>(a.workspace);
  uint64_t *keys0 = reinterpret_cast<uint64_t *>(ws);
  uint64_t *keys1 = reinterpret_cast<uint64_t *>(ws + plan.keys_bytes);
  float *aug_q = reinterpret_cast<float *>(ws + 2 * plan.keys_bytes);
  float *aug_k = reinterpret_cast<float *>(ws + 2 * plan.keys_bytes + plan.aug_bytes);
  float *scores = a.block_scores
                      ? a.block_scores
                      : reinterpret_cast<float *>(ws + 2 * plan.keys_bytes + 2 * plan.aug_bytes);
  cudaError_t e;

  // steps 1-2: norms and sort, per sorted tensor; identity otherwise
  const void *srcs[2] = {a.q, a.k};
  int32_t *perms[2] = {a.perm_q, a.perm_k};
  const bool sorted[2] = {sort_q, sort_k};
  int slot = 0;
  for (int t = 0; t < 2; ++t) {
    if (!sorted[t]) {
      k_iota<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, st>>>(perms[t], rows, L);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      continue;
    }
    uint64_t *k0 = keys0 + slot * rows;
    uint64_t *k1 = keys1 + slot * rows;
    ++slot;
    const int tpr = D / 8;
    const int64_t threads = rows * tpr;
    const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
    if (D == 128)
      k_sqnorm_keys<128><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(srcs[t]), k0,
                                               rows, L);
    else
      k_sqnorm_keys<64><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(srcs[t]), k0,
                                              rows, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the chunk sort reads k0 and writes k1; merges ping-pong k1 <-> k0
    if ((e = sort_sequences(k0, k1, k0, perms[t], static_cast<int>(bh), L, a.sort_window, st)) !=
        cudaSuccess)
      return e;
  }

  // steps 3-4: statistics on the (possibly) permuted blocks
  if (D == 128) {
    if ((e = launch_stats<128>(a.q, a.perm_q, bh, L, B, N, aug_q, 1, a.beta, st))) return e;
    if ((e = launch_stats<128>(a.k, a.perm_k, bh, L, B, N, aug_k, 0, a.beta, st))) return e;
  } else {
    if ((e = launch_stats<64>(a.q, a.perm_q, bh, L, B, N, aug_q, 1, a.beta, st))) return e;
    if ((e = launch_stats<64>(a.k, a.perm_k, bh, L, B, N, aug_k, 0, a.beta, st))) return e;
  }

  // steps 5-7: scores (the compensation terms are skipped when beta == 0:
  // they are exact zeros then)
  const int ks = (a.beta == 0.f) ? D : 3 * D;
  k_scores<<<dim3((N + 63) / 64, (N + 63) / 64, static_cast<unsigned>(bh)), 256, 0, st>>>(
      aug_q, aug_k, scores, N, ks, 3 * D);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // steps 8-11: top-kappa
  const int64_t qrows = bh * N;
  const size_t smem = static_cast<size_t>(kTopkWarps) * N * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    if ((e = cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem))) != cudaSuccess)
      return e;
  }
  k_topk<<<static_cast<unsigned>((qrows + kTopkWarps - 1) / kTopkWarps), kTopkWarps * 32, smem,
           st>>>(scores, qrows, N, a.kappa, a.block_idx, a.block_mask);
  return cudaGetLastError();
}

}  // namespace ba
