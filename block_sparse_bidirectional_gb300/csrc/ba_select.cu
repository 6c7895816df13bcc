// Selection stage of BA-Att ("Efficient Long-Context Modeling in Diffusion
// Language Models via Block Approximate Sparse Attention", Algorithm 1
// steps 1-11) for sm_103a.
//
//   k_sqnorm_keys   Eq. 9: fp32 squared norm of every Q / K row, packed with
//                   the token index into a 64-bit sort key.  One streaming
//                   pass over Q and K (16-byte vector loads, coalesced).
//   k_chunk_sort    Eq. 10, windows of up to 8192 keys: each thread sorts 8
//                   keys in registers (a 19-comparator network), the CTA
//                   merges the runs in shared memory (merge path, 9 levels)
//                   and emits pi (sorted position -> token index).  Keys are
//                   unique (index in the low word), so the result is the
//                   stable sort.
//   k_radix_pass    Eq. 10, longer windows: four stable 8-bit LSD radix
//                   passes over the norm bits, one cluster of 4 CTAs per
//                   window exchanging digit totals through distributed
//                   shared memory; the last pass emits pi.
//   k_block_stats   Algorithm 1 step 4: gathers the rows of sorted blocks
//                   through pi into shared memory (cp.async, double-buffered
//                   across the blocks a CTA walks); two-pass fp32 mean and
//                   population variance per feature; writes
//                     a = [Qbar/sqrt(d), beta/d*VarQ, beta/d*Qbar^2]
//                     b = [Kbar, Kbar^2 + VarK, VarK]
//                   so that a.b = Eq. 2 + beta * Eq. 14 (Eq. 13).
//   k_scores        l'[gq,gk] = a_gq . b_gk: a batched fp32 SIMT GEMM
//                   (128x128 tiles, 8x8 outputs per thread, or 64x64 and
//                   4x4 for small grids, in a conflict-free fragment layout,
//                   f32x2 FMAs).  Kept on the
//                   fp32 ALUs so the top-kappa decision is taken in fp32.
//   k_topk          steps 8-11: one warp per query-block row, keys held in
//                   registers; MSB-first radix
//                   select of the kappa-th largest score on order-preserving
//                   integer keys (warp reductions), ties to the lower block
//                   index; emits the ascending index list and the bitmask.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ba_common.cuh"
#include "ba_internal.h"

namespace ba {

// Windows of up to kChunkMax keys are sorted by one CTA (k_chunk_sort, 8 keys
// per thread, 512 or 1024 threads); longer ones by the clustered radix sort.
constexpr int kChunkMax = 8192;
constexpr int kStatsThreads = 256;
constexpr int kTopkWarps = 4;
constexpr int kNormRowsPerThread = 4;

// ---------------------------------------------------------------------------
// step 1-2a: squared norms -> sort keys.  grid = (.., sorted tensors)
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256, 8) k_sqnorm_keys(const __nv_bfloat16 *__restrict__ x0,
                                                     const __nv_bfloat16 *__restrict__ x1,
                                                     uint64_t *__restrict__ keys, int64_t rows,
                                                     int L) {
  constexpr int TPR = D / 8;            // threads per row, 8 bf16 (16 B) each
  constexpr int RPW = 256 / TPR;        // rows per 256-thread wave
  const __nv_bfloat16 *x = blockIdx.y == 0 ? x0 : x1;
  uint64_t *out = keys + static_cast<int64_t>(blockIdx.y) * rows;
  const int part = threadIdx.x % TPR;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * RPW * kNormRowsPerThread + threadIdx.x / TPR;
  // token index of row0 (rows of one thread are RPW apart)
  int tok0 = static_cast<int>(row0 % L);
  uint4 raw[kNormRowsPerThread];
#pragma unroll
  for (int u = 0; u < kNormRowsPerThread; ++u) {
    const int64_t row = row0 + u * RPW;
    // read once here (the block statistics gather these rows again much
    // later, long after they left L2): streaming loads
    raw[u] = (row < rows) ? __ldcs(reinterpret_cast<const uint4 *>(x + row * D) + part)
                          : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int u = 0; u < kNormRowsPerThread; ++u) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw[u]);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      acc = fmaf(f.x, f.x, acc);
      acc = fmaf(f.y, f.y, acc);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const int64_t row = row0 + u * RPW;
    if (row < rows && part == 0)
      out[row] = (static_cast<uint64_t>(__float_as_uint(acc)) << 32) | static_cast<uint32_t>(tok0);
    tok0 += RPW;
    while (tok0 >= L) tok0 -= L;
  }
}

// ---------------------------------------------------------------------------
// step 1-2, windows of up to kChunkMax keys: one CTA per window.
// grid = (1, windows, sorted sequences).  A thread sorts its 8 consecutive
// keys in registers; the CTA then merges the 512 runs in shared memory
// (merge path, 9 levels) and writes pi.  Keys are unique, so the order is
// the stable one.
// ---------------------------------------------------------------------------
struct SortGeom {
  int L;        // tokens per sequence
  int win;      // window length (== L for a whole-sequence sort); with a
                // split, the longer of the two windows
  int nwin;     // windows per sequence
  int bh;       // sequences per tensor
  int split;    // > 0: two windows, [0, split) and [split, L)
};

__device__ __forceinline__ int window_start(const SortGeom &g, int w) {
  return g.split > 0 ? (w == 0 ? 0 : g.split) : w * g.win;
}

__device__ __forceinline__ int window_len(const SortGeom &g, int w) {
  if (g.split > 0) return w == 0 ? g.split : g.L - g.split;
  const int start = w * g.win;
  return min(g.win, g.L - start);
}

// Shared-memory arrays of 64-bit keys are padded with one word per 8 so that
// threads walking runs that start 8 keys apart hit distinct banks.
__device__ __forceinline__ int spad(int i) { return i + (i >> 3); }
constexpr int spad_size(int n) { return n + (n >> 3); }

// merge_path_8 over padded shared-memory runs: A = s[a0 ..), B = s[b0 ..)
__device__ __forceinline__ void merge_path_8_smem(const uint64_t *s, int a0, int b0, int la,
                                                  int lb, int diag, int n, uint64_t *dst,
                                                  int d0) {
  int lo = max(0, diag - lb), hi = min(diag, la);
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s[spad(a0 + mid)] < s[spad(b0 + diag - 1 - mid)])
      lo = mid + 1;
    else
      hi = mid;
  }
  int i = lo, j = diag - lo;
  uint64_t va = (i < la) ? s[spad(a0 + i)] : ~0ull;
  uint64_t vb = (j < lb) ? s[spad(b0 + j)] : ~0ull;
  for (int t = 0; t < n; ++t) {
    const bool take_a = (i < la) && (j >= lb || va < vb);
    if (take_a) {
      dst[spad(d0 + t)] = va;
      ++i;
      va = (i < la) ? s[spad(a0 + i)] : ~0ull;
    } else {
      dst[spad(d0 + t)] = vb;
      ++j;
      vb = (j < lb) ? s[spad(b0 + j)] : ~0ull;
    }
  }
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads) k_chunk_sort(const uint64_t *__restrict__ keys_in,
                                                         int32_t *__restrict__ perm0,
                                                         int32_t *__restrict__ perm1, SortGeom g) {
  constexpr int kChunk = 8 * kThreads;  // keys per CTA
  extern __shared__ __align__(16) uint64_t sbuf[];  // 2 x padded kChunk
  uint64_t *sa = sbuf, *sb = sbuf + spad_size(kChunk);
  const int w = blockIdx.y;
  const int seq = blockIdx.z;
  const int wlen = window_len(g, w);
  const int c0 = blockIdx.x * kChunk;
  if (c0 >= wlen) return;  // uniform over the CTA
  const int n = min(kChunk, wlen - c0);
  const int64_t base = static_cast<int64_t>(seq) * g.L + window_start(g, w) + c0;
  // ---- each thread sorts its 8 consecutive keys in registers (Batcher's
  // odd-even merge network, 19 compare-exchanges) ----
  uint64_t r[8];
  const int e0 = threadIdx.x * 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = (e0 + i < n) ? keys_in[base + e0 + i] : ~0ull;
  auto cx = [&](int i, int j) {
    const uint64_t a = r[i], b = r[j];
    r[i] = a < b ? a : b;
    r[j] = a < b ? b : a;
  };
  cx(0, 1); cx(2, 3); cx(4, 5); cx(6, 7);
  cx(0, 2); cx(1, 3); cx(4, 6); cx(5, 7);
  cx(1, 2); cx(5, 6);
  cx(0, 4); cx(1, 5); cx(2, 6); cx(3, 7);
  cx(2, 4); cx(3, 5);
  cx(1, 2); cx(3, 4); cx(5, 6);
#pragma unroll
  for (int i = 0; i < 8; ++i) sa[spad(e0 + i)] = r[i];
  __syncthreads();

  // ---- merge the kThreads sorted runs: 8 -> 16 -> ... -> kChunk ----
  uint64_t *src = sa, *dst = sb;
  for (int width = 8; width < kChunk; width <<= 1) {
    const int o0 = threadIdx.x * 8;
    const int p0 = (o0 / (2 * width)) * 2 * width;
    merge_path_8_smem(src, p0, p0 + width, width, width, o0 - p0, 8, dst, o0);
    __syncthreads();
    uint64_t *t = src;
    src = dst;
    dst = t;
  }
  int32_t *perm = (seq < g.bh) ? perm0 : perm1;
  const int64_t pbase = static_cast<int64_t>(seq % g.bh) * g.L + window_start(g, w) + c0;
  for (int i = threadIdx.x; i < n; i += kThreads)
    perm[pbase + i] = static_cast<int32_t>(src[spad(i)] & 0xffffffffu);
}

// ---------------------------------------------------------------------------
// step 1-2, long windows: stable LSD radix sort on the 32 norm bits of the
// 64-bit keys (norm bits << 32 | token index), four passes of 8-bit digits.
// A cluster of kRadixCluster CTAs sorts one window: CTA r owns the r-th
// contiguous part of it and each of its warps a contiguous slice of that, so
// the order "CTA, warp, position" is the input order.  Per pass: every warp
// counts its digits (lanes with equal digits found with eight ballots, so
// one lane per digit adds); the CTAs exchange their digit totals through
// distributed shared memory; each (warp, digit) gets its first output
// position; a second sweep writes every key at that position plus its rank
// among the equal digits of the warp's slice (kept from the first sweep for
// parts that fit the shared-memory stage, else recounted per 32-key chunk).
// Equal norms keep the input
// (token index) order, the order the keys start in.  The last pass writes pi.
// grid = (kRadixCluster * windows, sorted sequences)
// ---------------------------------------------------------------------------
constexpr int kRadixThreads = 1024;
constexpr int kRadixWarps = kRadixThreads / 32;
constexpr int kRadixCluster = 4;
constexpr int kRadixBins = 256;
// Parts of up to kRadixStage keys (windows up to 4 x 16384 tokens) keep each
// warp's keys in registers across both sweeps (kRadixRegChunks chunks of 32
// per warp) and leave through a shared-memory stage in digit order, so each
// digit's keys go out as one contiguous, coalesced run; longer parts reload
// their keys and scatter them directly.
constexpr int kRadixRegChunks = 16;
constexpr int kRadixStage = kRadixWarps * kRadixRegChunks * 32;
constexpr size_t kRadixSmem = sizeof(int) * (kRadixWarps * kRadixBins + 3 * kRadixBins + kRadixBins / 32) +
                              sizeof(uint64_t) * kRadixStage + sizeof(uint16_t) * kRadixStage;

__global__ void __cluster_dims__(kRadixCluster, 1, 1) __launch_bounds__(kRadixThreads)
    k_radix_pass(const uint64_t *__restrict__ in, uint64_t *__restrict__ out, int32_t *__restrict__ perm0,
                 int32_t *__restrict__ perm1, SortGeom g, int shift, int final_pass) {
  namespace cg = cooperative_groups;
  extern __shared__ __align__(16) uint8_t rsm[];
  uint64_t *stage = reinterpret_cast<uint64_t *>(rsm);                  // [kRadixStage]
  int(*hist)[kRadixBins] = reinterpret_cast<int(*)[kRadixBins]>(stage + kRadixStage);  // [warps][bins]
  int *total = &hist[kRadixWarps][0];   // this CTA's digit counts (read by the cluster)
  int *lbase = total + kRadixBins;      // first staged position of each digit
  int *delta = lbase + kRadixBins;      // output position - staged position, per digit
  int *wsum = delta + kRadixBins;       // [kRadixBins / 32]
  // staged parts: each key's rank among the equal digits of its warp's slice
  uint16_t *lrank = reinterpret_cast<uint16_t *>(wsum + kRadixBins / 32);  // [kRadixStage]
  cg::cluster_group cluster = cg::this_cluster();
  const int r = static_cast<int>(cluster.block_rank());
  const int w = blockIdx.x / kRadixCluster;
  const int seq = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int wlen = window_len(g, w);
  const int64_t base = static_cast<int64_t>(seq) * g.L + window_start(g, w);
  // this CTA's part and this warp's slice of it
  const int p0 = static_cast<int>(static_cast<int64_t>(wlen) * r / kRadixCluster);
  const int p1 = static_cast<int>(static_cast<int64_t>(wlen) * (r + 1) / kRadixCluster);
  const int s0 = p0 + static_cast<int>(static_cast<int64_t>(p1 - p0) * warp / kRadixWarps);
  const int s1 = p0 + static_cast<int>(static_cast<int64_t>(p1 - p0) * (warp + 1) / kRadixWarps);
  // uniform over the cluster (all its parts differ in length by at most one)
  const bool staged = (wlen + kRadixCluster - 1) / kRadixCluster <= kRadixStage;
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint16_t *lrank_w = lrank + (s0 - p0);  // this warp's slice of the ranks
  auto digit = [&](uint64_t key) { return static_cast<int>((key >> (32 + shift)) & 0xFFu); };
  // lanes of `m` whose digit equals this lane's: eight ballots, one per
  // digit bit (a constant cost, whatever the number of distinct digits;
  // measured faster than match.any on the low, near-uniform digits)
  auto same_digit = [&](uint32_t m, int dig) {
    // a chunk of one digit (the common case for the exponent byte)
    if (__all_sync(m, dig == __shfl_sync(m, dig, __ffs(m) - 1))) return m;
    uint32_t peers = m;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t v = __ballot_sync(m, (dig >> b) & 1);
      peers &= ((dig >> b) & 1) ? v : ~v;
    }
    return peers;
  };
  for (int i = lane; i < kRadixBins; i += 32) hist[warp][i] = 0;
  __syncwarp();
  // ---- sweep 1: per-warp digit counts (staged: keys kept in registers) ----
  uint64_t kr[kRadixRegChunks];
  if (staged) {
#pragma unroll
    for (int u = 0; u < kRadixRegChunks; ++u) {
      const int i = s0 + u * 32 + lane;
      kr[u] = (i < s1) ? in[base + i] : 0ull;
    }
#pragma unroll
    for (int u = 0; u < kRadixRegChunks; ++u) {
      const int i = s0 + u * 32 + lane;
      if (s0 + u * 32 >= s1) break;  // uniform over the warp
      const bool act = i < s1;
      const uint32_t m = __ballot_sync(0xffffffffu, act);
      if (act) {
        const int dig = digit(kr[u]);
        const uint32_t peers = same_digit(m, dig);
        const int before = hist[warp][dig];
        lrank_w[u * 32 + lane] = static_cast<uint16_t>(before + __popc(peers & lt_mask));
        __syncwarp(m);  // every lane has read the count before its digit's leader updates it
        if ((peers & lt_mask) == 0u) hist[warp][dig] = before + __popc(peers);
      }
      __syncwarp();  // the next chunk's lanes see this update
    }
  } else {
    for (int c = s0; c < s1; c += 32) {
      const int i = c + lane;
      const bool act = i < s1;
      const uint32_t m = __ballot_sync(0xffffffffu, act);
      if (act) {
        const int dig = digit(in[base + i]);
        const uint32_t peers = same_digit(m, dig);
        if ((peers & lt_mask) == 0u) hist[warp][dig] += __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // ---- this CTA's totals; per-warp counts become exclusive prefixes ----
  if (threadIdx.x < kRadixBins) {
    const int d = threadIdx.x;
    int run = 0;
    for (int k = 0; k < kRadixWarps; ++k) {
      const int v = hist[k][d];
      hist[k][d] = run;
      run += v;
    }
    total[d] = run;
  }
  cluster.sync();  // every CTA's totals are visible to the cluster
  int before = 0, all = 0, mine = 0;
  if (threadIdx.x < kRadixBins) {
    const int d = threadIdx.x;
    for (int k = 0; k < kRadixCluster; ++k) {
      const int v = cluster.map_shared_rank(total, k)[d];
      all += v;
      if (k < r) before += v;
      if (k == r) mine = v;
    }
  }
  cluster.sync();  // the remote reads are done before any CTA moves on (or exits)
  // exclusive scans over the 256 digits: of the window's totals (global
  // positions) and of this CTA's totals (staged positions)
  if (threadIdx.x < kRadixBins) {
    int incl = all, incl_m = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      const int vm = __shfl_up_sync(0xffffffffu, incl_m, off);
      if (lane >= off) {
        incl += v;
        incl_m += vm;
      }
    }
    if (lane == 31) wsum[warp] = incl;
    total[threadIdx.x] = incl - all + before;
    lbase[threadIdx.x] = incl_m - mine;
    if (lane == 31) delta[warp] = incl_m;  // borrowed: the warp's sum of this CTA's totals
  }
  __syncthreads();
  int first = 0, lfirst = 0;
  if (threadIdx.x < kRadixBins) {
    int off = 0, off_m = 0;
    for (int k = 0; k < warp; ++k) {
      off += wsum[k];
      off_m += delta[k];
    }
    first = total[threadIdx.x] + off;      // this CTA's first output position for the digit
    lfirst = lbase[threadIdx.x] + off_m;   // its first staged position for the digit
  }
  __syncthreads();  // every thread has read delta[] (the warp sums) before it is overwritten
  if (threadIdx.x < kRadixBins) {
    const int d = threadIdx.x;
    if (staged) {
      delta[d] = first - lfirst;
      for (int k = 0; k < kRadixWarps; ++k) hist[k][d] += lfirst;
    } else {
      for (int k = 0; k < kRadixWarps; ++k) hist[k][d] += first;
    }
  }
  __syncthreads();
  // ---- sweep 2: rank in input order; stage and write out in digit runs ----
  int32_t *perm = (seq < g.bh) ? perm0 : perm1;
  const int64_t pbase = static_cast<int64_t>(seq % g.bh) * g.L + window_start(g, w);
  if (staged) {
#pragma unroll
    for (int u = 0; u < kRadixRegChunks; ++u) {
      const int i = s0 + u * 32 + lane;
      if (s0 + u * 32 >= s1) break;
      // the warp's first staged position of the digit plus the rank sweep 1 kept
      if (i < s1) stage[hist[warp][digit(kr[u])] + lrank_w[u * 32 + lane]] = kr[u];
    }
    __syncthreads();
    const int n = p1 - p0;
    for (int t = threadIdx.x; t < n; t += kRadixThreads) {
      const uint64_t key = stage[t];
      const int dest = t + delta[digit(key)];
      if (final_pass)
        perm[pbase + dest] = static_cast<int32_t>(key & 0xffffffffu);
      else
        out[base + dest] = key;
    }
  } else {
    for (int c = s0; c < s1; c += 32) {
      const int i = c + lane;
      const bool act = i < s1;
      const uint32_t m = __ballot_sync(0xffffffffu, act);
      if (act) {
        const uint64_t key = in[base + i];
        const int dig = digit(key);
        const uint32_t peers = same_digit(m, dig);
        const int dest = hist[warp][dig] + __popc(peers & lt_mask);
        __syncwarp(m);
        if ((peers & lt_mask) == 0u) hist[warp][dig] += __popc(peers);
        if (final_pass)
          perm[pbase + dest] = static_cast<int32_t>(key & 0xffffffffu);
        else
          out[base + dest] = key;
      }
      __syncwarp();
    }
  }
}

__global__ void k_iota(int32_t *__restrict__ perm, int64_t total, int L) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < total) perm[i] = static_cast<int32_t>(i % L);
}

// ---------------------------------------------------------------------------
// step 3-4: block statistics -> augmented vectors.
// grid = (ceil(N / kStatsBlocksPerCta), b*h, 2): z = 0 for Q (query side),
// 1 for K.  A CTA walks kStatsBlocksPerCta consecutive sorted blocks; the
// rows of the next block are gathered through pi into a second shared-memory
// stage with cp.async while the current block is reduced (two passes: mean,
// then mean squared deviation, one feature per thread and row slice).
// ---------------------------------------------------------------------------
constexpr int kStatsBlocksPerCta = 4;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D, int BK>
__global__ void __launch_bounds__(kStatsThreads) k_block_stats(
    const __nv_bfloat16 *__restrict__ xq, const __nv_bfloat16 *__restrict__ xk,
    const int32_t *__restrict__ perm_q, const int32_t *__restrict__ perm_k, int L, int N,
    float *__restrict__ aug_q, float *__restrict__ aug_k, float beta) {
  constexpr int VPR = D / 8;             // 16-byte vectors per row
  constexpr int QPR = D / 4;             // 4-feature groups per row
  constexpr int P = kStatsThreads / QPR; // row slices
  extern __shared__ __align__(16) unsigned char st_raw[];
  __nv_bfloat16 *stage[2] = {reinterpret_cast<__nv_bfloat16 *>(st_raw),
                             reinterpret_cast<__nv_bfloat16 *>(st_raw) + BK * D};
  int *s_src = reinterpret_cast<int *>(st_raw + 2 * BK * D * 2);  // [bpc][BK]
  __shared__ __align__(16) float red[P][D];
  __shared__ __align__(16) float s_mean[D];
  const bool qside = blockIdx.z == 0;
  const __nv_bfloat16 *x = qside ? xq : xk;
  const int32_t *perm = qside ? perm_q : perm_k;
  float *aug = qside ? aug_q : aug_k;
  const int64_t bh = blockIdx.y;
  const int g0 = blockIdx.x * kStatsBlocksPerCta;
  const int nblk = min(kStatsBlocksPerCta, N - g0);
  const __nv_bfloat16 *xs = x + bh * static_cast<int64_t>(L) * D;

  // source rows of every block this CTA reduces
  for (int i = threadIdx.x; i < nblk * BK; i += kStatsThreads) {
    const int r = g0 * BK + i;
    s_src[i] = (r < L) ? __ldg(perm + bh * static_cast<int64_t>(L) + r) : -1;
  }
  __syncthreads();
  auto issue = [&](int bi) {
    __nv_bfloat16 *dst = stage[bi & 1];
    for (int idx = threadIdx.x; idx < BK * VPR; idx += kStatsThreads) {
      const int r = idx / VPR, c = idx % VPR;
      const int src = s_src[bi * BK + r];
      if (src >= 0) cp_async16(dst + r * D + c * 8, xs + static_cast<int64_t>(src) * D + c * 8);
    }
    cp_async_commit();
  };
  issue(0);
  // a thread sums 4 features over the rows part, part + P, ...; a warp reads
  // whole rows (8-byte loads); the P partial sums of a feature are then
  // added in slice order by one thread
  const int quad = threadIdx.x % QPR, part = threadIdx.x / QPR;
  const int dim = threadIdx.x;  // feature owned in the combine step (< D)
  // four features of row r as two packed fp32 pairs (a bf16 is the top half
  // of its fp32), so the sums below run as f32x2 adds / fmas: the same IEEE
  // operation per feature, half the instructions
  auto load4 = [&](const __nv_bfloat16 *rows, int r, uint64_t &p01, uint64_t &p23) {
    const uint2 w = *reinterpret_cast<const uint2 *>(rows + r * D + quad * 4);
    p01 = f2_pack(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
    p23 = f2_pack(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
  };
  for (int bi = 0; bi < nblk; ++bi) {
    if (bi + 1 < nblk) {
      issue(bi + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const __nv_bfloat16 *rows = stage[bi & 1];
    const int g = g0 + bi;
    const int n = min(BK, L - g * BK);
    uint64_t a01 = f2_pack(0.f, 0.f), a23 = a01;
    for (int r = part; r < n; r += P) {
      uint64_t p01, p23;
      load4(rows, r, p01, p23);
      a01 = f2_add(a01, p01);
      a23 = f2_add(a23, p23);
    }
    float acc[4];
    f2_unpack(a01, acc[0], acc[1]);
    f2_unpack(a23, acc[2], acc[3]);
    *reinterpret_cast<float4 *>(&red[part][quad * 4]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    __syncthreads();
    if (threadIdx.x < D) {
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < P; ++q) sum += red[q][dim];
      s_mean[dim] = sum / static_cast<float>(n);
    }
    __syncthreads();
    const float4 m4 = *reinterpret_cast<const float4 *>(&s_mean[quad * 4]);
    const uint64_t nm01 = f2_pack(-m4.x, -m4.y), nm23 = f2_pack(-m4.z, -m4.w);
    a01 = f2_pack(0.f, 0.f);
    a23 = a01;
    for (int r = part; r < n; r += P) {
      uint64_t p01, p23;
      load4(rows, r, p01, p23);
      const uint64_t d01 = f2_add(p01, nm01), d23 = f2_add(p23, nm23);  // x - mean
      a01 = f2_fma(d01, d01, a01);
      a23 = f2_fma(d23, d23, a23);
    }
    f2_unpack(a01, acc[0], acc[1]);
    f2_unpack(a23, acc[2], acc[3]);
    *reinterpret_cast<float4 *>(&red[part][quad * 4]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    __syncthreads();
    if (threadIdx.x < D) {
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < P; ++q) sum += red[q][dim];
      const float var = sum / static_cast<float>(n);
      const float mean = s_mean[dim];
      float *o = aug + (bh * N + g) * static_cast<int64_t>(3 * D);
      if (qside) {
        const float cf = beta / static_cast<float>(D);
        o[dim] = mean * rsqrtf(static_cast<float>(D));
        o[D + dim] = cf * var;
        o[2 * D + dim] = cf * mean * mean;
      } else {
        o[dim] = mean;
        o[D + dim] = fmaf(mean, mean, var);
        o[2 * D + dim] = var;
      }
    }
    __syncthreads();  // the stage is refilled two iterations on
  }
}

// ---------------------------------------------------------------------------
// step 5-7: scores = A . B^T per (b,h); A, B are [N][KS] rows with stride 3D.
// grid = (ceil(N/TM), ceil(N/TM), b*h); TM x TM tiles (TM = 128: 8 x 8
// outputs per thread; TM = 64, for small grids: 4 x 4), packed f32x2 FMAs.
// A warp covers 4 x 8 threads of the 16 x 16 thread grid; a thread owns the
// row groups {4ty..4ty+3} (+ TM/2 when TM = 128) and the same pattern of
// columns, so each fragment load of a warp is one shared-memory wavefront
// (broadcast for A, 128 contiguous bytes for B).  Every output is one fma
// chain over k in order, the same for both tile sizes.
// ---------------------------------------------------------------------------
template <int TM>
__global__ void __launch_bounds__(256) k_scores(const float *__restrict__ A,
                                                const float *__restrict__ Bm,
                                                float *__restrict__ C, int N, int KS,
                                                int stride) {
  constexpr int BKK = 8, PAD = 4;
  constexpr int G = TM / 64;       // 4-row (4-column) groups per thread
  constexpr int R = 4 * G;         // rows (columns) per thread
  __shared__ __align__(16) float As[BKK][TM + PAD];
  __shared__ __align__(16) float Bs[BKK][TM + PAD];
  const int64_t bh = blockIdx.z;
  const float *Ab = A + bh * N * static_cast<int64_t>(stride);
  const float *Bb = Bm + bh * N * static_cast<int64_t>(stride);
  const int i0 = blockIdx.y * TM, j0 = blockIdx.x * TM;
  const int tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  const int tx = (warp % 2) * 8 + lane % 8, ty = (warp / 2) * 4 + lane / 8;
  // loader: TM = 128: every thread one float4 of A and one of B;
  // TM = 64: threads 0-127 load A, 128-255 load B
  const int lt = (TM == 128) ? tid : tid % 128;
  const int lr = lt / 2, lk = (lt % 2) * 4;
  const bool load_a = (TM == 128) || tid < 128, load_b = (TM == 128) || tid >= 128;
  uint64_t acc[R][R / 2];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int c = 0; c < R / 2; ++c) acc[r][c] = 0ull;
  const float *arow = Ab + (i0 + lr) * static_cast<int64_t>(stride) + lk;
  const float *brow = Bb + (j0 + lr) * static_cast<int64_t>(stride) + lk;
  const bool a_ok = load_a && i0 + lr < N, b_ok = load_b && j0 + lr < N;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  // kPF k-chunks in flight (registers): a CTA's chunks are a chain of L2
  // round trips, and the 64-wide tiles serve short grids with few CTAs to
  // hide them (the 128-wide tiles keep one: more would cost them their
  // second CTA per SM); KS / BKK (8, 16, 24 or 48) is a multiple of kPF
  constexpr int kPF = TM == 64 ? 4 : 1;
  float4 na4[kPF], nb4[kPF];
#pragma unroll
  for (int u = 0; u < kPF; ++u) {
    na4[u] = (a_ok && u * BKK < KS) ? *reinterpret_cast<const float4 *>(arow + u * BKK) : z4;
    nb4[u] = (b_ok && u * BKK < KS) ? *reinterpret_cast<const float4 *>(brow + u * BKK) : z4;
  }
  for (int k00 = 0; k00 < KS; k00 += kPF * BKK)
#pragma unroll
  for (int u = 0; u < kPF; ++u) {
    const int k0 = k00 + u * BKK;
    const float4 va = na4[u], vb = nb4[u];
    if (k0 + kPF * BKK < KS) {  // the chunk kPF ahead replaces this one
      na4[u] = a_ok ? *reinterpret_cast<const float4 *>(arow + k0 + kPF * BKK) : z4;
      nb4[u] = b_ok ? *reinterpret_cast<const float4 *>(brow + k0 + kPF * BKK) : z4;
    }
    if (load_a) {
      As[lk + 0][lr] = va.x; As[lk + 1][lr] = va.y; As[lk + 2][lr] = va.z; As[lk + 3][lr] = va.w;
    }
    if (load_b) {
      Bs[lk + 0][lr] = vb.x; Bs[lk + 1][lr] = vb.y; Bs[lk + 2][lr] = vb.z; Bs[lk + 3][lr] = vb.w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BKK; ++kk) {
      float av[R];
      uint64_t bp[R / 2];
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        const float4 a4 = *reinterpret_cast<const float4 *>(&As[kk][gi * 64 + ty * 4]);
        const float4 b4 = *reinterpret_cast<const float4 *>(&Bs[kk][gi * 64 + tx * 4]);
        av[4 * gi + 0] = a4.x; av[4 * gi + 1] = a4.y; av[4 * gi + 2] = a4.z; av[4 * gi + 3] = a4.w;
        bp[2 * gi + 0] = f2_pack(b4.x, b4.y);
        bp[2 * gi + 1] = f2_pack(b4.z, b4.w);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint64_t a2 = f2_pack(av[r], av[r]);
#pragma unroll
        for (int c = 0; c < R / 2; ++c) acc[r][c] = f2_fma(a2, bp[c], acc[r][c]);
      }
    }
    __syncthreads();
  }
  // row r: group r / 4 (offset 64 each), 4ty + r % 4; column pair c: group
  // c / 2, columns 4tx + 2 (c % 2), + 1
  float *Cb = C + bh * N * static_cast<int64_t>(N);
  const bool vec = (N % 4) == 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = i0 + (r / 4) * 64 + ty * 4 + r % 4;
    if (i >= N) continue;
    float *crow = Cb + i * static_cast<int64_t>(N);
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      const int j = j0 + gi * 64 + tx * 4;
      float x0, x1, x2, x3;
      f2_unpack(acc[r][2 * gi], x0, x1);
      f2_unpack(acc[r][2 * gi + 1], x2, x3);
      if (vec && j + 3 < N) {
        *reinterpret_cast<float4 *>(crow + j) = make_float4(x0, x1, x2, x3);
      } else {
        if (j < N) crow[j] = x0;
        if (j + 1 < N) crow[j + 1] = x1;
        if (j + 2 < N) crow[j + 2] = x2;
        if (j + 3 < N) crow[j + 3] = x3;
      }
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

// Keys of one row live in registers (KPL per lane, element e = i * 32 + lane).
// The row is split in two parts, elements [0, n_first) with budget
// kappa_first and [n_first, N) with budget kappa - kappa_first (isolated
// prefill / generation selection); n_first == N is the plain top-kappa.
// kRange = false: the part is the whole row; elements past N hold key 0,
// which no candidate (>= 1) counts, so no range test is needed.  The MSB-first
// search stops once exactly k keys lie at or above the threshold so far.
template <int KPL, bool kRange>
__device__ __forceinline__ void part_threshold(const uint32_t (&keys)[KPL], int lane, int lo, int hi,
                                               int k, uint32_t &T, int &need) {
  T = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    uint32_t cnt = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int e = i * 32 + lane;
      cnt += (!kRange || (e >= lo && e < hi)) && keys[i] >= cand;
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if (cnt >= static_cast<uint32_t>(k)) T = cand;
    // exactly k keys at or above T: they are the top k whatever T's lower
    // bits, and the keys equal to T (need below) are all of them taken
    if (cnt == static_cast<uint32_t>(k)) break;
  }
  uint32_t gt = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = i * 32 + lane;
    gt += (!kRange || (e >= lo && e < hi)) && keys[i] > T;
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  need = k - static_cast<int>(gt);  // >= 1 keys equal to T to take, lowest index first
}

template <int KPL>
__global__ void __launch_bounds__(kTopkWarps * 32) k_topk(const float *__restrict__ scores,
                                                          int64_t rows, int N, int kappa,
                                                          int n_first, int kappa_first,
                                                          int32_t *__restrict__ idx,
                                                          uint32_t *__restrict__ mask) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kTopkWarps + warp;
  if (row >= rows) return;  // warp-uniform; no block barrier below
  const float *src = scores + row * N;
  uint32_t keys[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = i * 32 + lane;
    keys[i] = (e < N) ? order_key(src[e]) : 0u;  // 0 sorts below every real key
  }
  uint32_t T0, T1 = 0;
  int need0, need1 = 0;
  const bool two = n_first < N;
  if (two) {
    part_threshold<KPL, true>(keys, lane, 0, n_first, kappa_first, T0, need0);
    part_threshold<KPL, true>(keys, lane, n_first, N, kappa - kappa_first, T1, need1);
  } else {
    part_threshold<KPL, false>(keys, lane, 0, N, kappa_first, T0, need0);
  }
  const int nwords = (N + 31) / 32;
  const uint32_t lt_mask = (1u << lane) - 1u;
  int taken0 = 0, taken1 = 0, base = 0;
#pragma unroll
  for (int wd = 0; wd < KPL; ++wd) {
    if (wd >= nwords) break;
    const int e = wd * 32 + lane;
    const bool in0 = e < n_first, in1 = two && e >= n_first && e < N;
    const uint32_t key = keys[wd];
    const bool eq0 = in0 && key == T0, eq1 = in1 && key == T1;
    const uint32_t eqb0 = __ballot_sync(0xffffffffu, eq0);
    const int rem0 = need0 - taken0;
    const bool sel_eq0 = eq0 && __popc(eqb0 & lt_mask) < rem0;
    taken0 += min(__popc(eqb0), max(rem0, 0));
    bool sel_eq1 = false;
    if (two) {
      const uint32_t eqb1 = __ballot_sync(0xffffffffu, eq1);
      const int rem1 = need1 - taken1;
      sel_eq1 = eq1 && __popc(eqb1 & lt_mask) < rem1;
      taken1 += min(__popc(eqb1), max(rem1, 0));
    }
    const uint32_t selb = __ballot_sync(
        0xffffffffu, (in0 && key > T0) || sel_eq0 || (in1 && key > T1) || sel_eq1);
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

// Sorts `nseq` sequences of L keys (windows of `win`), writing pi into
// perm0 (the first `bh` sequences) and perm1 (the rest).
static cudaError_t sort_sequences(const uint64_t *keys, uint64_t *buf0, uint64_t *buf1,
                                  int32_t *perm0, int32_t *perm1, int nseq, int64_t bh, int L,
                                  int win, int split, cudaStream_t st) {
  SortGeom g;
  g.L = L;
  g.bh = static_cast<int>(bh);
  g.split = (split > 0 && split < L) ? split : 0;
  if (g.split > 0) {
    g.win = max(g.split, L - g.split);
    g.nwin = 2;
  } else {
    g.win = (win <= 0 || win >= L) ? L : win;
    g.nwin = (L + g.win - 1) / g.win;
  }
  cudaError_t e;
  if (g.win > kChunkMax) {
    // long windows: four radix passes, keys -> buf0 -> buf1 -> buf0 -> pi
    static std::atomic<uint64_t> radix_configured{0};
    e = once_per_device(radix_configured, [] {
      return cudaFuncSetAttribute(k_radix_pass, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(kRadixSmem));
    });
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(kRadixCluster * g.nwin), static_cast<unsigned>(nseq));
    const uint64_t *src = keys;
    uint64_t *bufs[2] = {buf0, buf1};
    for (int pass = 0; pass < 4; ++pass) {
      k_radix_pass<<<grid, kRadixThreads, kRadixSmem, st>>>(src, bufs[pass & 1], perm0, perm1, g, 8 * pass,
                                                            pass == 3);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      src = bufs[pass & 1];
    }
    return cudaSuccess;
  }
  // one CTA covers the window: keys -> pi (4096 keys with 512 threads, up to
  // 8192 with 1024: at L = 8192 one launch instead of four radix passes whose
  // parts of 2048 keys are dominated by the cluster exchanges)
  static std::atomic<uint64_t> configured{0};
  e = once_per_device(configured, [] {
    cudaError_t r = cudaFuncSetAttribute(k_chunk_sort<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(2 * spad_size(4096) * sizeof(uint64_t)));
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(k_chunk_sort<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(2 * spad_size(8192) * sizeof(uint64_t)));
  });
  if (e != cudaSuccess) return e;
  if (g.win <= 4096)
    k_chunk_sort<512><<<dim3(1, g.nwin, nseq), 512, 2 * spad_size(4096) * sizeof(uint64_t), st>>>(keys, perm0,
                                                                                                perm1, g);
  else
    k_chunk_sort<1024><<<dim3(1, g.nwin, nseq), 1024, 2 * spad_size(8192) * sizeof(uint64_t), st>>>(keys, perm0,
                                                                                                  perm1, g);
  return cudaGetLastError();
}

template <int D, int BK>
static cudaError_t launch_stats(const SelectArgs &a, int64_t bh, int N, float *aug_q, float *aug_k,
                                cudaStream_t st) {
  const size_t smem = 2 * BK * D * 2 + kStatsBlocksPerCta * BK * sizeof(int);
  static std::atomic<uint64_t> configured{0};
  const cudaError_t e = once_per_device(configured, [smem] {
    return cudaFuncSetAttribute(k_block_stats<D, BK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem));
  });
  if (e != cudaSuccess) return e;
  const dim3 grid((N + kStatsBlocksPerCta - 1) / kStatsBlocksPerCta, static_cast<unsigned>(bh), 2);
  k_block_stats<D, BK><<<grid, kStatsThreads, smem, st>>>(
      static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k), a.perm_q,
      a.perm_k, a.seqlen, N, aug_q, aug_k, a.beta);
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

  // steps 1-2: norms and sort of the sorted tensors (one launch each for
  // both); identity permutations otherwise
  const void *srcs[2];
  int32_t *perms[2];
  int nsorted = 0;
  if (sort_q) { srcs[nsorted] = a.q; perms[nsorted++] = a.perm_q; }
  if (sort_k) { srcs[nsorted] = a.k; perms[nsorted++] = a.perm_k; }
  if (!sort_q) {
    k_iota<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, st>>>(a.perm_q, rows, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (!sort_k) {
    k_iota<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, st>>>(a.perm_k, rows, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (nsorted > 0) {
    const int rows_per_cta = (256 / (D / 8)) * kNormRowsPerThread;
    const dim3 grid(static_cast<unsigned>((rows + rows_per_cta - 1) / rows_per_cta), nsorted);
    const __nv_bfloat16 *x0 = static_cast<const __nv_bfloat16 *>(srcs[0]);
    const __nv_bfloat16 *x1 = static_cast<const __nv_bfloat16 *>(srcs[nsorted - 1]);
    if (D == 128)
      k_sqnorm_keys<128><<<grid, 256, 0, st>>>(x0, x1, keys0, rows, L);
    else
      k_sqnorm_keys<64><<<grid, 256, 0, st>>>(x0, x1, keys0, rows, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the chunk sort reads keys0 and writes keys1; merges ping-pong keys1 <-> keys0
    if (a.prefill_len == 0 || !sort_k) {
      if ((e = sort_sequences(keys0, keys1, keys0, perms[0], perms[nsorted - 1],
                              static_cast<int>(nsorted * bh), bh, L, a.sort_window, 0, st)) !=
          cudaSuccess)
        return e;
    } else {
      // isolated selection: keys are sorted inside [0, prefill) and
      // [prefill, L) so no sorted key block mixes the two ranges; queries
      // keep the caller's window
      const int64_t qoff = sort_q ? rows : 0;  // K's keys follow Q's
      if (sort_q && (e = sort_sequences(keys0, keys1, keys0, a.perm_q, a.perm_q,
                                        static_cast<int>(bh), bh, L, a.sort_window, 0, st)) !=
                        cudaSuccess)
        return e;
      if ((e = sort_sequences(keys0 + qoff, keys1 + qoff, keys0 + qoff, a.perm_k, a.perm_k,
                              static_cast<int>(bh), bh, L, 0, a.prefill_len, st)) != cudaSuccess)
        return e;
    }
  }

  // steps 3-4: statistics on the (possibly) permuted blocks, Q and K together
  if (D == 128 && B == 128) e = launch_stats<128, 128>(a, bh, N, aug_q, aug_k, st);
  else if (D == 128 && B == 64) e = launch_stats<128, 64>(a, bh, N, aug_q, aug_k, st);
  else if (D == 64 && B == 128) e = launch_stats<64, 128>(a, bh, N, aug_q, aug_k, st);
  else e = launch_stats<64, 64>(a, bh, N, aug_q, aug_k, st);
  if (e != cudaSuccess) return e;

  // steps 5-7: scores (the compensation terms are skipped when beta == 0:
  // they are exact zeros then)
  const int ks = (a.beta == 0.f) ? D : 3 * D;
  // 128-wide tiles unless that grid would leave more than half of the SMs
  // idle; there the 64-wide tiles (a quarter of the serial work per thread)
  // finish sooner (L = 8192, B = 64: 0.140 -> 0.134 ms for the selection),
  // while on a grid of one CTA per SM (L = 32768, B = 128) they lose to
  // L2 latency per k-chunk (0.377 -> 0.396 ms)
  const int64_t t128 = static_cast<int64_t>((N + 127) / 128) * ((N + 127) / 128) * bh;
  if (2 * t128 >= 152)
    k_scores<128><<<dim3((N + 127) / 128, (N + 127) / 128, static_cast<unsigned>(bh)), 256, 0, st>>>(
        aug_q, aug_k, scores, N, ks, 3 * D);
  else
    k_scores<64><<<dim3((N + 63) / 64, (N + 63) / 64, static_cast<unsigned>(bh)), 256, 0, st>>>(
        aug_q, aug_k, scores, N, ks, 3 * D);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // steps 8-11: top-kappa (keys of a row in registers: 32 * KPL >= N)
  const int64_t qrows = bh * N;
  const unsigned tgrid = static_cast<unsigned>((qrows + kTopkWarps - 1) / kTopkWarps);
  // isolated selection: the first prefill_len / B key blocks are the prefill part
  const int n_first = a.prefill_len > 0 ? a.prefill_len / B : N;
  const int k_first = a.prefill_len > 0 ? a.kappa_prefill : a.kappa;
  if (N <= 256)
    k_topk<8><<<tgrid, kTopkWarps * 32, 0, st>>>(scores, qrows, N, a.kappa, n_first, k_first,
                                                 a.block_idx, a.block_mask);
  else if (N <= 512)
    k_topk<16><<<tgrid, kTopkWarps * 32, 0, st>>>(scores, qrows, N, a.kappa, n_first, k_first,
                                                  a.block_idx, a.block_mask);
  else if (N <= 1024)
    k_topk<32><<<tgrid, kTopkWarps * 32, 0, st>>>(scores, qrows, N, a.kappa, n_first, k_first,
                                                  a.block_idx, a.block_mask);
  else
    k_topk<128><<<tgrid, kTopkWarps * 32, 0, st>>>(scores, qrows, N, a.kappa, n_first, k_first,
                                                   a.block_idx, a.block_mask);
  return cudaGetLastError();
}

}  // namespace ba
