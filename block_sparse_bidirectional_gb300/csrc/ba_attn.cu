// Block-sparse attention forward for sm_103a: BA-Att paper Algorithm 1
// step 12 ("Efficient Long-Context Modeling in Diffusion Language Models via
// Block Approximate Sparse Attention"), with the masked softmax of SparseD
// §3.1 Eq. 3-4, and the same kernel run dense (Eq. 1).
//
// One CTA owns a tile of 128 consecutive sorted query rows (one query block
// when B = 128, two when B = 64) and walks the key blocks its rows selected
// (for B = 64: the union of the two lists, each entry tagged with which of
// the two query blocks selected it; rows of the other block see -inf).
//
// Warp roles (256 threads):
//   warp 0       TMA producer: Q tile once, then K_j and V_j tiles of every
//                listed key block into a 2-stage shared-memory ring
//                (128-byte swizzle, 64-column boxes, 3-D maps so the ragged
//                last block reads zeros instead of the next head).
//   warp 1       tensor-memory allocation and the single MMA-issuing thread:
//                  S_j = Q K_j^T   -> TMEM (two S buffers, ping-pong), and
//                  O  += P_j V_j   -> TMEM, V read as an MN-major operand;
//                S_{j+1} is issued before waiting for P_j so the tensor core
//                works while the softmax runs.
//   warps 4-7    softmax + epilogue: thread t owns row t of the tile
//                (TMEM lane t).  Online softmax in the log2 domain with a
//                lazy rescale: O in TMEM is corrected only when the running
//                max grows by more than 2^8.  P (bf16) goes to shared memory
//                in the swizzled K-major layout the MMA reads.  At the end
//                O / l is written as bf16 to the ORIGINAL row pi_q(r), and
//                LSE = ln(sum exp(scale q.k)).
// Every wait is bounded; on a timeout the CTA records the site in the device
// error word, drains its in-flight copies / MMAs and frees tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ba_common.cuh"
#include "ba_internal.h"

namespace ba {

constexpr int kTileM = 128;
constexpr int kAttnThreads = 256;
constexpr int kStages = 2;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxBlocks = 4096;

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

constexpr int next_pow2_cols(int x) {
  int c = 32;
  while (c < x) c <<= 1;
  return c;
}

template <int D, int BK>
struct AttnLayout {
  static constexpr int kQBytes = kTileM * D * 2;
  static constexpr int kKVBytes = BK * D * 2;
  static constexpr int kPBytes = kTileM * BK * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  static constexpr int kOffP = kOffV + kStages * kKVBytes;
  static constexpr int kOffList = kOffP + kPBytes;
  static constexpr int kOffBitmap = kOffList + kMaxBlocks * 2;
  static constexpr int kOffBar = kOffBitmap + 2 * (kMaxBlocks / 32) * 4;
  static constexpr int kNumBars = 1 + 4 * kStages + 2 + 1 + 1 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64;
  static constexpr int kTmemCols = next_pow2_cols(2 * BK + D);
  // Shared memory is padded so that no more CTAs fit on an SM than its 512
  // tensor-memory columns can hold (an allocation would otherwise stall).
  static constexpr int kMaxCtasByTmem = 512 / kTmemCols;
  static constexpr int kMinAlloc = (228 * 1024) / (kMaxCtasByTmem + 1) + 1024;
  static constexpr int kAlloc = (kBytes + 1024 > kMinAlloc) ? kBytes + 1024 : kMinAlloc;
  static_assert(kTmemCols <= 512, "tensor memory budget");
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

struct AttnParams {
  int L;          // tokens per sequence
  int N;          // key blocks (and query blocks) of size BK
  int kappa;      // list length per query block (unused when dense)
  int dense;      // 1: every key block, no list
  const int32_t *block_idx;
  const int32_t *perm_q;  // sorted query position -> original row (nullable)
  __nv_bfloat16 *o;
  float *lse;
  float scale_log2;       // scale * log2(e)
};

template <int D, int BK>
__global__ void __launch_bounds__(kAttnThreads, 1)
    k_attn(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using Lay = AttnLayout<D, BK>;
  constexpr int G = kTileM / BK;  // query blocks per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + Lay::kOffQ;
  uint8_t *sK = smem + Lay::kOffK;
  uint8_t *sV = smem + Lay::kOffV;
  uint8_t *sP = smem + Lay::kOffP;
  uint16_t *list = reinterpret_cast<uint16_t *>(smem + Lay::kOffList);
  uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem + Lay::kOffBitmap);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kOffBar);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + kStages;
  uint64_t *v_full = k_empty + kStages;
  uint64_t *v_empty = v_full + kStages;
  uint64_t *s_full = v_empty + kStages;
  uint64_t *p_full = s_full + 2;
  uint64_t *o_done = p_full + 1;
  uint64_t *drain = o_done + 1;
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + Lay::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(&misc[2]);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tile = blockIdx.x;
  const int bh = blockIdx.y;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    misc[1] = 0;
    misc[2] = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&misc[0], Lay::kTmemCols);
    tc_fence_before();
  }

  // ---- the key-block list of this tile ------------------------------------
  if (!p.dense) {
    if (G == 1) {
      const int32_t *src = p.block_idx + (static_cast<int64_t>(bh) * p.N + tile) * p.kappa;
      for (int i = threadIdx.x; i < p.kappa; i += kAttnThreads)
        list[i] = static_cast<uint16_t>(min(max(src[i], 0), p.N - 1) | (1 << 12));
      if (threadIdx.x == 0) misc[1] = p.kappa;
    } else {
      const int nwords = (p.N + 31) / 32;
      for (int i = threadIdx.x; i < 2 * (kMaxBlocks / 32); i += kAttnThreads) bitmap[i] = 0u;
      __syncthreads();
      for (int g = 0; g < G; ++g) {
        const int gq = tile * G + g;
        if (gq >= p.N) break;
        const int32_t *src = p.block_idx + (static_cast<int64_t>(bh) * p.N + gq) * p.kappa;
        for (int i = threadIdx.x; i < p.kappa; i += kAttnThreads) {
          const int blk = src[i];
          if (blk < 0 || blk >= p.N) continue;  // ids are not validated on the host
          atomicOr(&bitmap[g * (kMaxBlocks / 32) + (blk >> 5)], 1u << (blk & 31));
        }
      }
      __syncthreads();
      if (warp == 0) {
        int base = 0;
        for (int w0 = 0; w0 < nwords; w0 += 32) {
          const int w = w0 + lane;
          const uint32_t m0 = (w < nwords) ? bitmap[w] : 0u;
          const uint32_t m1 = (w < nwords) ? bitmap[(kMaxBlocks / 32) + w] : 0u;
          uint32_t u = m0 | m1;
          const int cnt = __popc(u);
          int incl = cnt;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += t;
          }
          int pos = base + incl - cnt;
          while (u) {
            const int b = __ffs(u) - 1;
            u &= u - 1;
            const uint32_t sel = ((m0 >> b) & 1u) | (((m1 >> b) & 1u) << 1);
            list[pos++] = static_cast<uint16_t>((w * 32 + b) | (sel << 12));
          }
          base += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) misc[1] = base;
      }
    }
  }
  __syncthreads();
  tc_fence_after();
  const int n_iter = p.dense ? p.N : static_cast<int>(misc[1]);
  const uint32_t tmem = misc[0];

  if (warp == 0) {
    // ===================== TMA producer =====================================
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      int nk[kStages] = {}, nv[kStages] = {};
      mbar_arrive_expect_tx(q_full, Lay::kQBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(sQ + c * kTileM * 128, &tmQ, q_full, c * 64, tile * kTileM, bh);
      for (int j = 0; j < n_iter; ++j) {
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        const int blk = p.dense ? j : (list[j] & 0xFFF);
        if (j >= kStages && !mbar_wait(&k_empty[s], ph ^ 1u, kSiteKEmpty, abort_flag)) break;
        mbar_arrive_expect_tx(&k_full[s], Lay::kKVBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sK + s * Lay::kKVBytes + c * BK * 128, &tmK, &k_full[s], c * 64, blk * BK,
                      bh);
        ++nk[s];
        if (j >= kStages && !mbar_wait(&v_empty[s], ph ^ 1u, kSiteVEmpty, abort_flag)) break;
        mbar_arrive_expect_tx(&v_full[s], Lay::kKVBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sV + s * Lay::kKVBytes + c * BK * 128, &tmV, &v_full[s], c * 64, blk * BK,
                      bh);
        ++nv[s];
      }
      // drain: the last copy issued on each barrier has landed
      mbar_wait_drain(q_full, 0);
      for (int s = 0; s < kStages; ++s) {
        if (nk[s]) mbar_wait_drain(&k_full[s], (nk[s] - 1) & 1);
        if (nv[s]) mbar_wait_drain(&v_full[s], (nv[s] - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ===================== MMA issuer =======================================
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(kTileM, BK, 0, 0);
      const uint32_t idO = idesc_bf16_f32(kTileM, D, 0, 1);
      const uint32_t tS0 = tmem, tS1 = tmem + BK, tO = tmem + 2 * BK;
      const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK);
      const uint32_t v_addr = smem_u32(sV), p_addr = smem_u32(sP);
      bool ok = mbar_wait(q_full, 0, kSiteQFull, abort_flag);
      tc_fence_after();
      auto issue_s = [&](int j) -> bool {
        const int s = j % kStages;
        if (!mbar_wait(&k_full[s], (j / kStages) & 1, kSiteKFull, abort_flag)) return false;
        tc_fence_after();
        const uint32_t dst = (j & 1) ? tS1 : tS0;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t a = smem_desc_sw128(q_addr + (ks / 4) * kTileM * 128 + (ks % 4) * 32, 16, 1024);
          const uint64_t b = smem_desc_sw128(
              k_addr + s * Lay::kKVBytes + (ks / 4) * BK * 128 + (ks % 4) * 32, 16, 1024);
          mma_bf16_ss(dst, a, b, idS, ks > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[j & 1]);
        mma_commit(&k_empty[s]);
        return true;
      };
      if (ok && n_iter > 0) ok = issue_s(0);
      for (int j = 0; ok && j < n_iter; ++j) {
        if (j + 1 < n_iter && !(ok = issue_s(j + 1))) break;
        if (!(ok = mbar_wait(p_full, j & 1, kSitePFull, abort_flag))) break;
        const int s = j % kStages;
        if (!(ok = mbar_wait(&v_full[s], (j / kStages) & 1, kSiteVFull, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
          const uint64_t a = smem_desc_sw128(p_addr + (ks / 4) * kTileM * 128 + (ks % 4) * 32, 16, 1024);
          const uint64_t b = smem_desc_sw128(v_addr + s * Lay::kKVBytes + ks * 16 * 128, BK * 128, 1024);
          mma_bf16_ss(tO, a, b, idO, (j > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(o_done);
        mma_commit(&v_empty[s]);
      }
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else if (warp >= 4) {
    // ===================== softmax + epilogue ===============================
    const int r = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS0 = tmem + lane_base, tS1 = tS0 + BK, tO = tS0 + 2 * BK;
    const int row_sorted = tile * kTileM + r;
    const bool row_valid = row_sorted < p.L;
    const int my_g = r / BK;
    // l: sum of the exact fp32 weights (for the LSE); lr: sum of the
    // bf16-rounded weights the PV product consumes (normalises O, so O is an
    // exact convex combination of V rows up to fp32 accumulation)
    float m_used = -INFINITY, l = 0.f, lr = 0.f;
    bool ok = true;
    for (int j = 0; j < n_iter; ++j) {
      const uint32_t e = p.dense ? (static_cast<uint32_t>(j) | (3u << 12)) : list[j];
      const int blk = e & 0xFFF;
      const bool use = row_valid && ((e >> (12 + my_g)) & 1u);
      ok = mbar_wait(&s_full[j & 1], (j >> 1) & 1, kSiteSFull, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float sv[BK];
#pragma unroll
      for (int c = 0; c < BK / 32; ++c) tmem_ld32(((j & 1) ? tS1 : tS0) + c * 32, sv + c * 32);
      tmem_wait_ld();
      const int valid_cols = min(BK, p.L - blk * BK);
      float mx = -INFINITY;
      if (use) {
#pragma unroll
        for (int c = 0; c < BK; ++c)
          if (c < valid_cols) mx = fmaxf(mx, sv[c]);
      }
      const float m_cand = fmaxf(m_used, mx * p.scale_log2);
      if (j > 0) {
        ok = mbar_wait(o_done, (j - 1) & 1, kSiteODone, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      const bool need = m_cand > m_used + kRescaleLog2;
      const bool resc = need && (m_used != -INFINITY);
      float alpha = 1.f;
      if (need) {
        alpha = resc ? fast_exp2(m_used - m_cand) : 0.f;
        l *= alpha;
        lr *= alpha;
        m_used = m_cand;
      }
      if (__any_sync(0xffffffffu, resc)) {
        const float f = resc ? alpha : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float ov[32];
          tmem_ld32(tO + c * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] *= f;
          tmem_st32(tO + c * 32, ov);
        }
        tmem_wait_st();
      }
      // P_j (bf16) into shared memory, 128-byte swizzled, K-major
#pragma unroll
      for (int u16 = 0; u16 < BK / 8; ++u16) {
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = u16 * 8 + i;
          x[i] = (use && c < valid_cols) ? fast_exp2(fmaf(sv[c], p.scale_log2, -m_used)) : 0.f;
          l += x[i];
        }
        uint4 w;
        w.x = pack_bf16(x[0], x[1]);
        w.y = pack_bf16(x[2], x[3]);
        w.z = pack_bf16(x[4], x[5]);
        w.w = pack_bf16(x[6], x[7]);
        lr += bf16_lo(w.x) + bf16_hi(w.x) + bf16_lo(w.y) + bf16_hi(w.y) + bf16_lo(w.z) +
             bf16_hi(w.z) + bf16_lo(w.w) + bf16_hi(w.w);
        const int chunk = u16 / 8, u = u16 % 8;
        *reinterpret_cast<uint4 *>(sP + chunk * kTileM * 128 + r * 128 + ((u ^ (r & 7)) << 4)) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok && n_iter > 0) {
      ok = mbar_wait(o_done, (n_iter - 1) & 1, kSiteODone, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const int64_t orig = row_valid ? (p.perm_q ? p.perm_q[static_cast<int64_t>(bh) * p.L + row_sorted]
                                                 : row_sorted)
                                     : 0;
      const float inv_l = (lr > 0.f) ? 1.f / lr : 0.f;
      uint4 *orow = reinterpret_cast<uint4 *>(p.o + (static_cast<int64_t>(bh) * p.L + orig) * D);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float ov[32];
        tmem_ld32(tO + c * 32, ov);
        tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16(ov[q4 * 8 + 0] * inv_l, ov[q4 * 8 + 1] * inv_l);
            w.y = pack_bf16(ov[q4 * 8 + 2] * inv_l, ov[q4 * 8 + 3] * inv_l);
            w.z = pack_bf16(ov[q4 * 8 + 4] * inv_l, ov[q4 * 8 + 5] * inv_l);
            w.w = pack_bf16(ov[q4 * 8 + 6] * inv_l, ov[q4 * 8 + 7] * inv_l);
            orow[c * 4 + q4] = w;
          }
        }
      }
      if (row_valid)
        p.lse[static_cast<int64_t>(bh) * p.L + orig] = (m_used + log2f(l)) * 0.69314718055994531f;
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

// ---------------------------------------------------------------------------
// row gather: out[bh, r, :] = in[bh, perm[bh, r], :]   (K and V share perm_k)
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) k_permute_rows(const __nv_bfloat16 *__restrict__ in0,
                                                      const __nv_bfloat16 *__restrict__ in1,
                                                      const int32_t *__restrict__ perm,
                                                      __nv_bfloat16 *__restrict__ out0,
                                                      __nv_bfloat16 *__restrict__ out1,
                                                      int64_t rows, int L) {
  constexpr int VPR = D / 8;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gid / VPR;
  const int c = static_cast<int>(gid % VPR);
  if (row >= rows) return;
  const int64_t bh = row / L;
  const int64_t src = bh * L + __ldg(perm + row);
  reinterpret_cast<uint4 *>(out0 + row * D)[c] =
      __ldg(reinterpret_cast<const uint4 *>(in0 + src * D) + c);
  if (in1 != nullptr)
    reinterpret_cast<uint4 *>(out1 + row * D)[c] =
        __ldg(reinterpret_cast<const uint4 *>(in1 + src * D) + c);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

cudaError_t take_attn_error_word(uint32_t *word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(uint32_t));
}

size_t attn_workspace_bytes(int64_t bh, int L, int D, bool perm_q, bool perm_k) {
  const size_t t = align256(static_cast<size_t>(bh) * L * D * 2);
  return (perm_q ? t : 0) + (perm_k ? 2 * t : 0);
}

template <int D, int BK>
static cudaError_t launch_attn(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                               const AttnParams &p, int64_t bh, cudaStream_t st) {
  using Lay = AttnLayout<D, BK>;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(k_attn<D, BK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay::kAlloc);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const dim3 grid((p.L + kTileM - 1) / kTileM, static_cast<unsigned>(bh));
  k_attn<D, BK><<<grid, kAttnThreads, Lay::kAlloc, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

cudaError_t run_attention(const AttnArgs &a, cudaStream_t st) {
  const int64_t bh = static_cast<int64_t>(a.batch) * a.heads;
  const int L = a.seqlen, D = a.head_dim;
  const bool dense = a.block_idx == nullptr;
  const int BK = dense ? 128 : a.block;
  const int64_t rows = bh * L;
  const void *qs = a.q, *ks = a.k, *vs = a.v;
  unsigned char *ws = static_cast<unsigned char *>(a.workspace);
  const size_t t = align256(static_cast<size_t>(rows) * D * 2);
  cudaError_t e;
  if (a.perm_q) {
    __nv_bfloat16 *qp = reinterpret_cast<__nv_bfloat16 *>(ws);
    ws += t;
    const int64_t threads = rows * (D / 8);
    const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
    if (D == 128)
      k_permute_rows<128><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(a.q), nullptr,
                                                a.perm_q, qp, nullptr, rows, L);
    else
      k_permute_rows<64><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(a.q), nullptr,
                                               a.perm_q, qp, nullptr, rows, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    qs = qp;
  }
  if (a.perm_k) {
    __nv_bfloat16 *kp = reinterpret_cast<__nv_bfloat16 *>(ws);
    __nv_bfloat16 *vp = reinterpret_cast<__nv_bfloat16 *>(ws + t);
    const int64_t threads = rows * (D / 8);
    const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
    if (D == 128)
      k_permute_rows<128><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(a.k),
                                                static_cast<const __nv_bfloat16 *>(a.v), a.perm_k,
                                                kp, vp, rows, L);
    else
      k_permute_rows<64><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(a.k),
                                               static_cast<const __nv_bfloat16 *>(a.v), a.perm_k,
                                               kp, vp, rows, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ks = kp;
    vs = vp;
  }
  alignas(64) CUtensorMap mq, mk, mv;
  if ((e = encode_tensor_map_3d(&mq, qs, D, L, bh, 64, kTileM)) != cudaSuccess) return e;
  if ((e = encode_tensor_map_3d(&mk, ks, D, L, bh, 64, BK)) != cudaSuccess) return e;
  if ((e = encode_tensor_map_3d(&mv, vs, D, L, bh, 64, BK)) != cudaSuccess) return e;

  AttnParams p;
  p.L = L;
  p.N = (L + BK - 1) / BK;
  p.kappa = dense ? p.N : a.kappa;
  p.dense = dense ? 1 : 0;
  p.block_idx = a.block_idx;
  p.perm_q = a.perm_q;
  p.o = static_cast<__nv_bfloat16 *>(a.o);
  p.lse = a.lse;
  const float scale = (a.scale > 0.f) ? a.scale : 1.0f / sqrtf(static_cast<float>(D));
  p.scale_log2 = scale * 1.4426950408889634f;

  if (D == 128 && BK == 128) return launch_attn<128, 128>(mq, mk, mv, p, bh, st);
  if (D == 128 && BK == 64) return launch_attn<128, 64>(mq, mk, mv, p, bh, st);
  if (D == 64 && BK == 128) return launch_attn<64, 128>(mq, mk, mv, p, bh, st);
  if (D == 64 && BK == 64) return launch_attn<64, 64>(mq, mk, mv, p, bh, st);
  return cudaErrorInvalidValue;
}

}  // namespace ba
