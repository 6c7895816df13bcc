// Block-sparse attention forward for sm_103a: BA-Att paper Algorithm 1
// step 12 ("Efficient Long-Context Modeling in Diffusion Language Models via
// Block Approximate Sparse Attention"), with the masked softmax of SparseD
// §3.1 Eq. 3-4, and the same kernel run dense (Eq. 1).
//
// A CTA owns two tiles of 128 consecutive sorted query rows.  A tile is one
// query block when B = 128, two when B = 64 (then it walks the union of the
// two lists, each entry tagged with which block selected it; rows of the
// other block see -inf for that entry).  Key blocks are always consumed as
// 128-key slots: with B = 64 two list entries share a slot (two 64-row
// boxes), so every iteration has the shape of the B = 128 path.
//
// Warp roles (384 threads; setmaxnreg moves registers to the softmax warps):
//   warp 0       TMA producer: both Q tiles once, then every K_j and V_j
//                block the MMA thread will consume, in that order, into one
//                ring of shared-memory slots (128-byte swizzle, 64-column
//                boxes, 3-D maps so a ragged last block reads zeros instead
//                of the next head).  Dense mode: both tiles walk the same
//                blocks, so each load serves both.
//   warp 1       tensor-memory allocation and the single MMA-issuing thread:
//                  S_t = Q_t K_j^T        -> TMEM (one S buffer per tile)
//                  O_t += P_t V_j         -> TMEM, P_t read from TMEM as the A
//                                            operand, V as an MN-major operand
//                alternating tiles so the tensor core works on one tile
//                while the other tile's softmax runs.  S_t(j+1) is issued
//                right after PV_t(j) and overwrites P_t in place (tcgen05 MMAs
//                of one thread execute in order).  Descriptors are
//                precomputed 32-bit words plus one add per MMA.
//   warp 2 (3)   row gathers of Q', K', V' for this head's unclaimed slices
//                and one slice of a later head (warps 2-3 in the packed
//                64-token-block kernel).
//   warp 3       (unpacked kernels) stage confirmer: waits for the K/V copies
//                of each tile's next PV and S and adds the last arrival of
//                that tile's P-ready barrier, so the MMA thread waits on one
//                barrier per tile and iteration.
//   warps 4-7,   softmax + epilogue for tile 0 and tile 1: thread r owns row r
//   warps 8-11   (TMEM lane r).  Online softmax in the log2 domain with a lazy
//                rescale: O_t is corrected only when the running max grows by
//                more than 2^8, and then without waiting (PV_t(j-1) completed
//                before S_t(j) did).  P (bf16 pairs) is stored over S_t.  At
//                the end O / l is written as bf16 to the ORIGINAL row pi_q(r),
//                and LSE = ln(sum exp(scale q.k)).
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

constexpr int kTileM = 128;          // query rows per tile (TMEM lanes)
constexpr int kTiles = 2;            // query tiles per CTA (ping-pong)
constexpr int kAttnThreads = 384;    // 12 warps
// Registers per thread after setmaxnreg: warps 0-3 drop to kLow, warps 4-11
// rise to kHigh; 4*32*kLow + 8*32*kHigh must equal the launch's 384*168.
template <int BK> struct RegSplit { static constexpr int kLow = 72, kHigh = 216; };
static_assert(4 * 32 * RegSplit<128>::kLow + 8 * 32 * RegSplit<128>::kHigh == 384 * 168, "split");
constexpr int kSplitRegs(int lo, int hi) { return 4 * 32 * lo + 8 * 32 * hi; }
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

constexpr int next_pow2_cols(int x) {
  int c = 32;
  while (c < x) c <<= 1;
  return c;
}
constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int D, int BK>
struct AttnLayout {
  static constexpr int kG = kTileM / BK;               // query blocks per tile
  static constexpr int kQBytes = kTileM * D * 2;       // one Q tile
  static constexpr int kSlotBytes = BK * D * 2;        // one K or V block
  static constexpr int kListBytes = 0;  // tile lists are read from global memory
  static constexpr int kBarBytes = 512;
  static constexpr int kMaxDyn = 227 * 1024;
  static constexpr int kSlots =
      cmin(8, (kMaxDyn - 1024 - kBarBytes - kListBytes - kTiles * kQBytes) / kSlotBytes);
  static constexpr int kOffQ = 0;
  static constexpr int kOffSlots = kOffQ + kTiles * kQBytes;
  static constexpr int kOffList = kOffSlots + kSlots * kSlotBytes;
  static constexpr int kOffBar = kOffList + kListBytes;
  static constexpr int kBytes = kOffBar + kBarBytes;
  static constexpr int kTmemCols = next_pow2_cols(kTiles * (BK + D));
  // No more CTAs may share an SM than its 512 tensor-memory columns can hold.
  static constexpr int kMaxCtasByTmem = 512 / kTmemCols;
  static constexpr int kMinAlloc = (228 * 1024) / (kMaxCtasByTmem + 1) + 1024;
  static constexpr int kAlloc = (kBytes + 1024 > kMinAlloc) ? kBytes + 1024 : kMinAlloc;
  static_assert(kSlots >= 3, "shared memory ring too small");
  static_assert(kTmemCols <= 512, "tensor memory budget");
  static_assert(kAlloc <= kMaxDyn, "shared memory budget");
};

struct AttnParams {
  int L;          // tokens per sequence
  int N;          // key blocks (and query blocks) of size BK
  int kappa;      // list length per query block (unused when dense)
  int n_tiles;    // 128-row query tiles per sequence
  int npairs;     // CTAs (tile pairs) per sequence
  const uint16_t *pair_lists;  // [b*h][npairs][2][N]: per tile, common blocks first
  const int32_t *pair_counts;  // [b*h][npairs][4]: n0, n1, common, -
  const int32_t *perm_q;  // sorted query position -> original row (nullable)
  // Row gathers inside the kernel by warp 2 (unpacked) or warps 2-3
  // (packed) (claim != nullptr): head h's
  // rows are cut into nslices slices of slice_rows rows.  A slice is claimed
  // with an atomic ticket on claim[h] and counted in done[h] once written.
  // CTAs of head h - lookahead each claim one slice ahead of time, and CTAs
  // of head h claim every slice still unclaimed when they start, so a CTA
  // waits only on slices that running CTAs hold, whatever order the CTAs
  // are dispatched in.  Heads < lookahead were gathered by a kernel launched
  // before.
  const int32_t *perm_k;
  const __nv_bfloat16 *src_q, *src_k, *src_v;  // unpermuted inputs
  __nv_bfloat16 *dst_q, *dst_k, *dst_v;        // Q' (or null), K' and V' (or null)
  int *claim;
  int *done;
  int lookahead;
  int bh_total;
  int slice_rows;
  int nslices;
  __nv_bfloat16 *o;
  float *lse;
  float scale_log2;          // scale * log2(e)
  uint64_t issuer_wait_ns;   // wait limit of the MMA thread (the other roles: 2 s)
  int skip_load;             // failure-path test only: this K/V load is never issued; -1 otherwise
};

// A key-block entry: bits 0-11 block id, bit 12+g set when query block g of
// the tile selected it.  Sparse tiles read their entries from the pair list
// (k_pair_lists); dense tiles walk every block.
__device__ __forceinline__ uint32_t dense_entry(int j) { return static_cast<uint32_t>(j) | (3u << 12); }

// Copies rows [r_begin, r_end) of one head through a permutation into the
// gathered layout, for one tensor (s1 == nullptr) or for two that share it
// (K and V).  A thread owns 16 bytes of kU rows per step.  While a step's
// rows are in flight the thread loads the next step's permutation entries
// and asks L2 for the next step's rows (prefetches hold no register), and
// the entries two steps ahead are prefetched too, so a step mostly waits
// for L2, not for an index load followed by a DRAM row load.
template <int D, int kGatherThreads, int kU>
__device__ __forceinline__ void copy_rows(const __nv_bfloat16 *s0, const __nv_bfloat16 *s1,
                                          __nv_bfloat16 *d0, __nv_bfloat16 *d1, const int32_t *perm,
                                          int r_begin, int r_end, int L, int tid) {
  constexpr int VPR = D / 8;                 // 16-byte pieces per row
  constexpr int RPP = kGatherThreads / VPR;  // rows per pass of the gather threads
  constexpr int kStep = RPP * kU;
  const int c = tid % VPR;
  const int rs = r_begin + tid / VPR;
  // pointers of this head and piece; row offsets fit 32 bits (L * D < 2^31)
  const uint4 *x0 = reinterpret_cast<const uint4 *>(s0) + c;
  const uint4 *x1 = reinterpret_cast<const uint4 *>(s1) + c;
  uint4 *y0 = reinterpret_cast<uint4 *>(d0) + c;
  uint4 *y1 = reinterpret_cast<uint4 *>(d1) + c;
  int src[kU];
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int row = rs + u * RPP;
    src[u] = (row < r_end) ? min(max(__ldg(perm + row), 0), L - 1) : 0;
  }
  for (int r0 = rs; r0 < r_end; r0 += kStep) {
    uint4 a[kU], b[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (r0 + u * RPP < r_end) {
        a[u] = __ldg(x0 + src[u] * VPR);
        if (s1 != nullptr) b[u] = __ldg(x1 + src[u] * VPR);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {  // the next step's indices, in flight with the rows
      const int row = r0 + kStep + u * RPP;
      src[u] = (row < r_end) ? min(max(__ldg(perm + row), 0), L - 1) : 0;
    }
    if (c == 0 && r0 + 2 * kStep < r_end) prefetch_l2(perm + r0 + 2 * kStep);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (r0 + kStep + u * RPP < r_end) {
        prefetch_l2(x0 + src[u] * VPR);
        if (s1 != nullptr) prefetch_l2(x1 + src[u] * VPR);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int row = r0 + u * RPP;
      if (row < r_end) {
        y0[row * VPR] = a[u];
        if (s1 != nullptr) y1[row * VPR] = b[u];
      }
    }
  }
}

// One CTA's share of the row gathers of head hp: slice `pair` of Q' (through
// pi_q) and of K' and V' (through pi_k, one index load for both rows).
template <int D, int kGatherThreads>
__device__ __forceinline__ void gather_slice(const AttnParams &p, int hp, int pair, int tid) {
  const int64_t base = static_cast<int64_t>(hp) * p.L;
  const int64_t xb = base * D;
  const int r_begin = pair * p.slice_rows;
  const int r_end = min(p.L, r_begin + p.slice_rows);
  if (p.dst_q != nullptr)
    copy_rows<D, kGatherThreads, 2>(p.src_q + xb, nullptr, p.dst_q + xb, nullptr, p.perm_q + base, r_begin,
                                    r_end, p.L, tid);
  if (p.dst_k != nullptr)
    copy_rows<D, kGatherThreads, 2>(p.src_k + xb, p.dst_v != nullptr ? p.src_v + xb : nullptr, p.dst_k + xb,
                                    p.dst_v != nullptr ? p.dst_v + xb : nullptr, p.perm_k + base, r_begin, r_end,
                                    p.L, tid);
}

// Gathers run on kGatherThreads threads (one warp, or warps 2-3): a named
// barrier (id 1) of those threads, a ticket broadcast through shared memory.
template <int kGatherThreads>
__device__ __forceinline__ void gather_sync() {
  if (kGatherThreads == 32)
    __syncwarp();
  else
    asm volatile("bar.sync 1, %0;" ::"n"(kGatherThreads) : "memory");
}

// One ticket from `counter`, broadcast to the gather threads.
template <int kGatherThreads>
__device__ __forceinline__ int claim_slice(int *counter, volatile int *bcast, int tid) {
  if constexpr (kGatherThreads == 32) {
    int s = 0;
    if (tid == 0) s = atomicAdd(counter, 1);
    return __shfl_sync(0xffffffffu, s, 0);
  } else {
    if (tid == 0) *bcast = atomicAdd(counter, 1);
    gather_sync<kGatherThreads>();
    const int s = *bcast;
    gather_sync<kGatherThreads>();  // every thread has read it before the next ticket overwrites it
    return s;
  }
}

// Publish a written slice: after the barrier, one thread orders every gather
// thread's stores before its count (fence cumulativity) and counts the slice.
template <int kGatherThreads>
__device__ __forceinline__ void publish_slice(int *done, int tid) {
  gather_sync<kGatherThreads>();
  if (tid == 0) {
    __threadfence();
    atomicAdd(done, 1);
  }
  if (kGatherThreads == 32) __syncwarp();
}

template <int D, int BK, bool kDense, bool kPack>
__global__ void __launch_bounds__(kAttnThreads, 1)
    k_attn(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using Lay = AttnLayout<D, BK>;
  constexpr int S = Lay::kSlots;
  // Unpacked kernels (dense; 128-token blocks): warp 3 confirms every K/V
  // copy and adds the last arrival of P-ready, so the MMA thread waits on
  // P-ready alone, and warp 2 gathers rows.  Packed kernels (64-token
  // blocks): the MMA thread waits for each copy itself and warps 2-3 gather
  // (their CTAs are short, and one gather warp fell behind: 0.53 -> 1.13 ms
  // on the LLaDA shape).
  constexpr bool kConfirm = !kPack;
  constexpr int kGatherThreads = kConfirm ? 32 : 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + Lay::kOffQ;
  uint8_t *sSlot = smem + Lay::kOffSlots;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kOffBar);
  uint64_t *q_full = bars;
  uint64_t *slot_full = bars + 1;
  uint64_t *slot_empty = slot_full + S;
  uint64_t *s_full = slot_empty + S;   // [kTiles]
  uint64_t *p_full = s_full + kTiles;  // [kTiles]
  uint64_t *o_done = p_full + kTiles;  // [kTiles]
  uint64_t *drain = o_done + kTiles;
  uint32_t *misc = reinterpret_cast<uint32_t *>(drain + 1);  // tmem, n0, n1, abort, common, ticket
  volatile int *abort_flag = reinterpret_cast<volatile int *>(&misc[3]);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tile0 = blockIdx.x * kTiles;
  const int bh = blockIdx.y;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&slot_full[s], 1);
      mbar_init(&slot_empty[s], 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], kTileM + (kConfirm ? 1 : 0));  // the tile's softmax threads (and the confirmer)
      mbar_init(&o_done[t], 1);
    }
    mbar_init(drain, 1);
    misc[3] = 0;  // abort flag; misc[1], misc[2], misc[4] are the counts below
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&misc[0], Lay::kTmemCols);
    tc_fence_before();
  }

  // ---- per-tile entry counts ----------------------------------------------
  const int pair = blockIdx.x;
  const uint16_t *plist[kTiles];
  for (int t = 0; t < kTiles; ++t)
    plist[t] = kDense ? nullptr
                      : p.pair_lists + ((static_cast<int64_t>(bh) * p.npairs + pair) * kTiles + t) * p.N;
  if (threadIdx.x <= kTiles) {
    if (kDense) {
      if (threadIdx.x < kTiles)
        misc[1 + threadIdx.x] = (tile0 + static_cast<int>(threadIdx.x) < p.n_tiles) ? p.N : 0;
    } else {
      const int32_t *cnt = p.pair_counts + (static_cast<int64_t>(bh) * p.npairs + pair) * 4;
      misc[threadIdx.x < kTiles ? 1 + threadIdx.x : 4] = cnt[threadIdx.x];
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  // Packed mode (64-token blocks): list entries are taken two at a time, one
  // 128-key slot holding the two 64-key blocks, so iteration j covers
  // entries 2j and 2j + 1 (the second is a fully masked dummy past the end).
  const int ne[kTiles] = {static_cast<int>(misc[1]), static_cast<int>(misc[2])};
  const int n_t[kTiles] = {kPack ? (ne[0] + 1) / 2 : ne[0], kPack ? (ne[1] + 1) / 2 : ne[1]};
  const int nmax = max(n_t[0], n_t[1]);
  // Positions j < n_common hold the same block(s) in both tiles' lists
  // (dense: every position), so the K_j / V_j load is shared there.
  const int n_common = kDense ? (n_t[1] > 0 ? n_t[0] : 0)
                              : (kPack ? static_cast<int>(misc[4]) / 2 : static_cast<int>(misc[4]));

  if (warp < 4) {
    reg_dealloc<RegSplit<BK>::kLow>();
    if (warp == 0 && lane == 0) {
      // ===================== TMA producer ===================================
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      // this head's Q', K', V' rows: every slice is held by a running CTA; a
      // wait that runs out aborts the CTA before any load (nothing is
      // computed from rows that were not written)
      bool rows_ok = true;
      if (p.claim != nullptr && bh >= p.lookahead) {
        rows_ok = wait_counter_at_least(p.done + bh, p.nslices, kSiteRowsReady);
        if (!rows_ok) *abort_flag = 1;
      }
      uint32_t loaded = 0u, parity = 0u;  // per ring slot: ever loaded, parity of its loads
      if (rows_ok) {
      uint32_t qbytes = 0;
      for (int t = 0; t < kTiles; ++t) qbytes += n_t[t] > 0 ? Lay::kQBytes : 0;
      mbar_arrive_expect_tx(q_full, qbytes);
      for (int t = 0; t < kTiles; ++t) {
        if (n_t[t] == 0) continue;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sQ + t * Lay::kQBytes + c * kTileM * 128, &tmQ, q_full, c * 64,
                      (tile0 + t) * kTileM, bh);
      }
      int issued = 0;
      auto load = [&](bool is_v, int t, int j) -> bool {
        int blk, blk_b = 0;
        if (kPack) {
          blk = plist[t][2 * j] & 0xFFF;
          blk_b = (2 * j + 1 < ne[t]) ? (plist[t][2 * j + 1] & 0xFFF) : blk;
        } else {
          blk = kDense ? j : (plist[t][j] & 0xFFF);
        }
        const int s = issued % S;
        if (issued >= S && !mbar_wait(&slot_empty[s], ((issued / S) & 1) ^ 1u, kSiteKEmpty, abort_flag))
          return false;
        if (issued == p.skip_load) {  // failure-path test: this copy never happens
          ++issued;
          return true;
        }
        mbar_arrive_expect_tx(&slot_full[s], Lay::kSlotBytes);
        loaded |= 1u << s;
        parity ^= 1u << s;
        const CUtensorMap *map = is_v ? &tmV : &tmK;
        uint8_t *dst = sSlot + s * Lay::kSlotBytes;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          if (kPack) {
            // rows 0-63 from block a, rows 64-127 from block b (64-row boxes)
            tma_load_3d(dst + c * BK * 128, map, &slot_full[s], c * 64, blk * (BK / 2), bh);
            tma_load_3d(dst + c * BK * 128 + (BK / 2) * 128, map, &slot_full[s], c * 64,
                        blk_b * (BK / 2), bh);
          } else {
            tma_load_3d(dst + c * BK * 128, map, &slot_full[s], c * 64, blk * BK, bh);
          }
        }
        ++issued;
        return true;
      };
      // the same operand order in which the MMA thread consumes the slots
      bool ok = true;
      for (int t = 0; ok && t < kTiles; ++t)
        if (n_t[t] > 0 && !(t == 1 && 0 < n_common)) ok = load(false, t, 0);
      for (int j = 0; ok && j < nmax; ++j)
        for (int t = 0; ok && t < kTiles; ++t) {
          if (j >= n_t[t]) continue;
          if (!(t == 1 && j < n_common)) ok = load(true, t, j);
          if (ok && j + 1 < n_t[t] && !(t == 1 && j + 1 < n_common)) ok = load(false, t, j + 1);
        }
      // drain: the last copy issued into each slot has landed
      mbar_wait_drain(q_full, 0);
      }
      for (int s = 0; s < S; ++s)
        if ((loaded >> s) & 1u) mbar_wait_drain(&slot_full[s], ((parity >> s) & 1u) ^ 1u);
    } else if (warp == 1 && lane == 0) {
      // ===================== MMA issuer =====================================
      const uint32_t idS = idesc_bf16_f32(kTileM, BK, 0, 0);
      const uint32_t idO = idesc_bf16_f32(kTileM, D, 0, 1);
      const uint32_t q_addr = smem_u32(sQ), slot_addr = smem_u32(sSlot);
      int consumed = 0;
      const uint64_t lim = p.issuer_wait_ns;
      bool ok = mbar_wait(q_full, 0, kSiteQFull, abort_flag, lim);
      tc_fence_after();
      // prologue takes wait for their K copies here; in the loop of an
      // unpacked kernel a slot's copy is confirmed by the stage confirmer
      // (warp 3) before its P-ready arrival, so the P wait covers it
      auto take_wait = [&](int &slot) -> bool {
        slot = consumed % S;
        if (!mbar_wait(&slot_full[slot], (consumed / S) & 1, kSiteKFull, abort_flag, lim)) return false;
        tc_fence_after();
        ++consumed;
        return true;
      };
      auto take = [&](int &slot) -> bool {
        if (!kConfirm) return take_wait(slot);
        slot = consumed % S;
        ++consumed;
        return true;
      };
      // K-major Q and K (stride 1024 between 8-row groups), MN-major V
      // (leading offset = one 64-column chunk of a slot): each MMA adds a
      // constant to a precomputed low descriptor word, one add per operand on
      // the issuing thread's path instead of a full encoding
      constexpr uint32_t kHi = desc_sw128_hi(1024);
      const uint32_t q_lo = desc_sw128_lo(q_addr, 16);
      const uint32_t k_lo = desc_sw128_lo(slot_addr, 16);
      const uint32_t v_lo = desc_sw128_lo(slot_addr, BK * 128);
      auto mma_s = [&](int t, int slot) {
        const uint32_t a0 = q_lo + ((t * Lay::kQBytes) >> 4);
        const uint32_t b0 = k_lo + ((slot * Lay::kSlotBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t oa = ((ks / 4) * kTileM * 128 + (ks % 4) * 32) >> 4;
          const uint32_t ob = ((ks / 4) * BK * 128 + (ks % 4) * 32) >> 4;
          mma_ss_words<false>(tmem + t * BK, a0 + oa, b0 + ob, kHi, idS, ks > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[t]);
      };
      auto mma_pv = [&](int t, int slot, int j) {
        const uint32_t b0 = v_lo + ((slot * Lay::kSlotBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks)
          mma_ts_words<false>(tmem + kTiles * BK + t * D, tmem + t * BK + ks * 8, b0 + ((ks * 16 * 128) >> 4), kHi,
                              idO, (j > 0 || ks > 0) ? 1u : 0u);
      };
      int slot_k0 = 0, slot_v0 = 0;  // shared positions: slots loaded for tile 0, reused by tile 1
      for (int t = 0; ok && t < kTiles; ++t) {
        if (n_t[t] == 0) continue;
        const bool sh = 0 < n_common;
        int sl = slot_k0;
        if (!(sh && t == 1) && !(ok = take_wait(sl))) break;
        mma_s(t, sl);
        if (!sh || t == 1) mma_commit(&slot_empty[sl]);
        else slot_k0 = sl;
      }
      for (int j = 0; ok && j < nmax; ++j) {
        for (int t = 0; ok && t < kTiles; ++t) {
          if (j >= n_t[t]) continue;
          if (!(ok = mbar_wait(&p_full[t], j & 1, kSitePFull, abort_flag, lim))) break;
          tc_fence_after();
          const bool shv = j < n_common;
          int sv = slot_v0;
          if (!(shv && t == 1) && !(ok = take(sv))) break;
          mma_pv(t, sv, j);
          if (j + 1 == n_t[t]) mma_commit(&o_done[t]);
          if (!shv || t == 1) mma_commit(&slot_empty[sv]);
          else slot_v0 = sv;
          if (j + 1 < n_t[t]) {
            const bool shk = j + 1 < n_common;
            int sk = slot_k0;
            if (!(shk && t == 1) && !(ok = take(sk))) break;
            mma_s(t, sk);
            if (!shk || t == 1) mma_commit(&slot_empty[sk]);
            else slot_k0 = sk;
          }
        }
      }
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    } else if ((warp == 2 || (!kConfirm && warp == 3)) && p.claim != nullptr) {
      // ===================== row gathers ====================================
      const int tid = threadIdx.x - 64;
      volatile int *bcast = reinterpret_cast<volatile int *>(&misc[5]);
      if (bh >= p.lookahead) {
        // slices of this CTA's own head that nobody has claimed yet
        for (;;) {
          const int s = claim_slice<kGatherThreads>(p.claim + bh, bcast, tid);
          if (s >= p.nslices) break;
          gather_slice<D, kGatherThreads>(p, bh, s, tid);
          publish_slice<kGatherThreads>(p.done + bh, tid);
        }
      }
      // one slice of a later head, ahead of time
      const int hp = bh + p.lookahead;
      if (hp < p.bh_total) {
        const int s = claim_slice<kGatherThreads>(p.claim + hp, bcast, tid);
        if (s < p.nslices) {
          gather_slice<D, kGatherThreads>(p, hp, s, tid);
          publish_slice<kGatherThreads>(p.done + hp, tid);
        }
      }
    } else if (kConfirm && warp == 3 && lane == 0 && nmax > 0) {
      // ===================== stage confirmer ================================
      // Replays the MMA thread's order of slot takes; for each tile and
      // iteration j it waits for the copies of the slots PV_t(j) and S_t(j+1)
      // read (V_t(j), K_t(j+1)) and adds the last arrival the tile's P-ready
      // barrier needs, so the MMA thread waits on P-ready alone.  Slots both
      // tiles share are taken (and confirmed) by tile 0, whose group the MMA
      // thread issues first.  It arrives for iteration j only after the
      // barrier's phase of iteration j - 1 has completed.
      int taken = (n_common > 0) ? 1 : ((n_t[0] > 0) + (n_t[1] > 0));  // prologue takes (K_t(0))
      bool ok = true;
      for (int j = 0; ok && j < nmax; ++j) {
        int i = taken;
        const int v0 = (j < n_t[0]) ? i++ : -1;
        const int k0 = (j + 1 < n_t[0]) ? i++ : -1;
        const int v1 = (j < n_t[1] && j >= n_common) ? i++ : -1;
        const int k1 = (j + 1 < n_t[1] && j + 1 >= n_common) ? i++ : -1;
        taken = i;
        for (int t = 0; ok && t < kTiles; ++t) {
          if (j >= n_t[t]) continue;
          const int a = t == 0 ? v0 : v1, b = t == 0 ? k0 : k1;
          if (a >= 0) ok = mbar_wait(&slot_full[a % S], (a / S) & 1, kSiteKFull, abort_flag);
          if (ok && b >= 0) ok = mbar_wait(&slot_full[b % S], (b / S) & 1, kSiteKFull, abort_flag);
          if (ok && j > 0) ok = mbar_wait(&p_full[t], (j - 1) & 1, kSitePFull, abort_flag);
          if (ok) mbar_arrive(&p_full[t]);
        }
      }
    }
  } else {
    reg_alloc<RegSplit<BK>::kHigh>();
    // ===================== softmax + epilogue, one warpgroup per tile =======
    const int t = (warp - 4) >> 2;
    const int r = threadIdx.x - 128 * (t + 1);
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * BK;
    const uint32_t tO = tmem + lane_base + kTiles * BK + t * D;
    const int row_sorted = (tile0 + t) * kTileM + r;
    const bool row_valid = row_sorted < p.L;
    const int my_g = r / (kPack ? BK / 2 : BK);
    const float cl = p.scale_log2;
    const uint64_t cl2 = f2_pack(cl, cl);
    float m = -INFINITY;
    uint64_t l2 = f2_pack(0.f, 0.f);  // running sum of the fp32 weights (two halves)
    // Sum of the bf16 rounding errors of every block's largest weight: the O
    // normaliser l + lcorr matches the weights the PV product consumed for
    // the terms that dominate a row (a row's largest weight is some block's
    // largest), so a row that attends to one key returns that key's value.
    float lcorr = 0.f;
    bool ok = true;
    const int n = n_t[t];
    // The softmax needs an entry only to mask: the other query block's
    // entries (64-row blocks) or the ragged last key block.  With 128-row
    // blocks every entry of a tile's list is its own, so when L is a multiple
    // of 128 the list is never read here.
    const bool read_list = !kDense && (kPack || BK < kTileM || p.L % BK != 0);
    uint32_t my_e = 0;  // sparse: 32 list entries at a time, one per lane
    for (int j = 0; j < n; ++j) {
      uint32_t e, eb = 0;
      if (kPack) {
        // entries 2j, 2j + 1; a missing second entry reads 0 (no selection bit)
        if ((j & 15) == 0) my_e = (2 * j + lane < ne[t]) ? __ldg(plist[t] + 2 * j + lane) : 0u;
        e = __shfl_sync(0xffffffffu, my_e, (2 * j) & 31);
        eb = __shfl_sync(0xffffffffu, my_e, (2 * j + 1) & 31);
      } else if (read_list) {
        if ((j & 31) == 0) my_e = (j + lane < n) ? __ldg(plist[t] + j + lane) : 0u;
        e = __shfl_sync(0xffffffffu, my_e, j & 31);
      } else {
        e = kDense ? dense_entry(j) : 0u;  // sparse: block 0, never the ragged one
      }
      const int blk = e & 0xFFF;
      const bool sel = (!kPack && BK == kTileM) || ((e >> (12 + my_g)) & 1u);
      // packed: columns [0, BK/2) belong to block a (e), [BK/2, BK) to block b (eb)
      const int bsz = kPack ? BK / 2 : BK;
      const int valid_cols = min(bsz, p.L - blk * bsz);
      const bool sel_b = kPack && ((eb >> (12 + my_g)) & 1u);
      const int valid_b = kPack ? min(bsz, p.L - static_cast<int>(eb & 0xFFF) * bsz) : 0;
      ok = mbar_wait(&s_full[t], j & 1, kSiteSFull, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float sv[BK];
#pragma unroll
      for (int c = 0; c < BK / 32; ++c) tmem_ld32(tS + c * 32, sv + c * 32);
      tmem_wait_ld();
      float mx, mx_b = -INFINITY;
      if (kPack) {
        if (!sel || valid_cols < bsz) {
#pragma unroll
          for (int c = 0; c < BK / 2; ++c)
            if (!sel || c >= valid_cols) sv[c] = -INFINITY;
        }
        if (!sel_b || valid_b < bsz) {
#pragma unroll
          for (int c = 0; c < BK / 2; ++c)
            if (!sel_b || c >= valid_b) sv[BK / 2 + c] = -INFINITY;
        }
        mx = sv[0];
#pragma unroll
        for (int c = 1; c + 1 < BK / 2; c += 2) mx = max3f(mx, sv[c], sv[c + 1]);
        mx = fmaxf(mx, sv[BK / 2 - 1]);
        mx_b = sv[BK / 2];
#pragma unroll
        for (int c = BK / 2 + 1; c + 1 < BK; c += 2) mx_b = max3f(mx_b, sv[c], sv[c + 1]);
        mx_b = fmaxf(mx_b, sv[BK - 1]);
      } else {
        if (!sel || valid_cols < BK) {
#pragma unroll
          for (int c = 0; c < BK; ++c)
            if (!sel || c >= valid_cols) sv[c] = -INFINITY;
        }
        mx = sv[0];
#pragma unroll
        for (int c = 1; c + 1 < BK; c += 2) mx = max3f(mx, sv[c], sv[c + 1]);
        mx = fmaxf(mx, sv[BK - 1]);
      }
      // the two blocks' maxima (packed) keep their own rounding corrections
      const float mx_a = mx;
      if (kPack) mx = fmaxf(mx, mx_b);
      const float m_new = fmaxf(m, mx * cl);
      const bool need = m_new > m + kRescaleLog2;
      const bool resc = need && (m != -INFINITY);
      float alpha = 1.f;
      if (need) {
        alpha = resc ? fast_exp2(m - m_new) : 0.f;
        const uint64_t a2 = f2_pack(alpha, alpha), z2 = f2_pack(0.f, 0.f);
        l2 = f2_fma(l2, a2, z2);
        lcorr *= alpha;
        m = m_new;
      }
      // lazy rescale of O_t: PV_{j-1} has completed (it was issued before
      // S_j, whose completion we just waited for); warp-collective accesses
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
      }
      const float nm = (m == -INFINITY) ? 0.f : -m;
      const uint64_t nm2 = f2_pack(nm, nm);
      {
        // computed exactly as this element's P entry below (same fma, ex2, RN)
        const float pbm = fast_exp2(fmaf(mx_a, cl, nm));
        lcorr += __bfloat162float(__float2bfloat16_rn(pbm)) - pbm;
        if (kPack) {
          const float pbb = fast_exp2(fmaf(mx_b, cl, nm));
          lcorr += __bfloat162float(__float2bfloat16_rn(pbb)) - pbb;
        }
      }
      // P_j overwrites the first BK/2 columns of S_j (bf16 pairs), 32 at a time
#pragma unroll
      for (int h = 0; h < BK / 64; ++h) {
        uint32_t pw[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = h * 64 + 2 * i;
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(sv[c], sv[c + 1]), cl2, nm2), x0, x1);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          const uint32_t w = pack_bf16(p0, p1);
          pw[i] = w;
          l2 = f2_add(l2, f2_pack(p0, p1));
        }
        tmem_st32u(tS + h * 32, pw);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[t]);
    }
    if (ok && n > 0) {
      ok = mbar_wait(&o_done[t], 0, kSiteODone, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok && n > 0) {
      tc_fence_after();
      float la, lb;
      f2_unpack(l2, la, lb);
      const float l = la + lb;
      // (an out-of-range permutation entry is clamped: wrong rows, never a
      // write outside this head's output)
      const int64_t orig =
          row_valid ? (p.perm_q ? min(max(p.perm_q[static_cast<int64_t>(bh) * p.L + row_sorted], 0), p.L - 1)
                                : row_sorted)
                    : 0;
      const float lo = l + lcorr;
      const float inv = (lo > 0.f) ? 1.f / lo : 0.f;
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
            w.x = pack_bf16(ov[q4 * 8 + 0] * inv, ov[q4 * 8 + 1] * inv);
            w.y = pack_bf16(ov[q4 * 8 + 2] * inv, ov[q4 * 8 + 3] * inv);
            w.z = pack_bf16(ov[q4 * 8 + 4] * inv, ov[q4 * 8 + 5] * inv);
            w.w = pack_bf16(ov[q4 * 8 + 6] * inv, ov[q4 * 8 + 7] * inv);
            orow[c * 4 + q4] = w;
          }
        }
      }
      if (row_valid)
        p.lse[static_cast<int64_t>(bh) * p.L + orig] = (m + log2f(l)) * 0.69314718055994531f;
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
// row gathers in one launch: out[job][bh, r, :] = in[job][bh, perm[job][bh, r], :]
// (Q through pi_q; K and V through pi_k).  grid = (.., jobs); each thread
// moves 16 bytes of kGatherRows rows, all loads in flight before the stores.
// ---------------------------------------------------------------------------
constexpr int kGatherRows = 4;

struct GatherJobs {
  const __nv_bfloat16 *in[3];
  __nv_bfloat16 *out[3];
  const int32_t *perm[3];
};

template <int D>
__global__ void __launch_bounds__(256, 8) k_gather_rows(const GatherJobs jobs, int64_t rows, int L) {
  constexpr int VPR = D / 8;
  constexpr int RPW = 256 / VPR;
  // the job's pointers by selection (an indexed parameter array would be
  // copied to local memory)
  const int job = blockIdx.y;
  const __nv_bfloat16 *in = job == 0 ? jobs.in[0] : (job == 1 ? jobs.in[1] : jobs.in[2]);
  __nv_bfloat16 *out = job == 0 ? jobs.out[0] : (job == 1 ? jobs.out[1] : jobs.out[2]);
  const int32_t *perm = job == 0 ? jobs.perm[0] : (job == 1 ? jobs.perm[1] : jobs.perm[2]);
  const int c = threadIdx.x % VPR;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * RPW * kGatherRows + threadIdx.x / VPR;
  // first row of the head of each row, carried from row to row (rows of a
  // thread are RPW apart): one division per thread
  int64_t hb = row0 - row0 % L;
  int tk = static_cast<int>(row0 - hb);
  int64_t src[kGatherRows];
#pragma unroll
  for (int u = 0; u < kGatherRows; ++u) {
    const int64_t row = row0 + u * RPW;
    src[u] = (row < rows) ? hb + min(max(__ldg(perm + row), 0), L - 1) : -1;
    tk += RPW;
    while (tk >= L) {
      tk -= L;
      hb += L;
    }
  }
  uint4 v[kGatherRows];
#pragma unroll
  for (int u = 0; u < kGatherRows; ++u)
    if (src[u] >= 0) v[u] = __ldg(reinterpret_cast<const uint4 *>(in + src[u] * D) + c);
#pragma unroll
  for (int u = 0; u < kGatherRows; ++u)
    if (src[u] >= 0) reinterpret_cast<uint4 *>(out + (row0 + u * RPW) * D)[c] = v[u];
}

// ---------------------------------------------------------------------------
// tile-pair lists.  For each CTA (two 128-row query tiles) and each of its
// tiles: the key blocks the tile's query blocks selected (for B = 64 the
// union of two lists, each entry tagged with which query block selected it),
// ordered with the blocks both tiles selected first -- in the same order in
// both lists, so the attention kernel loads them once for both tiles -- then
// the tile's other blocks; ascending within each part.  (Online softmax does
// not depend on the order of the key blocks.)  One warp per pair.
// ---------------------------------------------------------------------------
constexpr int kPairWarps = 4;
constexpr int kPairWords = kMaxBlocks / 32;

template <int G>
__global__ void __launch_bounds__(kPairWarps * 32) k_pair_lists(
    const int32_t *__restrict__ idx, int N, int kappa, int n_tiles, int npairs, int64_t total,
    uint16_t *__restrict__ lists, int32_t *__restrict__ counts, int *__restrict__ ready,
    int n_ready) {
  __shared__ uint32_t bm[kPairWarps][kTiles][G][kPairWords];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  {
    // the attention kernel's per-head gather counters (claim, done) start from zero
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (ready != nullptr && i < n_ready) ready[i] = 0;
  }
  const int64_t gp = static_cast<int64_t>(blockIdx.x) * kPairWarps + warp;
  if (gp >= total) return;  // warp-uniform; no block barrier below
  const int64_t bh = gp / npairs;
  const int pair = static_cast<int>(gp % npairs);
  const int nwords = (N + 31) / 32;
  uint32_t(*b)[G][kPairWords] = bm[warp];
  for (int t = 0; t < kTiles; ++t)
    for (int g = 0; g < G; ++g)
      for (int w = lane; w < nwords; w += 32) b[t][g][w] = 0u;
  __syncwarp();
  for (int t = 0; t < kTiles; ++t) {
    const int tile = pair * kTiles + t;
    if (tile >= n_tiles) continue;
    for (int g = 0; g < G; ++g) {
      const int gq = tile * G + g;
      if (gq >= N) continue;
      const int32_t *src = idx + (bh * N + gq) * kappa;
      for (int i = lane; i < kappa; i += 32) {
        const int blk = __ldg(src + i);
        if (blk < 0 || blk >= N) continue;  // ids are not validated on the host
        atomicOr(&b[t][g][blk >> 5], 1u << (blk & 31));
      }
    }
  }
  __syncwarp();
  uint16_t *out[kTiles] = {lists + (gp * kTiles) * N, lists + (gp * kTiles + 1) * N};
  auto any = [&](int t, int w) {
    uint32_t m = 0u;
#pragma unroll
    for (int g = 0; g < G; ++g) m |= b[t][g][w];
    return m;
  };
  auto entry = [&](int t, int w, int bit) {
    uint32_t sel = 0u;
#pragma unroll
    for (int g = 0; g < G; ++g) sel |= ((b[t][g][w] >> bit) & 1u) << g;
    return static_cast<uint16_t>((w * 32 + bit) | (sel << 12));
  };
  int common = 0, n[kTiles] = {0, 0};
  // pass 0: blocks of both tiles; pass 1: tile 0 only; pass 2: tile 1 only
  for (int pass = 0; pass < 3; ++pass) {
    int pos = (pass == 0) ? 0 : common;
    for (int w0 = 0; w0 < nwords; w0 += 32) {
      const int w = w0 + lane;
      const uint32_t a0 = (w < nwords) ? any(0, w) : 0u, a1 = (w < nwords) ? any(1, w) : 0u;
      uint32_t m = (pass == 0) ? (a0 & a1) : (pass == 1) ? (a0 & ~a1) : (a1 & ~a0);
      const int cnt = __popc(m);
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      int q = pos + incl - cnt;
      while (m) {
        const int bit = __ffs(m) - 1;
        m &= m - 1;
        if (pass != 2) out[0][q] = entry(0, w, bit);
        if (pass != 1) out[1][q] = entry(1, w, bit);
        ++q;
      }
      pos += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (pass == 0) common = pos;
    else n[pass - 1] = pos;
  }
  if (lane == 0) {
    counts[gp * 4 + 0] = n[0];
    counts[gp * 4 + 1] = n[1];
    counts[gp * 4 + 2] = common;
    counts[gp * 4 + 3] = 0;
  }
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

// Workspace of the sparse call: Q' (perm_q), K' and V' (perm_k), then the
// tile-pair lists and their counts, then (with a permutation) the gather
// claim and done counters, one of each per head.
static size_t pair_list_bytes(int64_t bh, int L, int B) {
  const int64_t n = (L + B - 1) / B;
  const int64_t npairs = ((L + kTileM - 1) / kTileM + kTiles - 1) / kTiles;
  return align256(static_cast<size_t>(bh * npairs * kTiles * n) * sizeof(uint16_t)) +
         align256(static_cast<size_t>(bh * npairs * 4) * sizeof(int32_t));
}

size_t attn_workspace_bytes(int64_t bh, int L, int D, int B, bool perm_q, bool perm_k) {
  const size_t t = align256(static_cast<size_t>(bh) * L * D * 2);
  const size_t counters = (perm_q || perm_k) ? align256(static_cast<size_t>(2 * bh) * sizeof(int)) : 0;
  return (perm_q ? t : 0) + (perm_k ? 2 * t : 0) + pair_list_bytes(bh, L, B) + counters;
}

// Heads between an attention CTA and the head whose rows it gathers: far
// enough back in launch order (about two waves of CTAs) that a head's rows
// are complete before its first CTA starts.
static int gather_lookahead(int npairs) {
  static std::atomic<int> sms_cached[64];  // per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
  std::atomic<int> &slot = sms_cached[dev & 63];
  int sms = slot.load(std::memory_order_relaxed);
  if (sms == 0) {
    int n = 0;
    sms = (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) ? n : 152;
    slot.store(sms, std::memory_order_relaxed);
  }
  return (2 * sms + npairs - 1) / npairs;
}

// The in-kernel copies pay while a CTA's own attention work outlasts its
// share of them (one slice of a later head: 2 x 128 rows of each gathered
// tensor, read and written).  Measured on GB300 (d = 128, two 128-row tiles
// per CTA): a key-slot iteration takes ~1.7 us; one gather warp copies a
// CTA's share of Q', K' and V' in ~75 us, the packed kernel's two warps in
// about half that.  A 128-token-block CTA walks ~kappa slots, a 64-token one
// ~kappa / 2 (two entries per slot).  Both sides scale alike with d.  Below
// the balance (L = 32768 at 90% sparsity: kappa 26, 2.02 ms with the copies
// in the kernel) every head is gathered by the separate pass instead.
static bool gathers_hide_under_attention(int kappa, int BK, int njobs) {
  const int64_t slots = BK == 128 ? kappa : (kappa + 1) / 2;
  const int64_t warps = BK == 128 ? 1 : 2;
  const int64_t attn_tenths_us = slots * 17;
  const int64_t copy_tenths_us = 750 * njobs / (3 * warps);
  return attn_tenths_us >= copy_tenths_us;
}

template <int D, int BK, bool kDense, bool kPack = false>
static cudaError_t launch_attn(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                               const AttnParams &p, int64_t bh, cudaStream_t st) {
  using Lay = AttnLayout<D, BK>;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = once_per_device(configured, [] {
    cudaError_t r = cudaFuncSetAttribute(k_attn<D, BK, kDense, kPack>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kAlloc);
    if (r != cudaSuccess) return r;
    // setmaxnreg.inc draws on the registers the block is launched with: a
    // split larger than that pool would never be granted, so refuse it here
    cudaFuncAttributes fa;
    if ((r = cudaFuncGetAttributes(&fa, k_attn<D, BK, kDense, kPack>)) != cudaSuccess) return r;
    if (fa.numRegs * kAttnThreads < kSplitRegs(RegSplit<BK>::kLow, RegSplit<BK>::kHigh))
      return cudaErrorInvalidConfiguration;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const dim3 grid((p.n_tiles + kTiles - 1) / kTiles, static_cast<unsigned>(bh));
  k_attn<D, BK, kDense, kPack><<<grid, kAttnThreads, Lay::kAlloc, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

static cudaError_t run_attention_impl(const AttnArgs &a, cudaStream_t st, uint64_t issuer_wait_ns,
                                      int skip_load) {
  const int64_t bh = static_cast<int64_t>(a.batch) * a.heads;
  const int L = a.seqlen, D = a.head_dim;
  const bool dense = a.block_idx == nullptr;
  const int BK = dense ? 128 : a.block;
  const int64_t rows = bh * L;
  const void *qs = a.q, *ks = a.k, *vs = a.v;
  unsigned char *ws = static_cast<unsigned char *>(a.workspace);
  const size_t t = align256(static_cast<size_t>(rows) * D * 2);
  cudaError_t e;
  GatherJobs jobs;
  int njobs = 0;
  if (a.perm_q) {
    __nv_bfloat16 *qp = reinterpret_cast<__nv_bfloat16 *>(ws);
    ws += t;
    jobs.in[njobs] = static_cast<const __nv_bfloat16 *>(a.q);
    jobs.out[njobs] = qp;
    jobs.perm[njobs++] = a.perm_q;
    qs = qp;
  }
  if (a.perm_k) {
    __nv_bfloat16 *kp = reinterpret_cast<__nv_bfloat16 *>(ws);
    __nv_bfloat16 *vp = reinterpret_cast<__nv_bfloat16 *>(ws + t);
    jobs.in[njobs] = static_cast<const __nv_bfloat16 *>(a.k);
    jobs.out[njobs] = kp;
    jobs.perm[njobs++] = a.perm_k;
    jobs.in[njobs] = static_cast<const __nv_bfloat16 *>(a.v);
    jobs.out[njobs] = vp;
    jobs.perm[njobs++] = a.perm_k;
    ks = kp;
    vs = vp;
    ws += 2 * t;
  }
  uint16_t *pair_lists = nullptr;
  int32_t *pair_counts = nullptr;
  const int n_tiles = (L + kTileM - 1) / kTileM;
  const int npairs = (n_tiles + kTiles - 1) / kTiles;
  // Gathers: the first `lookahead` heads by k_gather_rows before the
  // attention kernel, the others inside it (claimed slices).
  int *counters = nullptr;
  const int lookahead = gather_lookahead(npairs);
  const bool in_kernel_gathers =
      !dense && njobs > 0 && lookahead < bh && gathers_hide_under_attention(a.kappa, BK, njobs);
  if (!dense) {
    const int64_t nblk = (L + BK - 1) / BK;
    pair_lists = reinterpret_cast<uint16_t *>(ws);
    const size_t list_bytes = align256(static_cast<size_t>(bh * npairs * kTiles * nblk) * sizeof(uint16_t));
    pair_counts = reinterpret_cast<int32_t *>(ws + list_bytes);
    if (in_kernel_gathers) counters = reinterpret_cast<int *>(ws + pair_list_bytes(bh, L, BK));
    const int64_t total = bh * npairs;
    const int n_ready = counters ? static_cast<int>(2 * bh) : 0;
    const int64_t by_pairs = (total + kPairWarps - 1) / kPairWarps;
    const int64_t by_counters = (n_ready + kPairWarps * 32 - 1) / (kPairWarps * 32);
    const unsigned grid = static_cast<unsigned>(by_pairs > by_counters ? by_pairs : by_counters);
    if (BK == 128)
      k_pair_lists<1><<<grid, kPairWarps * 32, 0, st>>>(a.block_idx, static_cast<int>(nblk), a.kappa,
                                                        n_tiles, npairs, total, pair_lists, pair_counts,
                                                        counters, n_ready);
    else
      k_pair_lists<2><<<grid, kPairWarps * 32, 0, st>>>(a.block_idx, static_cast<int>(nblk), a.kappa,
                                                        n_tiles, npairs, total, pair_lists, pair_counts,
                                                        counters, n_ready);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (njobs > 0) {
    const int64_t grows = in_kernel_gathers ? static_cast<int64_t>(lookahead) * L : rows;
    const int rows_per_cta = (256 / (D / 8)) * kGatherRows;
    const dim3 grid(static_cast<unsigned>((grows + rows_per_cta - 1) / rows_per_cta), njobs);
    if (D == 128)
      k_gather_rows<128><<<grid, 256, 0, st>>>(jobs, grows, L);
    else
      k_gather_rows<64><<<grid, 256, 0, st>>>(jobs, grows, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  alignas(64) CUtensorMap mq, mk, mv;
  if ((e = encode_tensor_map_3d(&mq, qs, D, L, bh, 64, kTileM)) != cudaSuccess) return e;
  // 64-token blocks are loaded as 64-row boxes, two per 128-key slot
  if ((e = encode_tensor_map_3d(&mk, ks, D, L, bh, 64, BK)) != cudaSuccess) return e;
  if ((e = encode_tensor_map_3d(&mv, vs, D, L, bh, 64, BK)) != cudaSuccess) return e;

  AttnParams p;
  p.L = L;
  p.N = (L + BK - 1) / BK;
  p.n_tiles = n_tiles;
  p.npairs = npairs;
  p.pair_lists = pair_lists;
  p.pair_counts = pair_counts;
  p.perm_q = a.perm_q;
  p.perm_k = a.perm_k;
  p.src_q = static_cast<const __nv_bfloat16 *>(a.q);
  p.src_k = static_cast<const __nv_bfloat16 *>(a.k);
  p.src_v = static_cast<const __nv_bfloat16 *>(a.v);
  p.dst_q = a.perm_q ? const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(qs)) : nullptr;
  p.dst_k = a.perm_k ? const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(ks)) : nullptr;
  p.dst_v = a.perm_k ? const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(vs)) : nullptr;
  p.claim = counters;
  p.done = counters ? counters + bh : nullptr;
  p.lookahead = lookahead;
  p.bh_total = static_cast<int>(bh);
  p.slice_rows = (L + npairs - 1) / npairs;
  p.nslices = npairs;
  p.issuer_wait_ns = issuer_wait_ns;
  p.skip_load = skip_load;
  p.o = static_cast<__nv_bfloat16 *>(a.o);
  p.lse = a.lse;
  const float scale = (a.scale > 0.f) ? a.scale : 1.0f / sqrtf(static_cast<float>(D));
  p.scale_log2 = scale * 1.4426950408889634f;

  if (dense) {
    if (D == 128) return launch_attn<128, 128, true>(mq, mk, mv, p, bh, st);
    if (D == 64) return launch_attn<64, 128, true>(mq, mk, mv, p, bh, st);
  } else {
    if (D == 128 && BK == 128) return launch_attn<128, 128, false>(mq, mk, mv, p, bh, st);
    if (D == 128 && BK == 64) return launch_attn<128, 128, false, true>(mq, mk, mv, p, bh, st);
    if (D == 64 && BK == 128) return launch_attn<64, 128, false>(mq, mk, mv, p, bh, st);
    if (D == 64 && BK == 64) return launch_attn<64, 128, false, true>(mq, mk, mv, p, bh, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t run_attention(const AttnArgs &a, cudaStream_t st) {
  return run_attention_impl(a, st, kWaitLimitNs, -1);
}

// The dense kernel with the second K/V copy of every CTA (V_0) never issued:
// the softmax withholds P-ready until that copy lands, so the MMA thread's
// bounded wait for P gives up after `limit_ns` and records kSitePFull; every
// role unwinds (copies and MMAs drained, tensor memory freed, nothing
// written).
cudaError_t run_attention_stall(const AttnArgs &a, uint64_t limit_ns, cudaStream_t st) {
  return run_attention_impl(a, st, limit_ns, 1);
}

}  // namespace ba
