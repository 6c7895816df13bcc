// Internal host-side interfaces between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace ba {

// One-time setup per device (a kernel's cudaFuncSetAttribute before its
// first launch on that device), safe when several host threads launch: a
// device's bit in `done` is set only after `setup` succeeded; two threads
// may both run `setup` for the same device, which is harmless because it is
// idempotent.
template <typename F>
inline cudaError_t once_per_device(std::atomic<uint64_t> &done, F &&setup) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  if ((e = setup()) != cudaSuccess) return e;
  if (bit != 0) done.fetch_or(bit, std::memory_order_release);
  return cudaSuccess;
}

struct SelectArgs {
  const void *q, *k;
  int batch, heads, seqlen, head_dim, block, kappa;
  float beta;
  int sort_mode, sort_window;
  int32_t *perm_q, *perm_k, *block_idx;
  uint32_t *block_mask;
  float *block_scores;
  void *workspace;
  // isolated selection (SparseD §3.3): > 0 splits the keys at this token
  // (a multiple of block); kappa_prefill of the kappa blocks per row come
  // from the first prefill_len / block key blocks
  int prefill_len = 0;
  int kappa_prefill = 0;
};

struct AttnArgs {
  const void *q, *k, *v;
  int batch, heads, seqlen, head_dim, block;
  const int32_t *perm_q, *perm_k, *block_idx;  // block_idx == nullptr: dense
  int kappa;
  float scale;
  void *o;
  float *lse;
  void *workspace;
};

// LoSA locality pruning and result reuse.
constexpr int kLosaMaxGroup = 1024;
cudaError_t run_active_tokens(const void *q_now, const void *q_prev, int64_t bh, int L, int D,
                              int group, int top_k, uint8_t *active, float *mse, cudaStream_t st);
cudaError_t run_reuse_rows(const void *o_new, const float *lse_new, const uint8_t *active,
                           int64_t rows, int D, void *o_cache, float *lse_cache, cudaStream_t st);

// Fidelity diagnostics (block mass, logit deviation, its bound, recall).
struct FidArgs {
  const void *q, *k;
  int batch, heads, seqlen, head_dim, block;
  const int32_t *perm_q, *perm_k;  // nullable: identity
  const float *lse;                // dense row LSE [b,h,L], original order
  float scale;
  const int32_t *block_idx;        // nullable unless recall is asked for
  int kappa;
  float *mass, *dev_max, *bound, *recall;
  void *workspace;
};

size_t fidelity_workspace_bytes(int64_t bh, int L, int D, int B);
cudaError_t run_fidelity(const FidArgs &a, cudaStream_t st);
cudaError_t take_fidelity_error_word(uint32_t *word);
cudaError_t run_selftest_wait(uint64_t limit_ns, cudaStream_t st);
cudaError_t take_selftest_error_word(uint32_t *word);

size_t select_workspace_bytes(int64_t bh, int L, int D, int B, int sort_mode);
cudaError_t run_select(const SelectArgs &a, cudaStream_t st);

size_t attn_workspace_bytes(int64_t bh, int L, int D, int B, bool perm_q, bool perm_k);
cudaError_t run_attention(const AttnArgs &a, cudaStream_t st);
// Dense attention whose second K/V stage is never loaded: exercises the
// attention kernel's bounded-wait unwind (see ba_selftest_attn_stall).
cudaError_t run_attention_stall(const AttnArgs &a, uint64_t limit_ns, cudaStream_t st);

// Checks pi_q, pi_k (nullable) and block_idx on the device, synchronises the
// stream and returns the failure bits (1 pi_q, 2 pi_k, 4 block_idx) in *word.
cudaError_t run_validate_selection(const int32_t *perm_q, const int32_t *perm_k, const int32_t *block_idx,
                                   int64_t bh, int L, int N, int kappa, uint32_t *word, cudaStream_t st);

cudaError_t run_merge_lse(const void *o1, const float *lse1, const void *o2, const float *lse2,
                          int64_t rows, int head_dim, void *o, float *lse, cudaStream_t st);

// Reads and clears the attention kernels' device error word (synchronous).
cudaError_t take_attn_error_word(uint32_t *word);

// Encodes a tiled TMA descriptor (driver entry point resolved at run time).
cudaError_t encode_tensor_map_3d(void *map_out, const void *base, uint64_t inner, uint64_t rows,
                                 uint64_t outer, uint32_t box_inner, uint32_t box_rows);

}  // namespace ba
