// C ABI of the BA-Att library: argument checks, workspace sizing, dispatch.
// The operations are specified in include/ba.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "../../include/ba.h"
#include "ba_common.cuh"
#include "ba_internal.h"

namespace ba {

namespace {

constexpr int kMaxBlocksPerSeq = 4096;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks common to every call.  Returns BA_OK or an error status.
int check_shape(int batch, int heads, int seqlen, int head_dim, int block) {
  if (batch < 1 || heads < 1 || seqlen < 1) return BA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return BA_ERR_UNSUPPORTED;
  if (block != 64 && block != 128) return BA_ERR_UNSUPPORTED;
  const int64_t rows = static_cast<int64_t>(batch) * heads * seqlen;
  if (rows * head_dim >= (static_cast<int64_t>(1) << 40)) return BA_ERR_UNSUPPORTED;
  if (rows >= (static_cast<int64_t>(1) << 31)) return BA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(batch) * heads > 65535) return BA_ERR_UNSUPPORTED;
  const int n = (seqlen + block - 1) / block;
  if (n > kMaxBlocksPerSeq) return BA_ERR_UNSUPPORTED;
  return BA_OK;
}

int map_cuda(cudaError_t e) { return e == cudaSuccess ? BA_OK : BA_ERR_CUDA; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn resolve_encode() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

}  // namespace

cudaError_t encode_tensor_map_3d(void *map_out, const void *base, uint64_t inner, uint64_t rows,
                                 uint64_t outer, uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = resolve_encode();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {inner, rows, outer};
  const cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(static_cast<CUtensorMap *>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace ba

using namespace ba;

extern "C" {

const char *ba_status_string(int status) {
  switch (status) {
    case BA_OK: return "BA_OK";
    case BA_ERR_INVALID_ARG: return "BA_ERR_INVALID_ARG: invalid argument";
    case BA_ERR_UNSUPPORTED: return "BA_ERR_UNSUPPORTED: shape or option not supported";
    case BA_ERR_WORKSPACE: return "BA_ERR_WORKSPACE: workspace too small or misaligned";
    case BA_ERR_CUDA: return "BA_ERR_CUDA: CUDA runtime or launch error";
    case BA_ERR_DEVICE_TIMEOUT: return "BA_ERR_DEVICE_TIMEOUT: a kernel gave up on a bounded wait";
    default: return "BA_ERR_UNKNOWN";
  }
}

const char *ba_version(void) { return "ba-gb300 0.1 sm_103a"; }

size_t ba_select_workspace_size(int batch, int heads, int seqlen, int head_dim, int block,
                                int kappa, int sort_mode, int sort_window) {
  (void)kappa;
  (void)sort_window;
  if (check_shape(batch, heads, seqlen, head_dim, block) != BA_OK) return 0;
  if (sort_mode < 0 || sort_mode > 3) return 0;
  return select_workspace_bytes(static_cast<int64_t>(batch) * heads, seqlen, head_dim, block,
                                sort_mode);
}

int ba_select(const void *q, const void *k, int batch, int heads, int seqlen, int head_dim,
              int block, int kappa, float beta, int sort_mode, int sort_window, int32_t *perm_q,
              int32_t *perm_k, int32_t *block_idx, uint32_t *block_mask, float *block_scores,
              void *workspace, size_t workspace_bytes, ba_stream_t stream) {
  int st = check_shape(batch, heads, seqlen, head_dim, block);
  if (st != BA_OK) return st;
  const int n = (seqlen + block - 1) / block;
  if (kappa < 1 || kappa > n) return BA_ERR_INVALID_ARG;
  if (!isfinite(beta)) return BA_ERR_INVALID_ARG;
  if (sort_mode < 0 || sort_mode > 3) return BA_ERR_INVALID_ARG;
  if (sort_window < 0 || (sort_window > 0 && sort_window % block != 0)) return BA_ERR_INVALID_ARG;
  if (!q || !k || !perm_q || !perm_k || !block_idx || !block_mask) return BA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(perm_q) || !aligned16(perm_k) ||
      !aligned16(block_idx) || !aligned16(block_mask) ||
      (block_scores && !aligned16(block_scores)))
    return BA_ERR_INVALID_ARG;
  const size_t need = ba_select_workspace_size(batch, heads, seqlen, head_dim, block, kappa,
                                               sort_mode, sort_window);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                   (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return BA_ERR_WORKSPACE;
  SelectArgs a;
  a.q = q;
  a.k = k;
  a.batch = batch;
  a.heads = heads;
  a.seqlen = seqlen;
  a.head_dim = head_dim;
  a.block = block;
  a.kappa = kappa;
  a.beta = beta;
  a.sort_mode = sort_mode;
  a.sort_window = sort_window;
  a.perm_q = perm_q;
  a.perm_k = perm_k;
  a.block_idx = block_idx;
  a.block_mask = block_mask;
  a.block_scores = block_scores;
  a.workspace = workspace;
  return map_cuda(run_select(a, reinterpret_cast<cudaStream_t>(stream)));
}

int ba_select_isolated(const void *q, const void *k, int batch, int heads, int seqlen,
                       int head_dim, int block, int prefill_len, int kappa_prefill,
                       int kappa_generation, float beta, int sort_mode, int sort_window,
                       int32_t *perm_q, int32_t *perm_k, int32_t *block_idx,
                       uint32_t *block_mask, float *block_scores, void *workspace,
                       size_t workspace_bytes, ba_stream_t stream) {
  int st = check_shape(batch, heads, seqlen, head_dim, block);
  if (st != BA_OK) return st;
  const int n = (seqlen + block - 1) / block;
  if (prefill_len <= 0 || prefill_len >= seqlen || prefill_len % block != 0)
    return BA_ERR_INVALID_ARG;
  const int n_pre = prefill_len / block, n_gen = n - n_pre;
  if (kappa_prefill < 1 || kappa_prefill > n_pre) return BA_ERR_INVALID_ARG;
  if (kappa_generation < 1 || kappa_generation > n_gen) return BA_ERR_INVALID_ARG;
  const int kappa = kappa_prefill + kappa_generation;
  if (!isfinite(beta)) return BA_ERR_INVALID_ARG;
  if (sort_mode < 0 || sort_mode > 3) return BA_ERR_INVALID_ARG;
  if (sort_window < 0 || (sort_window > 0 && sort_window % block != 0)) return BA_ERR_INVALID_ARG;
  if (!q || !k || !perm_q || !perm_k || !block_idx || !block_mask) return BA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(perm_q) || !aligned16(perm_k) ||
      !aligned16(block_idx) || !aligned16(block_mask) ||
      (block_scores && !aligned16(block_scores)))
    return BA_ERR_INVALID_ARG;
  const size_t need = ba_select_workspace_size(batch, heads, seqlen, head_dim, block, kappa,
                                               sort_mode, sort_window);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                   (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return BA_ERR_WORKSPACE;
  SelectArgs a;
  a.q = q;
  a.k = k;
  a.batch = batch;
  a.heads = heads;
  a.seqlen = seqlen;
  a.head_dim = head_dim;
  a.block = block;
  a.kappa = kappa;
  a.beta = beta;
  a.sort_mode = sort_mode;
  a.sort_window = sort_window;
  a.perm_q = perm_q;
  a.perm_k = perm_k;
  a.block_idx = block_idx;
  a.block_mask = block_mask;
  a.block_scores = block_scores;
  a.workspace = workspace;
  a.prefill_len = prefill_len;
  a.kappa_prefill = kappa_prefill;
  return map_cuda(run_select(a, reinterpret_cast<cudaStream_t>(stream)));
}

int ba_active_tokens(const void *q_now, const void *q_prev, int batch, int heads, int seqlen,
                     int head_dim, int group, int top_k, uint8_t *active, float *mse,
                     ba_stream_t stream) {
  if (batch < 1 || heads < 1 || seqlen < 1) return BA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return BA_ERR_UNSUPPORTED;
  if (group < 1 || group > kLosaMaxGroup || top_k < 1) return BA_ERR_INVALID_ARG;
  const int64_t bh = static_cast<int64_t>(batch) * heads;
  if (bh > 65535) return BA_ERR_UNSUPPORTED;
  if (!q_now || !q_prev || !active) return BA_ERR_INVALID_ARG;
  if (!aligned16(q_now) || !aligned16(q_prev) || (mse && !aligned16(mse))) return BA_ERR_INVALID_ARG;
  return map_cuda(run_active_tokens(q_now, q_prev, bh, seqlen, head_dim, group, top_k, active, mse,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int ba_reuse_rows(const void *o_new, const float *lse_new, const uint8_t *active, int64_t rows,
                  int head_dim, void *o_cache, float *lse_cache, ba_stream_t stream) {
  if (rows < 0) return BA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return BA_ERR_UNSUPPORTED;
  if (rows == 0) return BA_OK;
  if (!o_new || !lse_new || !active || !o_cache || !lse_cache) return BA_ERR_INVALID_ARG;
  if (!aligned16(o_new) || !aligned16(o_cache)) return BA_ERR_INVALID_ARG;
  return map_cuda(run_reuse_rows(o_new, lse_new, active, rows, head_dim, o_cache, lse_cache,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

size_t ba_block_fidelity_workspace_size(int batch, int heads, int seqlen, int head_dim, int block) {
  if (check_shape(batch, heads, seqlen, head_dim, block) != BA_OK) return 0;
  return fidelity_workspace_bytes(static_cast<int64_t>(batch) * heads, seqlen, head_dim, block);
}

int ba_block_fidelity(const void *q, const void *k, int batch, int heads, int seqlen,
                      int head_dim, int block, const int32_t *perm_q, const int32_t *perm_k,
                      const float *lse, float scale, const int32_t *block_idx, int kappa,
                      float *mass, float *dev_max, float *bound, float *recall, void *workspace,
                      size_t workspace_bytes, ba_stream_t stream) {
  int st = check_shape(batch, heads, seqlen, head_dim, block);
  if (st != BA_OK) return st;
  const int n = (seqlen + block - 1) / block;
  if (!isfinite(scale)) return BA_ERR_INVALID_ARG;
  if (!q || !k || !lse || !mass) return BA_ERR_INVALID_ARG;
  if (recall && (!block_idx || kappa < 1 || kappa > n)) return BA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(lse) || !aligned16(mass) ||
      (dev_max && !aligned16(dev_max)) || (bound && !aligned16(bound)) ||
      (recall && !aligned16(recall)) || (perm_q && !aligned16(perm_q)) ||
      (perm_k && !aligned16(perm_k)) || (block_idx && !aligned16(block_idx)))
    return BA_ERR_INVALID_ARG;
  const size_t need = ba_block_fidelity_workspace_size(batch, heads, seqlen, head_dim, block);
  if (workspace == nullptr || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return BA_ERR_WORKSPACE;
  FidArgs a;
  a.q = q;
  a.k = k;
  a.batch = batch;
  a.heads = heads;
  a.seqlen = seqlen;
  a.head_dim = head_dim;
  a.block = block;
  a.perm_q = perm_q;
  a.perm_k = perm_k;
  a.lse = lse;
  a.scale = scale;
  a.block_idx = block_idx;
  a.kappa = kappa;
  a.mass = mass;
  a.dev_max = dev_max;
  a.bound = bound;
  a.recall = recall;
  a.workspace = workspace;
  return map_cuda(run_fidelity(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t ba_sparse_attn_workspace_size(int batch, int heads, int seqlen, int head_dim, int block,
                                     int kappa, int has_perm_q, int has_perm_k) {
  (void)kappa;
  if (check_shape(batch, heads, seqlen, head_dim, block) != BA_OK) return 0;
  return attn_workspace_bytes(static_cast<int64_t>(batch) * heads, seqlen, head_dim, block,
                              has_perm_q != 0, has_perm_k != 0);
}

int ba_sparse_attn(const void *q, const void *k, const void *v, int batch, int heads, int seqlen,
                   int head_dim, int block, const int32_t *perm_q, const int32_t *perm_k,
                   const int32_t *block_idx, int kappa, float scale, void *o, float *lse,
                   void *workspace, size_t workspace_bytes, ba_stream_t stream) {
  int st = check_shape(batch, heads, seqlen, head_dim, block);
  if (st != BA_OK) return st;
  const int n = (seqlen + block - 1) / block;
  if (kappa < 1 || kappa > n) return BA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return BA_ERR_INVALID_ARG;
  if (!q || !k || !v || !block_idx || !o || !lse) return BA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(block_idx) || (perm_q && !aligned16(perm_q)) || (perm_k && !aligned16(perm_k)))
    return BA_ERR_INVALID_ARG;
  const size_t need = ba_sparse_attn_workspace_size(batch, heads, seqlen, head_dim, block, kappa,
                                                    perm_q != nullptr, perm_k != nullptr);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                   (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return BA_ERR_WORKSPACE;
  AttnArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.batch = batch;
  a.heads = heads;
  a.seqlen = seqlen;
  a.head_dim = head_dim;
  a.block = block;
  a.perm_q = perm_q;
  a.perm_k = perm_k;
  a.block_idx = block_idx;
  a.kappa = kappa;
  a.scale = scale;
  a.o = o;
  a.lse = lse;
  a.workspace = workspace;
  return map_cuda(run_attention(a, reinterpret_cast<cudaStream_t>(stream)));
}

int ba_attn_dense(const void *q, const void *k, const void *v, int batch, int heads, int seqlen,
                  int head_dim, float scale, void *o, float *lse, ba_stream_t stream) {
  int st = check_shape(batch, heads, seqlen, head_dim, 128);
  if (st != BA_OK) return st;
  if (!isfinite(scale)) return BA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return BA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return BA_ERR_INVALID_ARG;
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.batch = batch;
  a.heads = heads;
  a.seqlen = seqlen;
  a.head_dim = head_dim;
  a.block = 128;
  a.scale = scale;
  a.o = o;
  a.lse = lse;
  return map_cuda(run_attention(a, reinterpret_cast<cudaStream_t>(stream)));
}

int ba_merge_lse(const void *o1, const float *lse1, const void *o2, const float *lse2,
                 int64_t rows, int head_dim, void *o, float *lse, ba_stream_t stream) {
  if (rows < 0) return BA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return BA_ERR_UNSUPPORTED;
  if (rows == 0) return BA_OK;
  if (!o1 || !lse1 || !o2 || !lse2 || !o || !lse) return BA_ERR_INVALID_ARG;
  if (!aligned16(o1) || !aligned16(o2) || !aligned16(o) || !aligned16(lse1) || !aligned16(lse2) ||
      !aligned16(lse))
    return BA_ERR_INVALID_ARG;
  if (rows >= (static_cast<int64_t>(1) << 40) / head_dim) return BA_ERR_UNSUPPORTED;
  return map_cuda(run_merge_lse(o1, lse1, o2, lse2, rows, head_dim, o, lse,
                                reinterpret_cast<cudaStream_t>(stream)));
}

int ba_validate_selection(const int32_t *perm_q, const int32_t *perm_k, const int32_t *block_idx,
                          int batch, int heads, int seqlen, int block, int kappa, uint32_t *detail,
                          ba_stream_t stream) {
  if (detail) *detail = 0;
  int st = check_shape(batch, heads, seqlen, 64, block);
  if (st != BA_OK) return st;
  const int n = (seqlen + block - 1) / block;
  if (kappa < 1 || kappa > n) return BA_ERR_INVALID_ARG;
  if (!block_idx || !aligned16(block_idx) || (perm_q && !aligned16(perm_q)) || (perm_k && !aligned16(perm_k)))
    return BA_ERR_INVALID_ARG;
  uint32_t word = 0;
  if (run_validate_selection(perm_q, perm_k, block_idx, static_cast<int64_t>(batch) * heads, seqlen, n, kappa,
                             &word, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BA_ERR_CUDA;
  if (detail) *detail = word;
  return word ? BA_ERR_INVALID_ARG : BA_OK;
}

int ba_selftest_wait_timeout(uint32_t limit_us, ba_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return BA_ERR_INVALID_ARG;
  return map_cuda(run_selftest_wait(static_cast<uint64_t>(limit_us) * 1000ull,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int ba_selftest_attn_stall(const void *q, const void *k, const void *v, int batch, int heads,
                           int seqlen, int head_dim, uint32_t limit_us, void *o, float *lse,
                           ba_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return BA_ERR_INVALID_ARG;
  int st = check_shape(batch, heads, seqlen, head_dim, 128);
  if (st != BA_OK) return st;
  // stage 1 must exist: at least two 128-key slots
  if (seqlen <= 128) return BA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return BA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return BA_ERR_INVALID_ARG;
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.batch = batch;
  a.heads = heads;
  a.seqlen = seqlen;
  a.head_dim = head_dim;
  a.block = 128;
  a.o = o;
  a.lse = lse;
  return map_cuda(run_attention_stall(a, static_cast<uint64_t>(limit_us) * 1000ull,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

int ba_last_device_error(ba_stream_t stream, uint32_t *detail) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return BA_ERR_CUDA;
  uint32_t word = 0, fid = 0, self = 0;
  if (take_attn_error_word(&word) != cudaSuccess) return BA_ERR_CUDA;
  if (take_fidelity_error_word(&fid) != cudaSuccess) return BA_ERR_CUDA;
  if (take_selftest_error_word(&self) != cudaSuccess) return BA_ERR_CUDA;
  if (word == 0) word = fid;
  if (word == 0) word = self;
  if (detail) *detail = word;
  return (word & 1u) ? BA_ERR_DEVICE_TIMEOUT : BA_OK;
}

}  // extern "C"
