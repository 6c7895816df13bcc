/*
 * ba.h — C ABI of the BA-Att (Block Approximate Sparse Attention) hot path
 * for one NVIDIA GB300 GPU (sm_103a).
 *
 * The operations follow "Efficient Long-Context Modeling in Diffusion
 * Language Models via Block Approximate Sparse Attention" (the BA-Att paper):
 * Algorithm 1 takes Q, K, V, a block size B, a per-query-block budget kappa
 * and a compensation weight beta, and returns the block mask and the sparse
 * attention output.  The library adds the per-row log-sum-exp so that results
 * over disjoint key sets can be merged (the online-softmax merge of the LoSA
 * summary post, "merge and update").
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensors are dense, row-major, contiguous, on the device, in the layout
 *    [batch, heads, seqlen, head_dim] ("[b,h,L,d]"); bf16 means IEEE bfloat16
 *    bit patterns (uint16_t storage).  Every device pointer must be 16-byte
 *    aligned.  The caller owns every buffer; the library never allocates or
 *    frees device memory and keeps no state between calls except the device
 *    error word read by ba_last_device_error() and the fixed scratch array
 *    of ba_select_noalloc().
 *  - Blocks: N = ceil(L / B) query blocks and N key blocks (self-attention,
 *    L_q = L_k = L).  When B does not divide L the last block is short.
 *  - Attention is bidirectional (no causal mask).
 *  - Every call is asynchronous on `stream` (NULL = legacy default stream):
 *    host-side checks run first; on any error the call returns a status and
 *    launches nothing.  A CUDA launch failure returns BA_ERR_CUDA.
 *  - Supported: head_dim in {64, 128}; block in {64, 128}; 1 <= L;
 *    b*h*L < 2^31; N <= 4096.  Other values return BA_ERR_UNSUPPORTED.
 *  - Workspace: each call that needs scratch device memory takes a caller
 *    buffer of at least the size its *_workspace_size() query returns
 *    (256-byte aligned); a smaller one returns BA_ERR_WORKSPACE.
 */
#ifndef BA_H_
#define BA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so that this header needs no
 * CUDA header. */
typedef struct CUstream_st *ba_stream_t;

typedef enum {
  BA_OK = 0,
  BA_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned pointer */
  BA_ERR_UNSUPPORTED = 2,    /* valid but not implemented (head_dim, block, N) */
  BA_ERR_WORKSPACE = 3,      /* workspace smaller than required */
  BA_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
  BA_ERR_DEVICE_TIMEOUT = 5  /* a kernel gave up on a bounded wait */
} ba_status;

/* Which token sequences are norm-sorted before blocking (Algorithm 1 steps
 * 1-2; the ablation of the paper's Table 7: none / SortK / SortQ / both). */
typedef enum {
  BA_SORT_NONE = 0,
  BA_SORT_K = 1,
  BA_SORT_Q = 2,
  BA_SORT_QK = 3
} ba_sort_mode;

/* Human-readable name of a status. Never NULL. */
const char *ba_status_string(int status);

/* Library version string, e.g. "ba-gb300 0.1 sm_103a". */
const char *ba_version(void);

/*
 * Selection stage: BA-Att paper Algorithm 1 steps 1-11 (§3.1 Eq. 2, §3.3
 * Eq. 9-10, §3.4 Eq. 13-14).
 *
 *  1-2. s_i = ||Q_i||, s_j = ||K_j|| (computed as fp32 squared norms, which
 *       have the same order); a stable non-decreasing sort of each (b,h)
 *       sequence gives pi_q, pi_k (equal norms keep the lower index first).
 *       sort_window > 0 sorts each run of sort_window consecutive tokens on
 *       its own (the algorithm's "(windowed) sort"); 0 sorts the whole
 *       sequence.  sort_window must be 0 or a multiple of block.
 *  3-4. Consecutive groups of B sorted tokens form blocks; per block the fp32
 *       mean and population variance of every feature.
 *  5-7. l'[gq,gk] = Qbar.Kbar/sqrt(d)
 *                   + beta/d * sum_t(VarQ_t Kbar_t^2 + VarK_t Qbar_t^2
 *                                     + VarQ_t VarK_t), in fp32.
 *  8-11. Per query-block row, the kappa key blocks with the largest l'
 *       (equal scores: lower key-block index first); the row softmax of
 *       step 9 preserves this order and is not computed.
 *
 * Inputs:  q, k         bf16 [b,h,L,d], device.
 * Outputs (device, caller-allocated, fully overwritten):
 *   perm_q, perm_k  int32 [b,h,L]: sorted position -> original token index
 *                   (the identity when that sequence is not sorted).
 *   block_idx       int32 [b,h,N,kappa]: selected key blocks, ascending.
 *   block_mask      uint32 [b,h,N,ceil(N/32)]: bit (gk % 32) of word gk/32
 *                   is M[gq,gk] (1 = selected); unused high bits are 0.
 *   block_scores    fp32 [b,h,N,N] l' (may be NULL: not written).
 * kappa in [1, N]; beta finite (the paper's default is 1).
 */
size_t ba_select_workspace_size(int batch, int heads, int seqlen, int head_dim,
                                int block, int kappa, int sort_mode,
                                int sort_window);

int ba_select(const void *q, const void *k, int batch, int heads, int seqlen,
              int head_dim, int block, int kappa, float beta, int sort_mode,
              int sort_window, int32_t *perm_q, int32_t *perm_k,
              int32_t *block_idx, uint32_t *block_mask, float *block_scores,
              void *workspace, size_t workspace_bytes, ba_stream_t stream);

/*
 * ba_select without a workspace argument, for callers that cannot allocate
 * device memory when they select: for example a serving engine that reserves
 * the whole GPU heap for its own pool at start-up and allows no cudaMalloc
 * afterwards, or a plugin running inside a framework whose allocator it
 * cannot reach.  The paper has no counterpart to this call; it exists for
 * such deployments only.
 *
 * Same arguments, outputs and checks as ba_select, minus workspace and
 * workspace_bytes.  The scratch memory is a fixed array of
 * BA_SELECT_STATIC_SCRATCH_BYTES compiled into the library; every GPU that
 * loads the library holds that much device memory until the process exits.
 *  - Sizes whose ba_select_workspace_size() exceeds
 *    BA_SELECT_STATIC_SCRATCH_BYTES are rejected with BA_ERR_WORKSPACE before
 *    anything is launched (32 heads of L = 8192, d = 128, B = 64 fit).
 *  - The first call on a device looks up that device's copy of the array
 *    (cudaGetSymbolAddress with the device current) and caches it; make that
 *    first call before any stream capture begins.  The current device must be
 *    the device of `stream`; a stream of another device returns
 *    BA_ERR_INVALID_ARG and launches nothing.
 *  - The library allocates and frees nothing in this call.
 *  - Every call on a device shares the one array: calls whose work overlaps on
 *    the GPU (different streams, or different host threads) race on it and
 *    give undefined results.  Serialise them, e.g. on one stream.  Nothing has
 *    to be cleared between calls: every scratch element is written before it
 *    is read.
 */
#define BA_SELECT_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

int ba_select_noalloc(const void *q, const void *k, int batch, int heads,
                      int seqlen, int head_dim, int block, int kappa,
                      float beta, int sort_mode, int sort_window,
                      int32_t *perm_q, int32_t *perm_k, int32_t *block_idx,
                      uint32_t *block_mask, float *block_scores,
                      ba_stream_t stream);

/*
 * Isolated selection: ba_select with the key dimension split into a prefill
 * range [0, prefill_len) and a generation range [prefill_len, L), each with
 * its own budget, after SparseD §3.3 "Isolated Selection" (Eq. 5-6): every
 * query block keeps its kappa_prefill best key blocks among the prefill
 * blocks and its kappa_generation best among the generation blocks, so
 * generation tokens, whose scores are low in early denoising steps, are not
 * crowded out by prefill tokens.  Scores are BA-Att's (as in ba_select).
 * With a key sort (sort_mode 1 or 3) the keys are norm-sorted inside each
 * range separately, so no sorted key block mixes the two; queries are sorted
 * as in ba_select (sort_window applies to them only).
 *
 * prefill_len      tokens of the prefill part: a multiple of block with
 *                  0 < prefill_len < L, else BA_ERR_INVALID_ARG.
 * kappa_prefill    1 <= kappa_prefill <= prefill_len / block.
 * kappa_generation 1 <= kappa_generation <= N - prefill_len / block.
 * block_idx        int32 [b,h,N,kappa_prefill + kappa_generation], ascending
 *                  (prefill blocks first, as their ids are lower).
 * Other arguments, outputs, workspace (ba_select_workspace_size with kappa =
 * kappa_prefill + kappa_generation) and errors as in ba_select.  The result
 * feeds ba_sparse_attn with kappa = kappa_prefill + kappa_generation.
 */
int ba_select_isolated(const void *q, const void *k, int batch, int heads,
                       int seqlen, int head_dim, int block, int prefill_len,
                       int kappa_prefill, int kappa_generation, float beta,
                       int sort_mode, int sort_window, int32_t *perm_q,
                       int32_t *perm_k, int32_t *block_idx,
                       uint32_t *block_mask, float *block_scores,
                       void *workspace, size_t workspace_bytes,
                       ba_stream_t stream);

/*
 * Block-sparse attention: BA-Att paper Algorithm 1 step 12 (§2 block-sparse
 * attention; the masked softmax of SparseD §3.1 Eq. 3-4).  For the token at
 * sorted query position r (query block g = r / B):
 *     O[pi_q(r)]   = sum_{j in S(g)} softmax_j(scale * q . k_j) v_j
 *     lse[pi_q(r)] = ln sum_{j in S(g)} exp(scale * q . k_j)
 * where S(g) holds every token pi_k(p) whose sorted key position p lies in a
 * key block listed in block_idx[g].  Results are written in the ORIGINAL
 * token order (the paper's remap by pi_q^-1).
 *
 * q, k, v     bf16 [b,h,L,d], device.
 * perm_q, perm_k  int32 [b,h,L] as produced by ba_select, or NULL for the
 *             identity.  Each must be a permutation of 0..L-1 per (b,h)
 *             (not checked; an invalid one gives undefined results).
 * block_idx   int32 [b,h,N,kappa], strictly ascending ids < N per row (not
 *             checked on the device).
 * scale       logit scale; <= 0 selects 1/sqrt(d).
 * o           bf16 [b,h,L,d] output;  lse  fp32 [b,h,L] output (natural log).
 * Uses tcgen05 tensor-core MMAs (bf16 in, fp32 accumulate in tensor memory).
 */
size_t ba_sparse_attn_workspace_size(int batch, int heads, int seqlen,
                                     int head_dim, int block, int kappa,
                                     int has_perm_q, int has_perm_k);

int ba_sparse_attn(const void *q, const void *k, const void *v, int batch,
                   int heads, int seqlen, int head_dim, int block,
                   const int32_t *perm_q, const int32_t *perm_k,
                   const int32_t *block_idx, int kappa, float scale, void *o,
                   float *lse, void *workspace, size_t workspace_bytes,
                   ba_stream_t stream);

/*
 * LoSA locality pruning (the LoSA summary post, step 1): between two
 * denoising steps, per group of `group` consecutive tokens of each (b,h)
 * sequence (the block denoised in parallel; the last group may be short),
 * the `top_k` tokens whose query vectors changed most are active:
 *     mse[i]    = (1/d) sum_t (q_now[i,t] - q_prev[i,t])^2     (fp32)
 *     active[i] = 1 iff fewer than top_k tokens of i's group have a larger
 *                 mse, or an equal one at a lower index; else 0.
 * Stable tokens keep their cached attention result (see ba_reuse_rows);
 * active ones take a new one.
 *
 * q_now, q_prev  bf16 [b,h,L,d], device, 16-byte aligned.
 * group          1 <= group <= 1024; top_k >= 1 (top_k >= group: all active).
 * active         uint8 [b,h,L] output; mse: fp32 [b,h,L] output or NULL.
 * Errors: BA_ERR_INVALID_ARG (null or misaligned pointers, bad group or
 * top_k, empty shape), BA_ERR_UNSUPPORTED (d not 64/128, b*h > 65535).
 */
int ba_active_tokens(const void *q_now, const void *q_prev, int batch,
                     int heads, int seqlen, int head_dim, int group,
                     int top_k, uint8_t *active, float *mse,
                     ba_stream_t stream);

/*
 * The cache update of a LoSA step ("merge and update"): for every row r with
 * active[r] != 0, o_cache[r] = o_new[r] and lse_cache[r] = lse_new[r];
 * stable rows keep their cached values.  rows = b*h*L.
 * o_new, o_cache  bf16 [rows, d] (d = 64 or 128), device, 16-byte aligned;
 * lse_new, lse_cache fp32 [rows]; active uint8 [rows].  rows == 0 is a no-op.
 */
int ba_reuse_rows(const void *o_new, const float *lse_new,
                  const uint8_t *active, int64_t rows, int head_dim,
                  void *o_cache, float *lse_cache, ba_stream_t stream);

/*
 * Fidelity diagnostics of a block selection (BA-Att paper §3.1 Eq. 3 and
 * §3.2 Eq. 5-8), all over the sorted blocks that perm_q / perm_k define
 * (NULL = identity), with s_ij = q_i.k_j and the scale of the attention call
 * (<= 0 selects 1/sqrt(d)):
 *   mass[gq,gk]    = (1/|I(gq)|) sum_{i in I(gq), j in J(gk)} exp(scale s_ij - lse_i),
 *                    the oracle block mass of Eq. 3 (lse = the dense row
 *                    log-sum-exp, as ba_attn_dense writes it, original order);
 *   dev_max[gq,gk] = max_{i in I(gq), j in J(gk)} |scale s_ij - scale Qbar_gq.Kbar_gk|,
 *                    the largest token-vs-block logit deviation (Eq. 5);
 *   bound[gq,gk]   = scale (R^Q M^K + M^Q R^K + R^Q R^K), Eq. 7-8 (R the
 *                    block radii max ||x - mean||, M the block max norms);
 *   recall[gq]     = sum over the kappa blocks of block_idx[gq] of mass[gq,.],
 *                    the share of the dense attention mass a selection keeps.
 * Each row of mass sums to 1 up to rounding.
 *
 * q, k        bf16 [b,h,L,d], device.
 * lse         fp32 [b,h,L], device (required).
 * block_idx   int32 [b,h,N,kappa] (required when recall != NULL).
 * mass        fp32 [b,h,N,N] (required); dev_max, bound: fp32 [b,h,N,N] or
 *             NULL; recall: fp32 [b,h,N] or NULL.
 * workspace   ba_block_fidelity_workspace_size() bytes, 256-byte aligned:
 *             permuted row copies, block means, radii and norms, block logits.
 * Uses tcgen05 tensor-core MMAs for s (bf16 in, fp32 accumulate); mass and
 * dev_max are accumulated with atomics, so mass may differ in the last bits
 * between runs.  Errors as in ba_sparse_attn; bounded waits report through
 * ba_last_device_error.
 */
size_t ba_block_fidelity_workspace_size(int batch, int heads, int seqlen,
                                        int head_dim, int block);

int ba_block_fidelity(const void *q, const void *k, int batch, int heads,
                      int seqlen, int head_dim, int block,
                      const int32_t *perm_q, const int32_t *perm_k,
                      const float *lse, float scale,
                      const int32_t *block_idx, int kappa, float *mass,
                      float *dev_max, float *bound, float *recall,
                      void *workspace, size_t workspace_bytes,
                      ba_stream_t stream);

/*
 * Dense attention with the same kernel (every key block of every row, no
 * permutation): softmax(scale * Q K^T) V and its row LSE — the BA-Att
 * paper's Eq. 1, the dense reference its speedups are measured against.
 * Arguments as in ba_sparse_attn.  Needs no workspace.
 */
int ba_attn_dense(const void *q, const void *k, const void *v, int batch,
                  int heads, int seqlen, int head_dim, float scale, void *o,
                  float *lse, ba_stream_t stream);

/*
 * Merge of two attention results over DISJOINT key sets of the same rows, the
 * online-softmax combination of the LoSA summary post ("merge and update":
 * cached prefix attention joined with newly computed attention through the
 * log-normaliser):
 *     lse[r] = ln(exp(lse1[r]) + exp(lse2[r]))
 *     o[r]   = exp(lse1[r] - lse[r]) o1[r] + exp(lse2[r] - lse[r]) o2[r]
 * o1, o2, o   bf16 [rows, head_dim]; lse1, lse2, lse  fp32 [rows] (natural
 *             log, as ba_sparse_attn writes them).  Device pointers; o may
 *             be o1 or o2 and lse may be lse1 or lse2 (in place).
 * A part with lse = -inf (no keys) has weight 0; when both are -inf the row
 * gets o = 0, lse = -inf.  head_dim in {64, 128}; rows >= 0 (0: no-op).
 */
int ba_merge_lse(const void *o1, const float *lse1, const void *o2,
                 const float *lse2, int64_t rows, int head_dim, void *o,
                 float *lse, ba_stream_t stream);

/*
 * Checks a selection's outputs before they are used: BA-Att paper Algorithm 1
 * steps 1-2 make pi_q and pi_k permutations of each (b,h) sequence, and
 * steps 8-11 keep kappa distinct key blocks per query block (ba_select emits
 * them ascending).  ba_sparse_attn trusts these inputs: it never faults on
 * them (out-of-range entries are clamped or dropped), but then its result is
 * meaningless.  This call runs the checks on the device:
 *   perm_q, perm_k  int32 [b,h,L] or NULL (not checked): every entry in
 *                   [0, L) and no position twice in a sequence;
 *   block_idx       int32 [b,h,N,kappa] (required): every row strictly
 *                   ascending with ids in [0, N).
 * It is synchronous: it enqueues the checks on `stream`, waits for the
 * stream and returns BA_OK, or BA_ERR_INVALID_ARG with *detail (may be NULL)
 * set to the failed checks: bit 0 pi_q, bit 1 pi_k, bit 2 block_idx.  Not
 * for use during stream capture; concurrent calls share one device word and
 * must be serialised.  block is 64 or 128; shape limits as elsewhere
 * (BA_ERR_UNSUPPORTED / BA_ERR_INVALID_ARG before any launch).
 */
int ba_validate_selection(const int32_t *perm_q, const int32_t *perm_k,
                          const int32_t *block_idx, int batch, int heads,
                          int seqlen, int block, int kappa, uint32_t *detail,
                          ba_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device error word that
 * kernels set when a bounded wait gives up.  Returns BA_OK,
 * BA_ERR_DEVICE_TIMEOUT or BA_ERR_CUDA.  `detail` (may be NULL) receives the
 * raw word: bit 0 = timeout, bits 8-15 = the first site that gave up.
 */
int ba_last_device_error(ba_stream_t stream, uint32_t *detail);

/*
 * ba_selftest_wait_timeout: exercises the bounded-wait failure path that
 * ba_last_device_error reports, without a GPU fault.  Launches one warp on
 * `stream` that waits, for at most limit_us microseconds, for a phase of a
 * barrier on which nothing ever arrives; the wait gives up, records site 11
 * in the device error word and the kernel returns.  A following
 * ba_last_device_error() returns BA_ERR_DEVICE_TIMEOUT with detail
 * (11 << 8) | 1 and clears the word; the context stays usable.
 *   limit_us   1 .. 1000000; anything else returns BA_ERR_INVALID_ARG and
 *              launches nothing.
 * Returns BA_OK, or BA_ERR_CUDA if the launch fails.
 */
int ba_selftest_wait_timeout(uint32_t limit_us, ba_stream_t stream);

/*
 * ba_selftest_attn_stall: exercises the attention kernel's own failure path
 * (BA-Att paper Algorithm 1 step 12 is the kernel under test) without a GPU
 * fault.  Runs ba_attn_dense on the caller's buffers with one change: the
 * second K/V copy of every CTA (the first V block) is never issued.  The
 * softmax gives its first P-ready signal only once that copy has landed, so
 * the MMA-issuing thread's bounded wait for it runs out after limit_us
 * microseconds and records site 7 in the device error word.  Every role of
 * the CTA then unwinds: the copies and MMAs it issued complete, its tensor
 * memory is freed, and no O or LSE element is written.  A following
 * ba_last_device_error() returns BA_ERR_DEVICE_TIMEOUT with detail
 * (7 << 8) | 1 and clears the word; the context stays usable.
 *   q, k, v, o, lse, shape: as in ba_attn_dense; seqlen must exceed 128 (two
 *              key blocks), else BA_ERR_INVALID_ARG.
 *   limit_us   1 .. 1000000, else BA_ERR_INVALID_ARG.
 * Every CTA waits limit_us, in waves of one CTA per SM: keep the shape small.
 */
int ba_selftest_attn_stall(const void *q, const void *k, const void *v,
                           int batch, int heads, int seqlen, int head_dim,
                           uint32_t limit_us, void *o, float *lse,
                           ba_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BA_H_ */
