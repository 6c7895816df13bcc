"""Plain fp64 CPU oracle for Block Approximate Sparse Attention (BA-Att).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code, constants or helpers with the
CUDA library.

Sources (cited by page title and section/equation):

* "Efficient Long-Context Modeling in Diffusion Language Models via Block
  Approximate Sparse Attention" (the BA-Att paper), §2 Eq. 1 and block-sparse
  attention, §3.1 Eq. 2-3, §3.2 Eq. 5-8, §3.3 Eq. 9-10, §3.4 Eq. 11-14 and
  Algorithm 1.
* "SparseD: Sparse Attention for Diffusion Language Models", §3.1 Eq. 3-4
  (the 0 / -inf sparse mask added to the logits before the softmax).
* "SparseD: Sparse Attention for Diffusion Language Models", §3.3 "Isolated
  Selection", Eq. 5-6: prefill and generation keys are selected separately.
* The LoSA summary post ("merge and update" step): prefix and suffix attention
  results are combined through their log-normaliser (online softmax).

Everything is float64.  bf16 inputs are converted to float64 exactly by the
caller.  Loops run over (batch, head) and over query blocks; inside them the
only library primitives are matrix products, a stable argsort and lexsort.

Readings taken where the pages are silent or garbled (each one is restated
where it is used):

* Block statistics use the population variance (divide by n); Eq. 12 defines
  the covariance as an expectation over the block.
* The compensated logit is Eq. 13 with the Eq. 14 diagonal estimate, taken
  literally: l' = Qbar.Kbar / sqrt(d) + beta * (1/d) * sum_t(...three terms...).
* Top-kappa is ranked on l'; the softmax of Algorithm 1 step 9 is strictly
  increasing in each entry of a row, so it gives the same order.  Equal scores
  go to the lower key-block index.
* The norm sort is stable and non-decreasing (Eq. 10); equal norms keep the
  lower original index first.  ``window`` > 0 sorts each run of ``window``
  consecutive tokens on its own (Algorithm 1 step 1 says "(windowed) sort"
  without a size; 0 means one sort over the whole sequence).
* When L is not a multiple of B there are ceil(L/B) blocks and the last one
  is short; its statistics use its own token count.
* O and the log-sum-exp are returned in the original token order (Algorithm 1
  step 12, "remap ... via pi_q^-1").  LSE is the natural log of
  sum_j exp(scale * q.k_j) over the selected keys, scale = 1/sqrt(d) by
  default.
"""

from __future__ import annotations

import math

import numpy as np

SORT_NONE, SORT_K, SORT_Q, SORT_QK = 0, 1, 2, 3


# ---------------------------------------------------------------------------
# Norm-based ranking (BA-Att paper §3.3 Eq. 9-10; Algorithm 1 steps 1-2)
# ---------------------------------------------------------------------------

def token_norms(x: np.ndarray) -> np.ndarray:
    """Eq. 9: s_j = ||x_j||_2 for every token row of ``x`` [..., L, d]."""
    return np.sqrt(np.sum(x * x, axis=-1))


def norm_sort_permutation(s: np.ndarray, window: int = 0) -> np.ndarray:
    """Eq. 10: a permutation pi with s[pi[0]] <= s[pi[1]] <= ... (stable).

    ``s`` is one sequence of scores [L].  pi[r] is the original index of the
    token placed at sorted position r.  With ``window`` > 0 each run of
    ``window`` consecutive tokens is sorted independently.
    """
    L = s.shape[0]
    if window <= 0 or window >= L:
        return np.argsort(s, kind="stable").astype(np.int64)
    out = np.empty(L, dtype=np.int64)
    for w0 in range(0, L, window):
        w1 = min(L, w0 + window)
        out[w0:w1] = w0 + np.argsort(s[w0:w1], kind="stable")
    return out


def identity_permutation(L: int) -> np.ndarray:
    return np.arange(L, dtype=np.int64)


# ---------------------------------------------------------------------------
# Block partition and block statistics (Algorithm 1 steps 3-4; §3.1; Eq. 14)
# ---------------------------------------------------------------------------

def num_blocks(L: int, B: int) -> int:
    """Number of blocks: ceil(L / B); the last block may be short."""
    return -(-L // B)


def block_ranges(L: int, B: int):
    """Sorted-position ranges [start, end) of the consecutive blocks of size B."""
    return [(g * B, min(L, (g + 1) * B)) for g in range(num_blocks(L, B))]


def block_moments(x_sorted: np.ndarray, B: int):
    """Per-block mean and population variance per feature (Algorithm 1 step 4).

    ``x_sorted`` [L, d] is one sequence already in sorted order.  Returns
    (mean [N, d], var [N, d]).  Two passes: the mean first, then the mean of
    squared deviations (divide by the block's own token count).
    """
    L, d = x_sorted.shape
    ranges = block_ranges(L, B)
    mean = np.empty((len(ranges), d))
    var = np.empty((len(ranges), d))
    for g, (a, b) in enumerate(ranges):
        blk = x_sorted[a:b]
        mean[g] = blk.sum(axis=0) / (b - a)
        dev = blk - mean[g]
        var[g] = (dev * dev).sum(axis=0) / (b - a)
    return mean, var


def block_logits(qbar: np.ndarray, kbar: np.ndarray) -> np.ndarray:
    """Eq. 2 / Algorithm 1 step 5: l[gq, gk] = (Qbar_gq . Kbar_gk) / sqrt(d)."""
    d = qbar.shape[-1]
    return (qbar @ kbar.T) / math.sqrt(d)


def covariance_compensation(qbar, varq, kbar, vark) -> np.ndarray:
    """Eq. 14 / Algorithm 1 step 6: the diagonal-variance estimate of Delta.

    Delta[gq, gk] = (1/d) * sum_t ( VarQ[gq,t] * Kbar[gk,t]^2
                                  + VarK[gk,t] * Qbar[gq,t]^2
                                  + VarQ[gq,t] * VarK[gk,t] ).
    All three terms are kept, as printed.
    """
    d = qbar.shape[-1]
    t1 = varq @ (kbar * kbar).T
    t2 = (qbar * qbar) @ vark.T
    t3 = varq @ vark.T
    return (t1 + t2 + t3) / d


def compensated_logits(qbar, varq, kbar, vark, beta: float) -> np.ndarray:
    """Eq. 13 / Algorithm 1 step 7: l' = l + beta * Delta."""
    return block_logits(qbar, kbar) + beta * covariance_compensation(qbar, varq, kbar, vark)


def block_distribution(scores: np.ndarray) -> np.ndarray:
    """Algorithm 1 step 9 (and §3.1's m): row-wise softmax of the block logits."""
    z = scores - scores.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


# ---------------------------------------------------------------------------
# Top-kappa selection (Algorithm 1 steps 8-11)
# ---------------------------------------------------------------------------

def topk_blocks(scores: np.ndarray, kappa: int):
    """Keep the ``kappa`` highest-scoring key blocks of every query-block row.

    ``scores`` [Nq, Nk].  Ties go to the lower key-block index.  Returns
    (idx [Nq, kappa] ascending int64, mask [Nq, Nk] bool).
    """
    nq, nk = scores.shape
    if not 1 <= kappa <= nk:
        raise ValueError("kappa must lie in [1, Nk]")
    gk = np.broadcast_to(np.arange(nk), scores.shape)
    # lexsort: last key is primary -> descending score, then ascending index.
    order = np.lexsort((gk, -scores), axis=-1)
    idx = np.sort(order[:, :kappa], axis=-1).astype(np.int64)
    mask = np.zeros((nq, nk), dtype=bool)
    np.put_along_axis(mask, idx, True, axis=-1)
    return idx, mask


def kappa_for_sparsity(sparsity: float, nk: int) -> int:
    """Budget kappa for a requested sparsity: the fewest blocks whose density
    is at least (1 - sparsity), clamped to [1, Nk]."""
    k = math.ceil((1.0 - sparsity) * nk - 1e-9)
    return max(1, min(nk, k))


# ---------------------------------------------------------------------------
# Selection stage, one (batch, head) sequence, and batched
# ---------------------------------------------------------------------------

def select_one(q, k, B, kappa, beta=1.0, sort_mode=SORT_QK, window=0,
               perm_q=None, perm_k=None):
    """Algorithm 1 steps 1-11 for one sequence: q, k [L, d] float64.

    ``perm_q`` / ``perm_k`` override the sort (used to re-evaluate the later
    steps on a permutation produced elsewhere).  Returns a dict with the
    permutations, block moments, scores l', the index list and the mask.
    """
    L = q.shape[0]
    if perm_q is None:
        perm_q = (norm_sort_permutation(token_norms(q), window)
                  if sort_mode in (SORT_Q, SORT_QK) else identity_permutation(L))
    if perm_k is None:
        perm_k = (norm_sort_permutation(token_norms(k), window)
                  if sort_mode in (SORT_K, SORT_QK) else identity_permutation(L))
    perm_q = np.asarray(perm_q, dtype=np.int64)
    perm_k = np.asarray(perm_k, dtype=np.int64)
    qbar, varq = block_moments(q[perm_q], B)
    kbar, vark = block_moments(k[perm_k], B)
    scores = compensated_logits(qbar, varq, kbar, vark, beta)
    idx, mask = topk_blocks(scores, kappa)
    return dict(perm_q=perm_q, perm_k=perm_k, qbar=qbar, varq=varq, kbar=kbar,
                vark=vark, scores=scores, idx=idx, mask=mask)


def ba_select(Q, K, B, kappa, beta=1.0, sort_mode=SORT_QK, window=0,
              perm_q=None, perm_k=None):
    """Batched selection: Q, K [b, h, L, d] float64.

    Returns perm_q, perm_k [b, h, L]; idx [b, h, N, kappa]; mask [b, h, N, N];
    scores [b, h, N, N].
    """
    b, h, L, d = Q.shape
    N = num_blocks(L, B)
    out = dict(perm_q=np.empty((b, h, L), np.int64), perm_k=np.empty((b, h, L), np.int64),
               idx=np.empty((b, h, N, kappa), np.int64), mask=np.empty((b, h, N, N), bool),
               scores=np.empty((b, h, N, N)))
    for bi in range(b):
        for hi in range(h):
            r = select_one(Q[bi, hi], K[bi, hi], B, kappa, beta, sort_mode, window,
                           None if perm_q is None else perm_q[bi, hi],
                           None if perm_k is None else perm_k[bi, hi])
            for key in out:
                out[key][bi, hi] = r[key]
    return out


# ---------------------------------------------------------------------------
# Isolated selection (SparseD §3.3 "Isolated Selection", Eq. 5-6) over the
# BA-Att block scores
# ---------------------------------------------------------------------------
#
# SparseD splits the key dimension into prefill tokens [0, p) and generation
# tokens [p, L) and keeps the top share of each range on its own (Eq. 6), the
# selected set being the union of the two (Eq. 5).  Applied to BA-Att's block
# scores: p is a multiple of B, the key norm sort runs inside each range (so
# a sorted key block never mixes the two), and each query-block row keeps its
# kappa_pre best prefill blocks and its kappa_gen best generation blocks.

def split_sort_permutation(s: np.ndarray, split: int) -> np.ndarray:
    """Eq. 10's stable non-decreasing sort, run separately on [0, split) and
    [split, L): positions below ``split`` hold prefill tokens only."""
    L = s.shape[0]
    out = np.empty(L, dtype=np.int64)
    out[:split] = np.argsort(s[:split], kind="stable")
    out[split:] = split + np.argsort(s[split:], kind="stable")
    return out


def topk_blocks_isolated(scores: np.ndarray, n_pre: int, kappa_pre: int, kappa_gen: int):
    """Eq. 5-6: per row, the top ``kappa_pre`` of the first ``n_pre`` key
    blocks united with the top ``kappa_gen`` of the rest (ties to the lower
    index within each part).  Returns (idx [Nq, kappa_pre + kappa_gen]
    ascending, mask [Nq, Nk] bool)."""
    nq, nk = scores.shape
    idx_pre, _ = topk_blocks(scores[:, :n_pre], kappa_pre)
    idx_gen, _ = topk_blocks(scores[:, n_pre:], kappa_gen)
    idx = np.concatenate([idx_pre, idx_gen + n_pre], axis=1)
    mask = np.zeros((nq, nk), dtype=bool)
    np.put_along_axis(mask, idx, True, axis=-1)
    return idx, mask


def select_isolated_one(q, k, B, prefill_len, kappa_pre, kappa_gen, beta=1.0,
                        sort_mode=SORT_QK, window=0, perm_q=None, perm_k=None):
    """Isolated selection for one sequence (q, k [L, d] float64).  Queries
    are sorted as in ``select_one`` (``window`` applies to them); keys inside
    each of the two ranges.  ``perm_q`` / ``perm_k`` override the sorts."""
    L = q.shape[0]
    if prefill_len % B != 0 or not 0 < prefill_len < L:
        raise ValueError("prefill_len must be a multiple of B inside (0, L)")
    if perm_q is None:
        perm_q = (norm_sort_permutation(token_norms(q), window)
                  if sort_mode in (SORT_Q, SORT_QK) else identity_permutation(L))
    if perm_k is None:
        perm_k = (split_sort_permutation(token_norms(k), prefill_len)
                  if sort_mode in (SORT_K, SORT_QK) else identity_permutation(L))
    perm_q = np.asarray(perm_q, dtype=np.int64)
    perm_k = np.asarray(perm_k, dtype=np.int64)
    qbar, varq = block_moments(q[perm_q], B)
    kbar, vark = block_moments(k[perm_k], B)
    scores = compensated_logits(qbar, varq, kbar, vark, beta)
    idx, mask = topk_blocks_isolated(scores, prefill_len // B, kappa_pre, kappa_gen)
    return dict(perm_q=perm_q, perm_k=perm_k, qbar=qbar, varq=varq, kbar=kbar,
                vark=vark, scores=scores, idx=idx, mask=mask)


def ba_select_isolated(Q, K, B, prefill_len, kappa_pre, kappa_gen, beta=1.0,
                       sort_mode=SORT_QK, window=0, perm_q=None, perm_k=None):
    """Batched isolated selection, outputs shaped as in ``ba_select`` with
    kappa = kappa_pre + kappa_gen."""
    b, h, L, d = Q.shape
    N = num_blocks(L, B)
    kappa = kappa_pre + kappa_gen
    out = dict(perm_q=np.empty((b, h, L), np.int64), perm_k=np.empty((b, h, L), np.int64),
               idx=np.empty((b, h, N, kappa), np.int64), mask=np.empty((b, h, N, N), bool),
               scores=np.empty((b, h, N, N)))
    for bi in range(b):
        for hi in range(h):
            r = select_isolated_one(Q[bi, hi], K[bi, hi], B, prefill_len, kappa_pre, kappa_gen,
                                    beta, sort_mode, window,
                                    None if perm_q is None else perm_q[bi, hi],
                                    None if perm_k is None else perm_k[bi, hi])
            for key in out:
                out[key][bi, hi] = r[key]
    return out


# ---------------------------------------------------------------------------
# Block-sparse attention (Algorithm 1 step 12; §2; SparseD Eq. 3-4)
# ---------------------------------------------------------------------------

def sparse_attention_one(q, k, v, perm_q, perm_k, idx, B, scale=None, query_blocks=None):
    """Masked softmax attention for one sequence: q, k, v [L, d] float64.

    Query token i sits in sorted query block g = (position of i in perm_q)//B.
    Its key set is every original token perm_k[p] with p inside a selected key
    block of row g (idx[g]); all other logits get -inf (SparseD Eq. 4).  O and
    LSE are written at the original row i.  ``query_blocks`` restricts the
    work to some sorted query blocks; other rows are left as NaN.
    """
    L, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O = np.full((L, v.shape[1]), np.nan)
    lse = np.full(L, np.nan)
    qranges = block_ranges(L, B)
    kranges = block_ranges(L, B)
    blocks = range(len(qranges)) if query_blocks is None else query_blocks
    for g in blocks:
        a, b_ = qranges[g]
        rows = perm_q[a:b_]
        keys = np.concatenate([perm_k[kranges[j][0]:kranges[j][1]] for j in idx[g]])
        logits = scale * (q[rows] @ k[keys].T)
        m = logits.max(axis=1, keepdims=True)
        w = np.exp(logits - m)
        s = w.sum(axis=1, keepdims=True)
        O[rows] = (w @ v[keys]) / s
        lse[rows] = (m + np.log(s))[:, 0]
    return O, lse


def sparse_attention(Q, K, V, perm_q, perm_k, idx, B, scale=None, query_blocks=None):
    """Batched block-sparse attention: returns O [b, h, L, dv], LSE [b, h, L].

    ``query_blocks``, if given, maps (bi, hi) -> list of sorted query blocks.
    """
    b, h, L, d = Q.shape
    O = np.full((b, h, L, V.shape[-1]), np.nan)
    lse = np.full((b, h, L), np.nan)
    for bi in range(b):
        for hi in range(h):
            qb = None if query_blocks is None else query_blocks[(bi, hi)]
            O[bi, hi], lse[bi, hi] = sparse_attention_one(
                Q[bi, hi], K[bi, hi], V[bi, hi], perm_q[bi, hi], perm_k[bi, hi],
                idx[bi, hi], B, scale, qb)
    return O, lse


def dense_attention_one(q, k, v, scale=None, rows=None):
    """Eq. 1: softmax(scale * q k^T) v over every key, plus the row LSE."""
    d = q.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    qr = q if rows is None else q[rows]
    logits = scale * (qr @ k.T)
    m = logits.max(axis=1, keepdims=True)
    w = np.exp(logits - m)
    s = w.sum(axis=1, keepdims=True)
    return (w @ v) / s, (m + np.log(s))[:, 0]


def dense_attention(Q, K, V, scale=None):
    b, h, L, d = Q.shape
    O = np.empty((b, h, L, V.shape[-1]))
    lse = np.empty((b, h, L))
    for bi in range(b):
        for hi in range(h):
            O[bi, hi], lse[bi, hi] = dense_attention_one(Q[bi, hi], K[bi, hi], V[bi, hi], scale)
    return O, lse


# ---------------------------------------------------------------------------
# LSE merge (LoSA post, "merge and update": online-softmax combination)
# ---------------------------------------------------------------------------

def merge_lse(O1, lse1, O2, lse2):
    """Combine two attention results over disjoint key sets of the same rows.

    lse = log(exp(lse1) + exp(lse2)); O = exp(lse1 - lse) O1 + exp(lse2 - lse) O2.
    """
    lse = np.logaddexp(lse1, lse2)
    w1 = np.exp(lse1 - lse)[..., None]
    w2 = np.exp(lse2 - lse)[..., None]
    return w1 * O1 + w2 * O2, lse


# ---------------------------------------------------------------------------
# LoSA locality pruning and result reuse (the LoSA summary post, steps 1, 2
# and the cache update of step 4)
# ---------------------------------------------------------------------------
#
# Between two denoising steps most tokens' queries barely move.  Per block of
# ``group`` consecutive tokens (the block that is denoised in parallel), the
# ``top_k`` tokens whose query vectors changed most (mean squared error over
# the d features) are "active"; the rest are "stable" and keep the attention
# result (O and its log-normaliser) cached from the previous step.  Ties go to
# the lower token index; a short last group keeps min(top_k, its length).

def query_mse(q_now: np.ndarray, q_prev: np.ndarray) -> np.ndarray:
    """Per token: (1/d) * sum_t (q_now[t] - q_prev[t])^2, over the last axis."""
    diff = q_now - q_prev
    return np.mean(diff * diff, axis=-1)


def active_tokens(mse: np.ndarray, group: int, top_k: int) -> np.ndarray:
    """Boolean mask [L]: the top_k largest ``mse`` of every run of ``group``
    tokens (ties to the lower index)."""
    L = mse.shape[0]
    out = np.zeros(L, dtype=bool)
    for g0 in range(0, L, group):
        seg = mse[g0:g0 + group]
        order = np.lexsort((np.arange(len(seg)), -seg))
        out[g0 + order[:min(top_k, len(seg))]] = True
    return out


def reuse_rows(o_new, lse_new, o_cache, lse_cache, active):
    """The cache after a LoSA step: active rows take the new result, stable
    rows keep the cached one."""
    o = np.where(active[..., None], o_new, o_cache)
    lse = np.where(active, lse_new, lse_cache)
    return o, lse


# ---------------------------------------------------------------------------
# Fidelity diagnostics (BA-Att paper §3.1 Eq. 3 and §3.2 Eq. 7-8)
# ---------------------------------------------------------------------------

def oracle_block_mass(q, k, perm_q, perm_k, B, scale=None):
    """Eq. 3: m_hat[gq, gk] = (1/|I|) sum_{i in I(gq)} sum_{j in J(gk)} A_ij,
    with A the dense attention map of Eq. 1 and I, J the sorted blocks."""
    L, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    logits = scale * (q @ k.T)
    A = np.exp(logits - logits.max(axis=1, keepdims=True))
    A /= A.sum(axis=1, keepdims=True)
    qr, kr = block_ranges(L, B), block_ranges(L, B)
    out = np.empty((len(qr), len(kr)))
    for g, (a, b_) in enumerate(qr):
        rows = perm_q[a:b_]
        for j, (c, e) in enumerate(kr):
            out[g, j] = A[np.ix_(rows, perm_k[c:e])].sum() / (b_ - a)
    return out


def observed_deviation(q, k, perm_q, perm_k, B, scale=None):
    """§3.2: the largest |l_hat_ij - l_{gq,gk}| over the token pairs of each
    block pair, l_hat_ij = scale * q_i.k_j (Eq. 5's left side) and l the
    block logit of Eq. 2 with the same scale (1/sqrt(d) by default)."""
    L, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    qs, ks = q[perm_q], k[perm_k]
    qbar, _ = block_moments(qs, B)
    kbar, _ = block_moments(ks, B)
    rng = block_ranges(L, B)
    out = np.empty((len(rng), len(rng)))
    for g, (a, b_) in enumerate(rng):
        for j, (c, e) in enumerate(rng):
            tok = scale * (qs[a:b_] @ ks[c:e].T)
            out[g, j] = np.abs(tok - scale * (qbar[g] @ kbar[j])).max()
    return out


def deviation_bound(q, k, perm_q, perm_k, B):
    """Eq. 7-8: radii R, max norms M and the bound U[gq, gk] on |l_hat_ij - l|."""
    L, d = q.shape
    qs, ks = q[perm_q], k[perm_k]
    qbar, _ = block_moments(qs, B)
    kbar, _ = block_moments(ks, B)
    RQ = np.array([np.linalg.norm(qs[a:b_] - qbar[g], axis=1).max()
                   for g, (a, b_) in enumerate(block_ranges(L, B))])
    MQ = np.array([np.linalg.norm(qs[a:b_], axis=1).max() for a, b_ in block_ranges(L, B)])
    RK = np.array([np.linalg.norm(ks[a:b_] - kbar[g], axis=1).max()
                   for g, (a, b_) in enumerate(block_ranges(L, B))])
    MK = np.array([np.linalg.norm(ks[a:b_], axis=1).max() for a, b_ in block_ranges(L, B)])
    U = (RQ[:, None] * MK[None, :] + MQ[:, None] * RK[None, :] + RQ[:, None] * RK[None, :]) / math.sqrt(d)
    return dict(RQ=RQ, MQ=MQ, RK=RK, MK=MK, U=U)
