"""Comparison helpers for the GPU parity tests (test code, not the oracle).

The tolerances are the ones the method's acceptance criteria state:
  * block mask: bit-exact, except blocks whose score lies within 1e-4
    (relative) of the row's kappa-th score;
  * O: max |err| <= 2e-2 and mean |err| <= 2e-3 against the oracle evaluated
    on the GPU's permutation and mask (bf16 inputs, fp32 accumulation);
  * LSE: |err| <= 1e-3.
Block scores l' = a . b are fp32 dot products of length 3d on the GPU; their
rounding error grows with the dot product's condition sum_t |a_t b_t| (which
bounds |l'|), so they are compared to 2e-5 of max(row max |l'|, that sum).
Permutations come from fp32 squared norms on the GPU and fp64 norms in the
oracle: where norms are within rounding of each other several orders are
correct, so the check is that the GPU's pi is a permutation, sorted under the
fp64 norms up to a relative 1e-5, and equal to the oracle's pi except at
positions whose tokens have norms within that tolerance.
"""

from __future__ import annotations

import numpy as np

MASK_REL = 1e-4
SCORE_REL = 2e-5
O_MAX, O_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3
NORM_REL = 1e-5


def to64(t):
    return t.detach().to("cpu").double().numpy()


def check_perm(perm_gpu: np.ndarray, perm_oracle: np.ndarray, x64: np.ndarray, window: int = 0):
    """perm arrays [b,h,L]; x64 [b,h,L,d]."""
    b, h, L = perm_gpu.shape
    s = np.sum(x64 * x64, axis=-1)  # squared norms, same order as norms
    W = L if window <= 0 else window
    n_diff = 0
    for bi in range(b):
        for hi in range(h):
            p = perm_gpu[bi, hi].astype(np.int64)
            assert np.array_equal(np.sort(p), np.arange(L)), "not a permutation"
            for w0 in range(0, L, W):
                seg = p[w0:w0 + W]
                assert seg.min() >= w0 and seg.max() < w0 + W, "token left its sort window"
                ss = s[bi, hi, seg]
                assert np.all(ss[1:] >= ss[:-1] - NORM_REL * np.abs(ss[:-1])), "not sorted"
            po = perm_oracle[bi, hi]
            diff = np.nonzero(p != po)[0]
            n_diff += len(diff)
            if len(diff):
                a, c = s[bi, hi, p[diff]], s[bi, hi, po[diff]]
                assert np.all(np.abs(a - c) <= NORM_REL * np.maximum(np.abs(a), np.abs(c))), \
                    "permutation differs beyond norm ties"
    return n_diff


def check_mask(idx_gpu, mask_words_gpu, scores_oracle, kappa, scores_gpu=None):
    """idx [b,h,N,kappa] int, mask words [b,h,N,W] (int32 view of uint32),
    scores_oracle [b,h,N,N] fp64 on the GPU's permutation.  Returns the
    number of near-threshold differences tolerated."""
    b, h, N, _ = scores_oracle.shape
    words = mask_words_gpu.astype(np.int64) & 0xFFFFFFFF
    bits = ((words[..., :, None] >> np.arange(32)) & 1).reshape(b, h, N, -1)[..., :N].astype(bool)
    tolerated = 0
    for bi in range(b):
        for hi in range(h):
            for g in range(N):
                row = idx_gpu[bi, hi, g]
                assert len(row) == kappa
                assert np.all(np.diff(row) > 0), "index list not strictly ascending"
                assert row.min() >= 0 and row.max() < N
                m = np.zeros(N, bool)
                m[row] = True
                assert np.array_equal(m, bits[bi, hi, g]), "bitmask disagrees with index list"
                sc = scores_oracle[bi, hi, g]
                order = np.lexsort((np.arange(N), -sc))
                want = np.zeros(N, bool)
                want[order[:kappa]] = True
                if np.array_equal(want, m):
                    continue
                thr = sc[order[kappa - 1]]
                tol = MASK_REL * max(abs(thr), 1e-30)
                diff = np.nonzero(want != m)[0]
                near = np.abs(sc[diff] - thr) <= tol
                if scores_gpu is not None:
                    sg = scores_gpu[bi, hi, g]
                    og = np.lexsort((np.arange(N), -sg))
                    tg = sg[og[kappa - 1]]
                    near |= np.abs(sg[diff] - tg) <= MASK_REL * max(abs(tg), 1e-30)
                assert np.all(near), f"mask differs away from the threshold (b{bi} h{hi} row {g})"
                tolerated += len(diff)
    return tolerated


def check_topk_of_own_scores(idx_gpu, scores_gpu, kappa):
    """The GPU's list is exactly the top-kappa of its own fp32 scores (ties:
    lower index) — an integer decision taken in the kernel's precision."""
    b, h, N, _ = scores_gpu.shape
    for bi in range(b):
        for hi in range(h):
            sc = scores_gpu[bi, hi].astype(np.float32)
            order = np.lexsort((np.broadcast_to(np.arange(N), sc.shape), -sc), axis=-1)
            want = np.sort(order[:, :kappa], axis=-1)
            assert np.array_equal(want, idx_gpu[bi, hi]), f"top-kappa of own scores (b{bi} h{hi})"


def check_attention(o_gpu, lse_gpu, o_ref, lse_ref, rows=None):
    """o [.., L, d] / lse [.., L]; ``rows`` is a boolean mask of rows to compare."""
    if rows is not None:
        o_gpu, o_ref = o_gpu[rows], o_ref[rows]
        lse_gpu, lse_ref = lse_gpu[rows], lse_ref[rows]
    assert np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(lse_gpu))
    err = np.abs(o_gpu - o_ref)
    lerr = np.abs(lse_gpu - lse_ref)
    stats = dict(o_max=float(err.max()), o_mean=float(err.mean()), lse_max=float(lerr.max()))
    assert stats["o_max"] <= O_MAX, stats
    assert stats["o_mean"] <= O_MEAN, stats
    assert stats["lse_max"] <= LSE_TOL, stats
    return stats


def score_condition(Q64, K64, perm_q, perm_k, B, beta):
    """sum_t |a_t b_t| per block pair [b,h,N,N] for the augmented vectors of
    Eq. 13-14 (a = [Qbar/sqrt(d), beta/d VarQ, beta/d Qbar^2],
    b = [Kbar, Kbar^2 + VarK, VarK]), from the oracle's fp64 block moments on
    the given permutations."""
    import oracle.ba_oracle as O

    b, h, L, d = Q64.shape
    N = O.num_blocks(L, B)
    out = np.empty((b, h, N, N))
    for bi in range(b):
        for hi in range(h):
            qbar, varq = O.block_moments(Q64[bi, hi][perm_q[bi, hi]], B)
            kbar, vark = O.block_moments(K64[bi, hi][perm_k[bi, hi]], B)
            c = np.abs(qbar) @ np.abs(kbar).T / np.sqrt(d)
            c += abs(beta) / d * (varq @ (kbar * kbar + vark).T + (qbar * qbar) @ vark.T)
            out[bi, hi] = c
    return out


def check_scores(scores_gpu, scores_oracle, Q64, K64, perm_q, perm_k, B, beta):
    """|l'_gpu - l'_oracle| <= SCORE_REL * max(row max |l'|, sum_t |a_t b_t|)."""
    sg = scores_gpu.astype(np.float64)
    so = scores_oracle
    row = np.maximum(np.abs(so).max(axis=-1, keepdims=True), 1e-6)
    scale = np.maximum(row, score_condition(Q64, K64, perm_q, perm_k, B, beta))
    err = np.abs(sg - so)
    assert np.all(err <= SCORE_REL * scale), float((err / scale).max())
