"""CPU checks of the comparison helpers the GPU parity tests rely on."""

from __future__ import annotations

import numpy as np

import oracle.ba_oracle as O
from parity import SCORE_REL, check_scores, score_condition


def _inputs(seed, b=1, h=2, L=300, d=64):
    rng = np.random.default_rng(seed)
    Q = rng.normal(size=(b, h, L, d)) * 1.5
    K = rng.normal(size=(b, h, L, d)) * 1.5
    perm = np.stack([np.stack([rng.permutation(L) for _ in range(h)]) for _ in range(b)])
    return Q, K, perm


def test_condition_bounds_the_scores():
    """|l'| <= sum_t |a_t b_t| for every block pair, beta 0 and 1."""
    Q, K, perm = _inputs(1)
    for beta in (0.0, 1.0, 0.5):
        so = O.ba_select(Q, K, 64, 2, beta, O.SORT_NONE, perm_q=perm, perm_k=perm)["scores"]
        c = score_condition(Q, K, perm, perm, 64, beta)
        assert np.all(np.abs(so) <= c * (1 + 1e-12) + 1e-15)


def test_condition_is_exact_for_same_sign_terms():
    """With non-negative Q and K every term of a . b is non-negative, so the
    condition equals the score itself."""
    Q, K, perm = _inputs(2)
    Q, K = np.abs(Q), np.abs(K)
    so = O.ba_select(Q, K, 64, 2, 1.0, O.SORT_NONE, perm_q=perm, perm_k=perm)["scores"]
    c = score_condition(Q, K, perm, perm, 64, 1.0)
    assert np.allclose(c, so, rtol=1e-12, atol=0)


def test_single_token_blocks():
    """One token per block: no variance, the condition is sum |q_t k_t| / sqrt(d)."""
    Q, K, _ = _inputs(3, L=1, d=128)
    ident = np.zeros((1, 2, 1), dtype=np.int64)
    c = score_condition(Q, K, ident, ident, 128, 1.0)
    want = np.abs(Q[..., 0, :] * K[..., 0, :]).sum(-1) / np.sqrt(128)
    assert np.allclose(c[..., 0, 0], want, rtol=1e-12)


def test_check_scores_rejects_an_error_above_the_bound():
    Q, K, perm = _inputs(4)
    so = O.ba_select(Q, K, 64, 2, 1.0, O.SORT_NONE, perm_q=perm, perm_k=perm)["scores"]
    c = np.maximum(score_condition(Q, K, perm, perm, 64, 1.0),
                   np.abs(so).max(axis=-1, keepdims=True))
    check_scores(so + 0.5 * SCORE_REL * c, so, Q, K, perm, perm, 64, 1.0)
    bad = so.copy()
    bad[0, 1, 2, 3] += 3 * SCORE_REL * c[0, 1, 2, 3]
    try:
        check_scores(bad, so, Q, K, perm, perm, 64, 1.0)
    except AssertionError:
        return
    raise AssertionError("an error of 3x the bound was accepted")
