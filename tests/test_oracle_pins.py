"""Pins for the fp64 oracle: each check ties an oracle function to something
other than itself — a hand-worked example, a closed form, an exact identity,
a textbook library routine or brute force over tokens on tiny inputs.

The checks are plain functions so that ``test_planted_mistakes_are_caught``
can re-run them against deliberately broken copies of the oracle: every
plausible slip (a dropped term, a wrong normaliser, a flipped tie-break, a
missing scale, a swapped operand) must make at least one of them fail.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.ba_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_like(x):
    """Round float64 draws to bf16 values (the inputs the library sees)."""
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# checks
# ---------------------------------------------------------------------------

def check_hand_example():
    """The hand-worked L=4, d=2, B=2 example (BA-Att Algorithm 1, Eq. 2, 13, 14)."""
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        ex = json.load(f)
    Q = np.array(ex["Q"], float)
    K = np.array(ex["K"], float)
    d, B = ex["d"], ex["B"]
    for mode, part in ((O.SORT_NONE, ex["unsorted"]), (O.SORT_QK, ex["sorted"])):
        r = O.select_one(Q, K, B, kappa=1, beta=1.0, sort_mode=mode)
        if "perm_q" in part:
            assert r["perm_q"].tolist() == part["perm_q"]
            assert r["perm_k"].tolist() == part["perm_k"]
        for key in ("qbar", "varq", "kbar", "vark"):
            np.testing.assert_allclose(r[key], np.array(part[key]), rtol=0, atol=1e-12)
        expect = np.array(part["dot"]) / math.sqrt(d) + np.array(part["delta"])
        np.testing.assert_allclose(r["scores"], expect, rtol=0, atol=1e-12)
        assert r["idx"].tolist() == part["top1_beta1"]
        if "top1_beta0" in part:
            r0 = O.select_one(Q, K, B, kappa=1, beta=0.0, sort_mode=mode)
            np.testing.assert_allclose(r0["scores"], np.array(part["dot"]) / math.sqrt(d),
                                       rtol=0, atol=1e-12)
            assert r0["idx"].tolist() == part["top1_beta0"]


def check_sort_bruteforce():
    """Eq. 10: stable non-decreasing order, by brute force (duplicated rows make ties)."""
    rng = _rng(1)
    x = rng.standard_normal((23, 5))
    x[7] = x[3]
    x[19] = x[3]
    x[11] = -x[2]                      # same norm, different row
    s = O.token_norms(x)
    want = sorted(range(len(s)), key=lambda i: (math.sqrt(sum(v * v for v in x[i])), i))
    got = O.norm_sort_permutation(s).tolist()
    assert got == want
    for W in (4, 5, 8):
        got = O.norm_sort_permutation(s, window=W).tolist()
        want = []
        for w0 in range(0, len(s), W):
            want += sorted(range(w0, min(len(s), w0 + W)), key=lambda i: (s[i], i))
        assert got == want


def check_block_logit_bilinearity():
    """Eq. 2 equals the mean of the token logits over the block pair (ragged tail included)."""
    rng = _rng(2)
    L, d, B = 10, 3, 4
    q, k = rng.standard_normal((L, d)), rng.standard_normal((L, d))
    for mode in (O.SORT_NONE, O.SORT_QK):
        r = O.select_one(q, k, B, kappa=1, beta=0.0, sort_mode=mode)
        pq, pk = r["perm_q"], r["perm_k"]
        for gq, (a, b) in enumerate(O.block_ranges(L, B)):
            for gk, (c, e) in enumerate(O.block_ranges(L, B)):
                tot, n = 0.0, 0
                for i in pq[a:b]:
                    for j in pk[c:e]:
                        tot += sum(q[i, t] * k[j, t] for t in range(d)) / math.sqrt(d)
                        n += 1
                assert abs(r["scores"][gq, gk] - tot / n) < 1e-12


def check_compensation_identity():
    """Eq. 14 with population variances is exactly (1/d) sum_t Var_{i,j}(Q_it K_jt)
    over all token pairs of the block pair — brute force over pairs."""
    rng = _rng(3)
    L, d, B = 11, 4, 4
    q, k = rng.standard_normal((L, d)), rng.standard_normal((L, d)) * 1.7 + 0.3
    for mode in (O.SORT_NONE, O.SORT_QK):
        r0 = O.select_one(q, k, B, kappa=1, beta=0.0, sort_mode=mode)
        r1 = O.select_one(q, k, B, kappa=1, beta=1.0, sort_mode=mode)
        r2 = O.select_one(q, k, B, kappa=1, beta=2.5, sort_mode=mode)
        pq, pk = r1["perm_q"], r1["perm_k"]
        for gq, (a, b) in enumerate(O.block_ranges(L, B)):
            for gk, (c, e) in enumerate(O.block_ranges(L, B)):
                acc = 0.0
                for t in range(d):
                    prods = [q[i, t] * k[j, t] for i in pq[a:b] for j in pk[c:e]]
                    m = sum(prods) / len(prods)
                    acc += sum((p - m) ** 2 for p in prods) / len(prods)
                delta = acc / d
                assert abs((r1["scores"][gq, gk] - r0["scores"][gq, gk]) - delta) < 1e-12
                assert abs((r2["scores"][gq, gk] - r0["scores"][gq, gk]) - 2.5 * delta) < 1e-12


def check_deviation_bound():
    """Eq. 8: |l_hat_ij - l| <= U for every token pair of every block pair."""
    rng = _rng(4)
    L, d, B = 24, 6, 8
    q = rng.standard_normal((L, d)) * rng.uniform(0.2, 3.0, (L, 1))
    k = rng.standard_normal((L, d)) * rng.uniform(0.2, 3.0, (L, 1))
    for mode in (O.SORT_NONE, O.SORT_QK):
        r = O.select_one(q, k, B, kappa=1, beta=0.0, sort_mode=mode)
        bnd = O.deviation_bound(q, k, r["perm_q"], r["perm_k"], B)
        for gq, (a, b) in enumerate(O.block_ranges(L, B)):
            for gk, (c, e) in enumerate(O.block_ranges(L, B)):
                for i in r["perm_q"][a:b]:
                    for j in r["perm_k"][c:e]:
                        dev = abs(q[i] @ k[j] / math.sqrt(d) - r["scores"][gq, gk])
                        assert dev <= bnd["U"][gq, gk] + 1e-12


def check_deviation_hand_example():
    """Eq. 7-8 and the observed deviation on the hand-worked example: radii,
    max norms, U and the largest token-vs-block logit gap, each worked out
    by hand (tests/golden/hand_example.json, unsorted blocks)."""
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        ex = json.load(f)
    Q = np.array(ex["Q"], float)
    K = np.array(ex["K"], float)
    part = ex["unsorted"]
    ev = lambda x: eval(str(x), {"sqrt": math.sqrt})  # noqa: E731 (hand-written expressions)
    p = np.arange(4)
    bnd = O.deviation_bound(Q, K, p, p, 2)
    for key in ("RQ", "MQ", "RK", "MK"):
        np.testing.assert_allclose(bnd[key], [ev(x) for x in part["radii"][key]], atol=1e-12)
    want_u = np.array([[ev(x) for x in row] for row in part["U_times_sqrt_d"]]) / math.sqrt(2)
    np.testing.assert_allclose(bnd["U"], want_u, atol=1e-12)
    dev = O.observed_deviation(Q, K, p, p, 2)
    np.testing.assert_allclose(dev, np.array(part["max_dev_dot"], float) / math.sqrt(2), atol=1e-12)
    assert np.all(dev <= bnd["U"] + 1e-12)


def check_active_tokens():
    """LoSA locality pruning: the MSE is the plain per-token mean of squared
    differences (checked entry by entry in pure Python), each group keeps
    exactly min(top_k, group length) tokens, and those are the ones no other
    token of the group beats (larger MSE, or equal MSE and lower index) --
    brute force over integer-valued changes with ties."""
    rng = _rng(41)
    L, d = 37, 3
    prev = rng.integers(-2, 3, (L, d)).astype(float)
    now = prev + rng.integers(-1, 2, (L, d)).astype(float)
    mse = O.query_mse(now, prev)
    for i in range(L):
        assert mse[i] == sum((now[i, t] - prev[i, t]) ** 2 for t in range(d)) / d
    for group, k in ((8, 3), (5, 5), (16, 1), (37, 10)):
        act = O.active_tokens(mse, group, k)
        for g0 in range(0, L, group):
            idx = list(range(g0, min(L, g0 + group)))
            assert int(act[idx].sum()) == min(k, len(idx))
            for i in idx:
                beaten = sum(1 for j in idx if mse[j] > mse[i] or (mse[j] == mse[i] and j < i))
                assert act[i] == (beaten < k)
    # with exactly top_k moved tokens in every group, the active set is them
    now2 = prev.copy()
    moved = [1, 6, 9, 14, 17, 20, 25, 30, 33, 35]
    now2[moved] += 1.0
    act2 = O.active_tokens(O.query_mse(now2, prev), 8, 2)
    assert np.nonzero(act2)[0].tolist() == moved


def check_reuse_rows():
    """Active rows take the new result, stable rows keep the cache."""
    o_new, o_c = np.full((4, 2), 1.0), np.full((4, 2), 2.0)
    l_new, l_c = np.array([1.0, 1, 1, 1]), np.array([2.0, 2, 2, 2])
    act = np.array([True, False, True, False])
    o, l = O.reuse_rows(o_new, l_new, o_c, l_c, act)
    assert o[:, 0].tolist() == [1, 2, 1, 2] and l.tolist() == [1, 2, 1, 2]


def check_topk_bruteforce():
    """Algorithm 1 steps 8-11 by brute force, with exact ties (integer scores)."""
    rng = _rng(5)
    s = rng.integers(-3, 4, size=(9, 13)).astype(float)
    for kappa in (1, 4, 13):
        idx, mask = O.topk_blocks(s, kappa)
        for g in range(s.shape[0]):
            order = sorted(range(s.shape[1]), key=lambda j: (-s[g, j], j))
            want = sorted(order[:kappa])
            assert idx[g].tolist() == want
            assert mask[g].sum() == kappa and all(mask[g, j] for j in want)


def check_topk_equals_softmax_order():
    """Ranking by m' = softmax(l') (Algorithm 1 step 9-10) equals ranking by l'."""
    rng = _rng(6)
    s = rng.standard_normal((7, 40)) * 3
    m = O.block_distribution(s)
    np.testing.assert_allclose(m.sum(axis=1), 1.0, atol=1e-12)
    for kappa in (1, 10, 39):
        a, _ = O.topk_blocks(s, kappa)
        b, _ = O.topk_blocks(m, kappa)
        assert (a == b).all()


def check_all_blocks_is_dense_attention():
    """kappa = N: block-sparse attention is softmax attention over every key
    (Eq. 1), for any sort; compared against torch's SDPA in float64 and
    scipy's logsumexp."""
    from scipy.special import logsumexp
    rng = _rng(7)
    b, h, L, d, B = 1, 2, 40, 8, 8
    Q = _bf16_like(rng.standard_normal((b, h, L, d)))
    K = _bf16_like(rng.standard_normal((b, h, L, d)))
    V = _bf16_like(rng.standard_normal((b, h, L, d)))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V)).numpy()
    lse_ref = logsumexp(np.einsum("bhid,bhjd->bhij", Q, K) / math.sqrt(d), axis=-1)
    N = O.num_blocks(L, B)
    for mode in (O.SORT_NONE, O.SORT_K, O.SORT_Q, O.SORT_QK):
        sel = O.ba_select(Q, K, B, N, 1.0, mode)
        assert sel["mask"].all()
        out, lse = O.sparse_attention(Q, K, V, sel["perm_q"], sel["perm_k"], sel["idx"], B)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
    out, lse = O.dense_attention(Q, K, V)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def check_constant_v():
    """With V constant over tokens, O equals that constant whatever the mask."""
    rng = _rng(8)
    L, d, B = 37, 8, 8
    q, k = rng.standard_normal((L, d)), rng.standard_normal((L, d)) * 2
    row = rng.standard_normal(d)
    v = np.tile(row, (L, 1))
    r = O.select_one(q, k, B, kappa=2, beta=1.0, sort_mode=O.SORT_QK)
    out, _ = O.sparse_attention_one(q, k, v, r["perm_q"], r["perm_k"], r["idx"], B)
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-12)


def check_masked_softmax_bruteforce():
    """Token-level masked softmax with M_S in {0, -inf} (SparseD Eq. 3-4) by
    pure-Python loops, including the pi_q^-1 remap and a ragged last block."""
    rng = _rng(9)
    L, d, B, kappa = 14, 3, 4, 2
    q, k, v = (rng.standard_normal((L, d)) for _ in range(3))
    scale = 0.7
    r = O.select_one(q, k, B, kappa=kappa, beta=1.0, sort_mode=O.SORT_QK)
    out, lse = O.sparse_attention_one(q, k, v, r["perm_q"], r["perm_k"], r["idx"], B, scale=scale)
    pos_q = {int(t): p for p, t in enumerate(r["perm_q"])}
    pos_k = {int(t): p for p, t in enumerate(r["perm_k"])}
    for i in range(L):
        g = pos_q[i] // B
        logits = []
        for j in range(L):
            allowed = (pos_k[j] // B) in set(r["idx"][g].tolist())
            logits.append(scale * sum(q[i, t] * k[j, t] for t in range(d)) if allowed else -math.inf)
        m = max(logits)
        w = [math.exp(x - m) if x != -math.inf else 0.0 for x in logits]
        s = sum(w)
        for t in range(d):
            assert abs(out[i, t] - sum(w[j] * v[j, t] for j in range(L)) / s) < 1e-12
        assert abs(lse[i] - (m + math.log(s))) < 1e-12


def check_lse_merge():
    """Splitting each row's key blocks into two disjoint halves and merging the
    two results through their LSE (LoSA "merge and update") gives the single call."""
    rng = _rng(10)
    L, d, B, kappa = 48, 8, 8, 4
    q, k, v = (rng.standard_normal((L, d)) for _ in range(3))
    r = O.select_one(q, k, B, kappa=kappa, beta=1.0, sort_mode=O.SORT_QK)
    full, lse = O.sparse_attention_one(q, k, v, r["perm_q"], r["perm_k"], r["idx"], B)
    o1, l1 = O.sparse_attention_one(q, k, v, r["perm_q"], r["perm_k"], r["idx"][:, :2], B)
    o2, l2 = O.sparse_attention_one(q, k, v, r["perm_q"], r["perm_k"], r["idx"][:, 2:], B)
    om, lm = O.merge_lse(o1, l1, o2, l2)
    np.testing.assert_allclose(om, full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lm, lse, rtol=0, atol=1e-12)


def check_ragged_tail_moments():
    """L not a multiple of B: ceil(L/B) blocks, the last one short; its moments
    use its own count (population mean/variance of its rows, by hand)."""
    x = np.arange(30, dtype=float).reshape(10, 3) ** 1.5
    mean, var = O.block_moments(x, 4)
    assert mean.shape == (3, 3)
    tail = x[8:10]
    for t in range(3):
        m = (tail[0, t] + tail[1, t]) / 2
        assert abs(mean[2, t] - m) < 1e-12
        assert abs(var[2, t] - ((tail[0, t] - m) ** 2 + (tail[1, t] - m) ** 2) / 2) < 1e-12


def check_kappa_rule():
    assert O.kappa_for_sparsity(0.9, 256) == 26
    assert O.kappa_for_sparsity(0.75, 256) == 64
    assert O.kappa_for_sparsity(0.5, 512) == 256
    assert O.kappa_for_sparsity(0.5, 16) == 8
    assert O.kappa_for_sparsity(0.999, 16) == 1
    assert O.kappa_for_sparsity(0.0, 16) == 16


def check_block_mass():
    """Eq. 3: each query-block row of m_hat sums to 1; with B=1 it is A itself."""
    rng = _rng(11)
    L, d = 12, 4
    q, k = rng.standard_normal((L, d)), rng.standard_normal((L, d))
    p = np.arange(L)
    m = O.oracle_block_mass(q, k, p, p, 3)
    np.testing.assert_allclose(m.sum(axis=1), 1.0, atol=1e-12)
    A = O.oracle_block_mass(q, k, p, p, 1)
    logits = q @ k.T / 2.0
    ref = np.exp(logits) / np.exp(logits).sum(axis=1, keepdims=True)
    np.testing.assert_allclose(A, ref, atol=1e-12)


def check_isolated_sort():
    """The split sort is Eq. 10 inside each range: with the split in the
    middle it equals the windowed sort (window = L/2); for any split each
    range holds its own tokens, non-decreasing, equal norms by lower index
    (brute force over positions)."""
    rng = _rng(31)
    L = 24
    s = rng.integers(0, 5, L).astype(float)       # many equal norms
    np.testing.assert_array_equal(O.split_sort_permutation(s, L // 2),
                                  O.norm_sort_permutation(s, window=L // 2))
    for split in (4, 10, 20):
        p = O.split_sort_permutation(s, split)
        for lo, hi in ((0, split), (split, L)):
            seg = p[lo:hi]
            assert sorted(seg.tolist()) == list(range(lo, hi))
            for a, b in zip(seg[:-1], seg[1:]):
                assert s[a] < s[b] or (s[a] == s[b] and a < b)


def check_isolated_topk_bruteforce():
    """Eq. 5-6: each part's chosen set is, among all sets of its size inside
    its own key range, the one with the largest score sum, equal sums going
    to the lexicographically smallest index set (= ties to the lower index).
    Integer scores make the sums exact and create ties."""
    from itertools import combinations
    rng = _rng(32)
    nq, nk, n_pre = 5, 8, 3
    scores = rng.integers(-3, 4, (nq, nk)).astype(float)
    for kpre, kgen in ((1, 1), (2, 3), (3, 5)):
        idx, mask = O.topk_blocks_isolated(scores, n_pre, kpre, kgen)
        for r in range(nq):
            want = []
            for lo, hi, kk in ((0, n_pre, kpre), (n_pre, nk, kgen)):
                best = min(combinations(range(lo, hi), kk),
                           key=lambda c: (-sum(scores[r, j] for j in c), c))
                want += list(best)
            assert idx[r].tolist() == want
            assert mask[r].tolist() == [j in want for j in range(nk)]


def check_isolated_keeps_generation_block():
    """SparseD's motivation for isolating (§3.3): when prefill keys dominate
    the scores, a plain top-kappa spends the whole budget on prefill blocks,
    while the isolated selection still keeps the best generation block."""
    B, d = 4, 4
    e = np.eye(d)
    q = np.tile(e[0], (16, 1))                        # 4 query blocks along e0
    k = np.concatenate([np.tile(3 * e[0], (8, 1)),    # prefill blocks 0-1: strong
                        np.tile(-1 * e[0], (4, 1)),   # generation block 2: negative
                        np.tile(1 * e[0], (4, 1))])   # generation block 3: weak but best
    plain = O.select_one(q, k, B, 2, 0.0, O.SORT_NONE)
    assert plain["idx"].tolist() == [[0, 1]] * 4
    iso = O.select_isolated_one(q, k, B, 8, 1, 1, 0.0, O.SORT_NONE)
    assert iso["idx"].tolist() == [[0, 3]] * 4


ALL_CHECKS = [check_hand_example, check_sort_bruteforce, check_block_logit_bilinearity,
              check_compensation_identity, check_deviation_bound, check_topk_bruteforce,
              check_topk_equals_softmax_order, check_all_blocks_is_dense_attention,
              check_constant_v, check_masked_softmax_bruteforce, check_lse_merge,
              check_ragged_tail_moments, check_kappa_rule, check_block_mass,
              check_isolated_sort, check_isolated_topk_bruteforce, check_deviation_hand_example,
              check_active_tokens, check_reuse_rows,
              check_isolated_keeps_generation_block]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check()


def test_planted_selection_tiny():
    """Workload 1 (tiny): the four planted key blocks are among the top kappa=8
    of the chosen query block's row when tokens are not sorted, for beta 0 and 1."""
    import workloads
    w = workloads.get("tiny")
    q, k, v, meta = workloads.make_inputs(w)
    Q = q.double().numpy()
    K = k.double().numpy()
    for beta in (0.0, 1.0):
        r = O.select_one(Q[0, 0], K[0, 0], w.block, w.kappa(), beta, O.SORT_NONE)
        row = set(r["idx"][meta["query_block"]].tolist())
        assert set(meta["planted_key_blocks"]) <= row


def test_permutation_equivariance():
    """Relabelling tokens (the same permutation applied to Q, K, V rows)
    permutes the outputs the same way, including with sorting on."""
    rng = _rng(12)
    L, d, B = 32, 4, 8
    q, k, v = (rng.standard_normal((L, d)) for _ in range(3))
    perm = rng.permutation(L)
    r1 = O.select_one(q, k, B, 2, 1.0, O.SORT_QK)
    o1, l1 = O.sparse_attention_one(q, k, v, r1["perm_q"], r1["perm_k"], r1["idx"], B)
    r2 = O.select_one(q[perm], k[perm], B, 2, 1.0, O.SORT_QK)
    o2, l2 = O.sparse_attention_one(q[perm], k[perm], v[perm], r2["perm_q"], r2["perm_k"], r2["idx"], B)
    np.testing.assert_allclose(o2, o1[perm], atol=1e-12)
    np.testing.assert_allclose(l2, l1[perm], atol=1e-12)


# ---------------------------------------------------------------------------
# planted mistakes: each broken oracle must fail at least one check
# ---------------------------------------------------------------------------

def _moments_sample_var(x_sorted, B):
    mean, var = _ORIG["block_moments"](x_sorted, B)
    out = var.copy()
    for g, (a, b) in enumerate(O.block_ranges(x_sorted.shape[0], B)):
        n = b - a
        if n > 1:
            out[g] = var[g] * n / (n - 1)
    return mean, out


def _comp_drop_third(qbar, varq, kbar, vark):
    d = qbar.shape[-1]
    return (varq @ (kbar * kbar).T + (qbar * qbar) @ vark.T) / d


def _comp_sqrt_d(qbar, varq, kbar, vark):
    d = qbar.shape[-1]
    return _ORIG["covariance_compensation"](qbar, varq, kbar, vark) * d / math.sqrt(d)


def _comp_swapped(qbar, varq, kbar, vark):
    d = qbar.shape[-1]
    return (varq @ kbar.T + (qbar * qbar) @ vark.T + varq @ vark.T) / d


def _logits_no_scale(qbar, kbar):
    return qbar @ kbar.T


def _topk_high_index(scores, kappa):
    nq, nk = scores.shape
    gk = np.broadcast_to(-np.arange(nk), scores.shape)
    order = np.lexsort((gk, -scores), axis=-1)
    idx = np.sort(order[:, :kappa], axis=-1)
    mask = np.zeros((nq, nk), bool)
    np.put_along_axis(mask, idx, True, axis=-1)
    return idx, mask


def _sort_descending(s, window=0):
    return _ORIG["norm_sort_permutation"](-s, window)


def _sort_unstable(s, window=0):
    # equal norms in reverse index order
    return np.lexsort((-np.arange(len(s)), s))


def _attn_rows_unpermuted(q, k, v, perm_q, perm_k, idx, B, scale=None, query_blocks=None):
    return _ORIG["sparse_attention_one"](q, k, v, np.arange(len(perm_q)), perm_k, idx, B, scale, query_blocks)


def _attn_lse_no_max(q, k, v, perm_q, perm_k, idx, B, scale=None, query_blocks=None):
    out, lse = _ORIG["sparse_attention_one"](q, k, v, perm_q, perm_k, idx, B, scale, query_blocks)
    return out, lse - 1e-3


def _split_sort_whole(s, split):
    return _ORIG["norm_sort_permutation"](s, 0)


def _isolated_no_offset(scores, n_pre, kappa_pre, kappa_gen):
    nq, nk = scores.shape
    idx_pre, _ = O.topk_blocks(scores[:, :n_pre], kappa_pre)
    idx_gen, _ = O.topk_blocks(scores[:, n_pre:], kappa_gen)
    idx = np.concatenate([idx_pre, idx_gen], axis=1)
    mask = np.zeros((nq, nk), bool)
    np.put_along_axis(mask, np.clip(idx, 0, nk - 1), True, axis=-1)
    return idx, mask


def _isolated_joint(scores, n_pre, kappa_pre, kappa_gen):
    return O.topk_blocks(scores, kappa_pre + kappa_gen)


def _mse_sum(q_now, q_prev):
    diff = q_now - q_prev
    return np.sum(diff * diff, axis=-1)


def _active_high_tie(mse, group, top_k):
    L = mse.shape[0]
    out = np.zeros(L, dtype=bool)
    for g0 in range(0, L, group):
        seg = mse[g0:g0 + group]
        order = np.lexsort((-np.arange(len(seg)), -seg))
        out[g0 + order[:min(top_k, len(seg))]] = True
    return out


_ORIG = {n: getattr(O, n) for n in ("block_moments", "covariance_compensation", "block_logits",
                                      "topk_blocks", "norm_sort_permutation", "sparse_attention_one",
                                      "split_sort_permutation", "topk_blocks_isolated")}

MUTANTS = [
    ("block_moments", _moments_sample_var),
    ("covariance_compensation", _comp_drop_third),
    ("covariance_compensation", _comp_sqrt_d),
    ("covariance_compensation", _comp_swapped),
    ("block_logits", _logits_no_scale),
    ("topk_blocks", _topk_high_index),
    ("norm_sort_permutation", _sort_descending),
    ("norm_sort_permutation", _sort_unstable),
    ("sparse_attention_one", _attn_rows_unpermuted),
    ("sparse_attention_one", _attn_lse_no_max),
    ("split_sort_permutation", _split_sort_whole),
    ("topk_blocks_isolated", _isolated_no_offset),
    ("topk_blocks_isolated", _isolated_joint),
    ("query_mse", _mse_sum),
    ("active_tokens", _active_high_tie),
]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=lambda m: getattr(m, "__name__", str(m)))
def test_planted_mistakes_are_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(O, name, mutant)
    failed = []
    for check in ALL_CHECKS:
        try:
            check()
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant {mutant.__name__} of {name} passed every pin"
