"""GPU parity of the SparseD-style variants against the fp64 oracle:

* isolated selection ("SparseD: Sparse Attention for Diffusion Language
  Models", §3.3 "Isolated Selection", Eq. 5-6) over BA-Att's block scores,
  through ``ba_select_isolated``, and attention on its lists;
* reuse of one selection across denoising steps (SparseD §3.3): the
  permutations and block lists of one step's Q, K drive attention on the next
  step's Q, K, V.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import block_sparse_bidirectional_gb300 as bsb
import oracle.ba_oracle as O
import workloads
from parity import MASK_REL, NORM_REL, check_attention, check_perm, check_scores, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    bsb.load()
    return torch.device("cuda:0")


def _check_split_perm(perm_gpu, perm_oracle, x64, split):
    """Each range [0, split), [split, L) holds its own tokens, sorted under
    the fp64 norms up to NORM_REL, equal to the oracle except at norm ties."""
    s = np.sum(x64 * x64, axis=-1)
    b, h, L = perm_gpu.shape
    for bi in range(b):
        for hi in range(h):
            p = perm_gpu[bi, hi].astype(np.int64)
            for lo, hi_ in ((0, split), (split, L)):
                seg = p[lo:hi_]
                assert np.array_equal(np.sort(seg), np.arange(lo, hi_)), "token left its range"
                ss = s[bi, hi, seg]
                assert np.all(ss[1:] >= ss[:-1] - NORM_REL * np.abs(ss[:-1])), "not sorted"
            po = perm_oracle[bi, hi]
            diff = np.nonzero(p != po)[0]
            if len(diff):
                a, c = s[bi, hi, p[diff]], s[bi, hi, po[diff]]
                assert np.all(np.abs(a - c) <= NORM_REL * np.maximum(np.abs(a), np.abs(c)))


def _check_isolated_lists(g, so, n_pre, kpre, kgen):
    """Per row: the list is ascending, matches the bitmask, holds kpre prefill
    and kgen generation blocks; each part is exactly the top of the GPU's own
    fp32 scores in that part (ties to the lower index) and equals the
    oracle's part except for blocks within MASK_REL of the part's threshold."""
    idx, words, sg = g["block_idx"], g["block_mask"], g["block_scores"]
    b, h, N, kappa = idx.shape
    assert kappa == kpre + kgen
    w = words.astype(np.int64) & 0xFFFFFFFF
    bits = ((w[..., :, None] >> np.arange(32)) & 1).reshape(b, h, N, -1)[..., :N].astype(bool)
    tolerated = 0
    for bi in range(b):
        for hi in range(h):
            for r in range(N):
                row = idx[bi, hi, r]
                assert np.all(np.diff(row) > 0)
                m = np.zeros(N, bool)
                m[row] = True
                assert np.array_equal(m, bits[bi, hi, r])
                assert int(np.sum(row < n_pre)) == kpre
                for lo, hi_, kk in ((0, n_pre, kpre), (n_pre, N, kgen)):
                    got = row[(row >= lo) & (row < hi_)] - lo
                    own = sg[bi, hi, r, lo:hi_].astype(np.float32)
                    o_own = np.lexsort((np.arange(hi_ - lo), -own))
                    assert np.array_equal(np.sort(o_own[:kk]), got), "part is not the top of own scores"
                    sc = so[bi, hi, r, lo:hi_]
                    o_ref = np.lexsort((np.arange(hi_ - lo), -sc))
                    want = set(o_ref[:kk].tolist())
                    if want == set(got.tolist()):
                        continue
                    thr = sc[o_ref[kk - 1]]
                    thr_own = own[o_own[kk - 1]]
                    for j in want ^ set(got.tolist()):
                        near = abs(sc[j] - thr) <= MASK_REL * max(abs(thr), 1e-30)
                        near |= abs(float(own[j]) - thr_own) <= MASK_REL * max(abs(thr_own), 1e-30)
                        assert near, f"part differs away from its threshold (b{bi} h{hi} row {r})"
                        tolerated += 1
    return tolerated


def _isolated_and_check(q, k, B, prefill, kpre, kgen, beta, mode, window, dev):
    qd, kd = q.to(dev), k.to(dev)
    sel = bsb.ba_select_isolated(qd, kd, B, prefill, kpre, kgen, beta, mode, window, return_scores=True)
    torch.cuda.synchronize()
    g = {n: t.cpu().numpy() for n, t in sel.items()}
    Q64, K64 = to64(q), to64(k)
    own = O.ba_select_isolated(Q64, K64, B, prefill, kpre, kgen, beta, mode, window)
    L = q.shape[2]
    if mode & 1:
        _check_split_perm(g["perm_k"], own["perm_k"], K64, prefill)
    else:
        assert np.array_equal(g["perm_k"], np.broadcast_to(np.arange(L), g["perm_k"].shape))
    if mode & 2:
        check_perm(g["perm_q"], own["perm_q"], Q64, window)
    else:
        assert np.array_equal(g["perm_q"], np.broadcast_to(np.arange(L), g["perm_q"].shape))
    ora = O.ba_select_isolated(Q64, K64, B, prefill, kpre, kgen, beta, mode, window,
                               perm_q=g["perm_q"], perm_k=g["perm_k"])
    so = ora["scores"]
    check_scores(g["block_scores"], so, Q64, K64, g["perm_q"], g["perm_k"], B, beta)
    _check_isolated_lists(g, so, prefill // B, kpre, kgen)
    return sel, g


def _attn_and_check(q, k, v, B, sel, g, dev, query_blocks=None):
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = bsb.ba_sparse_attn(qd, kd, vd, B, sel["perm_q"], sel["perm_k"], sel["block_idx"])
    torch.cuda.synchronize()
    st, word = bsb.last_device_error()
    assert st == 0, hex(word)
    o_ref, lse_ref = O.sparse_attention(to64(q), to64(k), to64(v), g["perm_q"], g["perm_k"],
                                        g["block_idx"], B, query_blocks=query_blocks)
    rows = ~np.isnan(lse_ref)
    return check_attention(to64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, rows)


@pytest.mark.parametrize("mode", [0, 1, 3])
@pytest.mark.parametrize("shape", [
    # b, h, L, d, B, prefill, kappa_prefill, kappa_generation
    (1, 3, 4000, 128, 64, 1024, 4, 12),     # ragged generation tail
    (2, 2, 3072, 64, 128, 2048, 5, 2),      # prefill longer than generation
    (1, 2, 8192 + 640, 128, 128, 640, 1, 30),
])
def test_isolated_small(dev, shape, mode):
    b, h, L, d, B, pre, kpre, kgen = shape
    q, k, v = workloads.random_inputs(b, h, L, d, seed=4242 + L + mode, scale=1.5)
    for beta in (1.0, 0.0):
        sel, g = _isolated_and_check(q, k, B, pre, kpre, kgen, beta, mode, 0, dev)
    _attn_and_check(q, k, v, B, sel, g, dev)


def test_isolated_windowed_queries(dev):
    """sort_window applies to the queries; keys keep the two ranges."""
    q, k, v = workloads.random_inputs(1, 2, 4096, 128, seed=99, scale=2.0)
    sel, g = _isolated_and_check(q, k, 128, 1536, 3, 6, 1.0, 3, 1024, dev)
    _attn_and_check(q, k, v, 128, sel, g, dev)


def test_isolated_llada_shape(dev):
    """The LLaDA-shaped workload (b1 h32 L8192 d128 B64) with its first
    quarter as prompt: 50% of each part's key blocks kept.  Selection in
    full; attention on sampled query blocks."""
    w = workloads.get("llada")
    q, k, v, _ = workloads.make_inputs(w)
    pre = w.seqlen // 4
    n_pre = pre // w.block
    kpre, kgen = n_pre // 2, (w.nblocks - n_pre) // 2
    sel, g = _isolated_and_check(q, k, w.block, pre, kpre, kgen, 1.0, 3, 0, dev)
    rng = np.random.default_rng(7)
    qb = {(0, hi): sorted(set(rng.choice(w.nblocks, 12, replace=False).tolist()) | {0, w.nblocks - 1})
          for hi in range(w.heads)}
    _attn_and_check(q, k, v, w.block, sel, g, dev, query_blocks=qb)


def test_selection_reused_across_steps(dev):
    """SparseD §3.3 reuse: the selection made on one denoising step's Q, K
    serves the attention of later steps (here: the same tokens moved by a
    small random step).  The library takes permutations and lists as plain
    inputs, so the result must equal the oracle's attention of the new Q, K, V
    under the old permutations and lists."""
    q1, k1, v1 = workloads.random_inputs(1, 4, 4096, 128, seed=11, scale=1.5)
    sel = bsb.ba_select(q1.to(dev), k1.to(dev), 64, 16, 1.0, bsb.SORT_QK)
    torch.cuda.synchronize()
    g = {n: t.cpu().numpy() for n, t in sel.items()}
    gen = torch.Generator().manual_seed(12)
    for step in range(2):
        q2 = (q1.float() + 0.1 * torch.randn(q1.shape, generator=gen)).to(torch.bfloat16)
        k2 = (k1.float() + 0.1 * torch.randn(k1.shape, generator=gen)).to(torch.bfloat16)
        v2 = (v1.float() + 0.1 * torch.randn(v1.shape, generator=gen)).to(torch.bfloat16)
        _attn_and_check(q2, k2, v2, 64, sel, g, dev)
