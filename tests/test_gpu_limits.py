"""GPU parity at the largest supported block count (4096 key blocks per
sequence): the top-kappa path that keeps 128 keys per lane, the tile-pair
lists at their capacity, and the norm sort over half a million tokens.
Selection is checked in full against the oracle; attention on sampled query
blocks including the last one."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import block_sparse_bidirectional_gb300 as bsb
import oracle.ba_oracle as O
import workloads
from parity import check_attention, check_mask, check_perm, check_scores, check_topk_of_own_scores, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    bsb.load()
    return torch.device("cuda:0")


@pytest.mark.parametrize("d,B,kappa", [(128, 128, 8), (64, 64, 12)])
def test_max_block_count(dev, d, B, kappa):
    N = 4096
    L = N * B
    q, k, v = workloads.random_inputs(1, 1, L, d, seed=N + B, scale=1.5)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    sel = bsb.ba_select(qd, kd, B, kappa, 1.0, bsb.SORT_QK, return_scores=True)
    torch.cuda.synchronize()
    g = {n: t.cpu().numpy() for n, t in sel.items()}
    Q64, K64 = to64(q), to64(k)
    own = O.ba_select(Q64, K64, B, kappa, 1.0, O.SORT_QK)
    check_perm(g["perm_q"], own["perm_q"], Q64)
    check_perm(g["perm_k"], own["perm_k"], K64)
    ora = O.ba_select(Q64, K64, B, kappa, 1.0, O.SORT_QK, perm_q=g["perm_q"], perm_k=g["perm_k"])
    so = ora["scores"]
    check_scores(g["block_scores"], so, Q64, K64, g["perm_q"], g["perm_k"], B, 1.0)
    check_topk_of_own_scores(g["block_idx"], g["block_scores"], kappa)
    check_mask(g["block_idx"], g["block_mask"], so, kappa, g["block_scores"])
    o, lse = bsb.ba_sparse_attn(qd, kd, vd, B, sel["perm_q"], sel["perm_k"], sel["block_idx"])
    torch.cuda.synchronize()
    st, word = bsb.last_device_error()
    assert st == 0, hex(word)
    qb = {(0, 0): [0, 1, 777, 2048, N - 2, N - 1]}
    o_ref, lse_ref = O.sparse_attention(Q64, K64, to64(v), g["perm_q"], g["perm_k"], g["block_idx"], B,
                                        query_blocks=qb)
    rows = ~np.isnan(lse_ref)
    check_attention(to64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, rows)
