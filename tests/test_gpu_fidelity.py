"""GPU parity of the fidelity diagnostics (``ba_block_fidelity``) against the
fp64 oracle: the oracle block mass of BA-Att §3.1 Eq. 3, the largest
token-vs-block logit deviation of §3.2, its bound U of Eq. 7-8, and the
recall of a selected mask, over the GPU's own sorted blocks.

Tolerances: the mass takes the dense LSE from ``ba_attn_dense`` (within 1e-3
of the exact one), so each entry is within a relative 2e-3 (+1e-7) of the
oracle's, rows sum to 1 within 2e-3 and the recall is within 2e-3.  The
deviation and the bound are fp32 arithmetic on exact bf16 inputs: within
1e-3 relative of the oracle (+1e-4 absolute).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import block_sparse_bidirectional_gb300 as bsb
import oracle.ba_oracle as O
import workloads
from parity import to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    bsb.load()
    return torch.device("cuda:0")


def _run(q, k, v, B, kappa, mode, dev):
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    sel = bsb.ba_select(qd, kd, B, kappa, 1.0, mode)
    _, lse = bsb.ba_attn_dense(qd, kd, vd)
    fid = bsb.ba_block_fidelity(qd, kd, B, lse, sel["perm_q"], sel["perm_k"], sel["block_idx"])
    torch.cuda.synchronize()
    st, word = bsb.last_device_error()
    assert st == 0, hex(word)
    g = {n: t.cpu().numpy() for n, t in sel.items()}
    f = {n: t.cpu().numpy().astype(np.float64) for n, t in fid.items()}
    return g, f


def _compare(q, k, B, g, f, heads=None):
    Q64, K64 = to64(q), to64(k)
    b, h = Q64.shape[:2]
    for bi in range(b):
        for hi in (range(h) if heads is None else heads):
            pq, pk = g["perm_q"][bi, hi].astype(np.int64), g["perm_k"][bi, hi].astype(np.int64)
            m_ref = O.oracle_block_mass(Q64[bi, hi], K64[bi, hi], pq, pk, B)
            m = f["mass"][bi, hi]
            assert np.all(np.abs(m - m_ref) <= 2e-3 * m_ref + 1e-7), float(np.abs(m - m_ref).max())
            assert np.all(np.abs(m.sum(axis=1) - 1.0) <= 2e-3)
            d_ref = O.observed_deviation(Q64[bi, hi], K64[bi, hi], pq, pk, B)
            assert np.all(np.abs(f["dev_max"][bi, hi] - d_ref) <= 1e-3 * d_ref + 1e-4)
            u_ref = O.deviation_bound(Q64[bi, hi], K64[bi, hi], pq, pk, B)["U"]
            assert np.all(np.abs(f["bound"][bi, hi] - u_ref) <= 1e-3 * u_ref + 1e-4)
            assert np.all(f["dev_max"][bi, hi] <= f["bound"][bi, hi] * (1 + 1e-4) + 1e-4)  # Eq. 8
            idx = g["block_idx"][bi, hi]
            r_ref = np.take_along_axis(m_ref, idx.astype(np.int64), axis=1).sum(axis=1)
            assert np.all(np.abs(f["recall"][bi, hi] - r_ref) <= 2e-3)


@pytest.mark.parametrize("shape", [
    # b, h, L, d, B, kappa, sort mode
    (1, 2, 1000, 64, 64, 4, 3),
    (1, 2, 1536, 128, 128, 3, 3),
    (2, 1, 777, 128, 64, 5, 1),
    (1, 1, 2048, 128, 64, 8, 0),
])
def test_fidelity_small(dev, shape):
    b, h, L, d, B, kappa, mode = shape
    q, k, v = workloads.random_inputs(b, h, L, d, seed=600 + L + d, scale=1.5)
    g, f = _run(q, k, v, B, kappa, mode, dev)
    _compare(q, k, B, g, f)


def test_fidelity_every_block_recall_is_one(dev):
    """kappa = N keeps the whole dense mass: recall 1 for every row."""
    q, k, v = workloads.random_inputs(1, 2, 1024, 128, seed=3)
    g, f = _run(q, k, v, 128, 8, 3, dev)
    assert np.all(np.abs(f["recall"] - 1.0) <= 2e-3)


def test_fidelity_llada_heads(dev):
    """The LLaDA-shaped workload (L=8192, d=128, B=64, 50%), two heads
    compared in full against the oracle's dense map."""
    w = workloads.get("llada")
    q, k, v, _ = workloads.make_inputs(w)
    q, k, v = q[:, :2].contiguous(), k[:, :2].contiguous(), v[:, :2].contiguous()
    g, f = _run(q, k, v, w.block, w.kappa(), 3, dev)
    _compare(q, k, w.block, g, f)
