"""GPU parity of LoSA's locality pruning and result reuse (the LoSA summary
post, "locality pruning" and the cache update of "merge and update") against
the fp64 oracle, and one LoSA step composed with the block-sparse attention
and the LSE merge.

The active set is an integer decision taken in fp32 on the GPU: it must be
exactly the top_k of the GPU's own fp32 MSE per group (ties to the lower
index); the MSE must match the oracle's within 1e-5 relative; the active set
must equal the oracle's except where MSE values lie within 1e-5 of the
group's top_k-th value.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import block_sparse_bidirectional_gb300 as bsb
import oracle.ba_oracle as O
import workloads
from parity import check_attention, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    bsb.load()
    return torch.device("cuda:0")


def _moved(q, frac, seed):
    """A denoising-step analogue: a fraction of the tokens move a lot, the
    rest a little, some not at all (exact ties)."""
    gen = torch.Generator().manual_seed(seed)
    b, h, L, d = q.shape
    scale = torch.rand((b, h, L, 1), generator=gen)
    big = (torch.rand((b, h, L, 1), generator=gen) < frac).float()
    still = (torch.rand((b, h, L, 1), generator=gen) < 0.2).float()
    step = (0.02 + 2.0 * big) * scale * (1 - still)
    return (q.float() + step * torch.randn(q.shape, generator=gen)).to(torch.bfloat16)


def _check_active(act_g, mse_g, q_now, q_prev, group, top_k):
    mse_o = O.query_mse(to64(q_now), to64(q_prev))
    mse_g = mse_g.astype(np.float64)
    assert np.all(np.abs(mse_g - mse_o) <= 1e-5 * np.abs(mse_o) + 1e-12)
    b, h, L = act_g.shape
    for bi in range(b):
        for hi in range(h):
            own = O.active_tokens(mse_g[bi, hi].astype(np.float32).astype(np.float64), group, top_k)
            assert np.array_equal(own, act_g[bi, hi].astype(bool)), "not the top_k of own MSE"
            ref = O.active_tokens(mse_o[bi, hi], group, top_k)
            diff = np.nonzero(ref != own)[0]
            for i in diff:
                g0 = (i // group) * group
                seg = mse_o[bi, hi, g0:g0 + group]
                thr = np.sort(seg)[::-1][min(top_k, len(seg)) - 1]
                assert abs(mse_o[bi, hi, i] - thr) <= 1e-5 * abs(thr) + 1e-12


@pytest.mark.parametrize("shape,group,top_k", [
    ((1, 2, 1000, 128), 16, 5),
    ((2, 3, 777, 64), 32, 4),
    ((1, 1, 100, 128), 1024, 7),
    ((1, 2, 64, 64), 8, 8),
])
def test_active_tokens(dev, shape, group, top_k):
    b, h, L, d = shape
    q_prev, _, _ = workloads.random_inputs(b, h, L, d, seed=L + group)
    q_now = _moved(q_prev, 0.1, seed=L)
    act, mse = bsb.ba_active_tokens(q_now.to(dev), q_prev.to(dev), group, top_k, return_mse=True)
    torch.cuda.synchronize()
    _check_active(act.cpu().numpy(), mse.cpu().numpy(), q_now, q_prev, group, top_k)


def test_reuse_rows(dev):
    b, h, L, d = 1, 2, 500, 128
    gen = torch.Generator().manual_seed(3)
    o_new = torch.randn((b, h, L, d), generator=gen).to(torch.bfloat16)
    o_c = torch.randn((b, h, L, d), generator=gen).to(torch.bfloat16)
    l_new, l_c = torch.randn((b, h, L), generator=gen), torch.randn((b, h, L), generator=gen)
    act = (torch.rand((b, h, L), generator=gen) < 0.3).to(torch.uint8)
    oc, lc = o_c.to(dev), l_c.to(dev)
    bsb.ba_reuse_rows(o_new.to(dev), l_new.to(dev), act.to(dev), oc, lc)
    torch.cuda.synchronize()
    o_ref, l_ref = O.reuse_rows(to64(o_new), l_new.double().numpy(), to64(o_c), l_c.double().numpy(),
                                act.numpy().astype(bool))
    assert np.array_equal(to64(oc), o_ref) and np.array_equal(lc.cpu().double().numpy(), l_ref)


def test_losa_step(dev):
    """One LoSA-style step: the previous step's result is cached; the new
    step's active tokens take fresh block-sparse attention results, stable
    ones keep the cache; the cache then merges with a second partial result
    through the LSE.  Against the oracle composing the same steps."""
    b, h, L, d, B, kappa = 1, 2, 2048, 128, 128, 6
    q0, k, v = workloads.random_inputs(b, h, L, d, seed=21, scale=1.5)
    q1 = _moved(q0, 0.1, seed=22)
    qd0, qd1, kd, vd = q0.to(dev), q1.to(dev), k.to(dev), v.to(dev)
    sel = bsb.ba_select(qd0, kd, B, kappa)
    o_c, l_c = bsb.ba_sparse_attn(qd0, kd, vd, B, sel["perm_q"], sel["perm_k"], sel["block_idx"])
    o_n, l_n = bsb.ba_sparse_attn(qd1, kd, vd, B, sel["perm_q"], sel["perm_k"], sel["block_idx"])
    act, mse = bsb.ba_active_tokens(qd1, qd0, 32, 4, return_mse=True)
    bsb.ba_reuse_rows(o_n, l_n, act, o_c, l_c)
    # a second partial result (here: dense attention over the same keys)
    o2, l2 = bsb.ba_attn_dense(qd1, kd, vd)
    o_m, l_m = bsb.ba_merge_lse(o_c, l_c, o2, l2)
    torch.cuda.synchronize()
    g = {n: t.cpu().numpy() for n, t in sel.items()}
    Q0, Q1, K, V = to64(q0), to64(q1), to64(k), to64(v)
    oc_ref, lc_ref = O.sparse_attention(Q0, K, V, g["perm_q"], g["perm_k"], g["block_idx"], B)
    on_ref, ln_ref = O.sparse_attention(Q1, K, V, g["perm_q"], g["perm_k"], g["block_idx"], B)
    a = act.cpu().numpy().astype(bool)
    oc_ref, lc_ref = O.reuse_rows(on_ref, ln_ref, oc_ref, lc_ref, a)
    o2_ref, l2_ref = O.dense_attention(Q1, K, V)
    om_ref, lm_ref = O.merge_lse(oc_ref, lc_ref, o2_ref, l2_ref)
    check_attention(to64(o_m), l_m.cpu().numpy().astype(np.float64), om_ref, lm_ref)
    assert int(a.sum()) == b * h * (L // 32) * 4
