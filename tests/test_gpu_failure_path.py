"""The bounded-wait failure path on the GPU, without a fault: a wait that
runs out (nothing ever completes the barrier phase it waits for) must come
back as BA_ERR_DEVICE_TIMEOUT with its site, clear on reading, and leave the
context usable for the next calls."""

import numpy as np
import pytest
import torch

import block_sparse_bidirectional_gb300 as bsb
import oracle.ba_oracle as O
import workloads
from parity import check_attention, to64

pytestmark = pytest.mark.gpu

DEVICE_TIMEOUT = 5
SITE_SELFTEST = 11


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    bsb.load()
    return torch.device("cuda:0")


def test_wait_that_runs_out_reports_and_clears(dev):
    assert bsb.last_device_error() == (0, 0)
    bsb.selftest_wait_timeout(2000)          # 2 ms
    st, word = bsb.last_device_error()
    assert st == DEVICE_TIMEOUT
    assert word & 1 and (word >> 8) & 0xFF == SITE_SELFTEST
    assert bsb.last_device_error() == (0, 0)  # read once, then clear


def test_context_usable_after_a_timeout(dev):
    bsb.selftest_wait_timeout(1000)
    assert bsb.last_device_error()[0] == DEVICE_TIMEOUT
    q, k, v = workloads.random_inputs(1, 2, 1024, 128, seed=3)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    sel = bsb.ba_select(qd, kd, 128, 4, 1.0, bsb.SORT_QK)
    o, lse = bsb.ba_sparse_attn(qd, kd, vd, 128, sel["perm_q"], sel["perm_k"], sel["block_idx"])
    torch.cuda.synchronize()
    assert bsb.last_device_error() == (0, 0)
    g = {n: t.cpu().numpy() for n, t in sel.items()}
    o_ref, lse_ref = O.sparse_attention(to64(q), to64(k), to64(v), g["perm_q"], g["perm_k"],
                                        g["block_idx"], 128)
    check_attention(to64(o), lse.cpu().double().numpy(), o_ref, lse_ref)


SITE_P_FULL = 7  # the MMA thread's wait for P-ready, held back by a K/V copy never issued


def test_attention_kernel_unwinds_after_a_stalled_stage(dev):
    """The attention kernel's own bounded wait runs out (its MMA thread waits
    for a P-ready signal that a K/V copy which is never issued holds back):
    the site is reported, nothing is written, the word clears, and the next
    select + attention matches the oracle."""
    assert bsb.last_device_error() == (0, 0)
    q, k, v = workloads.random_inputs(1, 2, 1024, 128, seed=5)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, 7.0)
    lse = torch.full((1, 2, 1024), 7.0, dtype=torch.float32, device=dev)
    bsb.selftest_attn_stall(qd, kd, vd, o, lse, limit_us=1000)
    st, word = bsb.last_device_error()
    assert st == DEVICE_TIMEOUT
    assert word & 1 and (word >> 8) & 0xFF == SITE_P_FULL
    assert bsb.last_device_error() == (0, 0)
    # an aborted CTA writes no output
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())
    sel = bsb.ba_select(qd, kd, 128, 4, 1.0, bsb.SORT_QK)
    o2, lse2 = bsb.ba_sparse_attn(qd, kd, vd, 128, sel["perm_q"], sel["perm_k"], sel["block_idx"])
    od, lsed = bsb.ba_attn_dense(qd, kd, vd)
    torch.cuda.synchronize()
    assert bsb.last_device_error() == (0, 0)
    g = {n: t.cpu().numpy() for n, t in sel.items()}
    o_ref, lse_ref = O.sparse_attention(to64(q), to64(k), to64(v), g["perm_q"], g["perm_k"],
                                        g["block_idx"], 128)
    check_attention(to64(o2), lse2.cpu().double().numpy(), o_ref, lse_ref)
    od_ref, ld_ref = O.dense_attention(to64(q), to64(k), to64(v))
    check_attention(to64(od), lsed.cpu().double().numpy(), od_ref, ld_ref)
