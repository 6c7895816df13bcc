"""ba_validate_selection on the GPU: a selection from ba_select passes; each
kind of damage to it (a repeated or out-of-range permutation entry, a
descending, repeated or out-of-range block id) is reported with its bit, in
otherwise valid buffers (no bad addresses are ever passed)."""

from __future__ import annotations

import pytest
import torch

import block_sparse_bidirectional_gb300 as bsb
import workloads

pytestmark = pytest.mark.gpu

INVALID = 1
PQ, PK, IDX = 1, 2, 4


@pytest.fixture(scope="module")
def sel():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    q, k, _ = workloads.random_inputs(2, 3, 2000, 64, seed=41)   # ragged: N = 32, last block 16 tokens
    dev = torch.device("cuda:0")
    s = bsb.ba_select(q.to(dev), k.to(dev), 64, 9, 1.0, bsb.SORT_QK)
    torch.cuda.synchronize()
    return s


def check(s, expect_bits, **override):
    args = dict(perm_q=s["perm_q"], perm_k=s["perm_k"], block_idx=s["block_idx"])
    args.update(override)
    st, bits = bsb.ba_validate_selection(64, args["block_idx"], args["perm_q"], args["perm_k"])
    assert bits == expect_bits
    assert st == (INVALID if expect_bits else 0)


def test_selection_from_ba_select_passes(sel):
    check(sel, 0)
    check(sel, 0, perm_q=None, perm_k=None)   # identity permutations: nothing to check


def test_repeated_permutation_entry(sel):
    pq = sel["perm_q"].clone()
    pq[1, 2, 17] = pq[1, 2, 400]
    check(sel, PQ, perm_q=pq)
    pk = sel["perm_k"].clone()
    pk[0, 0, 0] = pk[0, 0, 1999]
    check(sel, PK, perm_k=pk)


def test_out_of_range_permutation_entry(sel):
    pq, pk = sel["perm_q"].clone(), sel["perm_k"].clone()
    pq[0, 1, 5] = 2000
    pk[1, 0, 7] = -1
    check(sel, PQ | PK, perm_q=pq, perm_k=pk)


def test_damaged_block_lists(sel):
    for damage in ("descending", "repeat", "too_large", "negative"):
        idx = sel["block_idx"].clone()
        row = idx[1, 2, 11]
        if damage == "descending":
            row[3], row[4] = row[4].item(), row[3].item()
        elif damage == "repeat":
            row[5] = row[4]
        elif damage == "too_large":
            row[-1] = 32
        else:
            row[0] = -3
        check(sel, IDX, block_idx=idx)
    assert bsb.last_device_error() == (0, 0)
