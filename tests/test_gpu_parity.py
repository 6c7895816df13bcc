"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on
the same seeded inputs.

Small shapes are compared in full (several tiles, ragged tails, both block
sizes and head dims, every sort mode, beta 0 and 1).  The five workload
shapes are run at full size in the launch configuration the benchmark times;
selection is checked in full and attention on sampled query blocks (16 random
per head plus the first and the last, the ragged one where L % B != 0).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import block_sparse_bidirectional_gb300 as bsb
import oracle.ba_oracle as O
import workloads
from parity import (check_attention, check_mask, check_perm, check_scores, check_topk_of_own_scores,
                    to64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    bsb.load()
    return torch.device("cuda:0")


def _select_and_check(q, k, B, kappa, beta, mode, window, dev):
    qd, kd = q.to(dev), k.to(dev)
    sel = bsb.ba_select(qd, kd, B, kappa, beta, mode, window, return_scores=True)
    torch.cuda.synchronize()
    g = {n: t.cpu().numpy() for n, t in sel.items()}
    Q64, K64 = to64(q), to64(k)
    own = O.ba_select(Q64, K64, B, kappa, beta, mode, window)
    if mode & 2:
        check_perm(g["perm_q"], own["perm_q"], Q64, window)
    else:
        assert np.array_equal(g["perm_q"], np.broadcast_to(np.arange(q.shape[2]), g["perm_q"].shape))
    if mode & 1:
        check_perm(g["perm_k"], own["perm_k"], K64, window)
    else:
        assert np.array_equal(g["perm_k"], np.broadcast_to(np.arange(q.shape[2]), g["perm_k"].shape))
    ora = O.ba_select(Q64, K64, B, kappa, beta, mode, window, perm_q=g["perm_q"], perm_k=g["perm_k"])
    so = ora["scores"]
    check_scores(g["block_scores"], so, Q64, K64, g["perm_q"], g["perm_k"], B, beta)
    check_topk_of_own_scores(g["block_idx"], g["block_scores"], kappa)
    check_mask(g["block_idx"], g["block_mask"], so, kappa, g["block_scores"])
    return sel, g


def _attn_and_check(q, k, v, B, sel, g, dev, query_blocks=None, scale=0.0):
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = bsb.ba_sparse_attn(qd, kd, vd, B, sel["perm_q"], sel["perm_k"], sel["block_idx"], scale)
    torch.cuda.synchronize()
    st, word = bsb.last_device_error()
    assert st == 0, hex(word)
    Q64, K64, V64 = to64(q), to64(k), to64(v)
    o_ref, lse_ref = O.sparse_attention(Q64, K64, V64, g["perm_q"], g["perm_k"], g["block_idx"], B,
                                        scale=(scale if scale > 0 else None), query_blocks=query_blocks)
    rows = ~np.isnan(lse_ref)
    return check_attention(to64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, rows)


SMALL = [
    # b, h, L, d, B, kappa
    (1, 2, 1024, 64, 64, 8),
    (2, 2, 1000, 128, 128, 4),
    (1, 3, 2048, 128, 64, 16),
    (1, 2, 777, 64, 128, 3),
    (1, 1, 64, 64, 64, 1),
    (1, 1, 50, 128, 64, 1),
    (1, 2, 4096, 128, 128, 32),
    (1, 1, 4160, 64, 64, 20),
    (1, 1, 1, 64, 64, 1),       # a single token: O = V, LSE = scale * q.k
    (2, 2, 1, 128, 128, 1),
    (1, 2, 129, 64, 64, 2),     # last block of one token (packed 64-token path)
    (1, 1, 4097, 128, 128, 5),  # last block of one token (128-token path)
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "b%d_h%d_L%d_d%d_B%d_k%d" % s)
@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_small_select_and_attention(dev, shape, mode):
    b, h, L, d, B, kappa = shape
    q, k, v = workloads.random_inputs(b, h, L, d, seed=1000 + L + d + B + mode, scale=1.5)
    for beta in (1.0, 0.0):
        sel, g = _select_and_check(q, k, B, kappa, beta, mode, 0, dev)
    _attn_and_check(q, k, v, B, sel, g, dev)


@pytest.mark.parametrize("beta", [0.5, 2.5])
@pytest.mark.parametrize("shape", [(1, 2, 2048, 128, 128, 6), (1, 2, 1500, 64, 64, 9)])
def test_beta_scaling(dev, shape, beta):
    """beta other than 0 and 1 (Eq. 13): scores, mask and attention."""
    b, h, L, d, B, kappa = shape
    q, k, v = workloads.random_inputs(b, h, L, d, seed=31 + L + int(10 * beta), scale=1.5)
    sel, g = _select_and_check(q, k, B, kappa, beta, 3, 0, dev)
    _attn_and_check(q, k, v, B, sel, g, dev)


@pytest.mark.parametrize("window", [128, 512])
def test_windowed_sort(dev, window):
    q, k, v = workloads.random_inputs(1, 2, 2048 + 128, 128, seed=77, scale=2.0)
    sel, g = _select_and_check(q, k, 128, 6, 1.0, 3, window, dev)
    _attn_and_check(q, k, v, 128, sel, g, dev)


@pytest.mark.parametrize("L,window", [(4097, 0), (8192, 0), (8193, 0), (16512, 8192), (25600, 12800)])
def test_sort_path_boundaries(dev, L, window):
    """Sorted sequences and windows on both sides of the one-CTA chunk sort's
    limits (4096 keys on 512 threads, 8192 on 1024) and the clustered radix
    sort beyond them: pi, the lists and the attention against the oracle."""
    q, k, v = workloads.random_inputs(1, 2, L, 128, seed=L + window, scale=1.5)
    sel, g = _select_and_check(q, k, 128, 4, 1.0, 3, window, dev)
    _attn_and_check(q, k, v, 128, sel, g, dev)


@pytest.mark.parametrize("B,kappa", [(128, 48), (64, 90)])
def test_in_kernel_gathers_many_heads(dev, B, kappa):
    """More heads than the gather look-ahead (ten heads at 32 tile pairs per
    head) and enough key blocks per CTA for the attention kernel to copy the
    later heads' rows itself: every query block against the oracle."""
    q, k, v = workloads.random_inputs(1, 12, 8192, 128, seed=B + kappa, scale=1.5)
    sel, g = _select_and_check(q, k, B, kappa, 1.0, 3, 0, dev)
    _attn_and_check(q, k, v, B, sel, g, dev)


def test_custom_scale(dev):
    q, k, v = workloads.random_inputs(1, 2, 1024, 128, seed=5)
    sel, g = _select_and_check(q, k, 128, 3, 1.0, 3, 0, dev)
    _attn_and_check(q, k, v, 128, sel, g, dev, scale=0.05)


@pytest.mark.parametrize("shape", [(1, 2, 1024, 64), (2, 3, 1000, 128), (1, 1, 77, 64), (1, 2, 3000, 128),
                                   (2, 1, 1, 128)])
def test_dense_against_oracle(dev, shape):
    b, h, L, d = shape
    q, k, v = workloads.random_inputs(b, h, L, d, seed=L * d)
    o, lse = bsb.ba_attn_dense(q.to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    o_ref, lse_ref = O.dense_attention(to64(q), to64(k), to64(v))
    check_attention(to64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref)


@pytest.mark.parametrize("B", [64, 128])
def test_every_block_selected_equals_dense(dev, B):
    """kappa = N with sorting on is ordinary attention (pins the remap)."""
    q, k, v = workloads.random_inputs(1, 2, 1536, 128, seed=B)
    N = -(-1536 // B)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    sel = bsb.ba_select(qd, kd, B, N, 1.0, 3)
    o_s, l_s = bsb.ba_sparse_attn(qd, kd, vd, B, sel["perm_q"], sel["perm_k"], sel["block_idx"])
    o_d, l_d = bsb.ba_attn_dense(qd, kd, vd)
    torch.cuda.synchronize()
    o_ref, lse_ref = O.dense_attention(to64(q), to64(k), to64(v))
    check_attention(to64(o_s), l_s.cpu().double().numpy(), o_ref, lse_ref)
    check_attention(to64(o_d), l_d.cpu().double().numpy(), o_ref, lse_ref)


def test_constant_v(dev):
    """Constant V comes back within one bf16 ulp: the weights are rounded to
    bf16 for the PV product and normalised by their exact fp32 sum."""
    q, k, _ = workloads.random_inputs(1, 2, 2048, 128, seed=9, scale=2.0)
    row = torch.randn(128, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    v = row.expand(1, 2, 2048, 128).contiguous()
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    sel = bsb.ba_select(qd, kd, 128, 5, 1.0, 3)
    o, _ = bsb.ba_sparse_attn(qd, kd, vd, 128, sel["perm_q"], sel["perm_k"], sel["block_idx"])
    torch.cuda.synchronize()
    ref = row.double().numpy()
    err = np.abs(to64(o) - ref)
    # one bf16 ulp of each value: 2^(floor(log2|v|) - 7)
    ulp = np.exp2(np.floor(np.log2(np.abs(ref) + 1e-30)) - 7)
    assert np.all(err <= ulp), float((err / ulp).max())


def test_lse_merge(dev):
    """Two calls over the two halves of every row's list, merged through their
    LSE, give the single call (the online-softmax merge)."""
    q, k, v = workloads.random_inputs(1, 2, 2048, 128, seed=11)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    sel = bsb.ba_select(qd, kd, 128, 8, 1.0, 3)
    idx = sel["block_idx"]
    o, l = bsb.ba_sparse_attn(qd, kd, vd, 128, sel["perm_q"], sel["perm_k"], idx)
    o1, l1 = bsb.ba_sparse_attn(qd, kd, vd, 128, sel["perm_q"], sel["perm_k"], idx[..., :4].contiguous())
    o2, l2 = bsb.ba_sparse_attn(qd, kd, vd, 128, sel["perm_q"], sel["perm_k"], idx[..., 4:].contiguous())
    torch.cuda.synchronize()
    om, lm = O.merge_lse(to64(o1), l1.cpu().double().numpy(), to64(o2), l2.cpu().double().numpy())
    check_attention(om, lm, to64(o), l.cpu().double().numpy())


def test_tiny_planted(dev):
    """Workload 1: the four planted key blocks are selected for the chosen
    query block (no sort), and everything matches the oracle."""
    w = workloads.get("tiny")
    q, k, v, meta = workloads.make_inputs(w)
    sel, g = _select_and_check(q, k, w.block, w.kappa(), 1.0, 0, 0, dev)
    row = set(g["block_idx"][0, 0, meta["query_block"]].tolist())
    assert set(meta["planted_key_blocks"]) <= row
    _attn_and_check(q, k, v, w.block, sel, g, dev)
    sel, g = _select_and_check(q, k, w.block, w.kappa(), 1.0, 3, 0, dev)
    _attn_and_check(q, k, v, w.block, sel, g, dev)


def _sample_blocks(b, h, N, seed, n=16):
    rng = np.random.default_rng(seed)
    out = {}
    for bi in range(b):
        for hi in range(h):
            pick = set(rng.choice(N, size=min(n, N), replace=False).tolist()) | {0, N - 1}
            out[(bi, hi)] = sorted(pick)
    return out


@pytest.mark.parametrize("name,sparsity", [("llada", 0.5), ("long32k", 0.5), ("long32k", 0.75),
                                           ("long32k", 0.9), ("ultra64k", 0.5), ("video", 0.5)])
def test_workload_full_size(dev, name, sparsity):
    w = workloads.get(name)
    q, k, v, _ = workloads.make_inputs(w)
    kappa = w.kappa(sparsity)
    sel, g = _select_and_check(q, k, w.block, kappa, 1.0, 3, 0, dev)
    qb = None if name == "llada" else _sample_blocks(w.batch, w.heads, w.nblocks, seed=w.seed)
    _attn_and_check(q, k, v, w.block, sel, g, dev, query_blocks=qb)


def test_dense_full_size_sampled(dev):
    """The dense kernel at the headline shape, on sampled rows of 4 heads."""
    w = workloads.get("ultra64k")
    q, k, v, _ = workloads.make_inputs(w)
    o, lse = bsb.ba_attn_dense(q.to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    o = o.cpu()
    lse = lse.cpu()
    rng = np.random.default_rng(4)
    for hi in (0, 7, 19, 31):
        rows = np.unique(np.concatenate([rng.choice(w.seqlen, 96, replace=False), [0, w.seqlen - 1]]))
        ref_o, ref_l = O.dense_attention_one(to64(q[0, hi]), to64(k[0, hi]), to64(v[0, hi]), rows=rows)
        check_attention(to64(o[0, hi, rows]), lse[0, hi, rows].double().numpy(), ref_o, ref_l)


def test_device_error_word_clean(dev):
    st, word = bsb.last_device_error()
    assert st == 0 and word == 0


def test_merge_lse_kernel_against_oracle(dev):
    """ba_merge_lse (LoSA merge) against the oracle's merge on random partial
    results, including rows whose key set was empty (LSE = -inf)."""
    gen = torch.Generator().manual_seed(21)
    for d in (64, 128):
        rows = 3001
        o1 = torch.randn((rows, d), generator=gen).to(torch.bfloat16)
        o2 = torch.randn((rows, d), generator=gen).to(torch.bfloat16)
        l1 = torch.randn(rows, generator=gen) * 4
        l2 = torch.randn(rows, generator=gen) * 4
        l1[::7] = -float("inf")
        l2[::11] = -float("inf")
        o, lse = bsb.ba_merge_lse(o1.to(dev), l1.to(dev), o2.to(dev), l2.to(dev))
        torch.cuda.synchronize()
        both = torch.isinf(l1) & torch.isinf(l2)
        one = ~both.numpy()
        # the merge is defined where at least one part has keys
        om, lm = O.merge_lse(to64(o1)[one], l1.double().numpy()[one], to64(o2)[one],
                             l2.double().numpy()[one])
        og, lg = to64(o), lse.cpu().double().numpy()
        # bf16 output: within one bf16 rounding of the fp64 merge
        assert np.all(np.abs(og[one] - om) <= np.abs(om) * 2.0 ** -8 + 1e-6)
        assert np.all(np.abs(lg[one] - lm) <= 1e-5 * np.maximum(1.0, np.abs(lm)))
        assert np.all(og[both.numpy()] == 0) and np.all(np.isneginf(lg[both.numpy()]))


def test_merge_lse_in_place_equals_out_of_place(dev):
    """ba_merge_lse writing over its first (or second) input gives the same
    bits as writing to fresh outputs (the in-place use include/ba.h allows)."""
    gen = torch.Generator().manual_seed(22)
    for d in (64, 128):
        rows = 4099
        o1 = torch.randn((rows, d), generator=gen).to(torch.bfloat16).to(dev)
        o2 = torch.randn((rows, d), generator=gen).to(torch.bfloat16).to(dev)
        l1 = (torch.randn(rows, generator=gen) * 4).to(dev)
        l2 = (torch.randn(rows, generator=gen) * 4).to(dev)
        l1[::7] = -float("inf")
        ref_o, ref_l = bsb.ba_merge_lse(o1, l1, o2, l2)
        a_o, a_l = o1.clone(), l1.clone()
        bsb.ba_merge_lse_into(a_o, a_l, o2, l2, a_o, a_l)      # over the first input
        b_o, b_l = o2.clone(), l2.clone()
        bsb.ba_merge_lse_into(o1, l1, b_o, b_l, b_o, b_l)      # over the second input
        torch.cuda.synchronize()
        for og, lg in ((a_o, a_l), (b_o, b_l)):
            assert torch.equal(og, ref_o)
            assert torch.equal(torch.nan_to_num(lg, neginf=-1e30), torch.nan_to_num(ref_l, neginf=-1e30))


def test_merge_lse_kernel_joins_split_lists(dev):
    """Attention over the two halves of every list, merged on the GPU, equals
    the single call over the whole list (within the attention tolerances)."""
    q, k, v = workloads.random_inputs(1, 4, 4096, 128, seed=31)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    sel = bsb.ba_select(qd, kd, 128, 12, 1.0, 3)
    idx = sel["block_idx"]
    o, l = bsb.ba_sparse_attn(qd, kd, vd, 128, sel["perm_q"], sel["perm_k"], idx)
    o1, l1 = bsb.ba_sparse_attn(qd, kd, vd, 128, sel["perm_q"], sel["perm_k"], idx[..., :5].contiguous())
    o2, l2 = bsb.ba_sparse_attn(qd, kd, vd, 128, sel["perm_q"], sel["perm_k"], idx[..., 5:].contiguous())
    om, lm = bsb.ba_merge_lse(o1, l1, o2, l2)
    torch.cuda.synchronize()
    check_attention(to64(om), lm.cpu().double().numpy(), to64(o), l.cpu().double().numpy())


def test_step_captures_in_a_cuda_graph(dev):
    """A whole select + sparse-attention step (norm pass, sort, statistics,
    scores, top-kappa, pair lists, gathers, attention) records into a CUDA
    graph and replays to the same bits as eager execution: the calls only
    enqueue kernels on the caller's stream and take every buffer from it."""
    b, h, L, d, B, kappa = 1, 4, 4096, 128, 128, 8
    q, k, v = workloads.random_inputs(b, h, L, d, seed=91, scale=1.5)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    N = -(-L // B)
    i32 = dict(dtype=torch.int32, device=dev)
    pq, pk = torch.empty((b, h, L), **i32), torch.empty((b, h, L), **i32)
    idx, mask = torch.empty((b, h, N, kappa), **i32), torch.empty((b, h, N, -(-N // 32)), **i32)
    wss = torch.empty(bsb.select_workspace_size(b, h, L, d, B, kappa), dtype=torch.uint8, device=dev)
    wsa = torch.empty(bsb.sparse_attn_workspace_size(b, h, L, d, B, kappa), dtype=torch.uint8, device=dev)
    o = torch.empty_like(qd)
    lse = torch.empty((b, h, L), dtype=torch.float32, device=dev)

    def step():
        bsb.ba_select_into(qd, kd, B, kappa, 1.0, bsb.SORT_QK, 0, pq, pk, idx, mask, None, wss)
        bsb.ba_sparse_attn_into(qd, kd, vd, B, pq, pk, idx, 0.0, o, lse, wsa)

    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        step()                       # eager, also configures the kernels once
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (pq, pk, idx, o, lse)]
    for t in (o, lse):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for a, r in zip((pq, pk, idx, o, lse), ref):
            assert torch.equal(a, r)
    st, word = bsb.last_device_error()
    assert st == 0, hex(word)
