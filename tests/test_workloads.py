"""The seeded input recipe (workloads/) does what the design notes state:
shapes and budgets of the five workloads, determinism per seed, the planted
blocks of the tiny workload, the Z-order token layout, the shared cluster
shifts, the sink keys, and the video neighbourhoods.  Small shapes run through
the same generator code."""

import math

import torch

import workloads as W


def test_workload_table():
    want = {  # name: (b, h, L, d, B, N, kappas)
        "tiny": (1, 1, 1024, 64, 64, 16, [8]),
        "llada": (1, 32, 8192, 128, 64, 128, [64]),
        "long32k": (1, 32, 32768, 128, 128, 256, [128, 64, 26]),
        "ultra64k": (1, 32, 65536, 128, 128, 512, [256]),
        "video": (1, 24, 32760, 128, 64, 512, [256]),
    }
    for name, (b, h, L, d, B, N, kappas) in want.items():
        w = W.get(name)
        assert (w.batch, w.heads, w.seqlen, w.head_dim, w.block, w.nblocks) == (b, h, L, d, B, N)
        assert [w.kappa(s) for s in w.sparsities] == kappas
    v = W.get("video")
    assert v.seqlen - (v.nblocks - 1) * v.block == 56      # the short last block
    assert 21 * 30 * 52 == v.seqlen


def test_kappa_rule():
    assert W.kappa_for(0.9, 256) == 26                     # at least the requested density
    assert W.kappa_for(0.5, 512) == 256
    assert W.kappa_for(1.0, 10) == 1 and W.kappa_for(0.0, 10) == 10


def test_deterministic_per_seed():
    a = W.make_inputs("tiny")
    b = W.make_inputs("tiny")
    c = W.make_inputs("tiny", seed=7)
    for x, y in zip(a[:3], b[:3]):
        assert x.dtype == torch.bfloat16 and x.is_contiguous() and torch.equal(x, y)
    assert not torch.equal(a[0], c[0])


def test_tiny_planted_blocks():
    w = W.get("tiny")
    q, k, _, meta = W.make_inputs(w)
    g, planted = meta["query_block"], meta["planted_key_blocks"]
    B = w.block
    assert len(set(planted)) == 4 and all(abs(j - g) >= 2 for j in planted)
    u = q[0, 0, g * B:(g + 1) * B].float().mean(0)
    u = u / u.norm()
    proj = [float(k[0, 0, j * B:(j + 1) * B].float().mean(0) @ u) for j in range(w.nblocks)]
    for j in range(w.nblocks):
        if j in planted:
            assert abs(proj[j] - 2.0) < 0.6                # +2 u, noise of a 64-token mean
        else:
            assert abs(proj[j]) < 0.6


def test_zorder_layout():
    assert W.zorder_frame_order(2, 2) == [(0, 0), (0, 1), (1, 0), (1, 1)]
    assert W.zorder_frame_order(2, 4)[:4] == [(0, 0), (0, 1), (1, 0), (1, 1)]
    cells = W.zorder_frame_order(30, 52)
    assert len(cells) == 30 * 52 and len(set(cells)) == 30 * 52
    assert all(0 <= y < 30 and 0 <= x < 52 for y, x in cells)


def _small(name, h, L, d, B):
    return W.Workload(name, 0, 1, h, L, d, B, (0.5,), 5)


def test_clustered_recipe():
    w = _small("llada-like", 2, 1024, 128, 64)
    gen = torch.Generator().manual_seed(11)
    q, k, _, _ = W._clustered(w, gen, segment=256, per_head_ids=False)
    amp = 1.5 * math.sqrt(128)
    for hi in range(2):
        for s in range(1, 4):                              # segments without sink keys
            qs = q[0, hi, 256 * s:256 * (s + 1)].mean(0)
            ks = k[0, hi, 256 * s:256 * (s + 1)].mean(0)
            assert abs(float(qs.norm()) - amp) < 2.0        # a shift of RMS 1.5 per coordinate
            assert float((qs - ks).norm()) < 2.0            # the same shift in Q and K
    # sink keys 0..63 are scaled by 3 (Q is not)
    r_k = float(k[0, :, :64].norm(dim=-1).mean() / k[0, :, 64:256].norm(dim=-1).mean())
    r_q = float(q[0, :, :64].norm(dim=-1).mean() / q[0, :, 64:256].norm(dim=-1).mean())
    assert abs(r_k - 3.0) < 0.3 and abs(r_q - 1.0) < 0.2


def _same_centre_pattern(q_head, segment):
    """Which pairs of segments carry the same cluster shift (cosine of the
    segment means close to 1)."""
    m = q_head.reshape(-1, segment, q_head.shape[-1]).float().mean(1)
    m = m / m.norm(dim=1, keepdim=True)
    return (m @ m.T) > 0.9


def test_clustered_ids_shared_or_per_head():
    """llada: one cluster id per segment for all heads, so every head has the
    same pattern of segments sharing a centre; long32k: per-head ids."""
    w = _small("x", 4, 8 * 512, 128, 128)
    q_sh, _, _, _ = W._clustered(w, torch.Generator().manual_seed(3), segment=512, per_head_ids=False)
    pats = [_same_centre_pattern(q_sh[0, hi], 512) for hi in range(4)]
    assert all(torch.equal(pats[0], p) for p in pats[1:])
    assert int(pats[0].sum()) > 8                       # 8 segments, 8 centres: some repeat
    q_ph, _, _, _ = W._clustered(w, torch.Generator().manual_seed(3), segment=512, per_head_ids=True)
    pats = [_same_centre_pattern(q_ph[0, hi], 512) for hi in range(4)]
    assert not all(torch.equal(pats[0], p) for p in pats[1:])


def test_video_neighbourhoods():
    w = _small("video-like", 2, 3 * 4 * 8, 128, 64)
    gen = torch.Generator().manual_seed(9)
    q, k, _, meta = W._video(w, gen, frames=3, rows=4, cols=8, nb=(3, 2, 4), scale=1.0)
    assert meta["cells"] == 1 * 2 * 2
    order = W.zorder_frame_order(4, 8)
    cell_of = {}
    for t in range(3):
        for i, (y, x) in enumerate(order):
            cell_of[t * 32 + i] = (y // 2) * 2 + x // 4
    amp = math.sqrt(128)
    for hi in range(2):
        means = []
        for c in range(4):
            toks = [i for i, cc in cell_of.items() if cc == c]
            assert len(toks) == 24
            mq = q[0, hi, toks].float().mean(0)
            mk = k[0, hi, toks].float().mean(0)
            assert abs(float(mq.norm()) - amp) < 3.5       # one shared unit direction, scale 1
            assert float((mq - mk).norm()) < 3.5
            means.append(mq / mq.norm())
        for a in range(4):
            for b in range(a + 1, 4):
                assert abs(float(means[a] @ means[b])) < 0.6  # different cells, different directions
