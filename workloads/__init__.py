"""Seeded synthetic inputs shaped like the BA-Att paper's workloads.

This module only draws random numbers and lays tokens out.  It holds none of
the method's arithmetic (no norms, pooling, scores or attention), so both the
CUDA path and the fp64 oracle can be fed from it without sharing any code.

All draws use a CPU ``torch.Generator`` seeded per workload, in float32, then
rounded to bf16 (round-to-nearest-even).  The bf16 tensors are the ground
truth: the GPU receives a copy, the oracle reads them as float64 exactly.

Workloads (the paper's §4 models stand behind each shape; no dataset or
weights are used):

1. ``tiny``   b1 h1 L=1024 d=64 B=64, 50% sparsity, N(0,1) Q/K/V with four
   planted key blocks shifted by +2 u, u the unit mean direction of one chosen
   query block (a known answer for the selection when no sort is applied).
2. ``llada``  b1 h32 L=8192 d=128 B=64, 50%: N(0,1) + a per-head rank-8
   cluster structure (per-coordinate RMS 1.5), one cluster id per 256-token
   segment shared by Q and K and by all heads, sink keys 0..63 scaled x3.
3. ``long32k`` b1 h32 L=32768 d=128 B=128, 50/75/90%: as ``llada`` with
   1024-token segments and per-head cluster ids and bases.
4. ``ultra64k`` b1 h32 L=65536 d=128 B=128, 50%: as ``long32k``.
5. ``video``  b1 h24 L=32760 (21 frames x 30 x 52 latents) d=128 B=64, 50%:
   frame-major, Z-order within a frame; tokens of one 3x6x4 (t,y,x)
   neighbourhood share a random unit direction (scale 1.0) plus N(0,1) noise.
"""

from __future__ import annotations

import dataclasses
import math

import torch

__all__ = ["Workload", "WORKLOADS", "get", "kappa_for", "make_inputs", "zorder_frame_order"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int          # 1-based position in the workload table
    batch: int
    heads: int
    seqlen: int
    head_dim: int
    block: int
    sparsities: tuple
    seed: int

    @property
    def nblocks(self) -> int:
        return -(-self.seqlen // self.block)

    def kappa(self, sparsity: float | None = None) -> int:
        s = self.sparsities[0] if sparsity is None else sparsity
        return kappa_for(s, self.nblocks)


def kappa_for(sparsity: float, nblocks: int) -> int:
    """Fewest key blocks whose density is at least 1 - sparsity, in [1, N]."""
    k = math.ceil((1.0 - sparsity) * nblocks - 1e-9)
    return max(1, min(nblocks, k))


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 1024, 64, 64, (0.5,), 20261),
    "llada": Workload("llada", 2, 1, 32, 8192, 128, 64, (0.5,), 20262),
    "long32k": Workload("long32k", 3, 1, 32, 32768, 128, 128, (0.5, 0.75, 0.9), 20263),
    "ultra64k": Workload("ultra64k", 4, 1, 32, 65536, 128, 128, (0.5,), 20264),
    "video": Workload("video", 5, 1, 24, 32760, 128, 64, (0.5,), 20265),
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def _plain(gen, b, h, L, d):
    return torch.randn((b, h, L, d), generator=gen, dtype=torch.float32)


def _orthonormal(gen, d, r):
    a = torch.randn((d, r), generator=gen, dtype=torch.float64)
    qmat, _ = torch.linalg.qr(a)
    return qmat.to(torch.float32)


def _tiny(w: Workload, gen):
    b, h, L, d, B = w.batch, w.heads, w.seqlen, w.head_dim, w.block
    q = _plain(gen, b, h, L, d)
    k = _plain(gen, b, h, L, d)
    v = _plain(gen, b, h, L, d)
    n = L // B
    g = int(torch.randint(0, n, (1,), generator=gen))
    far = [j for j in range(n) if abs(j - g) >= 2]
    pick = torch.randperm(len(far), generator=gen)[:4].tolist()
    planted = sorted(far[i] for i in pick)
    # direction of the chosen query block's mean, as drawn (bf16-rounded)
    qg = _bf16(q[0, 0, g * B:(g + 1) * B]).float().mean(dim=0)
    u = qg / qg.norm()
    for j in planted:
        k[0, 0, j * B:(j + 1) * B] += 2.0 * u
    meta = dict(query_block=g, planted_key_blocks=planted)
    return q, k, v, meta


def _clustered(w: Workload, gen, segment: int, per_head_ids: bool, rank: int = 8,
               n_clusters: int = 8, rms: float = 1.5, sink: int = 64, sink_scale: float = 3.0):
    b, h, L, d = w.batch, w.heads, w.seqlen, w.head_dim
    q = _plain(gen, b, h, L, d)
    k = _plain(gen, b, h, L, d)
    v = _plain(gen, b, h, L, d)
    nseg = -(-L // segment)
    shared_ids = torch.randint(0, n_clusters, (nseg,), generator=gen)
    amp = rms * math.sqrt(d)
    for hi in range(h):
        basis = _orthonormal(gen, d, rank)                  # U_h: d x rank
        z = torch.randn((n_clusters, rank), generator=gen)
        z = z / z.norm(dim=1, keepdim=True)
        centres = z @ basis.T                                # unit vectors, n_clusters x d
        ids = torch.randint(0, n_clusters, (nseg,), generator=gen) if per_head_ids else shared_ids
        tok_ids = ids.repeat_interleave(segment)[:L]
        shift = amp * centres[tok_ids]                       # L x d
        q[:, hi] += shift
        k[:, hi] += shift
    k[:, :, :sink] *= sink_scale
    meta = dict(segment=segment, per_head_ids=per_head_ids)
    return q, k, v, meta


def zorder_frame_order(rows: int, cols: int):
    """(y, x) cells of a rows x cols frame listed in Z-order (Morton order)
    over the enclosing power-of-two grid, skipping cells outside the frame
    (the token layout of the loglinear-sparse-dit README, image data)."""
    side_y = 1 << max(0, (rows - 1).bit_length())
    side_x = 1 << max(0, (cols - 1).bit_length())
    cells = []
    for y in range(side_y):
        for x in range(side_x):
            if y < rows and x < cols:
                code = 0
                for bit in range(16):
                    code |= ((x >> bit) & 1) << (2 * bit)
                    code |= ((y >> bit) & 1) << (2 * bit + 1)
                cells.append((code, y, x))
    cells.sort()
    return [(y, x) for _, y, x in cells]


def _video(w: Workload, gen, frames=21, rows=30, cols=52, nb=(3, 6, 4), scale=1.0):
    b, h, L, d = w.batch, w.heads, w.seqlen, w.head_dim
    assert frames * rows * cols == L
    order = zorder_frame_order(rows, cols)
    t = torch.arange(frames).repeat_interleave(rows * cols)
    yx = torch.tensor(order, dtype=torch.int64).repeat(frames, 1)
    ct = t // nb[0]
    cy = yx[:, 0] // nb[1]
    cx = yx[:, 1] // nb[2]
    ny, nx = -(-rows // nb[1]), -(-cols // nb[2])
    nt = -(-frames // nb[0])
    cell = (ct * ny + cy) * nx + cx                          # neighbourhood id per token
    q = _plain(gen, b, h, L, d)
    k = _plain(gen, b, h, L, d)
    v = _plain(gen, b, h, L, d)
    amp = scale * math.sqrt(d)
    for hi in range(h):
        u = torch.randn((nt * ny * nx, d), generator=gen)
        u = u / u.norm(dim=1, keepdim=True)
        shift = amp * u[cell]
        q[:, hi] += shift
        k[:, hi] += shift
    meta = dict(cells=nt * ny * nx)
    return q, k, v, meta


def make_inputs(w: Workload | str, seed: int | None = None):
    """Return (q, k, v, meta): bf16 CPU tensors [b, h, L, d] and a dict."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    if w.name == "tiny":
        q, k, v, meta = _tiny(w, gen)
    elif w.name == "llada":
        q, k, v, meta = _clustered(w, gen, segment=256, per_head_ids=False)
    elif w.name in ("long32k", "ultra64k"):
        q, k, v, meta = _clustered(w, gen, segment=1024, per_head_ids=True)
    elif w.name == "video":
        q, k, v, meta = _video(w, gen)
    else:
        raise KeyError(w.name)
    return _bf16(q).contiguous(), _bf16(k).contiguous(), _bf16(v).contiguous(), meta


def random_inputs(b, h, L, d, seed, dv=None, scale=1.0):
    """Plain N(0, scale^2) bf16 Q, K, V of an arbitrary shape (for sweeps and edge cases)."""
    gen = torch.Generator().manual_seed(seed)
    dv = d if dv is None else dv
    q = torch.randn((b, h, L, d), generator=gen) * scale
    k = torch.randn((b, h, L, d), generator=gen) * scale
    v = torch.randn((b, h, L, dv), generator=gen)
    return _bf16(q).contiguous(), _bf16(k).contiguous(), _bf16(v).contiguous()
