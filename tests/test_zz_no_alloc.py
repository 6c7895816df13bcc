"""ba_select_noalloc against ba_select, through the C ABI.

Some callers cannot allocate device memory when they run the selection (an
engine that owns the whole GPU heap, a plugin without access to its host's
allocator), so the library offers ba_select_noalloc, which uses a scratch
array compiled into the library instead of a caller workspace.  This file
checks that its outputs equal those of ba_select on two calls in a row (the
second call runs over whatever the first left in the shared array), and that
a size beyond the array is refused before anything is launched.

It sits in its own file, named to be collected last, and makes no use of
state left by other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

import block_sparse_bidirectional_gb300 as bsb
import workloads

pytestmark = pytest.mark.gpu

CAPACITY = 32 * 1024 * 1024     # BA_SELECT_STATIC_SCRATCH_BYTES in include/ba.h
SCORE_RTOL = 0.0                # same kernels, same inputs: identical results expected


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, q, k, B, kappa, beta, mode, window):
    b, h, L, d = q.shape
    N = -(-L // B)
    dev = q.device
    out = dict(perm_q=torch.empty((b, h, L), dtype=torch.int32, device=dev),
               perm_k=torch.empty((b, h, L), dtype=torch.int32, device=dev),
               block_idx=torch.empty((b, h, N, kappa), dtype=torch.int32, device=dev),
               block_mask=torch.empty((b, h, N, -(-N // 32)), dtype=torch.int32, device=dev),
               block_scores=torch.empty((b, h, N, N), dtype=torch.float32, device=dev))
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    st = lib.ba_select_noalloc(_ptr(q), _ptr(k), b, h, L, d, B, kappa, float(beta), mode, window,
                               _ptr(out["perm_q"]), _ptr(out["perm_k"]), _ptr(out["block_idx"]),
                               _ptr(out["block_mask"]), _ptr(out["block_scores"]), stream)
    return st, out


def _compare(ref, got):
    for name in ("perm_q", "perm_k", "block_idx", "block_mask"):
        assert torch.equal(ref[name].cpu(), got[name].cpu()), name
    np.testing.assert_allclose(got["block_scores"].cpu().numpy(), ref["block_scores"].cpu().numpy(),
                               rtol=SCORE_RTOL, atol=0.0)


def test_noalloc_matches_ba_select_on_two_calls():
    assert torch.cuda.is_available()
    lib = bsb.load()
    dev = torch.device("cuda:0")
    w = workloads.get("llada")                      # 32 heads, L = 8192, d = 128, B = 64
    q1, k1, _, _ = workloads.make_inputs(w)
    q2, k2, _ = workloads.random_inputs(2, 3, 1000, 64, seed=321, scale=1.5)
    cases = [(q1.to(dev), k1.to(dev), w.block, w.kappa(), 1.0, 3, 0),
             (q2.to(dev), k2.to(dev), 128, 3, 0.5, 1, 256)]
    for q, k, B, kappa, beta, mode, window in cases:
        b, h, L, d = q.shape
        assert bsb.select_workspace_size(b, h, L, d, B, kappa, mode, window) <= CAPACITY
        st, got = _noalloc(lib, q, k, B, kappa, beta, mode, window)
        assert st == 0, lib.ba_status_string(st)
        ref = bsb.ba_select(q, k, B, kappa, beta, mode, window, return_scores=True)
        torch.cuda.synchronize()
        _compare(ref, got)
    st, word = bsb.last_device_error()
    assert st == 0, hex(word)


def test_noalloc_refuses_sizes_beyond_its_array():
    lib = bsb.load()
    b, h, L, d, B, kappa = 1, 32, 65536, 128, 128, 256
    assert bsb.select_workspace_size(b, h, L, d, B, kappa, 3, 0) > CAPACITY
    fake = ctypes.c_void_p(0x10000000)   # never dereferenced: the size check comes first
    st = lib.ba_select_noalloc(fake, fake, b, h, L, d, B, kappa, 1.0, 3, 0, fake, fake, fake, fake,
                               None, None)
    assert st == 3  # BA_ERR_WORKSPACE
