"""Concurrent calls from several host threads, each on its own stream with its
own buffers and workspaces, give the same results as the calls made one
after another: the library keeps no state between calls apart from the
device error word.  (ctypes releases the GIL during the foreign calls.)"""

import threading

import pytest
import torch

import block_sparse_bidirectional_gb300 as bsb
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    bsb.load()
    return torch.device("cuda:0")


def _step(q, k, v, B, kappa):
    sel = bsb.ba_select(q, k, B, kappa, 1.0, bsb.SORT_QK)
    o, lse = bsb.ba_sparse_attn(q, k, v, B, sel["perm_q"], sel["perm_k"], sel["block_idx"])
    return sel["block_idx"], o, lse


def test_threads_match_serial(dev):
    shapes = [(1, 4, 4096, 128, 128, 8), (1, 3, 3000, 64, 64, 12), (2, 2, 2048, 128, 64, 10),
              (1, 2, 5000, 128, 128, 20)]
    inputs = []
    for i, (b, h, L, d, B, kappa) in enumerate(shapes):
        q, k, v = workloads.random_inputs(b, h, L, d, seed=900 + i, scale=1.5)
        inputs.append((q.to(dev), k.to(dev), v.to(dev), B, kappa))
    serial = []
    for args in inputs:
        serial.append(_step(*args))
    torch.cuda.synchronize()

    results = [None] * len(inputs)
    errors = []
    barrier = threading.Barrier(len(inputs))

    def worker(i):
        try:
            stream = torch.cuda.Stream(dev)
            with torch.cuda.stream(stream):
                barrier.wait()
                for _ in range(3):
                    out = _step(*inputs[i])
                stream.synchronize()
            results[i] = out
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(inputs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    torch.cuda.synchronize()
    for (idx_s, o_s, l_s), (idx_t, o_t, l_t) in zip(serial, results):
        assert torch.equal(idx_s, idx_t)
        assert torch.equal(o_s, o_t)
        assert torch.equal(l_s, l_t)
    assert bsb.last_device_error() == (0, 0)
