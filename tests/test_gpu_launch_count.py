"""The bench line's launch count: the library's kernels in one select +
sparse-attention step, counted by the PyTorch profiler, equal what
bench.launches_per_step claims (short and long sequences, sort QK)."""

from __future__ import annotations

import os
import sys

import pytest
import torch

import block_sparse_bidirectional_gb300 as bsb
import workloads

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def profiler_ready():
    """The first profiler session of a process may record no device activity
    while the tracer starts; one throwaway session over a small kernel."""
    from torch.profiler import ProfilerActivity, profile

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    x = torch.ones(1024, device="cuda:0")
    with profile(activities=[ProfilerActivity.CUDA]):
        (x * 2).sum().item()
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["llada", "long32k"])
def test_launches_per_step_matches_the_library(name, profiler_ready):
    from torch.profiler import ProfilerActivity, profile

    dev = torch.device("cuda:0")
    w = workloads.get(name)
    q, k, v, _ = workloads.make_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    kappa = w.kappa()

    def step():
        sel = bsb.ba_select(qd, kd, w.block, kappa, 1.0, bsb.SORT_QK)
        return bsb.ba_sparse_attn(qd, kd, vd, w.block, sel["perm_q"], sel["perm_k"], sel["block_idx"])

    step()  # outputs, workspaces and one-time attributes outside the profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        step()
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if e.device_type.name == "CUDA" and "ba::k_" in e.name]
    if not any(e.device_type.name == "CUDA" for e in prof.events()):
        pytest.skip("the profiler recorded no device activity on this machine")
    assert len(names) == bench.launches_per_step(w), names
