"""Benchmark of the BA-Att hot path on GB300: select + block-sparse attention.

One step = ba_select (norm sort, block statistics, compensated scores,
top-kappa) followed by ba_sparse_attn over one batch of the headline workload
(b1, 32 heads, L=65536, d=128, B=128, 50% sparsity, sort Q and K, beta 1),
synthetic seeded inputs resident in HBM.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload ultra64k] [--no-cpu-baseline]

With N > 1 (torchrun, one process per GPU) every rank runs its own batch
(heads are independent: weak scaling, no collective on the data path); the
ranks meet at a barrier around the timed region and rank 0 reports the
maximum time.  ``--impl reference`` times the fp64 CPU oracle on a bounded
sample of the same workload on the host cores.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ms & dense-equiv TFLOPS, select+sparse attn, L=64k 50% sparsity; select GB/s"
# The pages' own figure for this path, quoted as context only (other
# hardware, another baseline kernel, sparsity not stated): BA-Att §4.3,
# Fig. 4a; §1 gives the same 6.95x at 128K tokens.
PAGES_SPEEDUP = ("BA-Att (Sort) operator speedup over FlashAttention-2: up to 6.95x at 256K tokens "
                 "on an NVIDIA A100 80GB, Triton kernels, block 128 (BA-Att section 4.3, Fig. 4a); "
                 "context only, not comparable to this GB300 measurement")
UNIT = "TFLOPS (dense-equivalent 4*b*h*L^2*d per step / step time)"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p["bf16_tflops_sustained"]), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


# DRAM bytes (read + write) of one attention-kernel launch from the ncu
# traffic capture of the headline workload, valid only for the kernel source
# it was taken on (sha256 prefix of csrc/ba_attn.cu).
ATTN_TRAFFIC = {"ultra64k": dict(bytes=5344434432, kernel_sha="632145e13ebab681")}


def attn_traffic(workload: str):
    rec = ATTN_TRAFFIC.get(workload)
    if rec is None:
        return None
    import hashlib
    path = os.path.join(ROOT, "block_sparse_bidirectional_gb300", "csrc", "ba_attn.cu")
    with open(path, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return rec["bytes"] if sha == rec["kernel_sha"] else None


# ---- multi-GPU: one process per GPU, each on its own batch (weak scaling) ----
# Every (batch, head) is independent in every step of the path, so ranks
# exchange nothing on the data path: they meet at a barrier around the timed
# region and reduce their elapsed times with a max.

def rank_seed(w, rank: int) -> int:
    """Each rank draws its own batch of the workload."""
    return w.seed + rank


def rank_barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks_of(x: float, world: int, device) -> float:
    """The slowest rank's time (the whole job ends when it does)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_rank_step: float, ms_per_step: float) -> float:
    """Aggregate throughput: every rank's work over the max-over-ranks time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def dense_flops(w):
    return 4.0 * w.batch * w.heads * w.seqlen * w.seqlen * w.head_dim


def select_bytes(w, sort_q=True, sort_k=True, kappa=None):
    """Algorithmic bytes of the selection stage: Q and K are streamed once for
    the norms of each sorted tensor and once for the block statistics; small
    outputs (pi, index list, mask) are added."""
    t = w.batch * w.heads * w.seqlen * w.head_dim * 2
    reads = (2 if sort_q else 1) * t + (2 if sort_k else 1) * t
    N = w.nblocks
    kappa = w.kappa() if kappa is None else kappa
    writes = (2 * w.batch * w.heads * w.seqlen * 4
              + w.batch * w.heads * N * (kappa * 4 + ((N + 31) // 32) * 4))
    return reads + writes


def launches_per_step(w):
    """Kernels the library launches per step (select + sparse attention) for
    sort mode QK and no sort window: a norm pass (Q and K together), the sort
    of Q and K together (one chunk-sort launch for sequences of up to 8192
    tokens, else four radix passes), one statistics, one score and one
    top-kappa kernel; then the tile-pair list kernel, one row-gather kernel
    (Q, K, V) and the attention kernel."""
    sort = 1 if w.seqlen <= 8192 else 4
    select = 1 + sort + 3
    attn = 3
    return select + attn


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(n)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(mx) if mx else None,
                    reasons=sorted(reasons), samples=len(sm))


def cpu_oracle_sample(w, q, k, v, budget_s=12.0, seed=0, kappa=None):
    """Times the fp64 oracle on one head: its whole selection plus as many
    sampled query blocks of attention as fit in ``budget_s``; extrapolates
    to the head's full work and returns dense-equivalent TFLOPS."""
    import numpy as np

    import oracle.ba_oracle as O
    kappa = w.kappa() if kappa is None else kappa
    Q = q[0, 0].double().numpy()
    K = k[0, 0].double().numpy()
    V = v[0, 0].double().numpy()
    t0 = time.perf_counter()
    sel = O.select_one(Q, K, w.block, kappa, 1.0, O.SORT_QK)
    t_sel = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    order = rng.permutation(w.nblocks)
    done = 0
    t1 = time.perf_counter()
    while done < len(order) and (done < 4 or time.perf_counter() - t1 < budget_s):
        O.sparse_attention_one(Q, K, V, sel["perm_q"], sel["perm_k"], sel["idx"], w.block,
                               query_blocks=[int(order[done])])
        done += 1
    t_att = time.perf_counter() - t1
    per_head = t_sel + t_att / done * w.nblocks
    head_flops = 4.0 * w.seqlen * w.seqlen * w.head_dim
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    full = done == w.nblocks and w.heads * w.batch == 1
    return dict(value=head_flops / per_head / 1e12, unit=UNIT, cores=cores, kind="oracle",
                sample=(f"1 of {w.heads} heads: full selection ({t_sel:.2f} s) + {done} of "
                        f"{w.nblocks} query blocks of attention ({t_att:.2f} s), "
                        + ("the whole workload" if full else
                           f"extrapolated linearly to the head ({per_head:.1f} s) and the {w.heads} heads")
                        + "; fp64 numpy"),
                ms_per_step=per_head * w.heads * w.batch * 1e3, extrapolated=not full,
                seconds=t_sel + t_att)


def _oracle_head(job):
    """One head through the fp64 oracle: selection, then attention over every
    query block (a process-pool task)."""
    import numpy as np

    import oracle.ba_oracle as O
    Q, K, V, B, kappa = job
    t0 = time.perf_counter()
    sel = O.select_one(Q, K, B, kappa, 1.0, O.SORT_QK)
    O.sparse_attention_one(Q, K, V, sel["perm_q"], sel["perm_k"], sel["idx"], B,
                           query_blocks=list(range(-(-Q.shape[0] // B))))
    return time.perf_counter() - t0


def cpu_oracle_full(w, q, k, v, kappa, workers=None):
    """The fp64 oracle over the whole workload (every head, every query
    block), one head per task on a spawn-started process pool."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    workers = max(1, min(workers or cores, w.batch * w.heads))
    jobs = [(q[bb, hh].double().numpy(), k[bb, hh].double().numpy(), v[bb, hh].double().numpy(), w.block, kappa)
            for bb in range(w.batch) for hh in range(w.heads)]
    # one BLAS thread per worker process (the workers inherit the environment
    # when they are spawned; the parent's own BLAS is already set up)
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {key: os.environ.get(key) for key in keys}
    os.environ.update({key: "1" for key in keys})
    try:
        t0 = time.perf_counter()
        with mp.get_context("spawn").Pool(workers) as pool:
            per_head = pool.map(_oracle_head, jobs, chunksize=1)
        wall = time.perf_counter() - t0
    finally:
        for key, val in saved.items():
            if val is None:
                os.environ.pop(key, None)
            else:
                os.environ[key] = val
    return dict(ms_per_step=wall * 1e3, extrapolated=False, cores=workers,
                sample=(f"the whole workload: {len(jobs)} heads, selection + attention over every query block, "
                        f"one head per task on {workers} spawned processes (wall {wall:.1f} s, sum of head "
                        f"times {sum(per_head):.1f} s, pool start-up included); fp64 numpy"))


def run_reference(args):
    """The oracle as the reference arm, on the host cores of rank 0."""
    import workloads
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = workloads.get(args.workload)
    q, k, v, _ = workloads.make_inputs(w)
    values = []
    for i in range(args.warmup + args.steps):
        r = cpu_oracle_sample(w, q, k, v, budget_s=max(2.0, 60.0 / max(1, args.steps + args.warmup)), seed=i)
        if i >= args.warmup:
            values.append(r)
    val = statistics.median(x["value"] for x in values)
    head_ms = dense_flops(w) / w.heads / (val * 1e12) * 1e3
    out = dict(impl="reference", metric=METRIC, value=val, unit=UNIT, n_gpus=args.gpus, steps=args.steps,
               warmup=args.warmup, ms_per_step=head_ms * w.heads, higher_is_better=True,
               scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
               config=workload_config(w),
               cpu_baseline=dict(value=val, unit=UNIT, cores=values[-1]["cores"], kind="oracle",
                                 sample=values[-1]["sample"]),
               e2e=dict(value=val, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0),
               gpu_launches=0)
    print(json.dumps(out), flush=True)
    return 0


def workload_config(w):
    return dict(workload=(f"{w.name}: b{w.batch} h{w.heads} L{w.seqlen} d{w.head_dim} B{w.block} "
                          f"kappa{w.kappa()} ({int(w.sparsities[0] * 100)}% sparsity), sort QK, beta 1"),
                global_batch=w.batch, seq_len=w.seqlen, heads=w.heads, head_dim=w.head_dim,
                block=w.block, kappa=w.kappa(),
                l2=f"inputs {3 * w.batch * w.heads * w.seqlen * w.head_dim * 2 / 2**30:.2f} GiB > L2, no flush",
                parallelism="independent heads per GPU (no collective)")


def measure_workload(bsb, w, sparsity, dev, steps=5, dense_steps=2, cpu_budget_s=4.0, with_cpu=True):
    """One workload at one sparsity, as its own select + sparse attention
    step: stage times (CUDA events, median of ``steps``), attention TFLOP/s on
    the computed tiles and its fraction of the bf16 peak, selection GB/s,
    the library's dense kernel at the same shape, and a bounded sample of the
    fp64 oracle on the host cores."""
    import numpy as np
    import torch

    import workloads
    q, k, v, _ = workloads.make_inputs(w)
    kappa = w.kappa(sparsity)
    b, h, L, d, B, N = w.batch, w.heads, w.seqlen, w.head_dim, w.block, w.nblocks
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    i32 = dict(dtype=torch.int32, device=dev)
    perm_q, perm_k = torch.empty((b, h, L), **i32), torch.empty((b, h, L), **i32)
    idx = torch.empty((b, h, N, kappa), **i32)
    mask = torch.empty((b, h, N, (N + 31) // 32), **i32)
    ws_sel = torch.empty(bsb.select_workspace_size(b, h, L, d, B, kappa, 3, 0), dtype=torch.uint8, device=dev)
    ws_att = torch.empty(max(1, bsb.sparse_attn_workspace_size(b, h, L, d, B, kappa)), dtype=torch.uint8,
                         device=dev)
    o, lse = torch.empty_like(qd), torch.empty((b, h, L), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def sel():
        bsb.ba_select_into(qd, kd, B, kappa, 1.0, 3, 0, perm_q, perm_k, idx, mask, None, ws_sel)

    def att():
        bsb.ba_sparse_attn_into(qd, kd, vd, B, perm_q, perm_k, idx, 0.0, o, lse, ws_att)
    for _ in range(3):
        sel()
        att()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e in ev:
        e[0].record(stream)
        sel()
        e[1].record(stream)
        att()
        e[2].record(stream)
    torch.cuda.synchronize(dev)
    st, word = bsb.last_device_error(dev)
    if st != 0:
        raise RuntimeError(f"device error word {word:#x} ({w.name})")
    sel_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    att_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    step_ms = statistics.median(e[0].elapsed_time(e[2]) for e in ev)
    sizes = np.full(N, B, dtype=np.float64)
    sizes[-1] = L - (N - 1) * B
    pair_tokens = sizes[idx.cpu().numpy()].sum(axis=-1)
    flops = float(4.0 * d * (pair_tokens * sizes[None, None, :]).sum())
    od, lsed = torch.empty_like(qd), torch.empty_like(lse)
    bsb.ba_attn_dense_into(qd, kd, vd, 0.0, od, lsed)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(dense_steps):
        bsb.ba_attn_dense_into(qd, kd, vd, 0.0, od, lsed)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    dense_ms = e0.elapsed_time(e1) / dense_steps
    pk = peaks()
    att_tf = flops / (att_ms * 1e-3) / 1e12
    sb = select_bytes(w, kappa=kappa)
    out = dict(workload=f"{w.name}: b{b} h{h} L{L} d{d} B{B} kappa{kappa} ({int(round(sparsity * 100))}% sparsity)",
               step_ms=round(step_ms, 4), select_ms=round(sel_ms, 4), attn_ms=round(att_ms, 4),
               attn_actual_tflops=round(att_tf, 2), attn_frac_tensor_burst=round(att_tf / pk["bf16"], 4),
               step_frac_tensor_burst=round(flops / (step_ms * 1e-3) / 1e12 / pk["bf16"], 4),
               select_gbs=round(sb / (sel_ms * 1e-3) / 1e9, 1),
               select_frac_hbm_measured=round(sb / (sel_ms * 1e-3) / 1e9 / pk["hbm"], 4),
               dense_ms=round(dense_ms, 4),
               dense_frac_tensor_burst=round(4.0 * b * h * L * L * d / (dense_ms * 1e-3) / 1e12 / pk["bf16"], 4),
               speedup_vs_dense=round(dense_ms / step_ms, 3), density=round(flops / (4.0 * b * h * L * L * d), 4))
    if with_cpu:
        # the two smallest workloads in full; the others as one head's
        # selection in full plus sampled attention, extrapolated
        c = (cpu_oracle_full(w, q, k, v, kappa) if w.index <= 2
             else cpu_oracle_sample(w, q, k, v, budget_s=cpu_budget_s, kappa=kappa))
        out["cpu_oracle"] = dict(ms_per_step=round(c["ms_per_step"], 1), extrapolated=c["extrapolated"],
                                 cores=c["cores"], sample=c["sample"])
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ultra64k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dense-steps", type=int, default=3)
    ap.add_argument("--no-fidelity", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload detail (all five shapes, each sparsity)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch
    import torch.distributed as dist

    import block_sparse_bidirectional_gb300 as bsb
    import workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)

    def barrier():
        rank_barrier(world)

    def max_over_ranks(x):
        return max_over_ranks_of(x, world, dev)

    w = workloads.get(args.workload)
    kappa = w.kappa()
    q, k, v, _ = workloads.make_inputs(w, seed=rank_seed(w, rank))
    b, h, L, d, B = w.batch, w.heads, w.seqlen, w.head_dim, w.block
    N = w.nblocks
    bsb.load()
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    # outputs and workspaces allocated once, outside the timed region
    i32 = dict(dtype=torch.int32, device=dev)
    perm_q = torch.empty((b, h, L), **i32)
    perm_k = torch.empty((b, h, L), **i32)
    idx = torch.empty((b, h, N, kappa), **i32)
    mask = torch.empty((b, h, N, (N + 31) // 32), **i32)
    ws_sel = torch.empty(bsb.select_workspace_size(b, h, L, d, B, kappa, 3, 0), dtype=torch.uint8, device=dev)
    ws_att = torch.empty(bsb.sparse_attn_workspace_size(b, h, L, d, B, kappa), dtype=torch.uint8, device=dev)
    o = torch.empty_like(qd)
    lse = torch.empty((b, h, L), dtype=torch.float32, device=dev)

    def step_to(qx, kx, vx, ox, lx):
        bsb.ba_select_into(qx, kx, B, kappa, 1.0, 3, 0, perm_q, perm_k, idx, mask, None, ws_sel)
        bsb.ba_sparse_attn_into(qx, kx, vx, B, perm_q, perm_k, idx, 0.0, ox, lx, ws_att)

    def step(qx, kx, vx):
        step_to(qx, kx, vx, o, lse)

    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        step(qd, kd, vd)
    torch.cuda.synchronize(dev)
    st, word = bsb.last_device_error(dev)
    if st != 0:
        raise RuntimeError(f"device error word {word:#x} after warm-up")

    # algorithmic attention FLOPs from the emitted mask (4 d per selected
    # query-key pair; the ragged last block counts its real tokens)
    sizes = np.full(N, B, dtype=np.float64)
    sizes[-1] = L - (N - 1) * B
    idx_np = idx.cpu().numpy()
    pair_tokens = sizes[idx_np].sum(axis=-1)            # [b,h,N]: keys per query block
    attn_flops = float(4.0 * d * (pair_tokens * sizes[None, None, :]).sum())

    # ---- timed region: K steps, events per stage ----------------------------
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        bsb.ba_select_into(qd, kd, B, kappa, 1.0, 3, 0, perm_q, perm_k, idx, mask, None, ws_sel)
        ev[i][1].record(stream)
        bsb.ba_sparse_attn_into(qd, kd, vd, B, perm_q, perm_k, idx, 0.0, o, lse, ws_att)
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end))
    sel_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    att_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    st, word = bsb.last_device_error(dev)
    if st != 0:
        raise RuntimeError(f"device error word {word:#x} in the timed region")
    ms_step = total_ms / args.steps

    # ---- the library's dense kernel at the same shape -----------------------
    od = torch.empty_like(qd)
    lsed = torch.empty_like(lse)
    bsb.ba_attn_dense_into(qd, kd, vd, 0.0, od, lsed)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.dense_steps):
        bsb.ba_attn_dense_into(qd, kd, vd, 0.0, od, lsed)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    dense_ms = e0.elapsed_time(e1) / args.dense_steps
    del od, lsed

    # ---- LoSA locality pruning at the same shape (groups of 32, top 4) -------
    # reads the current and the previous query (2 x b*h*L*d bf16): HBM-bound
    q_prev = qd.clone()
    q_prev.view(-1)[::7] += 1
    act = torch.empty((b, h, L), dtype=torch.uint8, device=dev)
    lib = bsb.load()
    pq_ptr, pp_ptr = bsb._ptr(qd), bsb._ptr(q_prev)
    st_ptr = bsb._stream(dev)

    def losa():
        r = lib.ba_active_tokens(pq_ptr, pp_ptr, b, h, L, d, 32, 4, bsb._ptr(act), None, st_ptr)
        if r != 0:
            raise RuntimeError(f"ba_active_tokens status {r}")
    losa()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(5):
        losa()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    losa_ms = e0.elapsed_time(e1) / 5
    losa_bytes = 2 * qd.numel() * qd.element_size() + act.numel()
    del q_prev, act

    # ---- isolated selection (SparseD §3.3) at the same shape ----------------
    # the first quarter of the tokens as prompt, half of each part's key blocks
    pre = (L // 4) // B * B
    n_pre = pre // B
    kpre, kgen = max(1, n_pre // 2), max(1, (N - n_pre) // 2)
    idx_iso = torch.empty((b, h, N, kpre + kgen), **i32)
    ws_iso = torch.empty(bsb.select_workspace_size(b, h, L, d, B, kpre + kgen, 3, 0),
                         dtype=torch.uint8, device=dev)

    def iso():
        bsb.ba_select_isolated_into(qd, kd, B, pre, kpre, kgen, 1.0, 3, 0, perm_q, perm_k, idx_iso,
                                    mask, None, ws_iso)
    iso()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(5):
        iso()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    iso_ms = e0.elapsed_time(e1) / 5

    # ---- the selection's variants (the pages' ablation axes, Tab. 7) -------
    # beta = 0 drops the covariance term ("Ours (Sort)", the pages' fastest
    # operator); the sort modes choose which sequences are norm-sorted
    def time_select(beta, mode, reps=5):
        ws_v = torch.empty(bsb.select_workspace_size(b, h, L, d, B, kappa, mode, 0), dtype=torch.uint8,
                           device=dev)
        bsb.ba_select_into(qd, kd, B, kappa, beta, mode, 0, perm_q, perm_k, idx, mask, None, ws_v)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(reps):
            bsb.ba_select_into(qd, kd, B, kappa, beta, mode, 0, perm_q, perm_k, idx, mask, None, ws_v)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return round(e0.elapsed_time(e1) / reps, 4)
    variant_ms = dict(select_ms_beta0_sort_qk=time_select(0.0, 3),
                      select_ms_beta1_sort_k=time_select(1.0, 1),
                      select_ms_beta1_sort_q=time_select(1.0, 2),
                      select_ms_beta1_no_sort=time_select(1.0, 0))
    del idx_iso, ws_iso

    # ---- end to end through the public API from pinned host memory ----------
    # Every step uploads its inputs (Q, K, V) from pinned host memory and
    # downloads its result (O, LSE) inside the timed region.  Inputs and
    # outputs are double-buffered and the copies run on their own streams, so
    # step i+1's upload and step i's download overlap step i's compute and
    # each other; events order every reuse of a buffer.
    e2e_steps = max(3, min(args.steps, 10))
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    xin = [tuple(torch.empty_like(t) for t in (qd, kd, vd)) for _ in range(2)]
    xout = [(torch.empty_like(o), torch.empty_like(lse)) for _ in range(2)]
    hout = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(),
             torch.empty(lse.shape, dtype=lse.dtype).pin_memory()) for _ in range(2)]
    # one upload stream per input tensor (they can use several copy engines
    # at once) and one download stream
    ustreams = [torch.cuda.Stream(dev) for _ in range(3)]
    dstream = torch.cuda.Stream(dev)

    def e2e_run(n, start_event):
        ev_in = [[torch.cuda.Event() for _ in range(3)] for _ in range(n)]  # step i's inputs on the device
        ev_done = [torch.cuda.Event() for _ in range(n)]  # step i computed
        ev_out = [torch.cuda.Event() for _ in range(n)]   # step i's result on the host
        for us in ustreams:
            us.wait_event(start_event)
        dstream.wait_event(start_event)

        def upload(i):
            for c, (us, dst, src) in enumerate(zip(ustreams, xin[i % 2], (qh, kh, vh))):
                with torch.cuda.stream(us):
                    if i >= 2:
                        us.wait_event(ev_done[i - 2])     # this slot's inputs are consumed
                    dst.copy_(src, non_blocking=True)
                    ev_in[i][c].record(us)

        upload(0)
        for i in range(n):
            sl = i % 2
            if i + 1 < n:
                upload(i + 1)
            for c in range(3):
                stream.wait_event(ev_in[i][c])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])          # this slot's outputs are downloaded
            step_to(*xin[sl], *xout[sl])
            ev_done[i].record(stream)
            with torch.cuda.stream(dstream):
                dstream.wait_event(ev_done[i])
                hout[sl][0].copy_(xout[sl][0], non_blocking=True)
                hout[sl][1].copy_(xout[sl][1], non_blocking=True)
                ev_out[i].record(dstream)
        stream.wait_event(ev_out[n - 1])
        for us in ustreams:
            stream.wait_stream(us)

    w0 = torch.cuda.Event()
    w0.record(stream)
    e2e_run(2, w0)
    torch.cuda.synchronize(dev)
    barrier()
    e0.record(stream)
    e2e_run(e2e_steps, e0)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1)) / e2e_steps
    del xin, xout, hout

    # ---- fidelity diagnostics (BA-Att §3.1 Eq. 3, §3.2 Eq. 5-8) -------------
    # The share of the dense attention mass the headline selection keeps
    # (mean recall), with the norm sort and without it, and how well the
    # bound U of Eq. 8 tracks the observed token-vs-block logit deviation
    # (correlation over block pairs: a synthetic analogue of the paper's
    # Fig. 2).  Timed: one ba_block_fidelity call (S = Q K^T over every tile
    # pair on the tensor cores + the exp sums).
    fid = dict()
    if not args.no_fidelity:
        _, lse_dense = bsb.ba_attn_dense(qd, kd, vd)
        bsb.ba_select_into(qd, kd, B, kappa, 1.0, 3, 0, perm_q, perm_k, idx, mask, None, ws_sel)
        bsb.ba_block_fidelity(qd, kd, B, lse_dense, perm_q, perm_k, idx)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        f_sorted = bsb.ba_block_fidelity(qd, kd, B, lse_dense, perm_q, perm_k, idx)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        fid_ms = e0.elapsed_time(e1)
        sel0 = bsb.ba_select(qd, kd, B, kappa, 1.0, bsb.SORT_NONE)
        f_plain = bsb.ba_block_fidelity(qd, kd, B, lse_dense, sel0["perm_q"], sel0["perm_k"],
                                        sel0["block_idx"])
        torch.cuda.synchronize(dev)

        def corr(fd):
            x, y = fd["bound"].flatten().double(), fd["dev_max"].flatten().double()
            return float(torch.corrcoef(torch.stack([x, y]))[0, 1])
        s_flops = 2.0 * b * h * L * L * d
        fid = dict(fidelity_ms=round(fid_ms, 3),
                   fidelity_s_tflops=round(s_flops / (fid_ms * 1e-3) / 1e12, 1),
                   recall_mean_sorted=round(float(f_sorted["recall"].double().mean()), 4),
                   recall_mean_unsorted=round(float(f_plain["recall"].double().mean()), 4),
                   bound_dev_corr_sorted=round(corr(f_sorted), 4),
                   bound_dev_corr_unsorted=round(corr(f_plain), 4),
                   dev_over_bound_sorted=round(float((f_sorted["dev_max"] / f_sorted["bound"]).double().mean()), 4))
        del f_sorted, f_plain, sel0, lse_dense
    # ---- every workload of the table, each sparsity (its own step) ----------
    per_workload = {}
    if not args.no_workloads:
        with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
        for wn in ("tiny", "llada", "long32k", "video"):
            ww = workloads.get(wn)
            for sp in ww.sparsities:
                per_workload[f"{wn}@{int(round(sp * 100))}"] = measure_workload(bsb, ww, sp, dev, with_cpu=with_cpu)
                torch.cuda.empty_cache()
    h2d = 3 * q.numel() * q.element_size()
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()

    pk = peaks()
    flops_step = dense_flops(w)
    value = whole_job_tflops(world, flops_step, ms_step)
    att_tflops = attn_flops / (att_ms * 1e-3) / 1e12
    sel_b = select_bytes(w)
    sel_gbs = sel_b / (sel_ms * 1e-3) / 1e9
    out = dict(
        metric=METRIC, value=round(value, 3), unit=UNIT, n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=round(ms_step, 4), higher_is_better=True, scaling="weak",
        vs_baseline=None, dtype="bf16", data="synthetic", config=workload_config(w),
        roofline=dict(bound="tensor", achieved=round(att_tflops, 2), peak=pk["bf16"], unit="TFLOP/s",
                      frac=round(att_tflops / pk["bf16"], 4), traffic=attn_traffic(w.name),
                      kernel="ba_sparse_attn (tile-pair lists + row gathers + tcgen05 attention kernel)",
                      peak_kind=f"bf16 dense burst, {pk['source']}",
                      algorithmic_flops_per_launch=attn_flops),
        e2e=dict(value=round(whole_job_tflops(world, flops_step, e2e_ms), 3), unit=UNIT,
                 ms_per_step=round(e2e_ms, 3), h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                 steps=e2e_steps,
                 copies="double-buffered; uploads on three streams, downloads on a fourth, overlapping compute"),
        gpu_launches=launches_per_step(w) * args.steps,
        clocks=dict(sm_mhz=clk["sm_mhz"], sm_max_mhz=clk["sm_max_mhz"], reasons=clk["reasons"],
                    samples=clk["samples"]),
        detail=dict(
            select_ms=round(sel_ms, 4), attn_ms=round(att_ms, 4),
            select_gbs=round(sel_gbs, 1), select_bytes=sel_b,
            select_frac_hbm_measured=round(sel_gbs / pk["hbm"], 4),
            select_frac_hbm_nominal_8tbs=round(sel_gbs / 8000.0, 4),
            attn_actual_tflops=round(att_tflops, 2),
            attn_frac_tensor_burst=round(att_tflops / pk["bf16"], 4),
            attn_frac_tensor_sustained=round(att_tflops / pk["bf16_sus"], 4),
            dense_ms=round(dense_ms, 3),
            dense_tflops=round(flops_step / (dense_ms * 1e-3) / 1e12, 2),
            dense_frac_tensor_burst=round(flops_step / (dense_ms * 1e-3) / 1e12 / pk["bf16"], 4),
            speedup_vs_dense=round(dense_ms / ms_step, 3),
            # selection + sparse attention together, on the computed tiles
            step_actual_tflops=round(attn_flops / (ms_step * 1e-3) / 1e12, 2),
            step_frac_tensor_burst=round(attn_flops / (ms_step * 1e-3) / 1e12 / pk["bf16"], 4),
            pages_speedup_context=PAGES_SPEEDUP,
            isolated_select_ms=round(iso_ms, 4),
            **variant_ms,
            active_tokens_ms=round(losa_ms, 4),
            active_tokens_gbs=round(losa_bytes / (losa_ms * 1e-3) / 1e9, 1),
            # against the measured copy bandwidth (read + write); a read-mostly
            # kernel can exceed 1.0 of it
            active_tokens_frac_of_copy_bw=round(losa_bytes / (losa_ms * 1e-3) / 1e9 / peaks()["hbm"], 4),
            isolated_select=f"prefill {pre} tokens, kappa {kpre} + {kgen}, sort QK",
            **fid,
            density=round(attn_flops / flops_step, 4),
            workloads=per_workload),
    )
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = {kk: vv for kk, vv in cpu_oracle_sample(w, q, k, v).items() if kk != "seconds"}
    elif rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
