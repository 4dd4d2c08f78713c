"""The multi-rank decomposition of the shard step, on CPU with 2 gloo ranks.

Virtual rank r's RaggedShard slice is independent: the only exchange the
method needs between devices is one all-reduce of the fp64 sum of squares
before the group scale ("veScale-FSDP: Flexible and High-Performance FSDP at
Scale (MLSys 2026)" summary page, 核心方法 > Distributed Buffer; 结构感知训练
case study > 8-bit Adam: no metadata collective). Each process here owns half
of the virtual ranks (from libvsf's host-side rank slices), sums the squares
of its slices with the oracle, all-reduces, and must reach the single-process
norm and factor. It also checks the benchmark's max-over-ranks timing rule.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, max_norm, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from fsdp_buffer_layout_gb300 import vsf as V
        from synth import workloads as W
        w = W.tiny()
        descs = [V.make_desc(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors]
        plan = V.vsf_plan_create(descs, w.m, w.g_coll)
        try:
            per = w.m // world
            pieces = []
            for r in range(rank * per, (rank + 1) * per):
                for (t, e0, e1, _, _) in V.vsf_plan_rank_slices(plan, r):
                    pieces.append(np.ascontiguousarray(W.grad(w, 1, t)[e0:e1]))
            # this process's own plan: restricted to its window of ranks
            V.vsf_plan_restrict(plan, rank * per, (rank + 1) * per)
            mine = V.vsf_plan_get_info(plan)
        finally:
            V.vsf_plan_destroy(plan)
        counts = torch.tensor([mine.real, mine.n_qblocks, sum(p.size for p in pieces)],
                              dtype=torch.int64)
        assert counts[0] == counts[2]  # the window's real elements are its slices
        dist.all_reduce(counts)
        local = oracle.sumsq(pieces) if pieces else 0.0
        total = torch.tensor([local], dtype=torch.float64)
        dist.all_reduce(total)
        factor, norm = oracle.factor(float(total.item()), w.m, max_norm)
        t = torch.tensor([1.0 + rank], dtype=torch.float64)  # a per-rank "time"
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        out[rank] = (factor, norm, float(t.item()), len(pieces), int(counts[0]), int(counts[1]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("max_norm", [math.inf, 0.01])
def test_two_rank_norm_matches_single_process(max_norm):
    import oracle
    from synth import workloads as W
    w = W.tiny()
    whole = [W.grad(w, 1, t) for t in range(len(w.tensors))]
    want_f, want_n = oracle.factor(oracle.sumsq(whole), w.m, max_norm)
    from fsdp_buffer_layout_gb300 import vsf as V
    plan = V.vsf_plan_create([V.make_desc(t.shape, t.gran, t.block_rows, t.tile_cols)
                              for t in w.tensors], w.m, w.g_coll)
    try:
        info = V.vsf_plan_get_info(plan)
    finally:
        V.vsf_plan_destroy(plan)
    ctx = mp.get_context("spawn")
    with ctx.Manager() as man:
        out = man.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, max_norm, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in (0, 1):
        f, n, tmax, npieces, real, nq = res[rank]
        assert npieces > 0
        assert (real, nq) == (info.real, info.n_qblocks)  # the windows partition the plan
        assert abs(n - want_n) <= 1e-12 * want_n
        if math.isinf(max_norm):
            assert f == want_f == np.float32(0.25)
        else:
            assert abs(f - want_f) <= np.spacing(np.float32(want_f))
        assert tmax == 2.0  # every rank reports the slowest rank's time


def _sum_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from fsdp_buffer_layout_gb300.step import sum_all_reduce
        t = torch.tensor([0.5 * (rank + 1)], dtype=torch.float64)
        sum_all_reduce()(t)
        out[rank] = float(t.item())
    finally:
        dist.destroy_process_group()


def test_window_step_all_reduce_sums_over_processes():
    """sum_all_reduce, the exchange ShardStep.window_step calls, sums the
    one-element fp64 tensor of every process in place (gloo: 3 processes)."""
    world = 3
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_sum_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        assert [out[r] for r in range(world)] == [3.0] * world
