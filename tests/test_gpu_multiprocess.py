"""The shard step as several processes, each owning a window of the virtual
ranks, against one process running the whole plan.

Each process restricts the plan to its ranks [r0, r1) (vsf_plan_restrict),
runs pack, its window's fp64 sum of squares, a torch.distributed all-reduce
of that one scalar (gloo, through the host: the path's one exchange,
"veScale-FSDP: Flexible and High-Performance FSDP at Scale (MLSys 2026)"
summary page, 核心方法 > Distributed Buffer), the factor, the 8-bit AdamW and
unpack (ShardStep.window_step), for every step. The processes share this
machine's one GPU; no kernel waits on another process's kernel, the only
synchronisation is the host-side all-reduce between launches. Their windows,
stitched together, must equal the whole plan's buffers and scales byte for
byte, and every process's parameters must equal its packed bf16 copy on the
window's elements.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from synth import workloads as W

import gpu_harness as H

pytestmark = pytest.mark.gpu

KEYS = ("packed_grad", "master", "m_state", "v_state", "packed_bf16")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _host(x):
    if x.dtype == torch.bfloat16:
        x = x.view(torch.int16)
    return x.cpu().numpy()


def _worker(rank, world, port, name, windows, steps, outdir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from fsdp_buffer_layout_gb300 import vsf as V
        from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec, sum_all_reduce
        torch.cuda.set_device(0)
        case = H.case_from_workload(W.get(name), steps=steps)
        r0, r1 = windows[rank]
        specs = [TensorSpec(tuple(s[0]), s[1], s[2], s[3]) for s in case.specs]
        ss = ShardStep(specs, case.m, case.g_coll, max_norm=case.max_norm, ranks=(r0, r1))
        try:
            dev, S, offs = ss.device, ss.info.S, ss.offsets
            lo, hi = r0 * S, r1 * S
            for t in range(len(specs)):
                m, o = case.masters(t), offs[t]
                a, b = max(lo, o), min(hi, o + m.size)
                if a < b:
                    ss.master[a - lo:b - lo].copy_(torch.from_numpy(m[a - o:b - o]).to(dev))
            grads = [torch.empty(n, dtype=torch.int16, device=dev) for n in case.numels]
            params = [torch.zeros(n, dtype=torch.int16, device=dev) for n in case.numels]
            reduce = sum_all_reduce()
            factors = []
            for s in range(1, steps + 1):
                for t, g in enumerate(grads):
                    g.copy_(torch.from_numpy(case.grads(s, t).view(np.int16)))
                ss.window_step(grads, params, s, reduce)
                torch.cuda.synchronize()
                assert ss.device_error() == 0, "a bounded device wait ran out"
                factors.append(float(ss.factor[0].item()))
            bf = _host(ss.packed_bf16)
            for t, p in enumerate(params):  # copy-out of the window's elements
                o, n = offs[t], case.numels[t]
                a, b = max(lo, o), min(hi, o + n)
                if a < b:
                    assert np.array_equal(_host(p)[a - o:b - o], bf[a - lo:b - lo]), t
            nq = ss.info.n_qblocks
            bases = V.vsf_plan_qblocks(ss.plan, nq)["base"] if nq else []
            out = {k: _host(getattr(ss, k)) for k in KEYS}
            out.update(m_scale=_host(ss.m_scale)[:nq], v_scale=_host(ss.v_scale)[:nq],
                       qbase=np.array(bases, np.int64) + lo, factors=np.array(factors))
            np.savez(os.path.join(outdir, f"rank{rank}.npz"), **out)
        finally:
            ss.close()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,windows,steps", [
    ("tiny", [(0, 1), (1, 4)], 3),
    ("llama_layer", [(0, 3), (3, 8)], 2),
])
def test_processes_over_rank_windows_equal_the_whole_plan(name, windows, steps, tmp_path):
    world = len(windows)
    mp.spawn(_worker, args=(world, _free_port(), name, windows, steps, str(tmp_path)),
             nprocs=world, join=True)
    case = H.case_from_workload(W.get(name), steps=steps)
    want = H.run_gpu(case)
    S = want["S"]
    from fsdp_buffer_layout_gb300 import vsf as V
    p = V.vsf_plan_create([V.make_desc(*s) for s in case.specs], case.m, case.g_coll)
    try:
        nq = V.vsf_plan_get_info(p).n_qblocks
        index = {int(b): q for q, b in enumerate(V.vsf_plan_qblocks(p, nq)["base"])}
    finally:
        V.vsf_plan_destroy(p)
    seen = 0
    for rank, (r0, r1) in enumerate(windows):
        got = np.load(tmp_path / f"rank{rank}.npz")
        assert list(got["factors"]) == want["factors"], rank
        lo, hi = r0 * S, r1 * S
        for k in KEYS:
            assert H.bit_equal(got[k], want[k][lo:hi], bf16=(k == "packed_bf16")), (rank, k)
        ids = np.array([index[int(b)] for b in got["qbase"]], np.int64)
        assert H.bit_equal(got["m_scale"], want["m_scale"][ids]), rank
        assert H.bit_equal(got["v_scale"], want["v_scale"][ids]), rank
        seen += ids.size
    assert seen == len(want["m_scale"]), "the windows' blocks do not cover the plan"
