"""Benchmark of the fused shard step (pack -> group norm/scale -> 8-bit AdamW ->
unpack) through libvsf's C ABI on one GB300, one JSON line on stdout.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Metric: algorithmic HBM bytes of the step per second (GB/s) and parameters
updated per second, against the measured HBM copy bandwidth. Algorithmic
bytes per real element (bf16 gradients): pack 2+2, AdamW 2+1+1+4 read and
1+1+4+2 written, unpack 2+2, i.e. 24 B, plus 16 B of scales per
quantisation block. Padding is never touched, so it is not counted.

Default workload: the 24-layer Llama-style 1.3B model (m = 1024 virtual
ranks), the largest workload that fits one GPU. Every step gets fresh
gradients (two seeded sets alternate). The line also carries the copy ceiling
measured in the same run (device-to-device memcpy and a 128-bit copy kernel).

Timing: W untimed steps, then K steps between a barrier and a device
synchronise, CUDA events on the launch stream; the inputs (32 GB per step for
the 1.3B model, 4.9 GB for one Llama layer) are larger than L2, so no flush is
needed. Under torchrun
(N > 1) every rank runs an independent replica of the workload (the m
virtual ranks of one buffer live on one GPU); value = sum over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused shard-step HBM GB/s and params/s vs GB300 HBM roofline"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # HBM3e specification figure the measured copy is set against
MUON_METRIC = "distributed Muon step Newton-Schulz TFLOP/s vs GB300 bf16 tensor roofline"
GROUP_METRIC = "fused DBuffer group ops (zero, scale, add) HBM GB/s vs GB300 HBM roofline"
# algorithmic bytes per real element of each group op, in step order
GROUP_OPS = (("zero bf16", 2), ("scale bf16", 4), ("add bf16 += bf16", 6),
             ("add fp32 += bf16", 10))
FALLBACK_BF16_TFLOPS = 1900.0


def algorithmic_bytes(n_real: int, n_qblocks: int, grad_bytes: int = 2,
                      zero_copy: bool = False) -> dict:
    """Bytes the step must move per real element. Zero-copy mode (gradients
    and parameters are views of the packed buffers) drops copy-in and
    copy-out; its group norm reads the packed gradient once instead."""
    adam = n_real * (grad_bytes + 1 + 1 + 4 + 1 + 1 + 4 + 2) + 16 * n_qblocks
    if zero_copy:
        return dict(pack=n_real * grad_bytes, adam=adam, unpack=0,
                    step=n_real * grad_bytes + adam)
    return dict(pack=n_real * 2 * grad_bytes, adam=adam, unpack=n_real * 4,
                step=n_real * 2 * grad_bytes + adam + n_real * 4)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak(sustained: bool):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(path) as f:
            return float(json.load(f)[key]), f"measured (MEASURED_PEAKS.json {key})"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback 1.9 PFLOP/s bf16"


GEMM_BM, GEMM_BN = 256, 256  # output tile of libvsf's Newton-Schulz kernel (one CTA pair)


def sym_tiles(n: int) -> int:
    """Output tiles of one n x n symmetric product that libvsf computes: in
    column block J (256 columns) the row groups 0 .. J (256 rows each), the
    tiles that reach the diagonal or lie above it."""
    mb, nb = -(-n // GEMM_BM), -(-n // GEMM_BN)
    return sum(min(mb, J + 1) for J in range(nb))


def sym_fraction(n: int) -> float:
    """Share of a symmetric n x n product's FLOPs that libvsf's tensor-core
    kernel executes (its computed tiles over all tiles; about 1/2 for large n)."""
    mb, nb = -(-n // GEMM_BM), -(-n // GEMM_BN)
    return sym_tiles(n) / float(mb * nb)


def muon_flops(w, ns_steps: int = 5, executed: bool = False) -> float:
    """Newton-Schulz FLOPs of one Muon step over every matrix tensor of w.
    By the definition, per iteration: 2 n^2 k for the Gram matrix, 2 n^3 for
    its square, 2 n^2 k for the product with X (n = min(R, C), k = max(R, C)).
    executed=True counts what the tensor cores run: the two symmetric
    products only on the tiles that reach or lie above the diagonal."""
    total = 0.0
    for t in w.tensors:
        if len(t.shape) < 2:
            continue
        *lead, R, C = t.shape
        n, k = min(R, C), max(R, C)
        sym = sym_fraction(n) if executed else 1.0
        per = sym * (2.0 * n * n * k + 2.0 * n ** 3) + 2.0 * n * n * k
        total += float(np.prod(lead, dtype=np.float64)) * per
    return total * ns_steps


def sample_workload(w, fraction: float):
    """The same tensor list with every tensor cut to about `fraction` of its
    rows (whole atoms kept), for the CPU oracle's bounded sample."""
    from synth.workloads import GRAN_ELEM, TensorSpec
    ts = []
    for t in w.tensors:
        if t.gran == GRAN_ELEM:
            n = max(w.g_coll, int(round(t.numel * fraction / w.g_coll)) * w.g_coll)
            ts.append(TensorSpec(t.name, (min(n, t.numel),), t.gran))
        else:
            rows = max(t.block_rows, int(round(t.rows * fraction / t.block_rows)) * t.block_rows)
            rows = min(rows, t.rows)
            ts.append(TensorSpec(t.name, (rows, t.cols), t.gran, t.block_rows, t.tile_cols))
    return w.with_(tensors=tuple(ts))


# ---------------------------------------------------------------- CPU oracle

def oracle_steps(w, steps: int):
    """Runs the oracle's full step (pack, sumsq, factor, AdamW over every block,
    unpack) `steps` times on workload w; returns (seconds per step, real
    elements, quantisation blocks). Inputs are drawn outside the timing."""
    import oracle
    from synth import workloads as W
    d = oracle.Desc.from_workload(w)
    S, off = oracle.plan(d, w.m, w.g_coll)
    qb = oracle.qblocks(d, w.g_coll, off)
    total = w.m * S
    master = oracle.pack([W.master_init(w, t) for t in range(d.n)], off, total)
    ms, vs = np.zeros(total, np.int8), np.zeros(total, np.uint8)
    nq = len(qb["base"])
    msc, vsc = np.zeros(nq, np.float32), np.zeros(nq, np.float32)
    bf = np.zeros(total, np.uint16)
    hp = oracle.hparams(w)
    numels = [t.numel for t in w.tensors]
    times = []
    for s in range(1, steps + 1):
        grads = [W.grad(w, s, t) for t in range(d.n)]
        t0 = time.perf_counter()
        packed = oracle.pack(grads, off, total)
        f, _ = oracle.factor(oracle.sumsq(grads), w.m, w.max_norm)
        oracle.adam_all(qb, packed, f, True, ms, vs, msc, vsc, master, bf, s, hp)
        oracle.unpack(bf, numels, off)
        times.append(time.perf_counter() - t0)
    return sum(times) / len(times), w.numel, nq


def cpu_baseline(w, target_s: float = 12.0):
    """The oracle as it stands, single thread, on a bounded sample of w."""
    probe = sample_workload(w, min(1.0, 2e6 / w.numel))
    t_probe, n_probe, _ = oracle_steps(probe, 1)
    per_elem = t_probe / n_probe
    steps = 2
    frac = min(1.0, target_s / steps / per_elem / w.numel)
    sw = sample_workload(w, frac)
    t_step, n, nq = oracle_steps(sw, steps)
    b = algorithmic_bytes(n, nq)
    import oracle
    t0 = time.perf_counter()
    oracle.plan(oracle.Desc.from_workload(w), w.m, w.g_coll)  # the whole workload's layout
    plan_s = time.perf_counter() - t0
    return dict(value=round(b["step"] / t_step / 1e9, 4), unit="GB/s", plan_seconds=round(plan_s, 6),
                params_per_s=round(n / t_step, 1), cores=1, kind="oracle",
                sample=f"{w.name} with every tensor cut to {frac:.4f} of its rows "
                       f"({n} real elements, {nq} quantisation blocks), {steps} full steps, "
                       f"single thread; host has {os.cpu_count()} cores")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if bus_id:
            cmd += ["-i", bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(mx) if mx else None, reasons=reasons, samples=len(rows))


# ---------------------------------------------------------------- GPU arm

def host_link_ms(host_in, dev_in, host_out, dev_out, s_in, s_out, steps: int) -> float:
    """The host link's bound on one end-to-end step: the same copy-in and
    copy-out, issued concurrently on the two copy streams with no compute,
    `steps` times; milliseconds per step."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(s_in)
    s_out.wait_event(a)
    for _ in range(steps):
        with torch.cuda.stream(s_in):
            dev_in.copy_(host_in, non_blocking=True)
        with torch.cuda.stream(s_out):
            host_out.copy_(dev_out, non_blocking=True)
    s_in.wait_stream(s_out)
    b.record(s_in)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def fill_grads(w, step: int, out: np.ndarray, starts) -> None:
    """The seeded gradients of `step` for every tensor of w into out (bf16
    bits), tensor t at starts[t]; tensors are generated in parallel (the
    generator is C and releases the interpreter lock)."""
    from concurrent.futures import ThreadPoolExecutor
    from synth import workloads as W
    jobs = [(t, starts[t], spec.numel) for t, spec in enumerate(w.tensors)]
    with ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
        list(ex.map(lambda j: W.grad(w, step, j[0], out=out[j[1]:j[1] + j[2]]), jobs))


def copy_ceiling(dev, nbytes: int = 4 << 30, reps: int = 10) -> dict:
    """The copy ceiling of this GPU, measured in this run: the best of `reps`
    device-to-device copies of nbytes (counted as read + write) by
    cudaMemcpyAsync (torch's contiguous copy) and by libvsf's 128-bit copy
    kernel, and the larger of the two."""
    import torch
    from fsdp_buffer_layout_gb300 import vsf as V
    a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    b = torch.empty_like(a)
    a.fill_(1)
    st = torch.cuda.current_stream(dev)

    def best(fn):
        for _ in range(2):
            fn()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        return 2 * nbytes / (min(ts) * 1e-3) / 1e9

    memcpy = best(lambda: b.copy_(a))
    kernel = best(lambda: V.vsf_device_copy(b.data_ptr(), a.data_ptr(), nbytes, st.cuda_stream))
    del a, b
    torch.cuda.empty_cache()
    return dict(gbs=round(max(memcpy, kernel), 1), memcpy_d2d_gbs=round(memcpy, 1),
                copy_kernel_gbs=round(kernel, 1), bytes_per_copy=2 * nbytes, reps=reps,
                how="best of the reps, CUDA events on the launching stream")


def gpu_arm(args, rank: int, world: int):
    import torch
    import torch.distributed as dist
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    from synth import workloads as W

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    ceiling = copy_ceiling(dev)  # before the workload's buffers take the memory
    w = W.get(args.workload)
    if args.fraction < 1.0:  # a reduced case of the same tensors (profiling captures)
        w = sample_workload(w, args.fraction)
    specs = [TensorSpec(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors]
    stream = torch.cuda.Stream(dev)
    ss = ShardStep(specs, w.m, w.g_coll, max_norm=w.max_norm, stream=stream,
                   bulk_warps=args.bulk_warps)
    n_real, nq = ss.info.real, ss.info.n_qblocks
    nbytes = algorithmic_bytes(n_real, nq, zero_copy=args.zero_copy)

    # Per-tensor gradients and parameters, 16-byte aligned views of one buffer.
    # The workload's input stream gives every step fresh gradients: two sets
    # (the seeded gradients of steps 1 and 2) are generated up front, and the
    # steps alternate between them, on the device and, for the end-to-end
    # leg, in pinned host memory.
    starts, cur = [], 0
    for n in ss.numels:
        starts.append(cur)
        cur += (n + 7) // 8 * 8
    host_g2 = [torch.zeros(cur, dtype=torch.int16).pin_memory() for _ in range(2)]
    for i, h in enumerate(host_g2):
        fill_grads(w, i + 1, h.numpy().view(np.uint16), starts)
    for t in range(len(ss.numels)):
        ss.load_master(t, torch.from_numpy(W.master_init(w, t)).to(dev))
    dev_g2 = [h.to(dev) for h in host_g2]
    dev_p2 = [torch.empty(cur, dtype=torch.int16, device=dev) for _ in range(2)]
    host_g = host_g2[0]
    dev_g, dev_p = dev_g2[0], dev_p2[0]
    host_p = torch.empty(cur, dtype=torch.int16).pin_memory()
    grads2 = [[b[s0:s0 + n] for s0, n in zip(starts, ss.numels)] for b in dev_g2]
    params2 = [[b[s0:s0 + n] for s0, n in zip(starts, ss.numels)] for b in dev_p2]
    params = params2[0]
    gviews = pviews = None
    if args.zero_copy:
        # gradients and parameters live in the packed buffers (address map):
        # two gradient buffers hold the two gradient sets, and the steps (and
        # the end-to-end leg's double buffering) alternate between them
        zc_grad = [ss.packed_grad, torch.zeros_like(ss.packed_grad)]
        zc_bf = [ss.packed_bf16, torch.zeros_like(ss.packed_bf16)]
        gviews = [ss.views(b.view(torch.int16)) for b in zc_grad]
        pviews = [ss.views(b.view(torch.int16)) for b in zc_bf]
        for i in range(2):
            for v, g in zip(gviews[i], grads2[i]):
                v.copy_(g)

    def gviews_of(buf):
        return gviews[buf]
    torch.cuda.synchronize(dev)

    # pack (or norm pass) + norm finalize + AdamW kernels (+ unpack)
    launches_per_step = (2 if args.zero_copy else 3) + ss.adam_launches()
    step = 0

    def one_step(ev=None):
        nonlocal step
        step += 1
        gset = step % 2  # fresh gradients: the two sets alternate
        if ev is not None:
            ev[0].record(stream)
        if args.zero_copy:
            ss.zero_copy_norm(zc_grad[gset])
        else:
            ss.pack(grads2[gset])
            ss.group_norm_scale()
        if ev is not None:
            ev[1].record(stream)
        if args.zero_copy:
            ss.zero_copy_adam(step, zc_grad[gset])
        else:
            ss.adam(step)
        if ev is not None:
            ev[2].record(stream)
        if not args.zero_copy:
            ss.unpack(params)
        if ev is not None:
            ev[3].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
    torch.cuda.synchronize(dev)

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id  # type: ignore[attr-defined]
    except Exception:
        bus = None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(bus)
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for i in range(args.steps):
            one_step(evs[i])
        t_end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    if world > 1:
        tt = torch.tensor([total_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms_step = total_ms / args.steps
    k_pack = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    k_adam = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    k_unpack = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)

    # End to end through the C ABI with host buffers: every step copies its
    # gradients in from pinned host memory (the two gradient sets alternate)
    # and its bf16 parameters and norm back out, inside the timed region.
    # Steps are pipelined on three streams with two device buffer sets: the
    # copy-in of step k+1 and the copy-out of step k-1 overlap the compute of
    # step k. Each step's norm goes to a slot of its own, written by the
    # library's norm kernel and read back on the copy-out stream, so that no
    # copy is queued on the compute stream (a device-to-host copy there would
    # wait for the previous step's copy-out in the copy engine and serialise
    # the pipeline).
    # at least 40 steps, so that the pipeline's fill (one copy-in and one
    # compute before the first copy-out) is a small part of the figure
    e2e_steps = max(40, min(args.steps, 100))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dev_norms = torch.zeros(e2e_steps, 2, dtype=torch.float64, device=dev)
    host_norms = torch.empty(e2e_steps, 2, dtype=torch.float64).pin_memory()
    # timing events double as the ordering events: ev_in[k] ends step k's
    # copy-in, ev_done[k] its compute, ev_out[k] its copy-out
    ev_in = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    ev_done = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    ev_out = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    # buffer reuse distance: two device buffer sets in both modes
    dist_k = 2

    def e2e_step(k, ev_in, ev_done, ev_out, dev_norms, host_norms):
        """Step k of the pipeline: copy-in on s_in, compute, copy-out on s_out."""
        nonlocal step
        buf = k % 2
        hsrc = host_g2[k % 2]
        with torch.cuda.stream(s_in):
            if k >= dist_k:
                s_in.wait_event(ev_done[k - dist_k])  # compute k-d has read this buffer
            if args.zero_copy:
                for v, s0, n in zip(gviews_of(buf), starts, ss.numels):
                    v.copy_(hsrc[s0:s0 + n], non_blocking=True)
            else:
                dev_g2[buf].copy_(hsrc, non_blocking=True)
            ev_in[k].record(s_in)
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[k])
            if k >= dist_k:
                stream.wait_event(ev_out[k - dist_k])  # copy-out k-d has read this buffer
            step += 1
            if args.zero_copy:
                ss.zero_copy_step(step, zc_grad[buf], zc_bf[buf], norm=dev_norms[k])
            else:
                ss.pack(grads2[buf])
                ss.group_norm_scale(norm=dev_norms[k])
                ss.adam(step)
                ss.unpack(params2[buf])
            ev_done[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[k])
            if args.zero_copy:
                for v, s0, n in zip(pviews[buf], starts, ss.numels):
                    host_p[s0:s0 + n].copy_(v, non_blocking=True)
            else:
                host_p.copy_(dev_p2[buf], non_blocking=True)
            host_norms[k].copy_(dev_norms[k], non_blocking=True)
            ev_out[k].record(s_out)

    # two untimed pipelined steps first (first use of the pinned buffers and
    # of the copy streams), then the timed run
    warm = [[torch.cuda.Event() for _ in range(2)] for _ in range(3)]
    for k in range(2):
        e2e_step(k, warm[0], warm[1], warm[2], dev_norms, host_norms)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e_start.record(s_in)
    s_out.wait_event(e_start)
    stream.wait_event(e_start)
    for k in range(e2e_steps):
        e2e_step(k, ev_in, ev_done, ev_out, dev_norms, host_norms)
    s_out.wait_stream(stream)
    e_end.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_ms = e_start.elapsed_time(e_end) / e2e_steps
    # steady state: the period of copy-out completions over the second half
    # of the run; fill: until the first copy-out finished
    half = e2e_steps // 2
    steady_ms = (ev_out[half].elapsed_time(ev_out[e2e_steps - 1]) / (e2e_steps - 1 - half)
                 if e2e_steps - 1 > half else e2e_ms)
    fill_ms = e_start.elapsed_time(ev_out[0])
    if not all(math.isfinite(x) and x > 0 for x in host_norms[:, 0].tolist()):
        raise RuntimeError("end-to-end leg: a step's norm did not reach the host")
    if world > 1:
        tt = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_ms = float(tt.item())
    link_ms = host_link_ms(host_g, dev_g2[0], host_p, dev_p2[0], s_in, s_out, e2e_steps)

    peak, peak_kind = measured_peak()
    adam_gbs = nbytes["adam"] / (k_adam * 1e-3) / 1e9
    value = nbytes["step"] * world / (ms_step * 1e-3) / 1e9
    traffic = None
    if not args.bulk_warps and args.fraction == 1.0 and w.name in TRAFFIC:
        # DRAM bytes per algorithmic byte of the capture, scaled to this launch
        traffic = round(TRAFFIC[w.name]["ratio"] * nbytes["adam"], 0)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s",
        "params_per_s": round(n_real * world / (ms_step * 1e-3), 1),
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "real_params": n_real, "m": w.m, "g_coll": w.g_coll,
                   "S": ss.info.S, "padding_ratio": round(ss.info.padding_ratio, 5),
                   "n_qblocks": nq, "grad_dtype": "bf16", "state": "int8 m / uint8 v, fp32 master",
                   "bytes_per_step": nbytes["step"],
                   "l2": f"inputs larger than L2 ({nbytes['step'] / 1e9:.2f} GB per step), no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU, m virtual ranks",
                   "mode": "zero-copy views (no copy-in/out)" if args.zero_copy
                   else "copy-in / copy-out",
                   "kernel_ms": {"pack+norm": round(k_pack, 5), "adam8": round(k_adam, 5),
                                 "unpack": round(k_unpack, 5)},
                   "frac_of_peak_step": round(value / world / peak, 4),
                   "frac_of_nominal_8tbs_step": round(value / world / NOMINAL_HBM_GBS, 4),
                   "frac_of_copy_ceiling_step": round(value / world / ceiling["gbs"], 4),
                   "copy_ceiling": ceiling,
                   "inputs": "fresh gradients each step: two seeded sets (steps 1 and 2) "
                             "alternate, on the device and in pinned host memory",
                   "plan_seconds": round(ss.info.plan_seconds, 6),
                   "bulk_warps": ss.info.bulk_warps, "bulk_cluster": ss.info.bulk_cluster},
        "roofline": {"bound": "hbm", "achieved": round(adam_gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(adam_gbs / peak, 4),
                     "frac_of_copy_ceiling": round(adam_gbs / ceiling["gbs"], 4),
                     "algorithmic_bytes": nbytes["adam"],
                     # captured with the planner's own kernel shape
                     "traffic": traffic,
                     "traffic_unit": "bytes per launch",
                     "traffic_source": TRAFFIC[w.name]["capture"] if traffic else None,
                     "kernel": "vsf_adam8_step",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s"},
        "e2e": {"value": round(nbytes["step"] * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": int(host_g.numel() * 2),
                "d2h_bytes_per_step": int(host_p.numel() * 2 + 16),
                "host_link_ms_per_step": round(link_ms, 5),
                "frac_of_host_link_bound": round(link_ms / e2e_ms, 4),
                "steps": e2e_steps, "fill_ms": round(fill_ms, 4),
                "steady_ms_per_step": round(steady_ms, 5),
                "steady_frac_of_host_link_bound": round(link_ms / steady_ms, 4),
                "pipeline": "3 streams (copy-in, compute, copy-out), 2 device buffer sets"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    return line


def muon_arm(args, rank: int, world: int):
    """One Muon step = copy-in of the per-tensor gradients, vsf_muon_step
    (momentum, per-matrix norm, bf16 normalisation, 5 Newton-Schulz
    iterations of 3 GEMMs, update of master and bf16 copy), copy-out."""
    import torch
    import torch.distributed as dist
    from fsdp_buffer_layout_gb300 import vsf as V
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    from synth import workloads as W

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = W.get(args.workload)
    if args.fraction < 1.0:  # a reduced case (profiling captures)
        w = sample_workload(w, args.fraction)
    specs = [TensorSpec(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors]
    stream = torch.cuda.Stream(dev)
    ss = ShardStep(specs, w.m, w.g_coll, stream=stream)
    n_real = ss.info.real
    flops = muon_flops(w)
    flops_exec = muon_flops(w, executed=True)
    starts, cur = [], 0
    for n in ss.numels:
        starts.append(cur)
        cur += (n + 7) // 8 * 8
    host_g = torch.empty(cur, dtype=torch.int16).pin_memory()
    hg = host_g.numpy().view(np.uint16)
    for t, n in enumerate(ss.numels):
        W.grad(w, 1, t, out=hg[starts[t]:starts[t] + n])
        ss.load_master(t, torch.from_numpy(W.master_init(w, t)).to(dev))
    dev_g = host_g.to(dev)
    dev_p = torch.empty(cur, dtype=torch.int16, device=dev)
    host_p = torch.empty(cur, dtype=torch.int16).pin_memory()
    grads = [dev_g[s0:s0 + n] for s0, n in zip(starts, ss.numels)]
    params = [dev_p[s0:s0 + n] for s0, n in zip(starts, ss.numels)]
    n_mats = sum(1 for t in w.tensors if len(t.shape) >= 2)
    roots, balance = ss.muon_roots()

    def one_step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        ss.pack(grads)
        if ev is not None:
            ev[1].record(stream)
        ss.muon_step()
        if ev is not None:
            ev[2].record(stream)
        ss.unpack(params)
        if ev is not None:
            ev[3].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
    torch.cuda.synchronize(dev)
    if ss.device_error():
        raise RuntimeError("device error word set")
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id  # type: ignore[attr-defined]
    except Exception:
        bus = None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(bus)
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for i in range(args.steps):
            one_step(evs[i])
        t_end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    if world > 1:
        tt = torch.tensor([total_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms_step = total_ms / args.steps
    k_muon = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    k_copy = statistics.mean(e[0].elapsed_time(e[1]) + e[2].elapsed_time(e[3]) for e in evs)

    # End to end with host buffers: every step copies its gradients in from
    # pinned host memory and its bf16 parameters back out, inside the timed
    # region; copy-in of step k+1 and copy-out of step k-1 overlap the compute
    # of step k (three streams, two device buffer sets).
    e2e_steps = max(3, min(args.steps, 20))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dev_g2 = [dev_g, torch.empty_like(dev_g)]
    dev_p2 = [dev_p, torch.empty_like(dev_p)]
    grads2 = [[b[s0:s0 + n] for s0, n in zip(starts, ss.numels)] for b in dev_g2]
    params2 = [[b[s0:s0 + n] for s0, n in zip(starts, ss.numels)] for b in dev_p2]
    ev_in = [torch.cuda.Event() for _ in range(e2e_steps)]
    ev_done = [torch.cuda.Event() for _ in range(e2e_steps)]
    ev_out = [torch.cuda.Event() for _ in range(e2e_steps)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e_start.record(s_in)
    s_out.wait_event(e_start)
    stream.wait_event(e_start)
    for k in range(e2e_steps):
        buf = k % 2
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev_done[k - 2])
            dev_g2[buf].copy_(host_g, non_blocking=True)
            ev_in[k].record(s_in)
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[k])
            if k >= 2:
                stream.wait_event(ev_out[k - 2])
            ss.pack(grads2[buf])
            ss.muon_step()
            ss.unpack(params2[buf])
            ev_done[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[k])
            host_p.copy_(dev_p2[buf], non_blocking=True)
            ev_out[k].record(s_out)
    s_out.wait_stream(stream)
    e_end.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_ms = e_start.elapsed_time(e_end) / e2e_steps
    if world > 1:
        tt = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_ms = float(tt.item())

    peak, peak_src = measured_bf16_peak(sustained=True)
    achieved = flops_exec / (k_muon * 1e-3) / 1e12
    value = flops * world / (ms_step * 1e-3) / 1e12
    return {
        "metric": MUON_METRIC, "value": round(value, 2), "unit": "TFLOP/s",
        "params_per_s": round(n_real * world / (ms_step * 1e-3), 1),
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "optimizer": "muon", "real_params": n_real,
                   "matrix_tensors": n_mats, "chunks": ss.muon_chunks(), "m": w.m,
                   "ns_steps": 5,
                   "ns_flops_per_step": flops, "ns_flops_executed_per_step": flops_exec,
                   "root_load_balance": round(balance, 4),
                   "gemm": "libvsf tcgen05 kernel: bf16 x bf16 -> bf16, fp32 accumulation "
                           "in TMEM, 256x256 tiles per CTA pair (cta_group::2), symmetric "
                           "products on the tiles at or above the diagonal",
                   "l2": "working set (master, momentum, Newton-Schulz buffers) larger than "
                         "L2, no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU, m virtual ranks",
                   "kernel_ms": {"muon_step": round(k_muon, 5),
                                 "pack+unpack": round(k_copy, 5)}},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "vsf_muon_step (Newton-Schulz GEMM chain with its element-wise "
                               "kernels)",
                     "flops": "executed by the tensor cores (symmetric products on half "
                              "their tiles); value counts the definition's full products",
                     "peak_source": peak_src},
        "e2e": {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": int(host_g.numel() * 2),
                "d2h_bytes_per_step": int(host_p.numel() * 2)},
        "gpu_launches": (2 + V.vsf_muon_kernel_launches(ss.plan, 5)) * args.steps,
        "gpu_launches_note": "own kernels: copy-in, copy-out, and per batched chunk of "
                             "same-shape matrices momentum, normalise, update and 3 "
                             "Newton-Schulz products per iteration",
        "clocks": clocks,
    }


def group_ops_arm(args, rank: int, world: int):
    """One step = the four fused group ops over every real element of the
    DBuffer: zero and scale of the packed bf16 gradient, bf16 += bf16 (a
    second micro-batch's gradient) and fp32 += bf16 (gradient accumulation
    into an fp32 buffer), each one launch over all tensors."""
    import torch
    import torch.distributed as dist
    from fsdp_buffer_layout_gb300 import vsf as V
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    from synth import workloads as W

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = W.get(args.workload)
    stream = torch.cuda.Stream(dev)
    ss = ShardStep([TensorSpec(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors],
                   w.m, w.g_coll, stream=stream)
    n_real, total = ss.info.real, ss.info.total
    g = ss.packed_grad
    g2 = torch.zeros_like(g)
    acc = torch.zeros(total, dtype=torch.float32, device=dev)
    for t in range(len(w.tensors)):  # real elements: a seeded gradient in both bf16 buffers
        o, n = ss.offsets[t], ss.numels[t]
        x = torch.from_numpy(W.grad(w, 1, t).view(np.int16)).to(dev)
        g.view(torch.int16)[o:o + n].copy_(x)
        g2.view(torch.int16)[o:o + n].copy_(x)
    st = stream.cuda_stream
    ops = [lambda: V.vsf_group_zero(ss.plan, g.data_ptr(), V.VSF_BF16, st),
           lambda: V.vsf_group_scale(ss.plan, g2.data_ptr(), V.VSF_BF16, 0.5, st),
           lambda: V.vsf_group_add(ss.plan, g.data_ptr(), V.VSF_BF16, g2.data_ptr(), V.VSF_BF16,
                                   st),
           lambda: V.vsf_group_add(ss.plan, acc.data_ptr(), V.VSF_FP32, g2.data_ptr(), V.VSF_BF16,
                                   st)]
    nbytes = [n_real * b for _, b in GROUP_OPS]

    def one_step(ev=None):
        for i, op in enumerate(ops):
            if ev is not None:
                ev[i].record(stream)
            op()
        if ev is not None:
            ev[len(ops)].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id  # type: ignore[attr-defined]
    except Exception:
        bus = None
    sampler = ClockSampler(bus)
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)]
           for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for i in range(args.steps):
            one_step(evs[i])
        t_end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    if world > 1:
        tt = torch.tensor([total_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms_step = total_ms / args.steps
    op_ms = [statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) for i in range(len(ops))]

    # end to end: each step copies a micro-batch gradient in from pinned host
    # memory into a packed buffer, accumulates it into the fp32 buffer and
    # reads one accumulated value back; two gradient buffers, so the copy-in
    # of step k+1 overlaps the accumulation of step k
    host_g = g2.view(torch.int16).cpu().pin_memory()
    host_out = torch.empty(1, dtype=torch.float32).pin_memory()
    gbuf = [g2, torch.zeros_like(g2)]
    s_in = torch.cuda.Stream(dev)
    e2e_steps = max(3, min(args.steps, 50))
    ev_in = [torch.cuda.Event() for _ in range(e2e_steps)]
    ev_done = [torch.cuda.Event() for _ in range(e2e_steps)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e_start.record(s_in)
    stream.wait_event(e_start)
    for k in range(e2e_steps):
        b = gbuf[k % 2]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev_done[k - 2])
            b.view(torch.int16).copy_(host_g, non_blocking=True)
            ev_in[k].record(s_in)
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[k])
            V.vsf_group_add(ss.plan, acc.data_ptr(), V.VSF_FP32, b.data_ptr(), V.VSF_BF16, st)
            host_out.copy_(acc[:1], non_blocking=True)
            ev_done[k].record(stream)
    s_in.wait_stream(stream)
    e_end.record(s_in)
    torch.cuda.synchronize(dev)
    e2e_ms = e_start.elapsed_time(e_end) / e2e_steps

    peak, peak_kind = measured_peak()
    gbs = [b / (ms * 1e-3) / 1e9 for b, ms in zip(nbytes, op_ms)]
    value = sum(nbytes) * world / (ms_step * 1e-3) / 1e9
    return {
        "metric": GROUP_METRIC, "value": round(value, 2), "unit": "GB/s",
        "params_per_s": round(n_real * world / (ms_step * 1e-3), 1),
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "ops": {name: {"ms": round(ms, 5), "GB/s": round(x, 1),
                                                      "frac": round(x / peak, 4),
                                                      "bytes_per_elem": b}
                                               for (name, b), ms, x in zip(GROUP_OPS, op_ms, gbs)},
                   "real_params": n_real, "m": w.m, "g_coll": w.g_coll,
                   "l2": "buffers larger than L2, no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU, m virtual ranks"},
        "roofline": {"bound": "hbm", "achieved": round(gbs[3], 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs[3] / peak, 4), "traffic": None,
                     "kernel": "vsf_group_add (fp32 += bf16)",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s"},
        "e2e": {"value": round(nbytes[3] * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "workload": "H2D of one bf16 gradient, "
                "fp32 accumulate, D2H of one value; double-buffered",
                "h2d_bytes_per_step": int(host_g.numel() * 2), "d2h_bytes_per_step": 4},
        "gpu_launches": len(ops) * args.steps,
        "clocks": clocks,
    }


def group_ops_cpu_baseline(w, target_s: float = 6.0):
    """The oracle's group add (fp32 += bf16, single thread) on the workload's
    layout with every tensor cut to a fraction of its rows: a probe sizes the
    sample to about target_s seconds."""
    import oracle
    from synth import workloads as W

    def timed(frac):
        sw = sample_workload(w, frac)
        d = oracle.Desc.from_workload(sw)
        S, off = oracle.plan(d, sw.m, sw.g_coll)
        numels = [t.numel for t in sw.tensors]
        src = oracle.pack([W.grad(sw, 1, t) for t in range(d.n)], off, sw.m * S)
        dst = np.zeros(sw.m * S, np.float32)
        t0 = time.perf_counter()
        oracle.group_op(2, numels, off, dst, src)
        return time.perf_counter() - t0, sum(numels)

    sec, n = timed(min(1.0, 1e6 / w.numel))
    frac = min(1.0, target_s / (sec / n) / w.numel)
    sec, n = timed(frac)
    return dict(value=round(n * 10 / sec / 1e9, 4), unit="GB/s", cores=1, kind="oracle",
                sample=f"add fp32 += bf16 over {w.name} cut to {frac:.4f} of its rows ({n} real "
                       f"elements, {sec:.1f} s), single thread; host has {os.cpu_count()} cores")


def muon_cpu_baseline(w, threads: int | None = None):
    """The Muon oracle (numpy, fp64 products with bf16 rounding points) on
    one whole matrix tensor of w, run in a child process with a fixed BLAS
    thread count so that `cores` is the count it used."""
    threads = threads or os.cpu_count() or 1
    mats = [t for t in w.tensors if len(t.shape) >= 2]
    t = min(mats, key=lambda x: math.prod(x.shape))
    code = (
        "import json, math, time, numpy as np\n"
        "from oracle import muon\n"
        f"R, C = {t.shape[-2]}, {t.shape[-1]}\n"
        "rng = np.random.default_rng(0)\n"
        "g = muon.bf16_from_f32((rng.standard_normal((R, C)) * 1e-3).astype(np.float32))\n"
        "M = np.zeros((R, C), np.float32); p = np.zeros((R, C), np.float32)\n"
        "hp = dict(lr=0.02, momentum=0.95, weight_decay=0.01, eps=1e-7, ns_steps=5,"
        " ns_a=3.4445, ns_b=-4.7750, ns_c=2.0315)\n"
        "t0 = time.perf_counter(); muon.muon_matrix(g, M, p, hp)\n"
        "print(json.dumps(time.perf_counter() - t0))\n")
    env = dict(os.environ, OMP_NUM_THREADS=str(threads), OPENBLAS_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads), PYTHONPATH=ROOT)
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         check=True, cwd=ROOT)
    sec = float(out.stdout.strip().splitlines()[-1])
    R, C = t.shape[-2], t.shape[-1]
    n, k = min(R, C), max(R, C)
    fl = 5 * (4.0 * n * n * k + 2.0 * n ** 3)
    return dict(value=round(fl / sec / 1e12, 6), unit="TFLOP/s", cores=threads, kind="oracle",
                sample=f"one Muon step of one {R}x{C} matrix ({t.name}) of {w.name}, "
                       f"{sec:.2f} s, numpy BLAS with {threads} threads")


# DRAM traffic of vsf_adam8_step's bulk-copy kernel per algorithmic byte
# ((dram__bytes_read.sum + dram__bytes_write.sum) / (16 B per element + 16 B
# per quantisation block)), from ncu captures of reduced cases of each
# workload (every tensor cut to a fraction of its rows: the same block sizes,
# fewer blocks) summarised in profiles/adam8_tma_*.md. The line's `traffic`
# is this ratio times the full launch's algorithmic bytes. A workload without
# a capture of the current kernel has no entry (traffic null).
TRAFFIC: dict = {
    "llama_1p3b": dict(ratio=1.0013, capture="llama_1p3b cut to 0.1 of its rows: 2.0782 GB "
                       "DRAM for 2.0754 GB algorithmic, one launch (profiles/adam8_tma_traffic.md)"),
    "llama_layer": dict(ratio=0.9893, capture="llama_layer cut to 0.5 of its rows: 1.6018 GB "
                        "for 1.6191 GB, one launch (profiles/adam8_tma_traffic.md)"),
    "moe_layer": dict(ratio=0.9973, capture="moe_layer cut to 0.15 of its rows: 1.9061 GB for "
                      "1.9113 GB, one launch (profiles/adam8_tma_traffic.md)"),
    "dsv3_block": dict(ratio=0.9730, capture="dsv3_block cut to 0.5 of its rows: 2.0572 GB for "
                       "2.1142 GB, one launch (profiles/adam8_tma_traffic.md)"),
}


def reference_arm(args):
    from synth import workloads as W
    w = W.get(args.workload)
    budget = float(os.environ.get("VSF_REFERENCE_BUDGET_S", "90"))
    probe = sample_workload(w, min(1.0, 1e6 / w.numel))
    t_probe, n_probe, _ = oracle_steps(probe, 1)
    per_elem = t_probe / n_probe
    frac = min(1.0, max(1e-6, budget / (args.steps + args.warmup) / per_elem / w.numel))
    sw = sample_workload(w, frac)
    t_step, n, nq = oracle_steps(sw, args.steps + args.warmup)
    b = algorithmic_bytes(n, nq)
    value = b["step"] / t_step / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "params_per_s": round(n / t_step, 1), "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "real_params": w.numel, "m": w.m, "g_coll": w.g_coll,
                   "sample_real_params": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{w.name} cut to {frac:.5f} of its rows per step ({n} real "
                                   f"elements), single thread; host has {os.cpu_count()} cores"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def group_ops_reference_arm(args):
    """The oracle's group add (fp32 += bf16) on a bounded sample per step."""
    from synth import workloads as W
    w = W.get(args.workload)
    base = group_ops_cpu_baseline(w)
    return {
        "impl": "reference", "metric": GROUP_METRIC, "value": base["value"], "unit": "GB/s",
        "n_gpus": 1, "steps": 1, "warmup": 0, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "ops": "add fp32 += bf16"},
        "cpu_baseline": base,
        "e2e": {"value": base["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def muon_reference_arm(args):
    """The Muon oracle on one whole matrix per step (see muon_cpu_baseline)."""
    from synth import workloads as W
    w = W.get(args.workload)
    base = muon_cpu_baseline(w)
    return {
        "impl": "reference", "metric": MUON_METRIC, "value": base["value"], "unit": "TFLOP/s",
        "n_gpus": 1, "steps": 1, "warmup": 0, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "optimizer": "muon"},
        "cpu_baseline": base,
        "e2e": {"value": base["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="vsf", choices=["vsf", "reference"])
    ap.add_argument("--workload", default="llama_1p3b")
    ap.add_argument("--fraction", type=float, default=1.0,
                    help="cut every tensor to this fraction of its rows (reduced cases for "
                         "profiling captures; not a bench line)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--optimizer", default="adam8", choices=["adam8", "muon"],
                    help="adam8: the 8-bit AdamW shard step; muon: distributed Muon")
    ap.add_argument("--group-ops", action="store_true",
                    help="time the fused DBuffer group ops (zero, scale, add) instead")
    ap.add_argument("--zero-copy", action="store_true",
                    help="gradients/params as views of the packed buffers (no pack/unpack)")
    ap.add_argument("--bulk-warps", type=int, default=0, choices=[0, 4, 16],
                    help="force the bulk-copy AdamW kernel shape (0: the planner's choice)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            arm = (group_ops_reference_arm if args.group_ops else
                   muon_reference_arm if args.optimizer == "muon" else reference_arm)
            print(json.dumps(arm(args)), flush=True)
        return
    if args.optimizer == "muon" and args.zero_copy:
        ap.error("--zero-copy applies to the AdamW step")
    if world > 1:
        import torch
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)  # one GPU per rank, bound before NCCL starts
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    arm = group_ops_arm if args.group_ops else muon_arm if args.optimizer == "muon" else gpu_arm
    line = arm(args, rank, world)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline and args.group_ops:
            from synth import workloads as W
            line["cpu_baseline"] = group_ops_cpu_baseline(W.get(args.workload))
        elif world == 1 and not args.no_cpu_baseline:
            from synth import workloads as W
            line["cpu_baseline"] = (muon_cpu_baseline if args.optimizer == "muon"
                                    else cpu_baseline)(W.get(args.workload))
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
