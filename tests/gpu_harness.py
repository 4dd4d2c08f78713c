"""Shared driver for the GPU parity tests: runs the same seeded steps through
libvsf (via ShardStep) and through the oracle, and compares the results.

Tolerances (the shard-step spec): layout, copy-in and copy-out bit-exact;
master weights within 1e-6 max relative error; quantised moment codes may
differ by at most 1 at no more than 1e-4 of positions; scales and bf16
copies compared after the master check. The kernels are written to be
bit-exact (same fp32 op order, one rounding per operation), so the tests also
report how many elements match exactly.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

import oracle
import synth
from synth import workloads as W

MASTER_RTOL = 1e-6
CODE_FRAC = 1e-4


@dataclasses.dataclass
class Case:
    specs: list          # (shape, gran, block_rows, tile_cols)
    m: int
    g_coll: int
    steps: int
    grads: callable      # (step, t) -> np.uint16 (bf16 bits) or np.float32 array
    masters: callable    # t -> np.float32 array
    max_norm: float = math.inf
    quantized: bool = True
    grad_dtype: int = 0  # 0 bf16, 1 fp32
    world: int | None = None
    standalone_norm: bool = False
    bulk_warps: int = 0  # forced bulk-copy kernel shape (0: the planner's choice)

    @property
    def numels(self):
        return [int(np.prod(s[0])) for s in self.specs]


def case_from_workload(w: W.Workload, steps=None, **kw) -> Case:
    fp32 = kw.get("grad_dtype", 0) == 1
    return Case(specs=[(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors],
                m=w.m, g_coll=w.g_coll, steps=w.steps if steps is None else steps,
                grads=(lambda s, t: W.grad_f32(w, s, t)) if fp32 else (lambda s, t: W.grad(w, s, t)),
                masters=lambda t: W.master_init(w, t), **{"max_norm": w.max_norm, **kw})


def hp_dict():
    return dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _desc(case: Case) -> oracle.Desc:
    rows = [int(np.prod(s[0][:-1])) if len(s[0]) > 1 else 1 for s in case.specs]
    return oracle.Desc(rows, [s[0][-1] for s in case.specs], [s[1] for s in case.specs],
                       [s[2] for s in case.specs], [s[3] for s in case.specs])


def run_oracle(case: Case):
    d = _desc(case)
    S, off = oracle.plan(d, case.m, case.g_coll)
    qb = oracle.qblocks(d, case.g_coll, off)
    total = case.m * S
    nq = len(qb["base"])
    world = case.m if case.world is None else case.world
    master = oracle.pack([case.masters(t) for t in range(d.n)], off, total)
    if case.quantized:
        ms, vs = np.zeros(total, np.int8), np.zeros(total, np.uint8)
    else:
        ms, vs = np.zeros(total, np.float32), np.zeros(total, np.float32)
    msc, vsc = np.zeros(nq, np.float32), np.zeros(nq, np.float32)
    bf = np.zeros(total, np.uint16)
    factors, norms = [], []
    for s in range(1, case.steps + 1):
        grads = [case.grads(s, t) for t in range(d.n)]
        packed = oracle.pack(grads, off, total)
        f, norm = oracle.factor(oracle.sumsq(grads), world, case.max_norm)
        factors.append(f)
        norms.append(norm)
        oracle.adam_all(qb, packed, f, case.quantized, ms, vs, msc, vsc, master, bf, s, hp_dict())
    params = oracle.unpack(bf, case.numels, off)
    return dict(S=S, offsets=off, packed_grad=packed, master=master, m_state=ms, v_state=vs,
                m_scale=msc, v_scale=vsc, packed_bf16=bf, params=params, factors=factors,
                norms=norms)


def run_gpu(case: Case):
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    specs = [TensorSpec(tuple(s[0]), s[1], s[2], s[3]) for s in case.specs]
    ss = ShardStep(specs, case.m, case.g_coll, grad_dtype=case.grad_dtype,
                   quantized=case.quantized, max_norm=case.max_norm, world=case.world,
                   bulk_warps=case.bulk_warps)
    try:
        dev = ss.device
        for t in range(len(specs)):
            ss.load_master(t, torch.from_numpy(case.masters(t)).to(dev))
        gdt = torch.int16 if case.grad_dtype == 0 else torch.float32
        grads = [torch.empty(n, dtype=gdt, device=dev) for n in case.numels]
        params = [torch.empty(n, dtype=torch.int16, device=dev) for n in case.numels]
        factors, norms = [], []
        for s in range(1, case.steps + 1):
            for t, g in enumerate(grads):
                h = case.grads(s, t)
                g.copy_(torch.from_numpy(h.view(np.int16) if case.grad_dtype == 0 else h))
            ss.pack(grads)
            ss.group_norm_scale(standalone=case.standalone_norm)
            ss.adam(s)
            ss.unpack(params)
            torch.cuda.synchronize()
            assert ss.device_error() == 0, "a bounded device wait ran out"
            factors.append(float(ss.factor[0].item()))
            norms.append(float(ss.norm[0].item()))
        def host(x):
            if x.dtype == torch.bfloat16:
                x = x.view(torch.int16)
            return x.cpu().numpy()

        out = dict(S=ss.info.S, offsets=np.array(ss.offsets), packed_grad=host(ss.packed_grad),
                   master=host(ss.master), m_state=host(ss.m_state), v_state=host(ss.v_state),
                   m_scale=host(ss.m_scale)[:ss.info.n_qblocks],
                   v_scale=host(ss.v_scale)[:ss.info.n_qblocks],
                   packed_bf16=host(ss.packed_bf16).view(np.uint16),
                   params=[host(p).view(np.uint16) for p in params], factors=factors,
                   norms=norms, bulk_cluster=int(ss.info.bulk_cluster))
        if case.grad_dtype == 0:
            out["packed_grad"] = out["packed_grad"].view(np.uint16)
        return out
    finally:
        ss.close()


def run_gpu_windows(case: Case, windows):
    """The same steps with the DBuffer split into rank windows [r0, r1), one
    ShardStep per window (as separate processes would hold them), run one
    after another on one GPU. The norm's one exchange is the sum of the
    windows' fp64 sums of squares (on the device). Results are stitched into
    whole-buffer arrays: buffers by window, scales through the block table."""
    from fsdp_buffer_layout_gb300 import vsf as V
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    specs = [TensorSpec(tuple(s[0]), s[1], s[2], s[3]) for s in case.specs]
    sss = []
    try:
        for r0, r1 in windows:
            sss.append(ShardStep(specs, case.m, case.g_coll, grad_dtype=case.grad_dtype,
                                 quantized=case.quantized, max_norm=case.max_norm,
                                 world=case.world, ranks=(r0, r1)))
        dev = sss[0].device
        S, offs = sss[0].info.S, sss[0].offsets
        for ss, (r0, r1) in zip(sss, windows):
            lo, hi = r0 * S, r1 * S
            for t in range(len(specs)):
                m, o = case.masters(t), offs[t]
                a, b = max(lo, o), min(hi, o + m.size)
                if a < b:
                    ss.master[a - lo:b - lo].copy_(torch.from_numpy(m[a - o:b - o]).to(dev))
        gdt = torch.int16 if case.grad_dtype == 0 else torch.float32
        grads = [torch.empty(n, dtype=gdt, device=dev) for n in case.numels]
        params = [torch.empty(n, dtype=torch.int16, device=dev) for n in case.numels]
        factors, norms = [], []
        for s in range(1, case.steps + 1):
            for t, g in enumerate(grads):
                h = case.grads(s, t)
                g.copy_(torch.from_numpy(h.view(np.int16) if case.grad_dtype == 0 else h))
            for ss in sss:
                ss.pack(grads)
                ss.group_sumsq(standalone=case.standalone_norm)
            total = sss[0].sumsq[:1].clone()
            for ss in sss[1:]:
                total += ss.sumsq[:1]
            for ss in sss:
                ss.scale_from_sumsq(total)
                ss.adam(s)
                ss.unpack(params)
            torch.cuda.synchronize()
            for ss in sss:
                assert ss.device_error() == 0, "a bounded device wait ran out"
                assert float(ss.factor[0].item()) == float(sss[0].factor[0].item())
            factors.append(float(sss[0].factor[0].item()))
            norms.append(float(sss[0].norm[0].item()))

        def host(x):
            if x.dtype == torch.bfloat16:
                x = x.view(torch.int16)
            return x.cpu().numpy()

        total_elems = case.m * S
        out = dict(S=S, offsets=np.array(offs), factors=factors, norms=norms,
                   params=[host(p).view(np.uint16) for p in params])
        for k in ("packed_grad", "master", "m_state", "v_state", "packed_bf16"):
            parts = [host(getattr(ss, k)) for ss in sss]
            whole = np.zeros(total_elems, dtype=parts[0].dtype)
            for part, (r0, r1) in zip(parts, windows):
                whole[r0 * S:r1 * S] = part
            out[k] = whole
        out["packed_bf16"] = out["packed_bf16"].view(np.uint16)
        if case.grad_dtype == 0:
            out["packed_grad"] = out["packed_grad"].view(np.uint16)
        # scales: window block (tensor, base + r0*S) -> the whole plan's block index
        whole_plan = V.vsf_plan_create([V.make_desc(*s) for s in case.specs], case.m, case.g_coll)
        try:
            nq = V.vsf_plan_get_info(whole_plan).n_qblocks
            qb = V.vsf_plan_qblocks(whole_plan, nq)
        finally:
            V.vsf_plan_destroy(whole_plan)
        index = {(qb["tensor"][q], qb["base"][q]): q for q in range(nq)}
        for k in ("m_scale", "v_scale"):
            whole = np.zeros(nq, np.float32)
            for ss, (r0, r1) in zip(sss, windows):
                lq = V.vsf_plan_qblocks(ss.plan, ss.info.n_qblocks)
                vals = host(getattr(ss, k))
                for q in range(ss.info.n_qblocks):
                    whole[index[(lq["tensor"][q], lq["base"][q] + r0 * S)]] = vals[q]
            out[k] = whole
        return out
    finally:
        for ss in sss:
            ss.close()


def check_master(got, want, rtol=MASTER_RTOL):
    got = got.astype(np.float64)
    want = want.astype(np.float64)
    denom = np.maximum(np.abs(want), 1e-30)
    rel = np.abs(got - want) / denom
    bad = (rel > rtol) & ~(np.isnan(got) & np.isnan(want))
    assert not bad.any(), f"master: {int(bad.sum())} elements beyond {rtol} (max {rel.max():.3g})"
    return int((got == want).sum())


def check_codes(got, want, name):
    diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
    assert diff.max(initial=0) <= 1, f"{name}: code difference {diff.max()} > 1"
    frac = float((diff > 0).mean()) if diff.size else 0.0
    assert frac <= CODE_FRAC, f"{name}: {frac:.3g} of codes differ (> {CODE_FRAC})"
    return int((diff == 0).sum())


def bf16_nan(h: np.ndarray) -> np.ndarray:
    """Which bf16 bit patterns are NaNs (exponent all ones, fraction nonzero)."""
    h = h.view(np.uint16)
    return ((h & 0x7F80) == 0x7F80) & ((h & 0x007F) != 0)


def bit_equal(a: np.ndarray, b: np.ndarray, bf16: bool = False) -> bool:
    """Byte equality, except that two NaNs match whatever their bits: fp32
    arrays, and uint16 arrays of bf16 values when bf16=True. IEEE 754 fixes
    only that a rounded NaN is a NaN; the CPU and the GPU pick different
    bit patterns."""
    if a.dtype == np.float32:
        same = a.view(np.uint32) == b.view(np.uint32)
        same |= np.isnan(a) & np.isnan(b)
        return bool(same.all())
    if bf16:
        same = a.view(np.uint16) == b.view(np.uint16)
        same |= bf16_nan(a) & bf16_nan(b)
        return bool(same.all())
    return np.array_equal(a.view(np.uint8), b.view(np.uint8))


def compare(case: Case, g: dict, o: dict, exact: bool = True):
    """Spec tolerances; with exact=True also every byte equal."""
    assert g["S"] == o["S"]
    assert np.array_equal(g["offsets"], o["offsets"])
    assert np.array_equal(g["packed_grad"].view(np.uint8), o["packed_grad"].view(np.uint8)), \
        "copy-in differs"
    assert bit_equal(np.array(g["factors"], np.float32), np.array(o["factors"], np.float32)), \
        (g["factors"], o["factors"])
    for a, b in zip(g["norms"], o["norms"]):
        if math.isnan(b) or math.isinf(b):
            assert (math.isnan(a) and math.isnan(b)) or a == b, (a, b)
        else:
            n = sum(case.numels)
            assert abs(a - b) <= max(1e-12, n * 2.0 ** -53) * max(abs(b), 1e-300), (a, b)
    check_master(g["master"], o["master"])
    if case.quantized:
        check_codes(g["m_state"], o["m_state"], "m codes")
        check_codes(g["v_state"], o["v_state"], "v codes")
    else:
        check_master(g["m_state"], o["m_state"])
        check_master(g["v_state"], o["v_state"])
    if exact:
        for k in ("master", "m_state", "v_state", "m_scale", "v_scale", "packed_bf16"):
            assert bit_equal(g[k], o[k], bf16=k == "packed_bf16"), f"{k} not bit-exact"
    # copy-out is a byte copy of the library's own bf16 buffer ...
    for a, b in zip(g["params"], oracle.unpack(g["packed_bf16"], case.numels, g["offsets"])):
        assert np.array_equal(a, b), "copy-out differs from the packed bf16 buffer"
    # ... whose values match the oracle's (NaNs by class)
    for a, b in zip(g["params"], o["params"]):
        assert bit_equal(a, b, bf16=True), "copy-out differs"
