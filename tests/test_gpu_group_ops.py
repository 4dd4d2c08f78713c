"""Fused group ops (zero / scale / add over every tensor of the buffer) and
the zero-copy step (gradients and parameters as views of the packed buffers)
through the C ABI, against the oracle, bit for bit; padding never touched.
"veScale-FSDP: Flexible and High-Performance FSDP at Scale (MLSys 2026)"
summary page, 核心方法 > Distributed Buffer."""
import numpy as np
import pytest
import torch

import oracle
from synth import workloads as W

from gpu_harness import case_from_workload, compare, run_oracle

pytestmark = pytest.mark.gpu

SPECS = [((300, 1000), W.GRAN_ROWS, 32, 0), ((45, 77), W.GRAN_TILE, 8, 16),
         ((1000,), W.GRAN_ELEM, 0, 0), ((1,), W.GRAN_ELEM, 0, 0)]


def _step(specs, m, g):
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    return ShardStep([TensorSpec(*s) for s in specs], m, g)


@pytest.mark.parametrize("g_coll", [128, 3])
@pytest.mark.parametrize("dst_t,src_t", [("bf16", "bf16"), ("f32", "bf16"), ("f32", "f32"),
                                         ("bf16", "f32")])
def test_group_ops_match_oracle(g_coll, dst_t, src_t):
    from fsdp_buffer_layout_gb300 import vsf as V
    ss = _step(SPECS, 5, g_coll)
    try:
        total = ss.info.total
        rng = np.random.default_rng(3)

        def fresh(kind):
            x = (rng.standard_normal(total) * 1e-3).astype(np.float32)
            if kind == "bf16":
                return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            return x

        code = {"bf16": V.VSF_BF16, "f32": V.VSF_FP32}
        d0, s0 = fresh(dst_t), fresh(src_t)
        tdev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()  # noqa: E731
        d, sv = tdev(d0.copy()), tdev(s0)
        st = ss.stream.cuda_stream
        V.vsf_group_add(ss.plan, d.data_ptr(), code[dst_t], sv.data_ptr(), code[src_t], st)
        V.vsf_group_scale(ss.plan, d.data_ptr(), code[dst_t], 0.375, st)
        torch.cuda.synchronize()
        want = d0.copy()
        oracle.group_op(2, ss.numels, ss.offsets, want, s0)
        oracle.group_op(1, ss.numels, ss.offsets, want, alpha=0.375)
        got = d.cpu().numpy()
        got = got.view(np.uint16) if dst_t == "bf16" else got
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8))  # padding kept too
        V.vsf_group_zero(ss.plan, d.data_ptr(), code[dst_t], st)
        torch.cuda.synchronize()
        oracle.group_op(0, ss.numels, ss.offsets, want)
        got = d.cpu().numpy()
        got = got.view(np.uint16) if dst_t == "bf16" else got
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8))
    finally:
        ss.close()


def test_zero_copy_step_matches_oracle():
    """Gradients written straight into their views of the packed buffer;
    norm on the packed gradient and AdamW; parameters read from the views."""
    w = W.tiny()
    case = case_from_workload(w)
    o = run_oracle(case)
    ss = _step([(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors], w.m, w.g_coll)
    try:
        for t in range(len(w.tensors)):
            ss.load_master(t, torch.from_numpy(W.master_init(w, t)).cuda())
        gviews = ss.views(ss.packed_grad.view(torch.int16))
        pviews = ss.views(ss.packed_bf16.view(torch.int16))
        for s in range(1, case.steps + 1):
            for t, v in enumerate(gviews):
                v.copy_(torch.from_numpy(W.grad(w, s, t).view(np.int16)))
            ss.zero_copy_step(s)
        torch.cuda.synchronize()
        assert ss.device_error() == 0
        assert np.array_equal(ss.master.cpu().numpy().view(np.uint32), o["master"].view(np.uint32))
        assert np.array_equal(ss.m_state.cpu().numpy(), o["m_state"])
        assert np.array_equal(ss.v_state.cpu().numpy(), o["v_state"])
        for v, want in zip(pviews, o["params"]):
            assert np.array_equal(v.cpu().numpy().view(np.uint16), want)
    finally:
        ss.close()
