"""The seeded input generator: counter-based (any slice redraws identically),
the documented distributions, and the workload recipe."""
import numpy as np

import synth
from synth import workloads as W


def test_slices_redraw_identically():
    w = W.llama_layer()
    full = W.grad(w, 3, 6, 0, 100000)
    part = W.grad(w, 3, 6, 31337, 1000)
    assert np.array_equal(full[31337:32337], part)
    m_full = W.master_init(w, 2, 0, 5000)
    assert np.array_equal(m_full[4000:], W.master_init(w, 2, 4000, 1000))


def test_streams_differ_by_step_tensor_kind():
    w = W.llama_layer()
    a = W.grad(w, 1, 0, 0, 64)
    assert not np.array_equal(a, W.grad(w, 2, 0, 0, 64))
    assert not np.array_equal(a, W.grad(w, 1, 1, 0, 64))


def test_normal_moments():
    w = W.llama_layer()
    x = synth.bf16_to_f32(W.grad(w, 1, 0, 0, 1 << 20)).astype(np.float64)
    assert abs(x.mean()) < 5e-6 and abs(x.std() - 1e-3) < 1e-5
    p = W.master_init(w, 0, 0, 1 << 20).astype(np.float64)
    assert abs(p.std() - 0.02) < 2e-4


def test_student_t3_is_heavy_tailed():
    w = W.dsv3_block()
    x = synth.bf16_to_f32(W.grad(w, 1, 0, 0, 1 << 20)).astype(np.float64) / 1e-3
    # t(3): variance 3, P(|T| > 5.84) = 0.01
    assert 2.5 < x.var() < 3.6
    assert 0.008 < np.mean(np.abs(x) > 5.841) < 0.012


def test_zero_experts():
    w = W.moe_layer()
    ids = w.zero_expert_ids()
    assert len(ids) == 2 and len(set(ids)) == 2
    per = w.tensors[1].numel // 32
    e = ids[0]
    g = W.grad(w, 1, 1, e * per - 10, per + 20)
    assert g[:10].any() and not g[10:10 + per].any() and g[10 + per:].any()
    assert W.grad(w, 1, 2, 0, 100).any()  # the router is never zeroed


def test_workload_sizes():
    assert W.tiny().numel == 214016
    assert W.llama_layer().numel == 202383360
    assert W.moe_layer().numel == 796354560
    assert W.dsv3_block().numel == 264255488
    w = W.llama_1p3b()
    assert w.numel == 1345423360 and len(w.tensors) == 219
