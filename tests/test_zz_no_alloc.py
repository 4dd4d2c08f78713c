"""The allocation-free group norm (vsf_group_norm_scale_static) against the
planned path's vsf_group_norm_scale, through the C ABI.

Some callers cannot allocate device memory at the moment they need the
gradient norm (for instance a hook inside a framework's caching allocator, or
a runtime that owns the whole memory budget). The static entry point keeps
its scratch in a fixed array inside the library. This test calls it twice in
a row, with the same inputs, and checks both results against the existing
entry point: the factor bit for bit, the norm within 1e-12 relative (the
two reductions split the sum differently). It also checks the static entry
point against the oracle on fp32 and bf16 gradients of odd lengths. This
file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from synth import workloads as W

pytestmark = pytest.mark.gpu


def _static_call(lib, V, grads, dtype, hp, factor, norm, stream):
    ptrs = (ctypes.c_void_p * len(grads))(*[g.data_ptr() for g in grads])
    numel = (ctypes.c_int64 * len(grads))(*[g.numel() for g in grads])
    return lib.vsf_group_norm_scale_static(ptrs, numel, len(grads), dtype, ctypes.byref(hp),
                                           ctypes.c_void_p(factor.data_ptr()),
                                           ctypes.c_void_p(norm.data_ptr()),
                                           ctypes.c_void_p(stream))


@pytest.mark.parametrize("max_norm", [float("inf"), 0.01])
def test_static_norm_matches_planned_norm_twice(max_norm):
    from fsdp_buffer_layout_gb300 import vsf as V
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    lib = V.lib()
    lib.vsf_group_norm_scale_static.restype = ctypes.c_int32
    w = W.tiny()
    specs = [TensorSpec(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors]
    ss = ShardStep(specs, w.m, w.g_coll, max_norm=max_norm)
    try:
        grads = [torch.from_numpy(W.grad(w, 1, t).view(np.int16)).cuda() for t in range(4)]
        ss.pack(grads)
        ss.group_norm_scale()
        torch.cuda.synchronize()
        want_f, want_n = float(ss.factor[0].item()), float(ss.norm[0].item())
        for _ in range(2):
            factor = torch.full((4,), -1.0, dtype=torch.float32, device="cuda")
            norm = torch.full((2,), -1.0, dtype=torch.float64, device="cuda")
            rc = _static_call(lib, V, grads, V.VSF_BF16, ss.hp, factor, norm,
                              ss.stream.cuda_stream)
            assert rc == V.VSF_OK, V.vsf_last_error()
            torch.cuda.synchronize()
            got_f, got_n = float(factor[0].item()), float(norm[0].item())
            assert np.float32(got_f).view(np.uint32) == np.float32(want_f).view(np.uint32)
            assert abs(got_n - want_n) <= 1e-12 * want_n
    finally:
        ss.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("lengths", [(7, 1023, 4097), (3, 5, 1, 11), (100003, 8, 65537)])
def test_static_norm_matches_the_oracle(dtype, lengths):
    """fp32 as well as bf16 gradients; odd lengths, so that CTA spans start
    inside tensors at addresses that are not 16-byte aligned (the scalar
    head); a total of 20 elements, far below the grid of 4 CTAs per SM (every
    CTA but the last sums nothing); and a case of a few hundred thousand
    elements. Two calls in a row, each against the oracle's fp64 sum of
    squares (within its n 2^-53 summation bound) and its factor bit for bit,
    with the clip active and inactive."""
    import oracle
    from fsdp_buffer_layout_gb300 import vsf as V
    lib = V.lib()
    lib.vsf_group_norm_scale_static.restype = ctypes.c_int32
    rng = np.random.default_rng(sum(lengths))
    host = []
    for n in lengths:
        x = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        host.append(x if dtype == "fp32" else (x.view(np.uint32) >> 16).astype(np.uint16))
    tdt = torch.float32 if dtype == "fp32" else torch.int16
    grads = [torch.from_numpy(h.view(np.int16) if dtype == "bf16" else h).to("cuda", tdt)
             for h in host]
    sumsq = oracle.sumsq(host)
    code = V.VSF_FP32 if dtype == "fp32" else V.VSF_BF16
    stream = torch.cuda.current_stream().cuda_stream
    for max_norm in (float("inf"), 1e-5):
        want_f, want_n = oracle.factor(sumsq, 4, max_norm)
        hp = V.make_hparams(world=4, max_norm=max_norm)
        for _ in range(2):
            factor = torch.full((4,), -1.0, dtype=torch.float32, device="cuda")
            norm = torch.full((2,), -1.0, dtype=torch.float64, device="cuda")
            rc = _static_call(lib, V, grads, code, hp, factor, norm, stream)
            assert rc == V.VSF_OK, V.vsf_last_error()
            torch.cuda.synchronize()
            got_f, got_n = float(factor[0].item()), float(norm[0].item())
            assert np.float32(got_f).view(np.uint32) == np.float32(want_f).view(np.uint32)
            assert abs(got_n - want_n) <= max(1e-300, sum(lengths) * 2.0 ** -53 * want_n)


def test_static_norm_rejects_too_many_tensors():
    from fsdp_buffer_layout_gb300 import vsf as V
    lib = V.lib()
    lib.vsf_group_norm_scale_static.restype = ctypes.c_int32
    g = torch.zeros(8, dtype=torch.int16, device="cuda")
    hp = V.make_hparams(world=1)
    out = torch.zeros(4, dtype=torch.float32, device="cuda")
    ptrs = (ctypes.c_void_p * 1025)(*([g.data_ptr()] * 1025))
    numel = (ctypes.c_int64 * 1025)(*([8] * 1025))
    rc = lib.vsf_group_norm_scale_static(ptrs, numel, 1025, V.VSF_BF16, ctypes.byref(hp),
                                         ctypes.c_void_p(out.data_ptr()), None, None)
    assert rc == V.VSF_ERR_ARG
    assert "1024" in V.vsf_last_error()
