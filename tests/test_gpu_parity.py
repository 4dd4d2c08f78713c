"""GPU parity: every libvsf entry point through the C ABI against the oracle
on the same seeded inputs (pack, group norm/scale, 8-bit AdamW, unpack).
Small and ragged cases; the full-size workloads are in test_gpu_fullsize.py.
"""
import math

import numpy as np
import pytest
import torch

from synth import workloads as W

from gpu_harness import Case, case_from_workload, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _normal_case(specs, m, g, steps, seed=11, **kw):
    def grads(s, t):
        n = int(np.prod(specs[t][0]))
        from synth import DIST_NORMAL, KIND_GRAD, fill_bf16, key
        return fill_bf16(key(seed, s, t, KIND_GRAD), DIST_NORMAL, 1e-3, 0, np.empty(n, np.uint16))

    def masters(t):
        n = int(np.prod(specs[t][0]))
        from synth import DIST_NORMAL, KIND_PARAM, fill_f32, key
        return fill_f32(key(seed, 0, t, KIND_PARAM), DIST_NORMAL, 0.02, 0, np.empty(n, np.float32))

    return Case(specs=specs, m=m, g_coll=g, steps=steps, grads=grads, masters=masters, **kw)


def test_tiny_three_steps_bit_exact():
    case = case_from_workload(W.tiny())
    compare(case, run_gpu(case), run_oracle(case))


def test_tiny_clip_active():
    """max_norm 0.01 against a mean-gradient norm near 0.116: c < 1."""
    case = case_from_workload(W.tiny(), max_norm=0.01)
    o = run_oracle(case)
    assert all(f < 0.25 for f in o["factors"])
    compare(case, run_gpu(case), o)


def test_tiny_fp32_grads():
    case = case_from_workload(W.tiny(), grad_dtype=1)
    compare(case, run_gpu(case), run_oracle(case))


def test_tiny_fp32_state():
    case = case_from_workload(W.tiny(), quantized=False)
    compare(case, run_gpu(case), run_oracle(case))


def test_tiny_standalone_norm():
    case = case_from_workload(W.tiny(), steps=2, standalone_norm=True)
    compare(case, run_gpu(case), run_oracle(case))


RAGGED = [
    ((300, 1000), W.GRAN_ROWS, 32, 0),      # 9 full blocks + a 12-row tail
    ((45, 77), W.GRAN_TILE, 8, 16),         # ragged right and bottom tiles
    ((1000,), W.GRAN_ELEM, 0, 0),           # 7 full chunks + one of 104
    ((1,), W.GRAN_ELEM, 0, 0),              # a one-element tensor
    ((3, 5), W.GRAN_ROWS, 8, 0),            # atom longer than the tensor
    ((4, 256, 96), W.GRAN_ROWS, 64, 0),     # 3-D: rows = product of leading dims
    ((128, 4096), W.GRAN_TILE, 128, 128),   # 32 full 128x128 tiles
]


def test_ragged_mixed_several_steps():
    case = _normal_case(RAGGED, m=5, g=128, steps=4)
    assert _bulk_warps(case) == 4
    compare(case, run_gpu(case), run_oracle(case))


def test_unaligned_collective_unit_takes_scalar_paths():
    """g_coll = 3: offsets and blocks are not 16-byte aligned."""
    case = _normal_case(RAGGED[:5], m=3, g=3, steps=3)
    compare(case, run_gpu(case), run_oracle(case))


def test_single_rank_and_many_empty_ranks():
    one = _normal_case(RAGGED[:3], m=1, g=64, steps=2)
    compare(one, run_gpu(one), run_oracle(one))
    many = _normal_case(RAGGED[:2], m=64, g=128, steps=2)
    compare(many, run_gpu(many), run_oracle(many))


def test_S_equal_to_one_block():
    """Four 8192-element row blocks on four ranks: S is exactly one block,
    every rank holds one whole block and every boundary is a block edge."""
    case = _normal_case([((128, 256), W.GRAN_ROWS, 32, 0)], m=4, g=128, steps=3)
    o = run_oracle(case)
    assert o["S"] == 8192
    compare(case, run_gpu(case), o)


def test_all_zero_blocks_keep_zero_codes():
    specs = [((64, 256), W.GRAN_ROWS, 16, 0), ((512,), W.GRAN_ELEM, 0, 0)]
    case = _normal_case(specs, m=2, g=128, steps=3)
    base = case.grads
    case.grads = lambda s, t: np.zeros_like(base(s, t)) if t == 0 else base(s, t)
    g, o = run_gpu(case), run_oracle(case)
    compare(case, g, o)
    off = int(o["offsets"][0])
    assert not g["m_state"][off:off + 64 * 256].any()
    assert not g["v_state"][off:off + 64 * 256].any()


def _bulk_warps(case):
    """Consumer warps of the bulk-copy AdamW kernel shape the case's plan uses."""
    from fsdp_buffer_layout_gb300 import vsf as V
    p = V.vsf_plan_create([V.make_desc(*s) for s in case.specs], case.m, case.g_coll)
    try:
        return V.vsf_plan_get_info(p).bulk_warps
    finally:
        V.vsf_plan_destroy(p)


def test_large_blocks_use_clusters():
    """Blocks of 352,256 elements (a 32-row stripe of an 11008-column matrix):
    the wide kernel shape."""
    specs = [((96, 11008), W.GRAN_ROWS, 32, 0), ((256, 4096), W.GRAN_ROWS, 32, 0),
             ((4096,), W.GRAN_ELEM, 0, 0)]
    case = _normal_case(specs, m=4, g=128, steps=3)
    assert _bulk_warps(case) == 16
    compare(case, run_gpu(case), run_oracle(case))


@pytest.mark.parametrize("shape,block_rows,want", [
    ((512, 2880), 128, 4),   # 368,640-element blocks (MoE expert stripes): 4 equal shares
    ((508, 2896), 127, 4),   # 367,792 = 16 * 22,987: shares of unequal 16-element counts
    ((256, 7168), 128, 8),   # 917,504-element blocks
])
def test_large_units_use_clusters_of_four_and_eight(shape, block_rows, want):
    """Units whose phase-1 bytes would overflow the L2 budget in clusters of 2
    go to clusters of 4 or 8, each CTA taking an equal element range (to 16
    elements) of every unit, empty for most CTAs of a 16- or 48-element unit;
    bit-exact like every other path."""
    specs = [(shape, W.GRAN_ROWS, block_rows, 0), ((4096,), W.GRAN_ELEM, 0, 0),
             # 16- and 48-element blocks: most CTAs of a cluster get an empty
             # share of such a unit and still take part in its exchange
             ((8, 16), W.GRAN_ROWS, 1, 0), ((4, 48), W.GRAN_ROWS, 1, 0)]
    case = _normal_case(specs, m=4, g=128, steps=3)
    g = run_gpu(case)
    assert g["bulk_cluster"] == want, f"clusters of {g['bulk_cluster']}"
    compare(case, g, run_oracle(case))


def test_large_blocks_fp32_gradients():
    """fp32 gradients on large blocks: the bulk-copy ring then holds 2 slots
    of 80 KB instead of 3 of 64 KB, with clusters of 2 for the 352K-element
    blocks, and 128x128 tiles through the 2-D tensor copies."""
    specs = [((96, 11008), W.GRAN_ROWS, 32, 0), ((512, 512), W.GRAN_TILE, 128, 128),
             ((4096,), W.GRAN_ELEM, 0, 0)]
    case = _normal_case(specs, m=4, g=128, steps=3)
    case.grad_dtype = 1

    def grads(s, t):  # seeded fp32 gradients (full fp32 mantissas)
        from synth import DIST_NORMAL, KIND_GRAD, fill_f32, key
        n = int(np.prod(specs[t][0]))
        return fill_f32(key(11, s, t, KIND_GRAD), DIST_NORMAL, 1e-3, 0, np.empty(n, np.float32))

    case.grads = grads
    compare(case, run_gpu(case), run_oracle(case))


@pytest.mark.parametrize("warps", [4, 16])
def test_tiles_on_every_path(warps):
    """Full tiles of mapped tile tensors (2-D tensor copies: 128x128, 32x64),
    ragged bottom tiles and tiles wider than a copy box (register kernel),
    next to element chunks: all bit-exact, in both kernel shapes (a tensor of
    352,256-element row blocks selects the wide one; the copy boxes are then
    4 times taller)."""
    specs = [((256, 512), W.GRAN_TILE, 128, 128), ((96, 256), W.GRAN_TILE, 32, 64),
             ((200, 384), W.GRAN_TILE, 64, 128), ((64, 4096), W.GRAN_TILE, 16, 1024),
             ((1024,), W.GRAN_ELEM, 0, 0)]
    if warps == 16:
        specs.append(((64, 11008), W.GRAN_ROWS, 32, 0))
    case = _normal_case(specs, m=4, g=128, steps=3)
    assert _bulk_warps(case) == warps
    compare(case, run_gpu(case), run_oracle(case))


@pytest.mark.parametrize("warps", [4, 16])
def test_forced_kernel_shapes_match_the_oracle(warps):
    """One plan in each forced bulk-copy shape (vsf_plan_set_bulk_warps): the
    ragged set (the planner's narrow choice) plus 352K-element row blocks (its
    wide choice). Both shapes must be bit-exact against the oracle, hence
    equal to each other."""
    specs = RAGGED + [((64, 11008), W.GRAN_ROWS, 32, 0)]
    case = _normal_case(specs, m=5, g=128, steps=2, bulk_warps=warps)
    assert _bulk_warps(case) == 16  # the planner's own choice for this set
    compare(case, run_gpu(case), run_oracle(case))


def test_heavy_tails_student_t():
    w = W.dsv3_block()
    specs = [((512, 1024), W.GRAN_TILE, 128, 128), ((7168,), W.GRAN_ELEM, 0, 0)]

    def grads(s, t):
        n = int(np.prod(specs[t][0]))
        from synth import DIST_STUDENT_T3, KIND_GRAD, fill_bf16, key
        return fill_bf16(key(0, s, t, KIND_GRAD), DIST_STUDENT_T3, 1e-3, 0, np.empty(n, np.uint16))

    case = Case(specs=specs, m=8, g_coll=512, steps=5, grads=grads,
                masters=lambda t: W.master_init(w, t, 0, int(np.prod(specs[t][0]))))
    compare(case, run_gpu(case), run_oracle(case))


def test_misaligned_pointer_is_an_error_not_a_fault():
    from fsdp_buffer_layout_gb300 import vsf as V
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    ss = ShardStep([TensorSpec((64, 64), W.GRAN_ROWS, 8)], 2, 128)
    try:
        g = torch.zeros(64 * 64 + 8, dtype=torch.int16, device="cuda")
        with pytest.raises(V.VsfError) as e:
            V.vsf_pack(ss.plan, [g.data_ptr() + 2], V.VSF_BF16, ss.packed_grad.data_ptr(),
                       ss.stream.cuda_stream)
        assert e.value.status == V.VSF_ERR_ALIGN
        with pytest.raises(V.VsfError) as e:
            V.vsf_adam8_step(ss.plan, ss.packed_grad.data_ptr() + 4, V.VSF_BF16,
                             ss.factor.data_ptr(), ss.master.data_ptr(), ss.m_state.data_ptr(),
                             ss.v_state.data_ptr(), ss.m_scale.data_ptr(), ss.v_scale.data_ptr(),
                             ss.packed_bf16.data_ptr(), ss.hp, 1, ss.stream.cuda_stream)
        assert e.value.status == V.VSF_ERR_ALIGN
        with pytest.raises(V.VsfError) as e:
            V.vsf_adam8_step(ss.plan, ss.packed_grad.data_ptr(), V.VSF_BF16,
                             ss.factor.data_ptr(), ss.master.data_ptr(), ss.m_state.data_ptr(),
                             ss.v_state.data_ptr(), ss.m_scale.data_ptr(), ss.v_scale.data_ptr(),
                             ss.packed_bf16.data_ptr(), ss.hp, 0, ss.stream.cuda_stream)
        assert e.value.status == V.VSF_ERR_ARG
        torch.cuda.synchronize()
    finally:
        ss.close()


def test_padding_is_never_written():
    """Canary values in the padding survive a step (no write outside real elements)."""
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    w = W.tiny()
    specs = [TensorSpec(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors]
    ss = ShardStep(specs, w.m, w.g_coll)
    try:
        real = torch.zeros(ss.info.total, dtype=torch.bool, device="cuda")
        for o, n in zip(ss.offsets, ss.numels):
            real[o:o + n] = True
        pad = ~real
        assert int(pad.sum()) > 0
        for buf in (ss.packed_grad.view(torch.int16), ss.master, ss.m_state, ss.v_state,
                    ss.packed_bf16.view(torch.int16)):
            buf[pad] = 77 if buf.dtype != torch.float32 else 77.0
        grads = [torch.from_numpy(W.grad(w, 1, t).view(np.int16)).cuda() for t in range(4)]
        params = [torch.empty_like(g) for g in grads]
        ss.step(grads, params, 1)
        torch.cuda.synchronize()
        for buf in (ss.packed_grad.view(torch.int16), ss.master, ss.m_state, ss.v_state,
                    ss.packed_bf16.view(torch.int16)):
            assert bool((buf[pad] == 77).all())
    finally:
        ss.close()


def test_special_values_match_oracle():
    """NaN, +-inf, values that overflow bf16, fp32 and bf16 denormals, bf16
    rounding ties and -0 in masters and gradients: same bits as the oracle
    (NaN bits aside: any NaN matches any NaN), and NaN codes = 0."""
    specs = [((64, 64), W.GRAN_ROWS, 16, 0), ((256,), W.GRAN_ELEM, 0, 0)]
    case = _normal_case(specs, m=2, g=128, steps=2)
    base_g, base_m = case.grads, case.masters
    f32 = lambda x: np.array([x], np.float32)[0]  # noqa: E731
    specials_m = [np.nan, np.inf, -np.inf, 3.4e38, -3.3e38, 1e-40, -1e-45,
                  f32(1 + 2 ** -8), f32(1 + 3 * 2 ** -8), -0.0, 0.0]

    def masters(t):
        x = base_m(t).copy()
        if t == 0:
            x[:len(specials_m)] = specials_m        # block 0 of tensor 0
            x[1024 + 5] = f32(-(1 + 2 ** -8))       # a tie in block 1
        else:
            x[3] = np.nan
        return x

    def grads(s, t):
        x = base_g(s, t).copy()
        if t == 0:
            x[2048 + 1] = 0x7FC0                    # NaN in block 2
            x[3072 + 2] = 0x7F80                    # +inf in block 3
            x[1024 + 9] = 0x0001                    # bf16 denormal
            x[1024 + 10] = 0x8000                   # -0
            x[1024 + 11] = 0x7F7F                   # largest finite bf16
        else:
            x[200] = 0x0001
        return x

    case.masters, case.grads = masters, grads
    compare(case, run_gpu(case), run_oracle(case))


def test_tiny_block_scale_codes_stay_symmetric():
    """Blocks whose gradients are all bf16 subnormals of both signs: the new
    m scale (about 1e-40) is below 127 / FLT_MAX, so 127 / scale overflows
    and every nonzero moment saturates. The m codes must be +-127, never
    -128, in the bulk-copy kernel (row blocks), the register kernel
    (128-column tiles) and the element-chunk kernel alike."""
    specs = [((64, 64), W.GRAN_ROWS, 16, 0), ((256,), W.GRAN_ELEM, 0, 0),
             ((64, 256), W.GRAN_TILE, 16, 128)]
    case = _normal_case(specs, m=2, g=128, steps=3)
    base_g = case.grads

    def grads(s, t):
        x = base_g(s, t).copy()
        rng = np.random.default_rng((5, s, t))  # the same values on every call
        lo, hi = {0: (1024, 2048), 1: (128, 256), 2: (16 * 256, 32 * 256)}[t]
        mag = rng.integers(1, 0x80, hi - lo).astype(np.uint16)        # bf16 subnormals
        sign = (rng.integers(0, 2, hi - lo).astype(np.uint16) << 15)
        x[lo:hi] = mag | sign
        return x

    case.grads = grads
    o = run_oracle(case)
    assert not np.any(o["m_state"] == -128)
    assert np.count_nonzero(o["m_state"] == -127) > 500
    compare(case, run_gpu(case), o)
