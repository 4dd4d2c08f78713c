"""The library's planner (libvsf, host only) against the oracle's: the same
S, offsets and quantisation blocks, bit for bit, on every workload and on
random descriptor sets; planning time on every workload under the pages'
0.3 s ("veScale-FSDP: Flexible and High-Performance FSDP at Scale (MLSys
2026)" summary page, 核心方法 > Algorithm 1 and 实验 > Figure 11)."""
import numpy as np
import pytest

import oracle
from fsdp_buffer_layout_gb300 import vsf as V
from synth import workloads as W


def lib_plan(specs, m, g, order=V.VSF_ORDER_DEFAULT):
    descs = [V.make_desc(s[0], s[1], s[2], s[3]) for s in specs]
    p = V.vsf_plan_create(descs, m, g, order)
    try:
        info = V.vsf_plan_get_info(p)
        off = V.vsf_plan_offsets(p, len(specs))
        qb = V.vsf_plan_qblocks(p, info.n_qblocks)
        slices = [V.vsf_plan_rank_slices(p, r, ) for r in range(min(m, 64))]
        return info, off, qb, slices
    finally:
        V.vsf_plan_destroy(p)


def specs_of(w):
    return [(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors]


def desc_of(specs):
    rows = [int(np.prod(s[0][:-1])) if len(s[0]) > 1 else 1 for s in specs]
    cols = [s[0][-1] for s in specs]
    return oracle.Desc(rows, cols, [s[1] for s in specs], [s[2] for s in specs],
                       [s[3] for s in specs])


def compare(specs, m, g, order):
    info, off, qb, _ = lib_plan(specs, m, g, order)
    d = desc_of(specs)
    S, ooff = oracle.plan(d, m, g, order)
    assert info.S == S
    assert list(off) == [int(x) for x in ooff]
    oq = oracle.qblocks(d, g, ooff)
    for k in ("tensor", "base", "nrows", "ncols", "stride"):
        assert list(qb[k]) == [int(x) for x in oq[k]], k
    return info


@pytest.mark.parametrize("name", list(W.ALL))
def test_workloads_match_oracle(name):
    w = W.get(name)
    for order in (V.VSF_ORDER_DEFAULT, V.VSF_ORDER_BLOCK, V.VSF_ORDER_SHAPE, V.VSF_ORDER_BEST3):
        info = compare(specs_of(w), w.m, w.g_coll, order)
        assert info.plan_seconds < 0.3
        assert info.real == w.numel and info.total == w.m * info.S


@pytest.mark.parametrize("seed", range(150))
def test_random_match_oracle(seed):
    rng = np.random.default_rng(77 + seed)
    n = int(rng.integers(1, 9))
    specs = []
    for _ in range(n):
        kind = int(rng.integers(0, 3))
        shape = tuple(int(x) for x in rng.integers(1, 40, size=int(rng.integers(1, 4))))
        br = int(rng.integers(1, 9)) if kind else 0
        bc = int(rng.integers(1, 9)) if kind == 2 else 0
        specs.append((shape, kind, br, bc))
    m = int(rng.integers(1, 17))
    g = int(rng.choice([1, 2, 3, 8, 16, 128]))
    compare(specs, m, g, int(rng.integers(0, 4)))


def test_rank_slices_are_the_ragged_shards():
    w = W.moe_layer()
    info, off, qb, slices = lib_plan(specs_of(w), w.m, w.g_coll)
    S = info.S
    numel = [t.numel for t in w.tensors]
    atom = [1 if t.gran == W.GRAN_ELEM else t.block_rows * t.cols for t in w.tensors]
    held = [0] * len(numel)
    for r, sl in enumerate(slices):
        for (t, e0, e1, a0, a1) in sl:
            assert r * S <= off[t] + e0 < off[t] + e1 <= (r + 1) * S
            assert e0 % atom[t] == 0 and (e1 % atom[t] == 0 or e1 == numel[t])
            assert a0 == e0 // atom[t] and a1 == -(-e1 // atom[t])
            held[t] += e1 - e0
    assert held == numel  # the first 64 ranks hold everything here (m = 64)
    counts = [sum(e1 - e0 for (_, e0, e1, _, _) in sl) for sl in slices]
    assert len(set(counts)) > 1  # uneven (ragged) content with a uniform S


def test_bad_descriptors_are_rejected():
    with pytest.raises(V.VsfError) as e:
        V.vsf_plan_create([V.make_desc((4, 4), V.VSF_GRAN_ROWS, 0)], 2, 8)
    assert e.value.status == V.VSF_ERR_ARG
    with pytest.raises(V.VsfError):
        V.vsf_plan_create([V.make_desc((4, 0), V.VSF_GRAN_ELEM)], 2, 8)
    with pytest.raises(V.VsfError):
        V.vsf_plan_create([V.make_desc((4, 4), 7)], 2, 8)
    with pytest.raises(V.VsfError) as e:
        V.vsf_plan_create([V.make_desc((1 << 40, 1 << 40), V.VSF_GRAN_ELEM)], 2, 8)
    assert e.value.status == V.VSF_ERR_OVERFLOW


def test_size_limits_are_refused_not_truncated():
    """The kernels keep block extents in 32-bit fields: a quantisation block
    of 2^31 elements or more, or a tile tensor with 2^31 or more rows or
    columns, must be refused at plan time (VSF_ERR_OVERFLOW)."""
    big_rows = V.make_desc((2, (1 << 30) + 8), V.VSF_GRAN_ROWS, 2)  # one block of > 2^31
    with pytest.raises(V.VsfError) as e:
        V.vsf_plan_create([big_rows], 1, 8)
    assert e.value.status == V.VSF_ERR_OVERFLOW
    wide_tile = V.make_desc((1, (1 << 31) + 16), V.VSF_GRAN_TILE, 1, 16)
    with pytest.raises(V.VsfError) as e:
        V.vsf_plan_create([wide_tile], 1, 16)
    assert e.value.status == V.VSF_ERR_OVERFLOW
    # just below the limit is planned
    ok = V.vsf_plan_create([V.make_desc((1, (1 << 31) - 16), V.VSF_GRAN_ROWS, 1)], 1, 16)
    try:
        assert V.vsf_plan_get_info(ok).n_qblocks == 1
    finally:
        V.vsf_plan_destroy(ok)
