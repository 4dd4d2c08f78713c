"""Rank windows (vsf_plan_restrict): a process that owns virtual ranks
[r0, r1) of the DBuffer plans and runs only their part.

"veScale-FSDP: Flexible and High-Performance FSDP at Scale (MLSys 2026)"
summary page, 核心方法 > RaggedShard (no block crosses a rank boundary) and
> Distributed Buffer (each rank holds its own slice of the buffer). Host
logic only: the windows' quantisation-block tables must partition the whole
plan's table (same blocks, bases shifted by r0 * S), the window sizes and
real counts must equal the overlap of every tensor's span with the window,
computed here from the offsets alone, and calls that need whole tensors must
refuse a window.
"""
import random

import numpy as np
import pytest

from fsdp_buffer_layout_gb300 import vsf as V
from synth import workloads as W


def _plan(specs, m, g_coll):
    return V.vsf_plan_create([V.make_desc(*s) for s in specs], m, g_coll)


def _blocks(plan):
    info = V.vsf_plan_get_info(plan)
    qb = V.vsf_plan_qblocks(plan, info.n_qblocks)
    return [tuple(qb[k][i] for k in ("tensor", "base", "nrows", "ncols", "stride"))
            for i in range(info.n_qblocks)]


def _partitions(m):
    cuts = sorted({0, m, m // 3, m // 2, m - 1} - {0, m})
    yield [(0, m)]
    yield [(r, r + 1) for r in range(m)] if m <= 16 else [(0, 1), (1, m)]
    edges = [0] + cuts + [m]
    yield [(a, b) for a, b in zip(edges, edges[1:]) if a < b]


def _check(specs, m, g_coll):
    whole = _plan(specs, m, g_coll)
    try:
        info = V.vsf_plan_get_info(whole)
        S = info.S
        offs = V.vsf_plan_offsets(whole, len(specs))
        numel = [int(np.prod(s[0])) for s in specs]
        want = sorted(_blocks(whole))
        assert info.rank_begin == 0 and info.rank_end == m
    finally:
        V.vsf_plan_destroy(whole)
    for part in _partitions(m):
        got = []
        for r0, r1 in part:
            p = _plan(specs, m, g_coll)
            try:
                V.vsf_plan_restrict(p, r0, r1)
                wi = V.vsf_plan_get_info(p)
                assert (wi.rank_begin, wi.rank_end, wi.S) == (r0, r1, S)
                assert wi.total == (r1 - r0) * S
                lo, hi = r0 * S, r1 * S
                real = sum(max(0, min(hi, o + n) - max(lo, o)) for o, n in zip(offs, numel))
                assert wi.real == real
                for (t, base, nr, nc, st) in _blocks(p):
                    assert 0 <= base < wi.total  # inside the window, from its start
                    got.append((t, base + lo, nr, nc, st))
                assert V.vsf_plan_offsets(p, len(specs)) == offs  # the layout is unchanged
            finally:
                V.vsf_plan_destroy(p)
        assert sorted(got) == want, (part, len(got), len(want))


@pytest.mark.parametrize("name", list(W.ALL))
def test_windows_partition_the_workload_blocks(name):
    w = W.get(name)
    _check([(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors], w.m, w.g_coll)


def test_windows_partition_random_layouts():
    rng = random.Random(7)
    for _ in range(40):
        specs = []
        for _ in range(rng.randint(1, 6)):
            gran = rng.choice([V.VSF_GRAN_ELEM, V.VSF_GRAN_ROWS, V.VSF_GRAN_TILE])
            rows, cols = rng.randint(1, 40), rng.choice([8, 16, 24, 32, 64])
            br = rng.randint(1, 8)
            tc = rng.choice([8, 16, 32]) if gran == V.VSF_GRAN_TILE else 0
            shape = (rows * cols,) if gran == V.VSF_GRAN_ELEM else (rows, cols)
            specs.append((shape, gran, 0 if gran == V.VSF_GRAN_ELEM else br, tc))
        _check(specs, rng.randint(1, 9), rng.choice([1, 3, 8, 16, 128]))


def test_empty_window_has_no_blocks():
    # one tensor of two 8192-element atoms on 4 ranks: S = 8192, ranks 2 and 3 hold padding only
    specs = [((64, 256), V.VSF_GRAN_ROWS, 32, 0)]
    p = _plan(specs, 4, 128)
    try:
        V.vsf_plan_restrict(p, 2, 4)
        info = V.vsf_plan_get_info(p)
        assert (info.S, info.real, info.n_qblocks, info.total) == (8192, 0, 0, 16384)
    finally:
        V.vsf_plan_destroy(p)


def test_restrict_errors_and_whole_tensor_calls():
    specs = [((64, 256), V.VSF_GRAN_ROWS, 32, 0), ((100,), V.VSF_GRAN_ELEM, 0, 0)]
    p = _plan(specs, 4, 128)
    try:
        for r0, r1 in [(-1, 2), (2, 2), (3, 2), (0, 5)]:
            with pytest.raises(V.VsfError) as e:
                V.vsf_plan_restrict(p, r0, r1)
            assert e.value.status == V.VSF_ERR_ARG
        V.vsf_plan_restrict(p, 1, 3)
        V.vsf_plan_restrict(p, 0, 4)  # a second call replaces the window
        assert V.vsf_plan_get_info(p).rank_end == 4
        V.vsf_plan_restrict(p, 0, 2)
        with pytest.raises(V.VsfError) as e:
            V.vsf_plan_views(p, 1 << 20, 2, len(specs))
        assert e.value.status == V.VSF_ERR_STATE
    finally:
        V.vsf_plan_destroy(p)
