"""Which shape of the bulk-copy AdamW kernel a plan selects (host logic).

The kernel comes in two shapes with identical results: wide (16 consumer
warps, one CTA per SM) and narrow (4 consumer warps, four CTAs per SM). A
plan takes the narrow shape exactly when it has bulk-copy units and every
unit holds at most 49152 elements (48 Ki); the plan info reports the choice
as bulk_warps. Checked here on row-atom layouts, whose contiguous blocks are
the units, so that the largest unit is known from the shapes alone, on
rank windows, which choose again for the blocks they hold, and on tile
stripes that only the wide shape's taller copy box divides.
"""
import pytest

from fsdp_buffer_layout_gb300 import vsf as V
from synth import workloads as W

NARROW_MAX = 48 * 1024


def _info(specs, m=4, g_coll=128, window=None):
    p = V.vsf_plan_create([V.make_desc(*s) for s in specs], m, g_coll)
    try:
        if window is not None:
            V.vsf_plan_restrict(p, *window)
        return V.vsf_plan_get_info(p)
    finally:
        V.vsf_plan_destroy(p)


@pytest.mark.parametrize("rows,cols,block_rows,want", [
    (64, 1024, 32, 4),                    # 32768-element units
    (96, 1024, 48, 4),                    # exactly 49152: still narrow
    (2, NARROW_MAX + 16, 1, 16),          # 16 elements over the bound
    (98, 1024, 49, 16),                   # 50176
    (96, 11008, 32, 16),                  # 352256 (a Llama MLP stripe)
])
def test_shape_follows_the_largest_unit(rows, cols, block_rows, want):
    info = _info([((rows, cols), W.GRAN_ROWS, block_rows, 0)])
    assert info.n_bulk_units == rows // block_rows
    assert info.bulk_warps == want


def test_largest_unit_decides_for_the_whole_plan():
    small = ((64, 1024), W.GRAN_ROWS, 32, 0)
    big = ((64, 4096), W.GRAN_ROWS, 16, 0)  # 65536-element units
    assert _info([small]).bulk_warps == 4
    assert _info([small, big]).bulk_warps == 16


def test_no_bulk_units_reports_the_wide_shape():
    info = _info([((100000,), W.GRAN_ELEM, 0, 0)])
    assert info.n_bulk_units == 0 and info.bulk_warps == 16


def test_windows_choose_for_their_own_blocks():
    # S fits one 352256-element stripe per rank: ranks 0 and 1 hold the large
    # blocks, the rank where the second tensor starts only small ones
    specs = [((64, 11008), W.GRAN_ROWS, 32, 0), ((256, 1024), W.GRAN_ROWS, 32, 0)]
    whole = _info(specs)
    assert whole.bulk_warps == 16 and whole.S == 32 * 11008
    p = V.vsf_plan_create([V.make_desc(*s) for s in specs], 4, 128)
    try:
        r_small = V.vsf_plan_offsets(p, 2)[1] // whole.S
    finally:
        V.vsf_plan_destroy(p)
    assert r_small >= 2
    assert _info(specs, window=(0, 1)).bulk_warps == 16
    small = _info(specs, window=(r_small, r_small + 1))
    assert small.n_bulk_units == 8 and small.bulk_warps == 4


def test_workload_shapes():
    want = {"llama_layer": 16, "moe_layer": 16, "dsv3_block": 4, "llama_1p3b": 16}
    for name, warps in want.items():
        w = W.get(name)
        info = _info([(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors],
                     w.m, w.g_coll)
        assert info.bulk_warps == warps, name


@pytest.mark.parametrize("block_rows,want", [(8, 4), (16, 4), (12, 16), (20, 16)])
def test_tile_stripes_keep_their_bulk_copies(block_rows, want):
    # 128-column tiles go two to a 256-column copy box of min(block_rows, 32)
    # rows in the wide shape and min(block_rows, 8) in the narrow one; a
    # stripe the narrow box does not divide would leave the bulk-copy kernel,
    # so such a plan keeps the wide shape and all of its units
    specs = [((block_rows * 4, 1024), W.GRAN_TILE, block_rows, 128)]
    info = _info(specs, m=1, g_coll=128)
    assert info.n_bulk_units == 4 * 1024 // 256
    assert info.n_register_blocks == 0
    assert info.bulk_warps == want


def _plan(specs, m=4, g_coll=128):
    return V.vsf_plan_create([V.make_desc(*s) for s in specs], m, g_coll)


def test_forced_shape_and_back():
    specs = [((256, 512), W.GRAN_TILE, 128, 128), ((96, 11008), W.GRAN_ROWS, 32, 0)]
    p = _plan(specs)
    try:
        auto = V.vsf_plan_get_info(p)
        blocks = V.vsf_plan_qblocks(p, auto.n_qblocks)
        assert auto.bulk_warps == 16
        for warps, want in ((4, 4), (16, 16), (0, 16)):
            V.vsf_plan_set_bulk_warps(p, warps)
            info = V.vsf_plan_get_info(p)
            assert info.bulk_warps == want
            # the blocks and their routing are the same: only the kernel shape moves
            assert (info.n_bulk_units, info.n_register_blocks) == \
                (auto.n_bulk_units, auto.n_register_blocks)
            got = V.vsf_plan_qblocks(p, info.n_qblocks)
            assert got == blocks
    finally:
        V.vsf_plan_destroy(p)


def test_forced_narrow_moves_undivided_stripes_to_the_register_kernel():
    specs = [((48, 1024), W.GRAN_TILE, 12, 128)]  # 12-row stripes: the 8-row box does not divide
    p = _plan(specs, m=1)
    try:
        wide = V.vsf_plan_get_info(p)
        V.vsf_plan_set_bulk_warps(p, 4)
        narrow = V.vsf_plan_get_info(p)
        assert wide.bulk_warps == 16 and wide.n_bulk_units == 16 and wide.n_register_blocks == 0
        assert narrow.bulk_warps == 4 and narrow.n_bulk_units == 0
        assert narrow.n_register_blocks == 4 * 8  # every 12x128 tile, one block each
    finally:
        V.vsf_plan_destroy(p)


def test_forced_shape_survives_restrict_and_rejects_other_values():
    specs = [((64, 11008), W.GRAN_ROWS, 32, 0), ((256, 1024), W.GRAN_ROWS, 32, 0)]
    p = _plan(specs)
    try:
        V.vsf_plan_set_bulk_warps(p, 4)
        V.vsf_plan_restrict(p, 0, 1)
        assert V.vsf_plan_get_info(p).bulk_warps == 4
        for bad in (1, 8, 15, -4):
            with pytest.raises(V.VsfError) as e:
                V.vsf_plan_set_bulk_warps(p, bad)
            assert e.value.status == V.VSF_ERR_ARG
        assert V.vsf_plan_get_info(p).bulk_warps == 4
    finally:
        V.vsf_plan_destroy(p)


def test_cluster_size_is_reported_only_after_upload():
    """vsf_plan_info.bulk_cluster is chosen by vsf_plan_upload (it needs the
    GPU's occupancy); before upload it reads 0, and the reserved word is 0."""
    info = _info([((96, 11008), W.GRAN_ROWS, 32, 0)])
    assert info.bulk_cluster == 0
    assert info.reserved == 0
