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
