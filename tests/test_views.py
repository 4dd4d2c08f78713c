"""The persistent address map (vsf_plan_views): every tensor's view is the
packed buffer plus its planned offset, for 1-, 2- and 4-byte elements."""
import pytest

from fsdp_buffer_layout_gb300 import vsf as V
from synth import workloads as W


@pytest.mark.parametrize("name", ["tiny", "llama_1p3b"])
def test_views_are_offsets(name):
    w = W.get(name)
    p = V.vsf_plan_create([V.make_desc(t.shape, t.gran, t.block_rows, t.tile_cols)
                           for t in w.tensors], w.m, w.g_coll)
    try:
        off = V.vsf_plan_offsets(p, len(w.tensors))
        base = 1 << 40
        for es in (1, 2, 4):
            views = V.vsf_plan_views(p, base, es, len(w.tensors))
            assert views == [base + o * es for o in off]
        with pytest.raises(V.VsfError):
            V.vsf_plan_views(p, base, 3, len(w.tensors))
    finally:
        V.vsf_plan_destroy(p)
