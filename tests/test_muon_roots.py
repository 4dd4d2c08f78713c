"""SelectRoot of distributed Muon in libvsf (host) equals the oracle's greedy
on the same loads, for every workload; 1-D tensors get no root."""
import numpy as np
import pytest

from fsdp_buffer_layout_gb300 import vsf as V
from oracle import muon
from synth import workloads as W


@pytest.mark.parametrize("name", list(W.ALL))
def test_roots_match_oracle(name):
    w = W.get(name)
    p = V.vsf_plan_create([V.make_desc(t.shape, t.gran, t.block_rows, t.tile_cols)
                           for t in w.tensors], w.m, w.g_coll)
    try:
        roots, bal = V.vsf_muon_select_roots(p, len(w.tensors))
    finally:
        V.vsf_plan_destroy(p)
    mats = [i for i, t in enumerate(w.tensors) if len(t.shape) >= 2]
    want, total = muon.select_roots([muon.ns_flops(w.tensors[i].shape) for i in mats], w.m)
    for i, t in enumerate(w.tensors):
        assert roots[i] == (want[mats.index(i)] if i in mats else -1)
    assert abs(bal - max(total) / (sum(total) / w.m)) < 1e-9
