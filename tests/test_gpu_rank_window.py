"""Rank windows on the GPU: the shard step run as separate windows of
virtual ranks (one ShardStep per window, as separate processes would own
them) must reach the oracle's whole-buffer results bit for bit, the norm's
one exchange being a sum of the windows' fp64 sums of squares.

"veScale-FSDP: Flexible and High-Performance FSDP at Scale (MLSys 2026)"
summary page, 核心方法 > RaggedShard and > Distributed Buffer. The windows run
one after another on one GPU; nothing waits on another window's kernels.
"""
import math

import numpy as np
import pytest
import torch

from synth import workloads as W
import gpu_harness as H

pytestmark = pytest.mark.gpu


def _case(specs, m, g_coll, steps=3, **kw):
    w = W.Workload("window_case", tuple(W.TensorSpec(f"t{i}", tuple(s[0]), s[1], s[2], s[3])
                                        for i, s in enumerate(specs)), m=m, g_coll=g_coll,
                   steps=steps)
    return H.case_from_workload(w, **kw)


@pytest.mark.parametrize("windows", [[(0, 1), (1, 3), (3, 4)], [(0, 2), (2, 4)], [(0, 4)]])
def test_tiny_windows(windows):
    case = H.case_from_workload(W.tiny())
    H.compare(case, H.run_gpu_windows(case, windows), H.run_oracle(case))


@pytest.mark.parametrize("kw", [dict(max_norm=0.01), dict(standalone_norm=True),
                                dict(grad_dtype=1), dict(quantized=False)])
def test_tiny_windows_variants(kw):
    case = H.case_from_workload(W.tiny(), **kw)
    H.compare(case, H.run_gpu_windows(case, [(0, 1), (1, 4)]), H.run_oracle(case))


def test_windows_with_an_empty_window():
    # two 8192-element atoms on 4 ranks: ranks 2 and 3 hold padding only
    case = _case([((64, 256), W.GRAN_ROWS, 32, 0)], 4, 128)
    H.compare(case, H.run_gpu_windows(case, [(0, 1), (1, 2), (2, 4)]), H.run_oracle(case))


def test_windows_cut_tile_and_row_tensors():
    # 128x128 tiles (bulk-copy tile maps restricted to the window's stripes),
    # 32-row blocks, element chunks, on 8 ranks cut in three windows
    specs = [((1024, 1024), W.GRAN_TILE, 128, 128), ((768, 512), W.GRAN_ROWS, 32, 0),
             ((1000,), W.GRAN_ELEM, 0, 0), ((256, 96), W.GRAN_TILE, 32, 32)]
    case = _case(specs, 8, 512)
    H.compare(case, H.run_gpu_windows(case, [(0, 1), (1, 5), (5, 8)]), H.run_oracle(case))


@pytest.mark.parametrize("name,windows", [("dsv3_block", [(0, 7), (7, 128)]),
                                          ("llama_layer", [(0, 3), (3, 8)]),
                                          pytest.param("moe_layer", [(0, 10), (10, 64)],
                                                       marks=pytest.mark.slow),
                                          pytest.param("llama_1p3b",
                                                       [(0, 100), (100, 613), (613, 1024)],
                                                       marks=pytest.mark.slow)])
def test_full_size_windows_equal_the_whole_plan(name, windows):
    """At full size the windows must give what the whole plan gives on the
    GPU (itself bit-exact against the oracle in the full-size parity tests),
    for every byte of every buffer, over 2 steps."""
    case = H.case_from_workload(W.get(name), steps=2)
    got = H.run_gpu_windows(case, windows)
    want = H.run_gpu(case)
    assert got["factors"] == want["factors"]
    for k in ("packed_grad", "master", "m_state", "v_state", "m_scale", "v_scale",
              "packed_bf16"):
        assert H.bit_equal(got[k], want[k]), k
    for a, b in zip(got["params"], want["params"]):
        assert np.array_equal(a, b)
