"""Layout studies on top of the planner (host only, no GPU):

- ``sweep``: padding and planning time of a set of tensors over shard
  granularities (rows per atom) and group sizes m, the study of "veScale-FSDP:
  Flexible and High-Performance FSDP at Scale (MLSys 2026)" summary page,
  实验 > Figure 11 (planning quality: padding against granularity);
- ``choose_group_size``: the largest group size whose padding stays under a
  limit, the offline group-size simulation the same page proposes against
  padding spikes (设计取舍; 局限与 Future Work).

    python -m fsdp_buffer_layout_gb300.planning --workload moe_layer
"""
from __future__ import annotations

import argparse
import dataclasses

from . import vsf as V


@dataclasses.dataclass
class SweepPoint:
    rows_per_atom: int
    m: int
    S: int
    padding: float
    plan_seconds: float


def _descs(tensors, rows_per_atom):
    out = []
    for shape, gran, br, bc in tensors:
        if gran in (V.VSF_GRAN_ROWS, V.VSF_GRAN_TILE) and rows_per_atom:
            br = rows_per_atom
        out.append(V.make_desc(shape, gran, br, bc))
    return out


def plan_point(tensors, m: int, g_coll: int, rows_per_atom: int = 0,
               order: int = V.VSF_ORDER_DEFAULT) -> SweepPoint:
    """One plan. tensors: (shape, gran, block_rows, tile_cols); rows_per_atom
    (if non-zero) replaces block_rows of every row or tile tensor."""
    p = V.vsf_plan_create(_descs(tensors, rows_per_atom), m, g_coll, order)
    try:
        i = V.vsf_plan_get_info(p)
        return SweepPoint(rows_per_atom, m, int(i.S), float(i.padding_ratio),
                          float(i.plan_seconds))
    finally:
        V.vsf_plan_destroy(p)


def sweep(tensors, granularities, group_sizes, g_coll: int,
          order: int = V.VSF_ORDER_DEFAULT) -> list[SweepPoint]:
    return [plan_point(tensors, m, g_coll, r, order) for r in granularities for m in group_sizes]


def choose_group_size(tensors, group_sizes, g_coll: int, max_padding: float,
                      rows_per_atom: int = 0, order: int = V.VSF_ORDER_DEFAULT) -> int | None:
    """The largest m of `group_sizes` whose padding ratio is <= max_padding."""
    best = None
    for m in sorted(group_sizes):
        if plan_point(tensors, m, g_coll, rows_per_atom, order).padding <= max_padding:
            best = m
    return best


def _main():
    from synth import workloads as W
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="moe_layer")
    ap.add_argument("--rows", default="1,16,128")
    ap.add_argument("--m", default="8,16,32,64,128,256,512,1024")
    args = ap.parse_args()
    w = W.get(args.workload)
    tensors = [(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors]
    ms = [int(x) for x in args.m.split(",")]
    print(f"{w.name}: padding ratio (planning seconds) by rows per atom x group size m")
    print("rows\\m " + " ".join(f"{m:>14d}" for m in ms))
    for r in (int(x) for x in args.rows.split(",")):
        pts = [plan_point(tensors, m, w.g_coll, r) for m in ms]
        print(f"{r:6d} " + " ".join(f"{100 * p.padding:7.2f}% ({p.plan_seconds:.3f})" for p in pts))
    print("largest m with padding <= 3%:",
          {r: choose_group_size(tensors, ms, w.g_coll, 0.03, r) for r in (1, 16, 128)})


if __name__ == "__main__":
    _main()
