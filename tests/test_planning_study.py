"""The layout study helpers against the oracle planner (same S, hence same
padding, at every sweep point) and the group-size chooser's definition."""
import oracle
from fsdp_buffer_layout_gb300 import planning
from synth import workloads as W


def _oracle_padding(tensors, m, g, rows_per_atom):
    rows = [int(t[0][0]) if len(t[0]) == 1 else int(__import__("numpy").prod(t[0][:-1]))
            for t in tensors]
    rows = [1 if len(t[0]) == 1 else r for t, r in zip(tensors, rows)]
    cols = [t[0][-1] for t in tensors]
    br = [rows_per_atom if t[1] else 0 for t in tensors]
    d = oracle.Desc(rows, cols, [t[1] for t in tensors], br, [t[3] for t in tensors])
    S, _ = oracle.plan(d, m, g)
    real = sum(r * c for r, c in zip(rows, cols))
    return S, 1 - real / (m * S)


def test_sweep_matches_oracle():
    w = W.moe_layer()
    tensors = [(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors]
    for p in planning.sweep(tensors, [1, 16, 128], [8, 64, 256], w.g_coll):
        S, pad = _oracle_padding(tensors, p.m, w.g_coll, p.rows_per_atom)
        assert p.S == S and abs(p.padding - pad) < 1e-12
        assert p.plan_seconds < 0.3


def test_choose_group_size():
    w = W.dsv3_block()
    tensors = [(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors]
    ms = [8, 16, 32, 64, 128, 256]
    pick = planning.choose_group_size(tensors, ms, w.g_coll, 0.03, rows_per_atom=1)
    pads = {m: planning.plan_point(tensors, m, w.g_coll, 1).padding for m in ms}
    assert pick == max(m for m in ms if pads[m] <= 0.03)
    assert planning.choose_group_size(tensors, ms, w.g_coll, 0.0, rows_per_atom=128) is None
