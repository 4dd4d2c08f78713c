"""Pins of the oracle's layout planner against things other than itself.

Rule being pinned: "veScale-FSDP: Flexible and High-Performance FSDP at Scale
(MLSys 2026)" summary page, 核心方法 > Grouped communication (Algorithm 1) and
> RaggedShard. Pins: invariants checked by independent Python code, a Python
exhaustive search over all aligned offsets on micro instances, the closed
forms in tests/golden/layout_closed_forms.txt, and a pigeonhole closed form.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
from synth import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layout_closed_forms.txt")


def atom(rows, cols, gran, br):
    return 1 if gran == W.GRAN_ELEM else br * cols


def check_invariants(d, m, g, S, off):
    """Independent statement of Algorithm 1's constraints."""
    numel = d.rows * d.cols
    assert S % g == 0
    lb = -(-int(numel.sum()) // m)
    lb = -(-lb // g) * g
    assert S >= lb
    spans = []
    for t in range(d.n):
        b = atom(d.rows[t], d.cols[t], d.gran[t], d.block_rows[t])
        a = b * g // math.gcd(b, g)
        o, n = int(off[t]), int(numel[t])
        assert o % a == 0, "offset not aligned to lcm(g_coll, block)"
        assert 0 <= o and o + n <= m * S, "tensor outside the buffer"
        for k in range(o // S + 1, m + 1):
            if k * S >= o + n:
                break
            assert (k * S - o) % b == 0, "a rank boundary cuts a block"
        spans.append((o, o + n))
    spans.sort()
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0, "tensors overlap"


def py_exhaustive(sizes, atoms, aligns, m, g, s_max):
    """Smallest S with some aligned, non-overlapping, uncut placement (any order)."""
    n = len(sizes)
    lb = -(-sum(sizes) // m)
    lb = -(-lb // g) * g
    for S in range(lb, s_max + 1, g):
        cands = []
        for t in range(n):
            c = []
            for o in range(0, m * S - sizes[t] + 1, aligns[t]):
                if all((k * S - o) % atoms[t] == 0
                       for k in range(o // S + 1, m + 1) if k * S < o + sizes[t]):
                    c.append(o)
            cands.append(c)
        for combo in itertools.product(*cands):
            iv = sorted((o, o + sizes[t]) for t, o in enumerate(combo))
            if all(a[1] <= b[0] for a, b in zip(iv, iv[1:])):
                return S
    return -1


def random_desc(rng, n):
    rows, cols, gran, br, bc = [], [], [], [], []
    for _ in range(n):
        kind = rng.integers(0, 3)
        r, c = int(rng.integers(1, 9)), int(rng.integers(1, 9))
        rows.append(r)
        cols.append(c)
        gran.append(kind)
        br.append(int(rng.integers(1, 4)) if kind else 0)
        bc.append(int(rng.integers(1, 4)) if kind == 2 else 0)
    return oracle.Desc(rows, cols, gran, br, bc)


@pytest.mark.parametrize("seed", range(40))
def test_invariants_random(seed):
    rng = np.random.default_rng(seed)
    d = random_desc(rng, int(rng.integers(1, 7)))
    m = int(rng.integers(1, 6))
    g = int(rng.choice([1, 2, 4, 8]))
    for policy in (oracle.ORDER_DEFAULT, oracle.ORDER_BLOCK, oracle.ORDER_SHAPE,
                   oracle.ORDER_BEST3):
        S, off = oracle.plan(d, m, g, policy)
        check_invariants(d, m, g, S, off)


@pytest.mark.parametrize("seed", range(30))
def test_order_policies_place_as_read(seed):
    """The tensor orders of Algorithm 1's first step, as read: DEFAULT keeps the
    input order, BLOCK sorts by atom size and SHAPE by element count, both
    descending with ties in input order; BEST3 returns the plan of the first of
    the three (DEFAULT, BLOCK, SHAPE) that reaches the smallest S. Tensors are
    placed one after another, so sorting them by offset recovers the order a
    plan used."""
    rng = np.random.default_rng(1000 + seed)
    d = random_desc(rng, int(rng.integers(2, 7)))
    m = int(rng.integers(1, 6))
    g = int(rng.choice([1, 2, 4, 8]))
    block, _ = oracle.atoms(d, g)
    numel = d.numel
    want = {oracle.ORDER_DEFAULT: list(range(d.n)),
            oracle.ORDER_BLOCK: sorted(range(d.n), key=lambda t: (-int(block[t]), t)),
            oracle.ORDER_SHAPE: sorted(range(d.n), key=lambda t: (-int(numel[t]), t))}
    plans = {}
    for policy, order in want.items():
        S, off = oracle.plan(d, m, g, policy)
        assert [int(t) for t in np.argsort(off, kind="stable")] == order, policy
        S2, off2 = oracle.plan(d, m, g, order=order)
        assert S == S2 and list(off) == list(off2)
        plans[policy] = (S, list(off))
    S3, off3 = oracle.plan(d, m, g, oracle.ORDER_BEST3)
    best = min(S for S, _ in plans.values())
    first = next(p for p in (oracle.ORDER_DEFAULT, oracle.ORDER_BLOCK, oracle.ORDER_SHAPE)
                 if plans[p][0] == best)
    assert (S3, list(off3)) == plans[first]


@pytest.mark.parametrize("seed", range(60))
def test_greedy_over_orders_equals_exhaustive(seed):
    """min over orders of the greedy placement == the true optimum (micro cases)."""
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 4))
    m = int(rng.integers(1, 5))
    g = int(rng.choice([1, 2, 3, 4]))
    d = random_desc(rng, n)
    sizes = [int(x) for x in d.rows * d.cols]
    atoms = [atom(d.rows[t], d.cols[t], d.gran[t], d.block_rows[t]) for t in range(n)]
    aligns = [a * g // math.gcd(a, g) for a in atoms]
    s_max = -(-(sum(sizes) + sum(aligns)) // g) * g
    want = py_exhaustive(sizes, atoms, aligns, m, g, s_max)
    got, order = oracle.bruteforce_S(d, m, g)
    assert got == want
    assert oracle.exhaustive_S(d, m, g, s_max) == want
    S, off = oracle.plan(d, m, g, order=order)
    assert S == want
    check_invariants(d, m, g, S, off)


def test_feasibility_not_monotone_in_S():
    """One 2-block tensor (block 10), m=2, g=1: S=10 fits, S=11 does not."""
    d = oracle.Desc([2], [10], [W.GRAN_ROWS], [1], [0])
    assert oracle.exhaustive_S(d, 2, 1, 10) == 10
    S, off = oracle.plan(d, 2, 1)
    assert S == 10 and off[0] == 0


@pytest.mark.parametrize("blocks,b,m,g", [(3, 10, 2, 1), (7, 8, 3, 4), (64, 128, 8, 128),
                                          (100, 96, 7, 32), (5, 16, 16, 16)])
def test_single_tensor_pigeonhole(blocks, b, m, g):
    """One tensor of `blocks` atoms of b elements (g | b): S* = b * ceil(blocks / m)."""
    d = oracle.Desc([blocks], [b], [W.GRAN_ROWS], [1], [0])
    S, off = oracle.plan(d, m, g)
    assert S == b * -(-blocks // m)
    check_invariants(d, m, g, S, off)


def test_element_granular_only_is_balanced():
    """No atom can be cut: S equals the balanced lower bound when sizes are multiples of g."""
    d = oracle.Desc([1, 1, 1], [1024, 384, 640], [W.GRAN_ELEM] * 3, [0] * 3, [0] * 3)
    S, off = oracle.plan(d, 4, 128)
    assert S == 512
    assert list(off) == [0, 1024, 1408]


def test_one_rank_holds_everything_contiguously():
    d = oracle.Desc([4, 3], [8, 5], [W.GRAN_ROWS, W.GRAN_ELEM], [2, 0], [0, 0])
    S, off = oracle.plan(d, 1, 4)
    assert list(off) == [0, 32] and S == 48


def load_closed_forms():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, N, m, g, lb, S, pad = line.split()
        rows.append((name, int(N), int(m), int(g), int(lb), int(S), float(pad)))
    return rows


@pytest.mark.parametrize("row", load_closed_forms(), ids=lambda r: r[0])
def test_closed_form_workloads(row):
    name, N, m, g, lb, S_star, pad = row
    w = W.get(name)
    assert (w.numel, w.m, w.g_coll) == (N, m, g)
    d = oracle.Desc.from_workload(w)
    for policy in (oracle.ORDER_DEFAULT, oracle.ORDER_BLOCK, oracle.ORDER_SHAPE):
        S, off = oracle.plan(d, m, g, policy)
        assert S == S_star
        check_invariants(d, m, g, S, off)
    assert abs((1 - N / (m * S_star)) - pad) < 5e-5


def test_llama_layer_invariants_and_bound():
    w = W.llama_layer()
    d = oracle.Desc.from_workload(w)
    S, off = oracle.plan(d, w.m, w.g_coll)
    check_invariants(d, w.m, w.g_coll, S, off)
    assert S >= 25297920


def test_tiny_bruteforce_report():
    w = W.tiny()
    d = oracle.Desc.from_workload(w)
    S_def, off = oracle.plan(d, w.m, w.g_coll)
    S_opt, order = oracle.bruteforce_S(d, w.m, w.g_coll)
    check_invariants(d, w.m, w.g_coll, S_def, off)
    assert S_opt <= S_def
    assert S_def >= 53504


def test_qblocks_tile_the_tensors():
    """Quantisation blocks cover every real element once and never cross a rank."""
    for name in ("tiny", "llama_layer", "dsv3_block"):
        w = W.get(name)
        d = oracle.Desc.from_workload(w)
        S, off = oracle.plan(d, w.m, w.g_coll)
        qb = oracle.qblocks(d, w.g_coll, off)
        cover = {}
        for q in range(len(qb["base"])):
            t = int(qb["tensor"][q])
            first = int(qb["base"][q])
            last = first + (int(qb["nrows"][q]) - 1) * int(qb["stride"][q]) + int(qb["ncols"][q]) - 1
            assert first // S == last // S, "quant block crosses a rank boundary"
            cover[t] = cover.get(t, 0) + int(qb["nrows"][q]) * int(qb["ncols"][q])
        assert [cover[t] for t in range(d.n)] == [int(x) for x in d.rows * d.cols]
    w = W.tiny()
    d = oracle.Desc.from_workload(w)
    S, off = oracle.plan(d, w.m, w.g_coll)
    assert len(oracle.qblocks(d, w.g_coll, off)["base"]) == 8 + 8 + 128 + 1
