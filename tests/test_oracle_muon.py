"""Pins of the Muon oracle (oracle/muon.py) against things other than itself.

Method: "veScale-FSDP: Flexible and High-Performance FSDP at Scale (MLSys
2026)" summary page, 结构感知训练 case study > 分布式 Muon (Algorithm 2).
  - SVD identity: in exact arithmetic the matrix iteration acts on each
    singular value alone, NS(X) = U p(S) V^T with p the scalar quintic
    (numpy's SVD is the library routine);
  - transpose identity: the tall (right-hand) form equals transposing,
    iterating and transposing back;
  - band: with bf16 rounding the output's singular values stay in [0.5, 1.5];
  - SelectRoot's greedy: within Graham's (4/3 - 1/(3m)) bound of the optimum
    found by brute force, and Graham's own worst case for two machines;
  - momentum and update: the closed form of two Nesterov steps, decoupled
    weight decay on a non-zero master, the sqrt(R/C) scale of a tall matrix;
  - FLOPs: numpy's einsum_path count of the three products of an iteration.
"""
import importlib.util
import itertools
import math
import os

import numpy as np
import pytest

if os.environ.get("ORACLE_MUON"):  # a planted-mistake copy (tests/test_oracle_mutants.py)
    _spec = importlib.util.spec_from_file_location("muon_mutant", os.environ["ORACLE_MUON"])
    muon = importlib.util.module_from_spec(_spec)
    _spec.loader.exec_module(muon)
else:
    from oracle import muon

HP = dict(lr=0.02, momentum=0.95, weight_decay=0.01, eps=1e-7, ns_steps=5,
          ns_a=3.4445, ns_b=-4.7750, ns_c=2.0315)


def _grad(rng, shape):
    return muon.bf16_from_f32((rng.standard_normal(shape) * 1e-3).astype(np.float32))


@pytest.mark.parametrize("shape", [(48, 80), (80, 48), (64, 64)])
def test_svd_identity_exact(shape):
    rng = np.random.default_rng(0)
    g = rng.standard_normal(shape)
    x0 = g / np.linalg.norm(g)
    got = muon.newton_schulz(x0, exact=True)
    U, s, Vt = np.linalg.svd(x0, full_matrices=False)
    want = (U * muon.scalar_quintic(s)) @ Vt
    assert np.abs(got - want).max() < 1e-10


def test_tall_form_is_transposed_wide_form():
    rng = np.random.default_rng(1)
    x0 = rng.standard_normal((96, 40))
    x0 /= np.linalg.norm(x0)
    assert np.abs(muon.newton_schulz(x0, exact=True)
                  - muon.newton_schulz(x0.T, exact=True).T).max() < 1e-12


@pytest.mark.parametrize("shape", [(64, 128), (128, 64), (96, 96)])
def test_bf16_output_singular_values_in_band(shape):
    rng = np.random.default_rng(2)
    g = rng.standard_normal(shape).astype(np.float32)
    x0 = muon.bf16_from_f32(g / np.float32(np.linalg.norm(g))).astype(np.float64)
    s = np.linalg.svd(muon.newton_schulz(x0), compute_uv=False)
    assert 0.5 <= s.min() and s.max() <= 1.5


def test_scalar_quintic_fixed_band():
    s = muon.scalar_quintic(np.linspace(0.05, 1.0, 200))
    assert s.min() > 0.5 and s.max() < 1.3


def test_bf16_rounding_matches_torch():
    """Random values, and exact ties (low 16 bits 0x8000) with an even and an
    odd bf16 neighbour below, of both signs: round half to even."""
    torch = pytest.importorskip("torch")
    x = (np.random.default_rng(4).standard_normal(10000) * 3).astype(np.float32)
    hi = np.random.default_rng(5).integers(0x0080, 0x7F00, 2000, dtype=np.uint32)
    ties = ((hi << 16) | 0x8000).astype(np.uint32)
    ties = np.concatenate([ties, ties | 0x80000000]).view(np.float32)
    assert (hi & 1).min() == 0 and (hi & 1).max() == 1
    x = np.concatenate([x, ties])
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(muon.bf16_from_f32(x), want)


@pytest.mark.parametrize("seed", range(30))
def test_select_roots_within_graham_bound(seed):
    rng = np.random.default_rng(seed)
    loads = [float(x) for x in rng.integers(1, 50, size=int(rng.integers(2, 8)))]
    ranks = int(rng.integers(2, 4))
    root, total = muon.select_roots(loads, ranks)
    assert sorted(set(root)) == sorted(set(root)) and all(0 <= r < ranks for r in root)
    assert abs(sum(total) - sum(loads)) < 1e-9
    opt = min(max(sum(l for l, r in zip(loads, a) if r == k) for k in range(ranks))
              for a in itertools.product(range(ranks), repeat=len(loads)))
    assert max(total) <= (4 / 3 - 1 / (3 * ranks)) * opt + 1e-9


def test_muon_step_one_matrix_shapes_and_decay():
    rng = np.random.default_rng(5)
    g = muon.bf16_from_f32((rng.standard_normal((32, 64)) * 1e-3).astype(np.float32))
    hp = dict(lr=0.02, momentum=0.95, weight_decay=0.01, eps=1e-7, ns_steps=5,
              ns_a=3.4445, ns_b=-4.7750, ns_c=2.0315)
    M, p, bits, O = muon.muon_matrix(g, np.zeros_like(g), np.zeros_like(g), hp)
    assert np.array_equal(M, g)  # first step: momentum = gradient
    assert np.allclose(p, -np.float32(0.02) * O)  # zero master: the update alone
    s = np.linalg.svd(O.astype(np.float64), compute_uv=False)
    assert 0.5 <= s.min() and s.max() <= 1.5


def test_two_nesterov_steps_closed_form():
    """M1 = g1, M2 = mu g1 + g2, so U2 = g2 + mu M2 = (1 + mu) g2 + mu^2 g1.
    Step 2's exact-iteration output must be NS(U2 / ||U2||) up to the bf16
    rounding of X0 (2^-9 relative): 0.002 here, against 0.4 with the
    Nesterov term dropped."""
    rng = np.random.default_rng(7)
    g1, g2 = _grad(rng, (32, 64)), _grad(rng, (32, 64))
    z = np.zeros_like(g1)
    M1, p1, _, _ = muon.muon_matrix(g1, z, z, HP)
    M2, _, _, O2 = muon.muon_matrix(g2, M1, p1, HP, exact=True)
    mu = HP["momentum"]
    assert np.abs(M2 - (mu * g1.astype(np.float64) + g2)).max() < 1e-9
    U = (1 + mu) * g2.astype(np.float64) + mu * mu * g1.astype(np.float64)
    ref = muon.newton_schulz(U / np.linalg.norm(U), exact=True)
    assert np.linalg.norm(O2 - ref) / np.linalg.norm(ref) < 0.02


@pytest.mark.parametrize("shape", [(64, 32), (32, 64)])
def test_decay_and_shape_scale(shape):
    """Decoupled weight decay on a master of order 1, and the update scaled by
    sqrt(max(1, R/C)): sqrt(2) for the tall matrix, 1 for the wide one. The
    fp32 roundings are far below both effects (lr wd = 2e-4, (sqrt 2 - 1) lr)."""
    rng = np.random.default_rng(8)
    g = _grad(rng, shape)
    p0 = rng.uniform(0.5, 1.5, shape).astype(np.float32)
    _, p1, _, O = muon.muon_matrix(g, np.zeros_like(g), p0, HP)
    R, C = shape
    want = (p0.astype(np.float64) * (1 - HP["lr"] * HP["weight_decay"])
            - HP["lr"] * math.sqrt(max(1.0, R / C)) * O.astype(np.float64))
    assert np.abs(p1 - want).max() < 1e-6


def test_select_roots_graham_worst_case():
    """Graham's worst case of longest-processing-time for two machines: loads
    3, 3, 2, 2, 2 (given here out of order) end at 7 and 5 against an optimum
    of 6. Ties go to the lower rank."""
    root, total = muon.select_roots([2.0, 3.0, 2.0, 3.0, 2.0], 2)
    assert total == [7.0, 5.0]
    assert root == [0, 0, 1, 1, 0]


class _CountingProducts:
    """Matrix products by explicit loops, counting one multiply and one add
    per term."""

    def __init__(self):
        self.flops = 0

    def mm(self, a, b):
        p, q = a.shape
        r = b.shape[1]
        out = np.zeros((p, r))
        for i in range(p):
            for j in range(r):
                acc = 0.0
                for l in range(q):
                    acc += a[i, l] * b[l, j]
                    self.flops += 2
                out[i, j] = acc
        return out


@pytest.mark.parametrize("shape", [(3, 5), (5, 3), (4, 4), (2, 3, 5)])
def test_ns_flops_counts_the_products_of_one_iteration(shape):
    """One exact quintic iteration run with counted loop products (the
    Gram matrix of the smaller side, A A, then B X or X B) must give the
    oracle's one-iteration result, and its count must equal ns_flops."""
    *lead, R, C = shape
    a, b, c = muon.NS_COEFFS
    rng = np.random.default_rng(9)
    cp = _CountingProducts()
    for _ in range(math.prod(lead)):
        x = rng.standard_normal((R, C))
        x /= np.linalg.norm(x)
        if R > C:
            A = cp.mm(x.T, x)
            B = c * cp.mm(A, A) + b * A
            y = a * x + cp.mm(x, B)
        else:
            A = cp.mm(x, x.T)
            B = c * cp.mm(A, A) + b * A
            y = a * x + cp.mm(B, x)
        assert np.abs(y - muon.newton_schulz(x, steps=1, exact=True)).max() < 1e-12
    assert muon.ns_flops(shape) == cp.flops
