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
    found by brute force.
"""
import itertools

import numpy as np
import pytest

from oracle import muon


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
    torch = pytest.importorskip("torch")
    x = (np.random.default_rng(4).standard_normal(10000) * 3).astype(np.float32)
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
