"""TEST INFRASTRUCTURE: the plain CPU oracle of distributed Muon (numpy).

Only the test suite and the benchmark's CPU-baseline leg use this module; the
product library never imports it, and it imports nothing from the library.

Method: "veScale-FSDP: Flexible and High-Performance FSDP at Scale (MLSys
2026)" summary page, 结构感知训练 case study > 分布式 Muon (Algorithm 2):
SelectRoot() balances the matrices over ranks; Redistribute gathers a whole
2-D matrix on its root; the root runs Newton-Schulz; the result goes back to
the ragged shards; other ranks do nothing for that matrix. The pages give no
coefficients or op order. Readings used here (restating the public Muon
algorithm, Keller Jordan, 2024):
  - momentum mu = 0.95, Nesterov: M = mu M + g; U = g + mu M (fp32);
  - X0 = bf16(U * r), r = fp32(1 / (||U||_F + eps)), ||U||_F in fp64;
  - 5 quintic Newton-Schulz steps with (a, b, c) = (3.4445, -4.7750, 2.0315);
    a wide matrix (R <= C) uses A = X X^T, B = b A + c A A, X = a X + B X;
    a tall one the right-hand form A = X^T X, X = a X + X B, which equals
    transposing, iterating and transposing back; every product is exact (fp64)
    and each result is rounded to fp32 and then to bf16 (the GPU accumulates
    in fp32 and stores bf16);
  - update p = p (1 - lr wd) - fp32(lr sqrt(max(1, R/C))) O, then the bf16
    copy; tensors with more than 2 dims are batches of matrices (their
    leading dims index the matrices).
SelectRoot: longest-processing-time greedy over the Newton-Schulz FLOPs
(ties to the lower rank).
Parity status: the Newton-Schulz map is pinned to the SVD identity and to
the transpose identity in exact arithmetic; the momentum and update to the
closed form of two Nesterov steps, decoupled decay on a non-zero master and
the sqrt(R/C) scale of a tall matrix; the FLOP count to an iteration run with
counted products; SelectRoot to Graham's bound and his two-machine worst
case. The bf16 rounding points are a reading, pinned only by the output's
singular-value band.
"""
from __future__ import annotations

import math

import numpy as np

NS_COEFFS = (3.4445, -4.7750, 2.0315)


def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even), returned as fp32 values."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    # a NaN stays a NaN (the quiet NaN 0x7fc0; its bits are not compared)
    r = np.where(nan, np.uint64(0x7FC00000), r).astype(np.uint32)
    return r.view(np.float32)


def round_bf16(y: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (nearest even) -> bf16 (nearest even), as float64."""
    return bf16_from_f32(y.astype(np.float32)).astype(np.float64)


def newton_schulz(x0, steps: int = 5, coeffs=NS_COEFFS, exact: bool = False):
    """Quintic Newton-Schulz on one matrix (float64 array of bf16 values).
    exact=True skips every rounding (for the identities)."""
    a, b, c = coeffs
    rnd = (lambda y: y) if exact else round_bf16
    x = np.asarray(x0, dtype=np.float64)
    tall = x.shape[0] > x.shape[1]
    for _ in range(steps):
        A = rnd(x.T @ x) if tall else rnd(x @ x.T)
        B = rnd(c * (A @ A) + b * A)
        x = rnd(a * x + (x @ B if tall else B @ x))
    return x


def scalar_quintic(s, steps: int = 5, coeffs=NS_COEFFS):
    """The same iteration on one singular value: s -> a s + b s^3 + c s^5."""
    a, b, c = coeffs
    s = np.asarray(s, dtype=np.float64)
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def muon_matrix(g, M, p, step_hp, exact: bool = False):
    """One Muon step on one R x C matrix. g: bf16 values (fp32 array), M:
    fp32 momentum, p: fp32 master. Returns (M, p, bf16 bits, O). exact=True
    runs the Newton-Schulz iteration without its bf16 rounding (same X0): the
    distance between the two is the rounding noise of the bf16 iteration."""
    mu = np.float32(step_hp["momentum"])
    R, C = g.shape
    M = (mu * M + g).astype(np.float32)
    U = (g + mu * M).astype(np.float32)
    s = math.sqrt(float(np.sum(U.astype(np.float64) ** 2)))
    r = np.float32(1.0 / (s + step_hp["eps"]))
    X0 = bf16_from_f32((U * r).astype(np.float32)).astype(np.float64)
    O = newton_schulz(X0, step_hp["ns_steps"], (step_hp["ns_a"], step_hp["ns_b"],
                                                step_hp["ns_c"]), exact).astype(np.float32)
    decay = np.float32(1.0 - step_hp["lr"] * step_hp["weight_decay"])
    alpha = np.float32(step_hp["lr"] * math.sqrt(max(1.0, R / C)))
    p = (p * decay).astype(np.float32)
    p = (p - (alpha * O).astype(np.float32)).astype(np.float32)
    bits = bf16_from_f32(p).view(np.uint32) >> 16
    return M, p, bits.astype(np.uint16), O


def ns_flops(shape) -> float:
    """Newton-Schulz FLOPs of one step of a tensor (batch of matrices)."""
    *lead, R, C = shape
    n, k = min(R, C), max(R, C)
    per = 2.0 * n * n * k + 2.0 * n ** 3 + 2.0 * n * n * k
    return float(np.prod(lead, dtype=np.float64)) * per


def select_roots(loads, ranks: int):
    """Longest-processing-time greedy: tensors by load descending (ties by
    index), each to the least-loaded rank (ties to the lower rank)."""
    order = sorted(range(len(loads)), key=lambda i: (-loads[i], i))
    total = [0.0] * ranks
    root = [-1] * len(loads)
    for i in order:
        r = min(range(ranks), key=lambda j: (total[j], j))
        root[i] = r
        total[r] += loads[i]
    return root, total
