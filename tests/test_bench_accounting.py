"""The benchmark's accounting, against the stated per-element figures.

Algorithmic bytes per real element of the shard step (bf16 gradients): pack
2 read + 2 written, 8-bit AdamW 2 + 1 + 1 + 4 read and 1 + 1 + 4 + 2 written
plus 16 bytes of scales per quantisation block, unpack 2 + 2: 24 in all. With
fp32 gradients pack moves 8 and AdamW 18 (30 in all); in zero-copy mode the
step is the norm's read of the packed gradient plus AdamW (18). Muon's
executed share of a symmetric product: the 256 x 256 output tiles (one per
CTA pair) of the library's tensor-core kernel that hold an element on or
above the diagonal (checked by brute force), with the tile shape the
library's own.
"""
import os
import re

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("grad_bytes,zero_copy,per_elem", [(2, False, 24), (4, False, 30),
                                                          (2, True, 18)])
def test_algorithmic_bytes_per_element(grad_bytes, zero_copy, per_elem):
    N, Q = 1_000_003, 977
    b = bench.algorithmic_bytes(N, Q, grad_bytes=grad_bytes, zero_copy=zero_copy)
    assert b["step"] == per_elem * N + 16 * Q
    assert b["step"] == b["pack"] + b["adam"] + b["unpack"]
    assert b["adam"] == (grad_bytes + 14) * N + 16 * Q


def _sym_tiles_brute(n, bm=256, bn=256):
    """Tiles of an n x n output (bm x bn) that hold an element (i, j) with i <= j."""
    count = 0
    for I in range(-(-n // bm)):
        for J in range(-(-n // bn)):
            if any(i <= j for i in range(I * bm, min(n, I * bm + bm))
                   for j in (min(n, J * bn + bn) - 1,)):
                count += 1
    return count


@pytest.mark.parametrize("n", [32, 100, 128, 200, 256, 300, 1000, 2048, 2880, 4096])
def test_symmetric_tiles_are_those_touching_the_upper_triangle(n):
    assert bench.sym_tiles(n) == _sym_tiles_brute(n)
    assert 0.5 <= bench.sym_fraction(n) <= 1.0


def test_tile_shape_is_the_librarys():
    src = open(os.path.join(ROOT, "fsdp_buffer_layout_gb300", "csrc", "ns_gemm.cuh")).read()
    # kGemmBM is one CTA's half of the pair's tile
    bm = 2 * int(re.search(r"constexpr int kGemmBM = (\d+);", src).group(1))
    bn = int(re.search(r"constexpr int kGemmBN = (\d+);", src).group(1))
    assert (bench.GEMM_BM, bench.GEMM_BN) == (bm, bn)
    assert bench.sym_fraction(4096) == 136 / 256
