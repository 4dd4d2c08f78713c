"""The benchmark's accounting, against the stated per-element figures.

Algorithmic bytes per real element of the shard step (bf16 gradients): pack
2 read + 2 written, 8-bit AdamW 2 + 1 + 1 + 4 read and 1 + 1 + 4 + 2 written
plus 16 bytes of scales per quantisation block, unpack 2 + 2: 24 in all. With
fp32 gradients pack moves 8 and AdamW 18 (30 in all); in zero-copy mode the
step is the norm's read of the packed gradient plus AdamW (18). Muon's
executed share of a symmetric product: 1 below n = 1024 (or when n is not a
multiple of 16), 3/4 with one level of blocks (n = 1024..4095), 5/8 with two
(n >= 4096), with the blocking threshold the library's own.
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


@pytest.mark.parametrize("n,frac", [(512, 1.0), (1000, 1.0), (1024, 0.75), (2048, 0.75),
                                    (4080, 0.75), (4096, 0.625), (8192, 0.625)])
def test_symmetric_blocking_share(n, frac):
    assert bench.sym_fraction(n) == frac


def test_blocking_threshold_is_the_librarys():
    src = open(os.path.join(ROOT, "fsdp_buffer_layout_gb300", "csrc", "muon.cu")).read()
    lib_min = int(re.search(r"constexpr int64_t kSymBlockMin = (\d+);", src).group(1))
    lib_levels = int(re.search(r"#define VSF_SYM_LEVELS (\d+)", src).group(1))
    assert bench.SYM_BLOCK_MIN == lib_min
    # sym_fraction splits at most twice: one level more would reach 9/16 at 8192
    assert lib_levels == 2 and bench.sym_fraction(8192) == 0.625
