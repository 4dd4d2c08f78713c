"""The Newton–Schulz product of distributed Muon (vsf_ns_gemm, the tcgen05
tensor-core kernel inside vsf_muon_step) through the C ABI, against the same
product computed in fp64 on the CPU.

D = alpha * opA opB^T + beta * C with bf16 operands, fp32 accumulation and one
bf16 rounding. For every element the error is bounded by the fp32
accumulation error of a K-term dot product, gamma_K * sum_k |a_k b_k| with
gamma_K = K 2^-24 / (1 - K 2^-24) (Higham, Accuracy and Stability of
Numerical Algorithms, 2nd ed., eq. 3.5), taken twice because the tensor
cores' adder need not round to nearest, times |alpha|, plus the rounding of
alpha * acc and of the fused add, plus the final bf16 rounding (half a bf16
ulp, 2^-9 relative). A wrong operand layout, a dropped K slice or a
transposed tile fails it by orders of magnitude.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def _op(mat: torch.Tensor, mn: bool) -> torch.Tensor:
    """The logical operand (rows = M or N, columns = K) of a stored matrix."""
    return mat.transpose(-1, -2) if mn else mat


def _run(a_mn, b_mn, sym, M, N, K, batch, alpha, beta, seed, ld_pad=0, same=False):
    from fsdp_buffer_layout_gb300 import vsf as V
    g = torch.Generator().manual_seed(seed)
    # stored shapes: K-major operand rows x K, MN-major K x rows; ld_pad extra columns
    a_shape = (K, M) if a_mn else (M, K)
    b_shape = (K, N) if b_mn else (N, K)
    A = torch.randn(batch, a_shape[0], a_shape[1] + ld_pad, generator=g) * 0.5
    B = A if same else torch.randn(batch, b_shape[0], b_shape[1] + ld_pad, generator=g) * 0.5
    C = torch.randn(batch, M, N + ld_pad, generator=g)
    if sym:
        C = C[..., :N]
        C = (C + C.transpose(-1, -2)) * 0.5
        C = torch.cat([C, torch.zeros(batch, M, ld_pad)], dim=-1)
    Ab, Bb, Cb = _bf16(A), _bf16(B), _bf16(C)
    dA, dB, dC = Ab.cuda(), Bb.cuda(), Cb.cuda()
    D = torch.full((batch, M, N + ld_pad), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lda, ldb, ldc, ldd = A.shape[-1], B.shape[-1], C.shape[-1], D.shape[-1]
    V.vsf_ns_gemm(a_mn, b_mn, sym, M, N, K, batch, dA.data_ptr(), lda, dA[0].numel(),
                  dB.data_ptr(), ldb, dB[0].numel(), alpha, beta,
                  dC.data_ptr() if beta != 0.0 else None, ldc, dC[0].numel(), D.data_ptr(), ldd,
                  D[0].numel(), err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "a bounded wait of the GEMM ran out"
    assert torch.isnan(D.float()[..., N:]).all(), "wrote into the leading-dimension padding"
    got = D.float().cpu()[..., :N].double()
    opA = _op(Ab.double()[..., :a_shape[1]], a_mn)
    opB = _op(Bb.double()[..., :b_shape[1]], b_mn)
    exact = alpha * (opA @ opB.transpose(-1, -2)) + beta * Cb.double()[..., :N]
    absprod = abs(alpha) * (opA.abs() @ opB.abs().transpose(-1, -2))
    u = 2.0 ** -24
    gamma = K * u / (1 - K * u)
    bound = (2 * gamma + 3 * u) * absprod + 2 * u * abs(beta) * Cb.double()[..., :N].abs() \
        + 2.0 ** -8 * exact.abs() + 1e-30
    diff = (got - exact).abs()
    assert torch.isfinite(got).all(), "unwritten or non-finite outputs"
    worst = (diff / bound).max().item()
    assert worst <= 1.0, f"error {worst:.3g} x the bound"
    if sym:
        assert torch.equal(got, got.transpose(-1, -2)), "symmetric product not exactly symmetric"
    return got


# (a_mn, b_mn, sym): the four layouts Newton–Schulz uses
@pytest.mark.parametrize("M,K,batch", [(200, 1000, 2), (128, 64, 1), (1024, 2048, 3),
                                       (1000, 72, 1)])
def test_gram_wide_k_major_symmetric(M, K, batch):
    """A = X X^T: both operands the rows of X (K-major), half the tiles."""
    _run(False, False, True, M, M, K, batch, 1.0, 0.0, seed=M + K, same=True)


@pytest.mark.parametrize("M,K,batch", [(200, 1000, 2), (1024, 2048, 2), (300, 130, 1)])
def test_gram_tall_mn_major_symmetric(M, K, batch):
    """A = X^T X: both operands the columns of X (MN-major)."""
    _run(True, True, True, M, M, K, batch, 1.0, 0.0, seed=7 * M + K, same=True)


@pytest.mark.parametrize("n,batch", [(200, 2), (768, 1), (1024, 2)])
def test_square_of_symmetric_with_scaled_add(n, batch):
    """B = c A A + b A on a symmetric A (K-major rows on both sides)."""
    from oracle import muon
    g = torch.Generator().manual_seed(n)
    X = torch.randn(batch, n, 3 * n // 2, generator=g)
    A = X @ X.transpose(-1, -2) / n
    # the operand is symmetric; the same storage serves as opA, opB and C
    from fsdp_buffer_layout_gb300 import vsf as V
    Ab = _bf16(A).cuda()
    D = torch.empty_like(Ab)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, b, c = muon.NS_COEFFS
    V.vsf_ns_gemm(False, False, True, n, n, n, batch, Ab.data_ptr(), n, n * n, Ab.data_ptr(), n,
                  n * n, c, b, Ab.data_ptr(), n, n * n, D.data_ptr(), n, n * n, err.data_ptr(),
                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    A64 = Ab.double().cpu()
    exact = c * (A64 @ A64) + b * A64
    got = D.double().cpu()
    u = 2.0 ** -24
    bound = (2 * n * u / (1 - n * u) + 3 * u) * abs(c) * (A64.abs() @ A64.abs()) \
        + 2 * u * abs(b) * A64.abs() + 2.0 ** -8 * exact.abs() + 1e-30
    assert ((got - exact).abs() / bound).max().item() <= 1.0
    assert torch.equal(got, got.transpose(-1, -2))


@pytest.mark.parametrize("M,N,K,batch", [(200, 1000, 200, 2), (1024, 2048, 1024, 2),
                                         (130, 520, 130, 1)])
def test_update_wide_k_by_mn(M, N, K, batch):
    """X' = a X + B X: opA = B's rows (K-major), opB = X's columns (MN-major)."""
    _run(False, True, False, M, N, K, batch, 1.0, 3.4445, seed=M * 3 + N)


@pytest.mark.parametrize("M,N,K,batch", [(1000, 200, 200, 2), (2048, 1024, 1024, 2),
                                         (333, 96, 96, 3)])
def test_update_tall_k_by_k(M, N, K, batch):
    """X' = a X + X B: opA = X's rows, opB = B's rows (both K-major)."""
    _run(False, False, False, M, N, K, batch, 1.0, 3.4445, seed=M + 5 * N)


LAYOUTS = [(False, False, True), (False, False, False), (True, True, True), (False, True, False)]


@pytest.mark.parametrize("layout", LAYOUTS)
def test_unaligned_leading_dimension_takes_the_cuda_core_kernel(layout):
    """Leading dimensions that are not multiples of 8 (K + 5 = 34, M + 5 = 50,
    N + 5 = 42) cannot be addressed by the tensor copies; the CUDA-core kernel
    has the same contract."""
    a_mn, b_mn, sym = layout
    M = 45
    N = M if sym else 37
    for ld in (29 + 5, M + 5, N + 5):
        assert ld % 8 != 0
    _run(a_mn, b_mn, sym, M, N, 29, 2, 1.0, 0.0 if sym else -0.5, seed=3, ld_pad=5, same=sym)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_padded_leading_dimension_on_the_tensor_cores(layout):
    """Rows padded beyond the matrix (K + 3 = 32, M + 3 = 48, N + 3 = 40: still
    multiples of 8): the tensor copies read only the logical extent, and
    nothing past it is written."""
    a_mn, b_mn, sym = layout
    M = 45
    N = M if sym else 37
    _run(a_mn, b_mn, sym, M, N, 29, 2, 1.0, 0.0 if sym else -0.5, seed=4, ld_pad=3, same=sym)


def test_alpha_scales_the_product():
    got1 = _run(False, False, False, 256, 256, 128, 1, 1.0, 0.0, seed=11)
    got2 = _run(False, False, False, 256, 256, 128, 1, -2.0, 0.0, seed=11)
    # -2 * x is exact in bf16 whenever x is
    assert torch.equal(got2, -2.0 * got1)
