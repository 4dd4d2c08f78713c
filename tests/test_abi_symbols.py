"""libvsf.so loads without a GPU and exports every function include/vsf.h declares."""
import ctypes
import os
import re

import pytest

from fsdp_buffer_layout_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "vsf.h")


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vsf_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ctypes.CDLL(_build.LIB)


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), f"{n} missing from libvsf.so"


def test_status_strings(lib):
    lib.vsf_status_string.restype = ctypes.c_char_p
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert lib.vsf_status_string(s)


def test_per_step_calls_reject_unuploaded_plan():
    from fsdp_buffer_layout_gb300 import vsf as V
    p = V.vsf_plan_create([V.make_desc((64, 64), V.VSF_GRAN_ROWS, 8)], 2, 128)
    try:
        with pytest.raises(V.VsfError) as e:
            V.vsf_pack(p, [256], V.VSF_BF16, 256, 0)
        assert e.value.status == V.VSF_ERR_STATE
    finally:
        V.vsf_plan_destroy(p)


def test_wait_selftest_refuses_a_limit_above_one_second():
    """Host-side argument check of the bounded-wait self-test (no launch)."""
    from fsdp_buffer_layout_gb300 import vsf as V
    with pytest.raises(V.VsfError) as e:
        V.vsf_selftest_wait_timeout(1 << 20, 2_000_000_000, 0)
    assert e.value.status == V.VSF_ERR_ARG


def test_device_copy_rejects_bad_arguments_before_any_launch():
    """The copy-ceiling kernel's host checks: NULL pointers, a size that is not
    a multiple of 16 bytes, misaligned pointers; a zero size is a no-op."""
    from fsdp_buffer_layout_gb300 import vsf as V
    for dst, src, n, want in ((0, 256, 16, V.VSF_ERR_ARG), (256, 0, 16, V.VSF_ERR_ARG),
                              (256, 512, 24, V.VSF_ERR_ARG), (264, 512, 32, V.VSF_ERR_ALIGN),
                              (256, 520, 32, V.VSF_ERR_ALIGN)):
        with pytest.raises(V.VsfError) as e:
            V.vsf_device_copy(dst, src, n, 0)
        assert e.value.status == want, (dst, src, n)
    V.vsf_device_copy(256, 512, 0, 0)  # nothing to copy, nothing launched


def test_ns_gemm_rejects_bad_arguments_before_any_launch():
    """vsf_ns_gemm's host checks: NULL operands, a missing C with beta != 0,
    unsupported operand layouts, symmetric products of unequal sides, sizes
    out of range."""
    from fsdp_buffer_layout_gb300 import vsf as V
    ok = dict(a_mn=False, b_mn=False, sym=False, M=64, N=64, K=64, batch=1, A=256, lda=64,
              sa=4096, B=256, ldb=64, sb=4096, alpha=1.0, beta=0.0, C=None, ldc=64, sc=4096,
              D=1 << 20, ldd=64, sd=4096, d_err=512, stream=0)
    bad = [dict(A=0), dict(D=0), dict(d_err=0), dict(beta=1.0),
           dict(a_mn=True, b_mn=False),              # MN x K is not a supported layout
           dict(a_mn=True, b_mn=True, sym=False),    # MN x MN only for symmetric products
           dict(sym=True, N=32),                     # symmetric needs M = N
           dict(M=0), dict(K=0), dict(batch=0), dict(batch=70000), dict(lda=0)]
    for change in bad:
        args = dict(ok, **change)
        with pytest.raises(V.VsfError) as e:
            V.vsf_ns_gemm(**args)
        assert e.value.status == V.VSF_ERR_ARG, change
