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
