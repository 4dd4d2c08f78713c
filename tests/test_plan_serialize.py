"""Checkpointing a plan through the C ABI (vsf_plan_serialize /
vsf_plan_deserialize), host only.

A serialized plan holds the planner's inputs (descriptors, m, g_coll, the
order policy used), the rank window and the forced kernel shape, plus the S
and offsets they produced; loading plans again and checks the layout. The
checks here: a round trip gives the same layout and tables on every
workload, also for a rank window, a forced shape and the best-of-three
order; a corrupted, truncated or foreign buffer is refused with an argument
error; a buffer whose stored layout differs from what the planner gives is
refused with a state error.
"""
import ctypes
import struct

import numpy as np
import pytest

from fsdp_buffer_layout_gb300 import vsf as V
from synth import workloads as W

HEADER = struct.Struct("<IIiiqiiiiq")  # magic, version, n, m, g_coll, order, r0, r1, warps, S


def _plan(w, order=V.VSF_ORDER_DEFAULT):
    return V.vsf_plan_create([V.make_desc(t.shape, t.gran, t.block_rows, t.tile_cols)
                              for t in w.tensors], w.m, w.g_coll, order)


def _layout(plan, n):
    info = V.vsf_plan_get_info(plan)
    nq = info.n_qblocks
    tables = [np.array(a) for a in V.vsf_plan_qblocks(plan, nq)] if nq else []
    return (info.S, info.total, info.real, nq, info.rank_begin, info.rank_end, info.bulk_warps,
            info.order_used, tuple(V.vsf_plan_offsets(plan, n)), tables)


def _same(a, b):
    assert a[:9] == b[:9]
    assert len(a[9]) == len(b[9]) and all(np.array_equal(x, y) for x, y in zip(a[9], b[9]))


def _fnv1a(data: bytes) -> int:
    h = 0xcbf29ce484222325
    for c in data:
        h ^= c
        h = (h * 0x100000001b3) & 0xffffffffffffffff
    return h


def _reseal(body: bytes) -> bytes:
    return body + struct.pack("<Q", _fnv1a(body))


@pytest.mark.parametrize("name", sorted(W.ALL))
def test_round_trip_gives_the_same_layout(name):
    w = W.get(name)
    p = _plan(w)
    try:
        data = V.vsf_plan_serialize(p)
        q = V.vsf_plan_deserialize(data)
        try:
            _same(_layout(p, len(w.tensors)), _layout(q, len(w.tensors)))
            assert V.vsf_plan_serialize(q) == data
        finally:
            V.vsf_plan_destroy(q)
    finally:
        V.vsf_plan_destroy(p)


def test_window_forced_shape_and_best_of_three_survive():
    w = W.llama_layer()
    p = _plan(w, V.VSF_ORDER_BEST3)
    try:
        V.vsf_plan_restrict(p, 2, 5)
        V.vsf_plan_set_bulk_warps(p, 4)
        q = V.vsf_plan_deserialize(V.vsf_plan_serialize(p))
        try:
            a, b = _layout(p, len(w.tensors)), _layout(q, len(w.tensors))
            _same(a, b)
            assert b[4:7] == (2, 5, 4)
        finally:
            V.vsf_plan_destroy(q)
    finally:
        V.vsf_plan_destroy(p)


def test_size_query_and_small_buffer():
    p = _plan(W.tiny())
    try:
        L = V.lib()
        need = ctypes.c_size_t(0)
        assert L.vsf_plan_serialize(p, None, ctypes.byref(need)) == V.VSF_OK
        n = len(W.tiny().tensors)
        assert need.value == HEADER.size + n * (ctypes.sizeof(V.vsf_tensor_desc) + 8) + 8
        small = ctypes.c_size_t(need.value - 1)
        buf = ctypes.create_string_buffer(need.value)
        assert L.vsf_plan_serialize(p, buf, ctypes.byref(small)) == V.VSF_ERR_ARG
        assert small.value == need.value
        assert L.vsf_plan_serialize(None, buf, ctypes.byref(small)) == V.VSF_ERR_ARG
    finally:
        V.vsf_plan_destroy(p)


def _refused(data: bytes, status: int):
    with pytest.raises(V.VsfError) as e:
        q = V.vsf_plan_deserialize(data)
        V.vsf_plan_destroy(q)
    assert e.value.status == status


def test_damaged_buffers_are_refused():
    p = _plan(W.tiny())
    try:
        data = V.vsf_plan_serialize(p)
    finally:
        V.vsf_plan_destroy(p)
    flipped = bytearray(data)
    flipped[HEADER.size + 20] ^= 0x40  # inside a descriptor: checksum no longer matches
    _refused(bytes(flipped), V.VSF_ERR_ARG)
    _refused(data[:-1], V.VSF_ERR_ARG)
    _refused(data[:10], V.VSF_ERR_ARG)
    _refused(b"\0" * len(data), V.VSF_ERR_ARG)
    fields = list(HEADER.unpack_from(data))
    fields[1] = 2  # a version this library does not know, resealed
    _refused(_reseal(HEADER.pack(*fields) + data[HEADER.size:-8]), V.VSF_ERR_ARG)
    fields = list(HEADER.unpack_from(data))
    fields[2] += 1  # tensor count that does not match the size
    _refused(_reseal(HEADER.pack(*fields) + data[HEADER.size:-8]), V.VSF_ERR_ARG)


def test_stored_layout_that_the_planner_does_not_give_is_refused():
    p = _plan(W.tiny())
    try:
        data = V.vsf_plan_serialize(p)
        S = V.vsf_plan_get_info(p).S
    finally:
        V.vsf_plan_destroy(p)
    fields = list(HEADER.unpack_from(data))
    fields[9] = S + 128  # another S
    _refused(_reseal(HEADER.pack(*fields) + data[HEADER.size:-8]), V.VSF_ERR_STATE)
    body = bytearray(data[:-8])
    off = len(body) - 8  # the last tensor's offset
    struct.pack_into("<q", body, off, struct.unpack_from("<q", body, off)[0] + 128)
    _refused(_reseal(bytes(body)), V.VSF_ERR_STATE)
