"""TEST INFRASTRUCTURE: Python access to the plain CPU oracle (``oracle.cpp``).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg use this package. The product library never imports it, and it
never imports the product library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GRAN_ELEM, GRAN_ROWS, GRAN_TILE = 0, 1, 2
ORDER_DEFAULT, ORDER_BLOCK, ORDER_SHAPE, ORDER_BEST3 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile liboracle.so (single thread, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", _SRC, "-o", _LIB_PATH + ".tmp"],
                   check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return None if a is None else a.ctypes.data


def lib():
    """The oracle library: liboracle.so, built on first use, or the library
    named by ORACLE_LIBRARY (the mutation test's planted-mistake builds)."""
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(os.environ.get("ORACLE_LIBRARY") or build())
            vp, i64, i32, dbl, c_int = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                        ctypes.c_double, ctypes.c_int)
            desc = [c_int, vp, vp, vp, vp, vp]
            L.orc_atoms.restype = c_int
            L.orc_atoms.argtypes = desc + [i64, vp, vp]
            L.orc_plan.restype = c_int
            L.orc_plan.argtypes = desc + [i64, i64, c_int, vp, vp, vp]
            L.orc_bruteforce_S.restype = i64
            L.orc_bruteforce_S.argtypes = desc + [i64, i64, vp]
            L.orc_exhaustive_S.restype = i64
            L.orc_exhaustive_S.argtypes = desc + [i64, i64, i64]
            L.orc_qblocks.restype = i64
            L.orc_qblocks.argtypes = desc + [i64, vp, vp, vp, vp, vp, vp]
            L.orc_pack.restype = None
            L.orc_pack.argtypes = [c_int, vp, vp, vp, c_int, vp]
            L.orc_unpack.restype = None
            L.orc_unpack.argtypes = [c_int, vp, vp, vp, c_int, vp]
            L.orc_sumsq.restype = dbl
            L.orc_sumsq.argtypes = [c_int, vp, vp, c_int]
            L.orc_factor.restype = ctypes.c_float
            L.orc_factor.argtypes = [dbl, c_int, dbl, vp]
            L.orc_adam_block.restype = None
            L.orc_adam_block.argtypes = [i64, vp, c_int, ctypes.c_float, c_int, vp, vp, vp, vp,
                                         vp, vp, vp, vp, dbl, dbl, dbl, dbl, dbl, c_int]
            L.orc_adam_all.restype = None
            L.orc_adam_all.argtypes = [i64, vp, vp, vp, vp, vp, c_int, ctypes.c_float, c_int,
                                       vp, vp, vp, vp, vp, vp, dbl, dbl, dbl, dbl, dbl, c_int]
            L.orc_quantize_m.argtypes = [i64, vp, vp, vp, vp]
            L.orc_quantize_v.argtypes = [i64, vp, vp, vp, vp]
            L.orc_group_op.restype = None
            L.orc_group_op.argtypes = [c_int, c_int, vp, vp, vp, c_int, vp, c_int, ctypes.c_float]
            L.orc_bf16_round.restype = ctypes.c_uint16
            L.orc_bf16_round.argtypes = [ctypes.c_float]
            _lib = L
    return _lib


class Desc:
    """Flat descriptor arrays for a list of (rows, cols, gran, block_rows, tile_cols)."""

    def __init__(self, rows, cols, gran, block_rows, tile_cols):
        self.rows = np.ascontiguousarray(rows, dtype=np.int64)
        self.cols = np.ascontiguousarray(cols, dtype=np.int64)
        self.gran = np.ascontiguousarray(gran, dtype=np.int32)
        self.block_rows = np.ascontiguousarray(block_rows, dtype=np.int64)
        self.tile_cols = np.ascontiguousarray(tile_cols, dtype=np.int64)
        self.n = len(self.rows)

    @classmethod
    def from_workload(cls, w):
        return cls([t.rows for t in w.tensors], [t.cols for t in w.tensors],
                   [t.gran for t in w.tensors], [t.block_rows for t in w.tensors],
                   [t.tile_cols for t in w.tensors])

    def args(self):
        return (self.n, _p(self.rows), _p(self.cols), _p(self.gran), _p(self.block_rows),
                _p(self.tile_cols))

    @property
    def numel(self):
        return self.rows * self.cols


def atoms(d: Desc, g_coll: int):
    block = np.zeros(d.n, np.int64)
    align = np.zeros(d.n, np.int64)
    if lib().orc_atoms(*d.args(), g_coll, _p(block), _p(align)) != 0:
        raise ValueError("bad descriptor")
    return block, align


def plan(d: Desc, m: int, g_coll: int, policy: int = ORDER_DEFAULT, order=None):
    """Returns (S, offsets)."""
    S = np.zeros(1, np.int64)
    off = np.zeros(d.n, np.int64)
    o = None if order is None else np.ascontiguousarray(order, dtype=np.int32)
    rc = lib().orc_plan(*d.args(), m, g_coll, policy, _p(o), _p(S), _p(off))
    if rc != 0:
        raise ValueError(f"orc_plan failed ({rc})")
    return int(S[0]), off


def bruteforce_S(d: Desc, m: int, g_coll: int):
    order = np.zeros(d.n, np.int32)
    S = lib().orc_bruteforce_S(*d.args(), m, g_coll, _p(order))
    return int(S), order


def exhaustive_S(d: Desc, m: int, g_coll: int, max_S: int) -> int:
    return int(lib().orc_exhaustive_S(*d.args(), m, g_coll, max_S))


def qblocks(d: Desc, g_coll: int, offsets):
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    n = lib().orc_qblocks(*d.args(), g_coll, _p(off), None, None, None, None, None)
    if n < 0:
        raise ValueError("bad descriptor")
    t = np.zeros(n, np.int32)
    base, nr, nc, st = (np.zeros(n, np.int64) for _ in range(4))
    lib().orc_qblocks(*d.args(), g_coll, _p(off), _p(t), _p(base), _p(nr), _p(nc), _p(st))
    return dict(tensor=t, base=base, nrows=nr, ncols=nc, stride=st)


def _ptrs(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def pack(tensors, offsets, total: int):
    """tensors: list of uint16 (bf16 bits) or float32 arrays -> packed array of `total`."""
    dt = tensors[0].dtype
    esize = dt.itemsize
    packed = np.zeros(total, dtype=dt)
    numel = np.array([t.size for t in tensors], np.int64)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    lib().orc_pack(len(tensors), _ptrs(tensors), _p(numel), _p(off), esize, _p(packed))
    return packed


def unpack(packed, numels, offsets):
    outs = [np.empty(int(n), dtype=packed.dtype) for n in numels]
    numel = np.array(numels, np.int64)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    lib().orc_unpack(len(outs), _ptrs(outs), _p(numel), _p(off), packed.dtype.itemsize,
                     _p(packed))
    return outs


def sumsq(tensors) -> float:
    is_bf16 = int(tensors[0].dtype == np.uint16)
    numel = np.array([t.size for t in tensors], np.int64)
    return float(lib().orc_sumsq(len(tensors), _ptrs(tensors), _p(numel), is_bf16))


def factor(sumsq_value: float, world: int, max_norm: float):
    norm = np.zeros(1, np.float64)
    f = lib().orc_factor(sumsq_value, world, max_norm, _p(norm))
    return float(np.float32(f)), float(norm[0])


def adam_block(g, quantized, factor_f32, state, step, hp):
    """One block. state: dict with p (float32), and either mq/vq (int8/uint8) +
    m_scale/v_scale (float) or m/v (float32). Returns a new dict plus 'bf16'."""
    s = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in state.items()}
    n = s["p"].size
    bf = np.zeros(n, np.uint16)
    ms = np.array([s.get("m_scale", 0.0)], np.float32)
    vs = np.array([s.get("v_scale", 0.0)], np.float32)
    lib().orc_adam_block(n, _p(g), int(g.dtype == np.uint16), factor_f32, int(quantized),
                         _p(s.get("mq")), _p(s.get("vq")), _p(ms), _p(vs), _p(s.get("m")),
                         _p(s.get("v")), _p(s["p"]), _p(bf), hp["lr"], hp["beta1"], hp["beta2"],
                         hp["eps"], hp["weight_decay"], step)
    if quantized:
        s["m_scale"], s["v_scale"] = float(ms[0]), float(vs[0])
    s["bf16"] = bf
    return s


def adam_all(blocks, packed_grad, factor_f32, quantized, m_state, v_state, m_scale, v_scale,
             master, packed_bf16, step, hp):
    """In place over the packed buffers."""
    lib().orc_adam_all(len(blocks["base"]), _p(blocks["base"]), _p(blocks["nrows"]),
                       _p(blocks["ncols"]), _p(blocks["stride"]), _p(packed_grad),
                       int(packed_grad.dtype == np.uint16), factor_f32, int(quantized),
                       _p(m_state), _p(v_state), _p(m_scale), _p(v_scale), _p(master),
                       _p(packed_bf16), hp["lr"], hp["beta1"], hp["beta2"], hp["eps"],
                       hp["weight_decay"], step)


def quantize_m(x):
    x = np.ascontiguousarray(x, np.float32)
    codes = np.zeros(x.size, np.int8)
    deq = np.zeros(x.size, np.float32)
    s = np.zeros(1, np.float32)
    lib().orc_quantize_m(x.size, _p(x), _p(codes), _p(s), _p(deq))
    return codes, float(s[0]), deq


def quantize_v(x):
    x = np.ascontiguousarray(x, np.float32)
    codes = np.zeros(x.size, np.uint8)
    deq = np.zeros(x.size, np.float32)
    s = np.zeros(1, np.float32)
    lib().orc_quantize_v(x.size, _p(x), _p(codes), _p(s), _p(deq))
    return codes, float(s[0]), deq


def group_op(op: int, numels, offsets, dst, src=None, alpha: float = 1.0):
    """In place on dst (uint16 bf16 bits or float32): 0 zero, 1 scale, 2 add."""
    numel = np.array(numels, np.int64)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    lib().orc_group_op(op, len(numel), _p(numel), _p(off), _p(dst), int(dst.dtype == np.uint16),
                       _p(src), int(src is not None and src.dtype == np.uint16), alpha)
    return dst


def bf16_round(x: float) -> int:
    return int(lib().orc_bf16_round(x))


def hparams(w) -> dict:
    return dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay)
