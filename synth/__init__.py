"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

The C generator (``synth.c``) is counter based: element ``i`` of the stream
``synth_key(seed, step, tensor, kind)`` is a pure function of those numbers, so
the tests can redraw any sampled block on its own. Nothing here computes any
part of the shard step itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

KIND_PARAM = 0
KIND_GRAD = 1
DIST_NORMAL = 0
DIST_STUDENT_T3 = 1


def build(force: bool = False) -> str:
    """Compile libsynth.so next to its source (gcc, OpenMP when available)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC,
            "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            u64, i32, dbl = ctypes.c_uint64, ctypes.c_int32, ctypes.c_double
            L.synth_key.restype = u64
            L.synth_key.argtypes = [u64, u64, u64, u64]
            L.synth_fill_f32.restype = None
            L.synth_fill_f32.argtypes = [u64, ctypes.c_int, dbl, u64, u64, ctypes.c_void_p]
            L.synth_fill_bf16.restype = None
            L.synth_fill_bf16.argtypes = [u64, ctypes.c_int, dbl, u64, u64, ctypes.c_void_p]
            L.synth_zero_u16.argtypes = [ctypes.c_void_p, u64]
            L.synth_zero_f32.argtypes = [ctypes.c_void_p, u64]
            L.synth_pick.restype = i32
            L.synth_pick.argtypes = [u64, i32, i32, ctypes.c_void_p]
            L.synth_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def key(seed: int, step: int, tensor: int, kind: int) -> int:
    return int(lib().synth_key(seed, step, tensor, kind))


def fill_f32(k: int, dist: int, scale: float, start: int, out: np.ndarray) -> np.ndarray:
    assert out.dtype == np.float32 and out.flags.c_contiguous
    lib().synth_fill_f32(k, dist, scale, start, out.size, out.ctypes.data)
    return out


def fill_bf16(k: int, dist: int, scale: float, start: int, out: np.ndarray) -> np.ndarray:
    """bf16 values as raw uint16 bit patterns."""
    assert out.dtype == np.uint16 and out.flags.c_contiguous
    lib().synth_fill_bf16(k, dist, scale, start, out.size, out.ctypes.data)
    return out


def pick(k: int, n: int, count: int) -> list[int]:
    out = np.zeros(max(count, 1), dtype=np.int32)
    rc = lib().synth_pick(k, n, count, out.ctypes.data)
    if rc != 0:
        raise ValueError("pick: count > n")
    return [int(x) for x in out[:count]]


def threads() -> int:
    return int(lib().synth_threads())


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for test arithmetic)."""
    return (u16.astype(np.uint32) << 16).view(np.float32)
