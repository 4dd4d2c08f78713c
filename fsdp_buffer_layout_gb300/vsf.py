"""Thin ctypes binding of libvsf (``include/vsf.h``): the same function names,
argument marshalling only. Device pointers and streams are passed as ints
(``tensor.data_ptr()``, ``stream.cuda_stream``). Every failure raises
VsfError with the library's message; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

VSF_OK, VSF_ERR_ARG, VSF_ERR_INFEASIBLE, VSF_ERR_OVERFLOW = 0, -1, -2, -3
VSF_ERR_ALIGN, VSF_ERR_CUDA, VSF_ERR_STATE = -4, -5, -6
VSF_GRAN_ELEM, VSF_GRAN_ROWS, VSF_GRAN_TILE = 0, 1, 2
VSF_ORDER_DEFAULT, VSF_ORDER_BLOCK, VSF_ORDER_SHAPE, VSF_ORDER_BEST3 = 0, 1, 2, 3
VSF_BF16, VSF_FP32 = 0, 1


class VsfError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"[{status}] {msg}")
        self.status = status


class vsf_tensor_desc(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int32), ("gran", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 8), ("block_rows", ctypes.c_int64),
                ("tile_cols", ctypes.c_int64)]


class vsf_adam_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double),
                ("max_norm", ctypes.c_double), ("world", ctypes.c_int32),
                ("quantized", ctypes.c_int32)]


class vsf_plan_info(ctypes.Structure):
    _fields_ = [("S", ctypes.c_int64), ("total", ctypes.c_int64), ("real", ctypes.c_int64),
                ("n_qblocks", ctypes.c_int64), ("n_tensors", ctypes.c_int32),
                ("m", ctypes.c_int32), ("g_coll", ctypes.c_int64),
                ("padding_ratio", ctypes.c_double), ("plan_seconds", ctypes.c_double),
                ("order_used", ctypes.c_int32), ("bulk_warps", ctypes.c_int32),
                ("n_bulk_units", ctypes.c_int64), ("n_register_blocks", ctypes.c_int64),
                ("n_element_chunks", ctypes.c_int64), ("rank_begin", ctypes.c_int32),
                ("rank_end", ctypes.c_int32), ("bulk_cluster", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class vsf_muon_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("momentum", ctypes.c_double),
                ("weight_decay", ctypes.c_double), ("eps", ctypes.c_double),
                ("ns_a", ctypes.c_double), ("ns_b", ctypes.c_double), ("ns_c", ctypes.c_double),
                ("ns_steps", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    """libvsf.so, or the library named by VSF_LIBRARY (the bounds-checking
    build, libvsf_bounds.so)."""
    return os.environ.get("VSF_LIBRARY") or _build.LIB


def lib():
    """Loads libvsf.so. Raises if it has not been built: there is no fallback."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"libvsf is not built ({path}); "
                                   "run `python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(path)
            vp, i32, i64, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32
            P = ctypes.POINTER
            L.vsf_plan_create.restype = st
            L.vsf_plan_create.argtypes = [P(vsf_tensor_desc), i32, i32, i64, i32, P(vp)]
            L.vsf_plan_destroy.restype = None
            L.vsf_plan_destroy.argtypes = [vp]
            L.vsf_plan_serialize.restype = st
            L.vsf_plan_serialize.argtypes = [vp, vp, P(ctypes.c_size_t)]
            L.vsf_plan_deserialize.restype = st
            L.vsf_plan_deserialize.argtypes = [vp, ctypes.c_size_t, P(vp)]
            L.vsf_plan_get_info.restype = st
            L.vsf_plan_get_info.argtypes = [vp, P(vsf_plan_info)]
            L.vsf_plan_offsets.restype = st
            L.vsf_plan_offsets.argtypes = [vp, vp]
            L.vsf_plan_qblocks.restype = st
            L.vsf_plan_qblocks.argtypes = [vp, vp, vp, vp, vp, vp]
            L.vsf_plan_rank_slices.restype = st
            L.vsf_plan_rank_slices.argtypes = [vp, i32, i32, P(i32), vp, vp, vp, vp, vp]
            L.vsf_plan_device_error_offset.restype = st
            L.vsf_plan_device_error_offset.argtypes = [vp, P(ctypes.c_size_t)]
            L.vsf_plan_workspace_bytes.restype = ctypes.c_size_t
            L.vsf_plan_workspace_bytes.argtypes = [vp]
            L.vsf_plan_upload.restype = st
            L.vsf_plan_upload.argtypes = [vp, vp, ctypes.c_size_t, vp]
            L.vsf_pack.restype = st
            L.vsf_pack.argtypes = [vp, P(vp), i32, vp, vp]
            L.vsf_selftest_wait_timeout.restype = st
            L.vsf_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint64, vp]
            L.vsf_device_copy.restype = st
            L.vsf_device_copy.argtypes = [vp, vp, ctypes.c_size_t, vp]
            L.vsf_ns_gemm.restype = st
            L.vsf_ns_gemm.argtypes = [i32, i32, i32, i64, i64, i64, i64, vp, i64, i64, vp, i64,
                                      i64, ctypes.c_float, ctypes.c_float, vp, i64, i64, vp, i64,
                                      i64, vp, vp]
            L.vsf_plan_restrict.restype = st
            L.vsf_plan_restrict.argtypes = [vp, i32, i32]
            L.vsf_plan_set_bulk_warps.restype = st
            L.vsf_plan_set_bulk_warps.argtypes = [vp, i32]
            L.vsf_group_sumsq.restype = st
            L.vsf_group_sumsq.argtypes = [vp, vp, i32, vp, vp]
            L.vsf_group_scale_from_sumsq.restype = st
            L.vsf_group_scale_from_sumsq.argtypes = [vp, P(vsf_adam_hparams), vp, vp, vp]
            L.vsf_group_norm_scale.restype = st
            L.vsf_group_norm_scale.argtypes = [vp, vp, i32, P(vsf_adam_hparams), vp, vp, vp]
            L.vsf_adam8_step.restype = st
            L.vsf_adam8_step.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp,
                                         P(vsf_adam_hparams), i32, vp]
            L.vsf_unpack.restype = st
            L.vsf_unpack.argtypes = [vp, vp, P(vp), vp]
            L.vsf_group_zero.restype = st
            L.vsf_group_zero.argtypes = [vp, vp, i32, vp]
            L.vsf_group_scale.restype = st
            L.vsf_group_scale.argtypes = [vp, vp, i32, ctypes.c_float, vp]
            L.vsf_group_add.restype = st
            L.vsf_group_add.argtypes = [vp, vp, i32, vp, i32, vp]
            L.vsf_plan_views.restype = st
            L.vsf_plan_views.argtypes = [vp, vp, i32, P(vp)]
            L.vsf_group_norm_scale_static.restype = st
            L.vsf_group_norm_scale_static.argtypes = [P(vp), vp, i32, i32, P(vsf_adam_hparams),
                                                      vp, vp, vp]
            L.vsf_muon_select_roots.restype = st
            L.vsf_muon_select_roots.argtypes = [vp, vp, P(ctypes.c_double)]
            L.vsf_muon_workspace_bytes.restype = ctypes.c_size_t
            L.vsf_muon_workspace_bytes.argtypes = [vp]
            L.vsf_muon_chunk_count.restype = ctypes.c_int32
            L.vsf_muon_chunk_count.argtypes = [vp]
            L.vsf_muon_kernel_launches.restype = ctypes.c_int64
            L.vsf_muon_kernel_launches.argtypes = [vp, ctypes.c_int32]
            L.vsf_muon_step.restype = st
            L.vsf_muon_step.argtypes = [vp, vp, vp, vp, vp, P(vsf_muon_hparams), vp,
                                        ctypes.c_size_t, vp]
            L.vsf_status_string.restype = ctypes.c_char_p
            L.vsf_status_string.argtypes = [st]
            L.vsf_last_error.restype = ctypes.c_char_p
            L.vsf_last_error.argtypes = []
            _lib = L
    return _lib


def _check(status: int):
    if status != VSF_OK:
        msg = lib().vsf_last_error().decode(errors="replace")
        raise VsfError(status, msg or lib().vsf_status_string(status).decode())


def make_desc(shape, gran, block_rows=0, tile_cols=0) -> vsf_tensor_desc:
    d = vsf_tensor_desc()
    d.ndim = len(shape)
    d.gran = gran
    for i, s in enumerate(shape):
        d.shape[i] = int(s)
    d.block_rows = int(block_rows)
    d.tile_cols = int(tile_cols)
    return d


def make_hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
                 max_norm=float("inf"), world=1, quantized=1) -> vsf_adam_hparams:
    return vsf_adam_hparams(lr, beta1, beta2, eps, weight_decay, max_norm, world, quantized)


def _ptr_array(ptrs):
    return (ctypes.c_void_p * len(ptrs))(*[int(p) for p in ptrs])


def vsf_plan_create(descs, m: int, g_coll: int, order: int = VSF_ORDER_DEFAULT) -> int:
    arr = (vsf_tensor_desc * len(descs))(*descs)
    out = ctypes.c_void_p()
    _check(lib().vsf_plan_create(arr, len(descs), m, g_coll, order, ctypes.byref(out)))
    return out.value


def vsf_plan_destroy(plan: int) -> None:
    lib().vsf_plan_destroy(plan)


def vsf_plan_serialize(plan: int) -> bytes:
    """The plan as bytes (its inputs, rank window, forced shape, S, offsets)."""
    n = ctypes.c_size_t(0)
    _check(lib().vsf_plan_serialize(plan, None, ctypes.byref(n)))
    buf = ctypes.create_string_buffer(n.value)
    _check(lib().vsf_plan_serialize(plan, buf, ctypes.byref(n)))
    return buf.raw[:n.value]


def vsf_plan_deserialize(data: bytes) -> int:
    """A new plan from vsf_plan_serialize's bytes (planned again and checked)."""
    out = ctypes.c_void_p()
    _check(lib().vsf_plan_deserialize(data, len(data), ctypes.byref(out)))
    return out.value


def vsf_selftest_wait_timeout(d_err: int, limit_ns: int, stream: int) -> None:
    _check(lib().vsf_selftest_wait_timeout(d_err, limit_ns, stream))


def vsf_ns_gemm(a_mn: bool, b_mn: bool, sym: bool, M: int, N: int, K: int, batch: int,
                A: int, lda: int, sa: int, B: int, ldb: int, sb: int, alpha: float, beta: float,
                C, ldc: int, sc: int, D: int, ldd: int, sd: int, d_err: int, stream: int) -> None:
    _check(lib().vsf_ns_gemm(int(a_mn), int(b_mn), int(sym), M, N, K, batch, A, lda, sa, B, ldb,
                             sb, alpha, beta, C, ldc, sc, D, ldd, sd, d_err, stream))


def vsf_device_copy(dst: int, src: int, nbytes: int, stream: int) -> None:
    _check(lib().vsf_device_copy(dst, src, nbytes, stream))


def vsf_plan_restrict(plan: int, rank_begin: int, rank_end: int) -> None:
    _check(lib().vsf_plan_restrict(plan, rank_begin, rank_end))


def vsf_plan_set_bulk_warps(plan: int, warps: int) -> None:
    _check(lib().vsf_plan_set_bulk_warps(plan, warps))


def vsf_group_sumsq(plan: int, packed_grad, dtype: int, d_sumsq: int, stream: int) -> None:
    _check(lib().vsf_group_sumsq(plan, packed_grad, dtype, d_sumsq, stream))


def vsf_group_scale_from_sumsq(d_sumsq: int, hp: vsf_adam_hparams, d_factor: int, d_norm,
                               stream: int) -> None:
    _check(lib().vsf_group_scale_from_sumsq(d_sumsq, ctypes.byref(hp), d_factor, d_norm, stream))


def vsf_plan_get_info(plan: int) -> vsf_plan_info:
    info = vsf_plan_info()
    _check(lib().vsf_plan_get_info(plan, ctypes.byref(info)))
    return info


def vsf_plan_offsets(plan: int, n: int):
    out = (ctypes.c_int64 * n)()
    _check(lib().vsf_plan_offsets(plan, out))
    return list(out)


def vsf_plan_qblocks(plan: int, nq: int):
    arrs = [(ctypes.c_int32 * nq)()] + [(ctypes.c_int64 * nq)() for _ in range(4)]
    _check(lib().vsf_plan_qblocks(plan, *arrs))
    keys = ("tensor", "base", "nrows", "ncols", "stride")
    return {k: list(a) for k, a in zip(keys, arrs)}


def vsf_plan_rank_slices(plan: int, rank: int):
    count = ctypes.c_int32()
    _check(lib().vsf_plan_rank_slices(plan, rank, 0, ctypes.byref(count), None, None, None,
                                      None, None))
    n = count.value
    t = (ctypes.c_int32 * max(n, 1))()
    a = [(ctypes.c_int64 * max(n, 1))() for _ in range(4)]
    _check(lib().vsf_plan_rank_slices(plan, rank, n, ctypes.byref(count), t, *a))
    return [(t[i], a[0][i], a[1][i], a[2][i], a[3][i]) for i in range(n)]


def vsf_plan_device_error_offset(plan: int) -> int:
    out = ctypes.c_size_t()
    _check(lib().vsf_plan_device_error_offset(plan, ctypes.byref(out)))
    return int(out.value)


def vsf_plan_workspace_bytes(plan: int) -> int:
    return int(lib().vsf_plan_workspace_bytes(plan))


def vsf_plan_upload(plan: int, d_workspace: int, nbytes: int, stream: int) -> None:
    _check(lib().vsf_plan_upload(plan, d_workspace, nbytes, stream))


def vsf_pack(plan: int, grads, dtype: int, packed_grad: int, stream: int) -> None:
    _check(lib().vsf_pack(plan, _ptr_array(grads), dtype, packed_grad, stream))


def vsf_group_norm_scale(plan: int, packed_grad, dtype: int, hp: vsf_adam_hparams,
                         d_factor: int, d_norm, stream: int) -> None:
    _check(lib().vsf_group_norm_scale(plan, packed_grad, dtype, ctypes.byref(hp), d_factor,
                                      d_norm, stream))


def vsf_adam8_step(plan: int, packed_grad: int, grad_dtype: int, d_factor: int, master: int,
                   m_state: int, v_state: int, m_scale, v_scale, packed_bf16: int,
                   hp: vsf_adam_hparams, step: int, stream: int) -> None:
    _check(lib().vsf_adam8_step(plan, packed_grad, grad_dtype, d_factor, master, m_state,
                                v_state, m_scale, v_scale, packed_bf16, ctypes.byref(hp), step,
                                stream))


def vsf_unpack(plan: int, packed_bf16: int, params, stream: int) -> None:
    _check(lib().vsf_unpack(plan, packed_bf16, _ptr_array(params), stream))


def vsf_group_zero(plan: int, buf: int, dtype: int, stream: int) -> None:
    _check(lib().vsf_group_zero(plan, buf, dtype, stream))


def vsf_group_scale(plan: int, buf: int, dtype: int, alpha: float, stream: int) -> None:
    _check(lib().vsf_group_scale(plan, buf, dtype, alpha, stream))


def vsf_group_add(plan: int, dst: int, dst_dtype: int, src: int, src_dtype: int,
                  stream: int) -> None:
    _check(lib().vsf_group_add(plan, dst, dst_dtype, src, src_dtype, stream))


def vsf_plan_views(plan: int, packed: int, elem_bytes: int, n: int):
    out = (ctypes.c_void_p * n)()
    _check(lib().vsf_plan_views(plan, packed, elem_bytes, out))
    return [int(x or 0) for x in out]


def vsf_group_norm_scale_static(grads, numel, dtype: int, hp: vsf_adam_hparams, d_factor: int,
                                d_norm, stream) -> None:
    arr = _ptr_array(grads)
    n = (ctypes.c_int64 * len(numel))(*[int(x) for x in numel])
    _check(lib().vsf_group_norm_scale_static(arr, n, len(grads), dtype, ctypes.byref(hp),
                                             d_factor, d_norm, stream))


def make_muon_hparams(lr=0.02, momentum=0.95, weight_decay=0.01, eps=1e-7, ns_a=3.4445,
                      ns_b=-4.7750, ns_c=2.0315, ns_steps=5) -> vsf_muon_hparams:
    return vsf_muon_hparams(lr, momentum, weight_decay, eps, ns_a, ns_b, ns_c, ns_steps, 0)


def vsf_muon_select_roots(plan: int, n: int):
    roots = (ctypes.c_int32 * n)()
    bal = ctypes.c_double()
    _check(lib().vsf_muon_select_roots(plan, roots, ctypes.byref(bal)))
    return list(roots), bal.value


def vsf_muon_workspace_bytes(plan: int) -> int:
    return int(lib().vsf_muon_workspace_bytes(plan))


def vsf_muon_chunk_count(plan: int) -> int:
    return int(lib().vsf_muon_chunk_count(plan))


def vsf_muon_kernel_launches(plan: int, ns_steps: int = 5) -> int:
    return int(lib().vsf_muon_kernel_launches(plan, ns_steps))


def vsf_muon_step(plan: int, packed_grad: int, momentum: int, master: int, packed_bf16: int,
                  hp: vsf_muon_hparams, d_workspace: int, ws_bytes: int, stream: int) -> None:
    _check(lib().vsf_muon_step(plan, packed_grad, momentum, master, packed_bf16, ctypes.byref(hp),
                               d_workspace, ws_bytes, stream))


def vsf_status_string(status: int) -> str:
    return lib().vsf_status_string(status).decode()


def vsf_last_error() -> str:
    return lib().vsf_last_error().decode(errors="replace")
