"""Thin ctypes binding of libqmm (include/qmm.h).

Argument marshalling only: every ``qmm_*`` function here has the C entry
point's name and argument order; tensors become device pointers
(``data_ptr()``), ``None`` becomes NULL, ints pass through, and the stream
defaults to torch's current CUDA stream.  A nonzero status raises
``QmmError``.  All arithmetic runs in the CUDA kernels of libqmm.so; if the
library is missing this module raises on import -- there is no fallback.

A few helpers at the bottom allocate outputs with torch and call the entry
points (``quantize_q8_0``, ``quantize_q4_0``, ``gemv``, ``gemm``, ...).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmm.so")
QK = 32

STATUS = {0: "QMM_OK", 1: "QMM_ERR_ARG", 2: "QMM_ERR_SHAPE", 3: "QMM_ERR_ALIGN", 4: "QMM_ERR_DEVICE",
          5: "QMM_ERR_CUDA", 6: "QMM_ERR_TIMEOUT", 7: "QMM_ERR_BAD_EXPERT_ID", 8: "QMM_ERR_WORKSPACE",
          9: "QMM_ERR_SCRATCH_LIMIT"}


class QmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib.qmm_status_string(status).decode()} (status {status})")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"libqmm.so not built at {LIB_PATH}: run __graft_entry__.build() "
                      "(no CPU fallback exists)")

_lib = ctypes.CDLL(LIB_PATH)

_P, _I64, _I32, _INT, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int, ctypes.c_size_t

class GemvOp(ctypes.Structure):
    """qmm_gemv_op of include/qmm.h (one batch-1 GEMV of a decode step)."""
    _fields_ = [("w_qs", ctypes.c_void_p), ("w_d", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("x", ctypes.c_void_p), ("norm_w", ctypes.c_void_p), ("xq", ctypes.c_void_p),
                ("xd", ctypes.c_void_p), ("residual", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("yq", ctypes.c_void_p), ("yd", ctypes.c_void_p), ("norm_eps", ctypes.c_float),
                ("flags", ctypes.c_int32)]


class StorePlane(ctypes.Structure):
    """qmm_store_plane of include/qmm.h (one plane of every expert)."""
    _fields_ = [("host", ctypes.c_void_p), ("host_stride", ctypes.c_int64), ("dev", ctypes.c_void_p),
                ("bytes", ctypes.c_int64)]


# name -> argtypes (the trailing stream is a void*)
SIGNATURES = {
    "qmm_quantize_q4_0": [_P, _I64, _I64, _I64, _P, _P, _P],
    "qmm_repack_q4_0": [_P, _I64, _I64, _P, _P, _P],
    "qmm_quantize_q8_0": [_P, _I64, _I64, _I64, _P, _P, _P],
    "qmm_swiglu_quantize_q8_0": [_P, _P, _I64, _I64, _I64, _P, _P, _P, _P],
    "qmm_gemv_q4_0_q8_0": [_P, _P, _I64, _I64, _P, _P, _P, _P],
    "qmm_gemv_q4_0_f32": [_P, _P, _I64, _I64, _P, _P, _P, _P, _P, _INT, _P],
    "qmm_gemv_fused": [_P, _P, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _INT, _P],
    "qmm_gemm_q4_0_q8_0": [_P, _P, _I64, _I64, _I64, _P, _P, _P, _I64, _P],
    "qmm_gemm_workspace_size": [_I64, _I64, ctypes.POINTER(_SZ)],
    "qmm_gemm_q4_0_q8_0_ws": [_P, _P, _I64, _I64, _I64, _P, _P, _P, _I64, _P, _SZ, _P],
    "qmm_debug_block_dots": [_P, _I64, _I64, _I64, _P, _P, _P],
    "qmm_debug_gemm_kernel": [_INT, ctypes.POINTER(_INT)],
    "qmm_debug_stream_wait": [ctypes.c_uint64, _INT, ctypes.POINTER(ctypes.c_uint64)],
    "qmm_gemv_fused_op": [ctypes.POINTER(GemvOp), _INT, _P],
    "qmm_gemv_fused_ops": [ctypes.POINTER(GemvOp), _I32, _INT, _P],
    "qmm_moe_workspace_size": [_I32, _I32, _I32, ctypes.POINTER(_SZ)],
    "qmm_moe_gemv": [_P, _P, _I32, _I64, _I64, _P, _I32, _I32, _P, _P, _INT, _P, _P, _SZ, _P],
    "qmm_moe_gemv_static": [_P, _P, _I32, _I64, _I64, _P, _I32, _I32, _P, _P, _INT, _P, _P],
    "qmm_moe_combine": [_P, _P, _I32, _I32, _I64, _P, _P],
    "qmm_moe_router_topk": [_P, _I32, _I32, _I32, _P, _P, _P, _SZ, _P],
    "qmm_moe_layer_f32": [_P, _I32, _I32, _I32, _P, _P, _P, _P, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "qmm_quantize_rowwise": [_P, _I64, _I64, _I64, _I32, _P, _P, _P],
    "qmm_lru_create": [_I32, _I32, ctypes.POINTER(_P)],
    "qmm_lru_request": [_P, _P, _I32, _I32, _P, _P, _P, _P],
    "qmm_lru_stats": [_P, _P, _P, _P, _P],
    "qmm_lru_slot_of": [_P, _I32, _P],
    "qmm_store_create": [_I32, _I32, ctypes.POINTER(StorePlane), _I32, _P, ctypes.POINTER(_P)],
    "qmm_store_request": [_P, _P, _I32, _P, _P],
    "qmm_store_release": [_P, _P],
    "qmm_store_prefetch": [_P, _P, _I32, _P],
    "qmm_store_map_ids": [_P, _P, _I64, _P, _P],
    "qmm_store_stats": [_P, _P, _P, _P, _P, _P],
    "qmm_gemv_rowwise_q8_0": [_P, _P, _I32, _I64, _I64, _P, _P, _P, _P],
    "qmm_gemv_q4_0_f32_fma": [_P, _P, _I64, _I64, _P, _P, _P],
    "qmm_moe_gemv_pregrouped": [_P, _P, _I32, _I64, _I64, _I32, _I32, _P, _P, _INT, _P, _P, _SZ, _P],
    "qmm_moe_gemv_gate_up": [_P, _P, _I32, _I64, _I64, _I32, _I32, _P, _P, _P, _INT, _P, _P, _SZ, _P],
    "qmm_moe_group_ids": [_P, _I32, _I32, _I32, _P, _SZ, _P],
    "qmm_moe_gemv_pregrouped_f32": [_P, _P, _I32, _I64, _I64, _I32, _I32, _P, _INT, _P, _P, _SZ, _P],
    "qmm_last_device_error": [_P],
}
for _name, _args in SIGNATURES.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
for _name in ("qmm_lru_destroy", "qmm_store_destroy"):
    getattr(_lib, _name).argtypes = [_P]
    getattr(_lib, _name).restype = None
_lib.qmm_status_string.argtypes = [ctypes.c_int]
_lib.qmm_status_string.restype = ctypes.c_char_p
_lib.qmm_abi_version.argtypes = []
_lib.qmm_abi_version.restype = ctypes.c_int


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, where: str):
    if st != 0:
        raise QmmError(st, where)


def status_string(status: int) -> str:
    return _lib.qmm_status_string(status).decode()


def abi_version() -> int:
    return _lib.qmm_abi_version()


def library_handle():
    return _lib


# ------------------------------------------------------------------ raw entry points
def qmm_quantize_q4_0(w, N, K, ldw, qs, d, stream=None):
    _check(_lib.qmm_quantize_q4_0(_ptr(w), N, K, ldw, _ptr(qs), _ptr(d), _stream(stream)), "qmm_quantize_q4_0")


def qmm_repack_q4_0(blocks, N, K, qs, d, stream=None):
    _check(_lib.qmm_repack_q4_0(_ptr(blocks), N, K, _ptr(qs), _ptr(d), _stream(stream)), "qmm_repack_q4_0")


def qmm_quantize_q8_0(x, M, K, ldx, q, d, stream=None):
    _check(_lib.qmm_quantize_q8_0(_ptr(x), M, K, ldx, _ptr(q), _ptr(d), _stream(stream)), "qmm_quantize_q8_0")


def qmm_swiglu_quantize_q8_0(gate, up, rows, K, ld, q, d, h_out=None, stream=None):
    _check(_lib.qmm_swiglu_quantize_q8_0(_ptr(gate), _ptr(up), rows, K, ld, _ptr(q), _ptr(d), _ptr(h_out),
                                         _stream(stream)), "qmm_swiglu_quantize_q8_0")


def qmm_gemv_q4_0_q8_0(w_qs, w_d, N, K, xq, xd, y, stream=None):
    _check(_lib.qmm_gemv_q4_0_q8_0(_ptr(w_qs), _ptr(w_d), N, K, _ptr(xq), _ptr(xd), _ptr(y), _stream(stream)),
           "qmm_gemv_q4_0_q8_0")


X_SWIGLU, Y_SWIGLU_PAIRS, CHAIN = 1, 2, 4  # flags of qmm_gemv_q4_0_f32


def qmm_gemv_q4_0_f32(w_qs, w_d, N, K, x, residual, y, xq_out=None, xd_out=None, flags=0, stream=None):
    _check(_lib.qmm_gemv_q4_0_f32(_ptr(w_qs), _ptr(w_d), N, K, _ptr(x), _ptr(residual), _ptr(y), _ptr(xq_out),
                                  _ptr(xd_out), int(flags), _stream(stream)), "qmm_gemv_q4_0_f32")


def qmm_gemv_fused(w_qs, w_d, N, K, x, xq, xd, residual, y, yq, yd, flags=0, stream=None):
    _check(_lib.qmm_gemv_fused(_ptr(w_qs), _ptr(w_d), N, K, _ptr(x), _ptr(xq), _ptr(xd), _ptr(residual), _ptr(y),
                               _ptr(yq), _ptr(yd), int(flags), _stream(stream)), "qmm_gemv_fused")


def qmm_gemm_q4_0_q8_0(w_qs, w_d, N, K, M, xq, xd, y, ldy, stream=None):
    _check(_lib.qmm_gemm_q4_0_q8_0(_ptr(w_qs), _ptr(w_d), N, K, M, _ptr(xq), _ptr(xd), _ptr(y), ldy,
                                   _stream(stream)), "qmm_gemm_q4_0_q8_0")


def qmm_gemm_workspace_size(K, M) -> int:
    out = _SZ(0)
    _check(_lib.qmm_gemm_workspace_size(K, M, ctypes.byref(out)), "qmm_gemm_workspace_size")
    return out.value


def qmm_gemm_q4_0_q8_0_ws(w_qs, w_d, N, K, M, xq, xd, y, ldy, workspace, workspace_bytes, stream=None):
    _check(_lib.qmm_gemm_q4_0_q8_0_ws(_ptr(w_qs), _ptr(w_d), N, K, M, _ptr(xq), _ptr(xd), _ptr(y), ldy,
                                      _ptr(workspace), workspace_bytes, _stream(stream)), "qmm_gemm_q4_0_q8_0_ws")


GEMM_KERNEL_AUTO, GEMM_KERNEL_MMA, GEMM_KERNEL_TMEM, GEMM_KERNEL_STREAM, GEMM_KERNEL_MMA_GROUPS = 0, 1, 2, 3, 4


def qmm_debug_gemm_kernel(kernel):
    """Select the small-batch GEMM kernel; returns the previous setting."""
    prev = ctypes.c_int(0)
    _check(_lib.qmm_debug_gemm_kernel(kernel, ctypes.byref(prev)), "qmm_debug_gemm_kernel")
    return prev.value


def qmm_debug_stream_wait(limit_ns, withhold_last_copy=False):
    """Bound of the streaming kernel's device waits (ns) and the withheld-copy
    test mode; returns the previous bound."""
    prev = ctypes.c_uint64(0)
    _check(_lib.qmm_debug_stream_wait(int(limit_ns), int(bool(withhold_last_copy)), ctypes.byref(prev)),
           "qmm_debug_stream_wait")
    return prev.value


def qmm_debug_block_dots(w_qs, N, K, M, xq, dots, stream=None):
    _check(_lib.qmm_debug_block_dots(_ptr(w_qs), N, K, M, _ptr(xq), _ptr(dots), _stream(stream)),
           "qmm_debug_block_dots")


def gemv_op(w_qs, w_d, N, K, x=None, xq=None, xd=None, residual=None, y=None, yq=None, yd=None, flags=0,
            norm_w=None, norm_eps=1e-5):
    """A qmm_gemv_op from tensors (or None / raw pointers)."""
    return GemvOp(_ptr(w_qs), _ptr(w_d), N, K, _ptr(x), _ptr(norm_w), _ptr(xq), _ptr(xd), _ptr(residual), _ptr(y),
                  _ptr(yq), _ptr(yd), float(norm_eps), int(flags))


def qmm_gemv_fused_op(op, flags=0, stream=None):
    _check(_lib.qmm_gemv_fused_op(ctypes.byref(op), int(flags), _stream(stream)), "qmm_gemv_fused_op")


def gemv_op_array(ops):
    """A contiguous qmm_gemv_op array (for qmm_gemv_fused_ops) from GemvOp structs."""
    return (GemvOp * len(ops))(*ops)


def qmm_gemv_fused_ops(op_array, n, flags=0, stream=None):
    _check(_lib.qmm_gemv_fused_ops(op_array, int(n), int(flags), _stream(stream)), "qmm_gemv_fused_ops")


def qmm_moe_workspace_size(E, T, k) -> int:
    out = _SZ(0)
    _check(_lib.qmm_moe_workspace_size(E, T, k, ctypes.byref(out)), "qmm_moe_workspace_size")
    return out.value


def qmm_moe_gemv(w_qs, w_d, E, N, K, ids, T, k, xq, xd, x_per_slot, y, workspace, workspace_bytes, stream=None):
    _check(_lib.qmm_moe_gemv(_ptr(w_qs), _ptr(w_d), E, N, K, _ptr(ids), T, k, _ptr(xq), _ptr(xd), int(x_per_slot),
                             _ptr(y), _ptr(workspace), workspace_bytes, _stream(stream)), "qmm_moe_gemv")


def qmm_moe_gemv_static(w_qs, w_d, E, N, K, ids, T, k, xq, xd, x_per_slot, y, stream=None):
    _check(_lib.qmm_moe_gemv_static(_ptr(w_qs), _ptr(w_d), E, N, K, _ptr(ids), T, k, _ptr(xq), _ptr(xd),
                                    int(x_per_slot), _ptr(y), _stream(stream)), "qmm_moe_gemv_static")


def qmm_quantize_rowwise(w, N, K, ldw, bits, w_q, w_s, stream=None):
    _check(_lib.qmm_quantize_rowwise(_ptr(w), N, K, ldw, bits, _ptr(w_q), _ptr(w_s), _stream(stream)),
           "qmm_quantize_rowwise")


def qmm_gemv_rowwise_q8_0(w_q, w_s, bits, N, K, xq, xd, y, stream=None):
    _check(_lib.qmm_gemv_rowwise_q8_0(_ptr(w_q), _ptr(w_s), bits, N, K, _ptr(xq), _ptr(xd), _ptr(y), _stream(stream)),
           "qmm_gemv_rowwise_q8_0")


def qmm_gemv_q4_0_f32_fma(w_qs, w_d, N, K, x, y, stream=None):
    _check(_lib.qmm_gemv_q4_0_f32_fma(_ptr(w_qs), _ptr(w_d), N, K, _ptr(x), _ptr(y), _stream(stream)),
           "qmm_gemv_q4_0_f32_fma")


def _i32_array(values):
    values = [int(v) for v in values]
    return (ctypes.c_int32 * max(1, len(values)))(*values), len(values)


class Lru:
    """qmm_lru: the store's host-side LRU policy on its own (no device)."""

    def __init__(self, n_keys, n_slots):
        h = ctypes.c_void_p()
        _check(_lib.qmm_lru_create(n_keys, n_slots, ctypes.byref(h)), "qmm_lru_create")
        self._h = h

    def request(self, keys, use=True):
        """Returns (slot of each key, [(key, slot) loads in order])."""
        arr, n = _i32_array(keys)
        slots = (ctypes.c_int32 * max(1, n))()
        lk = (ctypes.c_int32 * max(1, n))()
        ls = (ctypes.c_int32 * max(1, n))()
        nl = ctypes.c_int32()
        _check(_lib.qmm_lru_request(self._h, arr, n, 1 if use else 0, slots, lk, ls, ctypes.byref(nl)),
               "qmm_lru_request")
        return list(slots[:n]), list(zip(lk[:nl.value], ls[:nl.value]))

    def slot_of(self, key):
        s = ctypes.c_int32()
        _check(_lib.qmm_lru_slot_of(self._h, key, ctypes.byref(s)), "qmm_lru_slot_of")
        return s.value

    def stats(self):
        v = [ctypes.c_int64() for _ in range(4)]
        _check(_lib.qmm_lru_stats(self._h, *[ctypes.byref(x) for x in v]), "qmm_lru_stats")
        return dict(zip(("hits", "misses", "evictions", "prefetched"), (x.value for x in v)))

    def __del__(self):
        if getattr(self, "_h", None):
            _lib.qmm_lru_destroy(self._h)
            self._h = None


class ExpertStore:
    """qmm_store: experts in host memory, n_slots of them resident on the
    device.  planes: list of (host tensor [E][...] pinned, device arena
    tensor [n_slots][...]), each expert's plane contiguous."""

    def __init__(self, E, n_slots, planes, dev_slot_of):
        arr = (StorePlane * len(planes))()
        for i, (host, dev) in enumerate(planes):
            nbytes = dev[0].numel() * dev.element_size()
            arr[i] = StorePlane(host.data_ptr(), host[0].numel() * host.element_size(), dev.data_ptr(), nbytes)
        h = ctypes.c_void_p()
        _check(_lib.qmm_store_create(E, n_slots, arr, len(planes), _ptr(dev_slot_of), ctypes.byref(h)),
               "qmm_store_create")
        self._h, self._keep = h, (planes, dev_slot_of)

    def request(self, ids, compute_stream=None, copy_stream=None):
        arr, n = _i32_array(ids)
        _check(_lib.qmm_store_request(self._h, arr, n, _stream(compute_stream), _stream(copy_stream)),
               "qmm_store_request")

    def release(self, compute_stream=None):
        _check(_lib.qmm_store_release(self._h, _stream(compute_stream)), "qmm_store_release")

    def prefetch(self, ids, copy_stream=None):
        arr, n = _i32_array(ids)
        _check(_lib.qmm_store_prefetch(self._h, arr, n, _stream(copy_stream)), "qmm_store_prefetch")

    def map_ids(self, ids, slot_ids, stream=None):
        _check(_lib.qmm_store_map_ids(self._h, _ptr(ids), ids.numel(), _ptr(slot_ids), _stream(stream)),
               "qmm_store_map_ids")

    def stats(self):
        v = [ctypes.c_int64() for _ in range(5)]
        _check(_lib.qmm_store_stats(self._h, *[ctypes.byref(x) for x in v]), "qmm_store_stats")
        return dict(zip(("hits", "misses", "evictions", "prefetched", "bytes_copied"), (x.value for x in v)))

    def __del__(self):
        if getattr(self, "_h", None):
            _lib.qmm_store_destroy(self._h)
            self._h = None


def qmm_moe_router_topk(logits, T, E, k, ids, gates, workspace=None, workspace_bytes=0, stream=None):
    _check(_lib.qmm_moe_router_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(gates), _ptr(workspace),
                                    workspace_bytes if workspace is not None else 0, _stream(stream)),
           "qmm_moe_router_topk")


def qmm_moe_layer_f32(logits, T, E, k, gu_qs, gu_d, down_qs, down_d, H, F, x, ids, gates, h, z, y, workspace,
                      workspace_bytes, stream=None):
    _check(_lib.qmm_moe_layer_f32(_ptr(logits), T, E, k, _ptr(gu_qs), _ptr(gu_d), _ptr(down_qs), _ptr(down_d), H, F,
                                  _ptr(x), _ptr(ids), _ptr(gates), _ptr(h), _ptr(z), _ptr(y), _ptr(workspace),
                                  workspace_bytes, _stream(stream)),
           "qmm_moe_layer_f32")


def qmm_moe_gemv_pregrouped(w_qs, w_d, E, N, K, T, k, xq, xd, x_per_slot, y, workspace, workspace_bytes,
                            stream=None):
    _check(_lib.qmm_moe_gemv_pregrouped(_ptr(w_qs), _ptr(w_d), E, N, K, T, k, _ptr(xq), _ptr(xd), int(x_per_slot),
                                        _ptr(y), _ptr(workspace), workspace_bytes, _stream(stream)),
           "qmm_moe_gemv_pregrouped")


def qmm_moe_gemv_gate_up(w_qs, w_d, E, N, K, T, k, x, xq, xd, x_per_slot, h, workspace, workspace_bytes,
                         stream=None):
    _check(_lib.qmm_moe_gemv_gate_up(_ptr(w_qs), _ptr(w_d), E, N, K, T, k, _ptr(x), _ptr(xq), _ptr(xd),
                                     int(x_per_slot), _ptr(h), _ptr(workspace), workspace_bytes, _stream(stream)),
           "qmm_moe_gemv_gate_up")


def qmm_moe_group_ids(ids, T, k, E, workspace, workspace_bytes, stream=None):
    _check(_lib.qmm_moe_group_ids(_ptr(ids), T, k, E, _ptr(workspace), workspace_bytes, _stream(stream)),
           "qmm_moe_group_ids")


def qmm_moe_gemv_pregrouped_f32(w_qs, w_d, E, N, K, T, k, x, x_per_slot, y, workspace, workspace_bytes, stream=None):
    _check(_lib.qmm_moe_gemv_pregrouped_f32(_ptr(w_qs), _ptr(w_d), E, N, K, T, k, _ptr(x), int(x_per_slot), _ptr(y),
                                            _ptr(workspace), workspace_bytes, _stream(stream)),
           "qmm_moe_gemv_pregrouped_f32")


def qmm_moe_combine(z, gates, T, k, N, y, stream=None):
    _check(_lib.qmm_moe_combine(_ptr(z), _ptr(gates), T, k, N, _ptr(y), _stream(stream)), "qmm_moe_combine")


def qmm_last_device_error(stream=None) -> int:
    """Returns the status code (does not raise), after synchronising the stream."""
    return _lib.qmm_last_device_error(_stream(stream))


# ------------------------------------------------------------------ helpers (allocate with torch)
def q4_0_planes(N: int, K: int, device="cuda"):
    """Empty Q4_0 planes for an N x K matrix: (qs uint8 [N][K/2], d int16-as-fp16-bits [N][K/32])."""
    return (torch.empty(N, K // 2, dtype=torch.uint8, device=device),
            torch.empty(N, K // QK, dtype=torch.int16, device=device))


def quantize_q4_0(w: torch.Tensor):
    N, K = w.shape
    qs, d = q4_0_planes(N, K, w.device)
    qmm_quantize_q4_0(w, N, K, w.stride(0), qs, d)
    return qs, d


def quantize_rowwise(w: torch.Tensor, bits: int):
    """Per-row-scale int4 (bits=4) or int2 (bits=2) container of w [N][K]:
    (codes uint8 [N][K*bits/8], scales fp32 [N])."""
    N, K = w.shape
    q = torch.empty(N, K * bits // 8, dtype=torch.uint8, device=w.device)
    s = torch.empty(N, dtype=torch.float32, device=w.device)
    qmm_quantize_rowwise(w, N, K, w.stride(0), bits, q, s)
    return q, s


def quantize_q8_0(x: torch.Tensor):
    if x.dim() == 1:
        x = x[None]
    M, K = x.shape
    q = torch.empty(M, K, dtype=torch.int8, device=x.device)
    d = torch.empty(M, K // QK, dtype=torch.int16, device=x.device)
    qmm_quantize_q8_0(x, M, K, x.stride(0), q, d)
    return q, d


def gemv(qs, d, xq, xd, out=None):
    N, K = qs.shape[0], qs.shape[1] * 2
    y = out if out is not None else torch.empty(N, dtype=torch.float32, device=qs.device)
    qmm_gemv_q4_0_q8_0(qs, d, N, K, xq, xd, y)
    return y


def gemm(qs, d, xq, xd, out=None, workspace=None):
    """y = the GEMM of qmm_gemm_q4_0_q8_0; with `workspace` (a uint8 device
    tensor of at least qmm_gemm_workspace_size(K, M) bytes) through
    qmm_gemm_q4_0_q8_0_ws."""
    N, K = qs.shape[0], qs.shape[1] * 2
    M = xq.shape[0]
    y = out if out is not None else torch.empty(M, N, dtype=torch.float32, device=qs.device)
    if workspace is None:
        qmm_gemm_q4_0_q8_0(qs, d, N, K, M, xq, xd, y, y.stride(0))
    else:
        qmm_gemm_q4_0_q8_0_ws(qs, d, N, K, M, xq, xd, y, y.stride(0), workspace, workspace.numel())
    return y
