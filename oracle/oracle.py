"""Python face of the CPU oracle (``qmm_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the test suite, by the smoke check and
by the bench's CPU-baseline / reference leg, never by the product library.
It shares no code with the CUDA path.

Every function takes and returns numpy arrays; the arithmetic lives in the C
file, whose header cites the passages each routine follows:

* Q4_0 block format -- TinyLLaMA C++ guide (kenji.blog), section 6.1.
* Block quantization ``w ~ Delta*q``, ``Delta = max|w|/7``, quantized dot
  ``y ~ Delta*Delta_x*sum q*q_x`` -- llama.cpp guide (kenji.blog/id), section 2.2.
* Q8_0-style int8 activations, sigmoid router -- Colibri page
  (kerneldigest.dev), system architecture.
* SwiGLU -- TinyLLaMA C++ guide, section 4.4.
* Per-row-scale int4/int2 containers -- Colibri page, system architecture
  (layout and scale rule are readings).
* Q4_0 x fp32 dequantize-then-FMA -- TinyLLaMA C++ guide, section 6.2.

Parity status: the fp16 conversion, both quantizers, the block dots, both
output paths, SwiGLU, RMSNorm and the router are pinned by the CPU tests.  The
router's normalisation over the k and its tie-break are a reading of a silent
page; the router is pinned to that reading (stable argsort, library sigmoid).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_LIB = os.path.join(_HERE, "libqmm_oracle.so")
_lock = threading.Lock()
_lib = None

QK = 32


def build(force: bool = False) -> str:
    """Compile the oracle with plain gcc (IEEE float: no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int64
            lib.oq_f32_to_f16.restype = ctypes.c_uint16
            lib.oq_f32_to_f16.argtypes = [ctypes.c_float]
            lib.oq_f16_to_f32.restype = ctypes.c_float
            lib.oq_f16_to_f32.argtypes = [ctypes.c_uint16]
            for name, args in {
                "oq_f32_to_f16_array": [P, P, I],
                "oq_f16_to_f32_array": [P, P, I],
                "oq_quantize_q8_0": [P, I, I, I, P, P],
                "oq_quantize_q4_0": [P, I, I, I, P, P],
                "oq_pack_q4_0_blocks": [P, P, I, I, P],
                "oq_unpack_q4_0_blocks": [P, I, I, P, P],
                "oq_block_dots": [P, I, I, P, I, P],
                "oq_matmul_int": [P, P, I, I, P, P, I, P, I, P, P, ctypes.c_int],
                "oq_matmul_dequant": [P, P, I, I, P, P, I, P],
                "oq_router_topk": [P, I, I, I, P, P],
                "oq_swiglu": [P, P, I, P],
                "oq_moe_combine": [P, P, I, I, I, P],
                "oq_rmsnorm": [P, P, I, ctypes.c_double, P],
                "oq_quantize_rowwise": [P, I, I, I, ctypes.c_int, P, P],
                "oq_pack_rowwise": [P, I, I, ctypes.c_int, P],
                "oq_unpack_rowwise": [P, I, I, ctypes.c_int, P],
                "oq_matmul_rowwise_int": [P, P, I, I, P, P, I, P, P],
                "oq_matmul_q4_0_f32": [P, P, I, I, P, I, P, P],
            }.items():
                f = getattr(lib, name)
                f.restype = None
                f.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- fp16
def f32_to_f16_bits(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().oq_f32_to_f16_array(_p(x), _p(out), x.size)
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    _load().oq_f16_to_f32_array(_p(h), _p(out), h.size)
    return out


# ---------------------------------------------------------------- quantizers
def quantize_q8_0(x):
    """x [M][K] fp32 -> (q int8 [M][K], d fp16-bits uint16 [M][K/32])."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None]
    M, K = x.shape
    assert K % QK == 0
    q = np.empty((M, K), np.int8)
    d = np.empty((M, K // QK), np.uint16)
    _load().oq_quantize_q8_0(_p(x), M, K, K, _p(q), _p(d))
    return q, d


def quantize_q4_0(w):
    """w [N][K] fp32 -> (signed q int8 [N][K] in [-8,7], d fp16-bits [N][K/32])."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % QK == 0
    q = np.empty((N, K), np.int8)
    d = np.empty((N, K // QK), np.uint16)
    _load().oq_quantize_q4_0(_p(w), N, K, K, _p(q), _p(d))
    return q, d


def pack_q4_0_blocks(q, d) -> np.ndarray:
    """Signed q + scales -> the page's 18-byte blocks, uint8 [N][K/32][18]."""
    q = _c(q, np.int8)
    d = _c(d, np.uint16)
    N, K = q.shape
    out = np.empty((N, K // QK, 18), np.uint8)
    _load().oq_pack_q4_0_blocks(_p(q), _p(d), N, K, _p(out))
    return out


def unpack_q4_0_blocks(blocks, N, K):
    blocks = _c(blocks, np.uint8)
    q = np.empty((N, K), np.int8)
    d = np.empty((N, K // QK), np.uint16)
    _load().oq_unpack_q4_0_blocks(_p(blocks), N, K, _p(q), _p(d))
    return q, d


# ---------------------------------------------------------------- products
def block_dots(qw, qx) -> np.ndarray:
    """int32 [M][N][K/32] per-block integer dots."""
    qw = _c(qw, np.int8)
    qx = _c(qx, np.int8)
    if qx.ndim == 1:
        qx = qx[None]
    N, K = qw.shape
    M = qx.shape[0]
    out = np.empty((M, N, K // QK), np.int32)
    _load().oq_block_dots(_p(qw), N, K, _p(qx), M, _p(out))
    return out


def matmul_int(qw, dw, qx, dx, rows=None, nthreads: int = 1):
    """Integer block-dot path, float64 combine.

    Returns (y, S), both float64 [M][nrows]; S = sum_b |dw*dx*dot| is the
    scale of the fp32 tolerance.  ``rows`` selects output rows (default all).
    """
    qw = _c(qw, np.int8)
    dw = _c(dw, np.uint16)
    qx = _c(qx, np.int8)
    dx = _c(dx, np.uint16)
    if qx.ndim == 1:
        qx, dx = qx[None], dx[None]
    N, K = qw.shape
    M = qx.shape[0]
    assert qx.shape[1] == K and dw.shape == (N, K // QK) and dx.shape == (M, K // QK)
    if rows is None:
        nrows, rp = N, None
    else:
        rows = _c(rows, np.int64)
        assert rows.min() >= 0 and rows.max() < N
        nrows, rp = rows.size, _p(rows)
    y = np.empty((M, nrows), np.float64)
    S = np.empty((M, nrows), np.float64)
    _load().oq_matmul_int(_p(qw), _p(dw), N, K, _p(qx), _p(dx), M, rp, nrows, _p(y), _p(S), int(nthreads))
    return y, S


def matmul_dequant(qw, dw, qx, dx) -> np.ndarray:
    """Dequantize-then-multiply path, float64 [M][N]."""
    qw = _c(qw, np.int8)
    dw = _c(dw, np.uint16)
    qx = _c(qx, np.int8)
    dx = _c(dx, np.uint16)
    if qx.ndim == 1:
        qx, dx = qx[None], dx[None]
    N, K = qw.shape
    M = qx.shape[0]
    y = np.empty((M, N), np.float64)
    _load().oq_matmul_dequant(_p(qw), _p(dw), N, K, _p(qx), _p(dx), M, _p(y))
    return y


# ---------------------------------------------------------------- per-row containers
def quantize_rowwise(w, bits: int):
    """Per-row-scale int4 (bits=4) or int2 (bits=2) codes of w [N][K] (Colibri
    page's per-row-scale container): (q int8 [N][K], s fp32 [N])."""
    assert bits in (2, 4)
    w = _c(w, np.float32)
    N, K = w.shape
    q = np.empty((N, K), np.int8)
    s = np.empty(N, np.float32)
    _load().oq_quantize_rowwise(_p(w), N, K, K, bits, _p(q), _p(s))
    return q, s


def pack_rowwise(q, bits: int) -> np.ndarray:
    """Codes u = q + 2^(bits-1), 8/bits per byte, low bits first: uint8 [N][K*bits/8]."""
    q = _c(q, np.int8)
    N, K = q.shape
    out = np.empty((N, K * bits // 8), np.uint8)
    _load().oq_pack_rowwise(_p(q), N, K, bits, _p(out))
    return out


def unpack_rowwise(packed, K: int, bits: int) -> np.ndarray:
    packed = _c(packed, np.uint8)
    N = packed.shape[0]
    q = np.empty((N, K), np.int8)
    _load().oq_unpack_rowwise(_p(packed), N, K, bits, _p(q))
    return q


def matmul_rowwise_int(qw, s, qx, dx):
    """Per-row codes x Q8_0 activations: (y, S) float64 [M][N]."""
    qw = _c(qw, np.int8)
    s = _c(s, np.float32)
    qx = _c(qx, np.int8)
    dx = _c(dx, np.uint16)
    if qx.ndim == 1:
        qx, dx = qx[None], dx[None]
    N, K = qw.shape
    M = qx.shape[0]
    assert s.shape == (N,) and qx.shape[1] == K and dx.shape == (M, K // QK)
    y = np.empty((M, N), np.float64)
    S = np.empty((M, N), np.float64)
    _load().oq_matmul_rowwise_int(_p(qw), _p(s), N, K, _p(qx), _p(dx), M, _p(y), _p(S))
    return y, S


def matmul_q4_0_f32(qw, dw, x):
    """Q4_0 weights x fp32 activations, dequantize-then-multiply (TinyLLaMA
    guide 6.2): (y, S) float64 [M][N]."""
    qw = _c(qw, np.int8)
    dw = _c(dw, np.uint16)
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None]
    N, K = qw.shape
    M = x.shape[0]
    assert dw.shape == (N, K // QK) and x.shape[1] == K
    y = np.empty((M, N), np.float64)
    S = np.empty((M, N), np.float64)
    _load().oq_matmul_q4_0_f32(_p(qw), _p(dw), N, K, _p(x), M, _p(y), _p(S))
    return y, S


# ---------------------------------------------------------------- MoE
def router_topk(logits, k: int):
    """Sigmoid scores, top-k (ties -> lower index), gates normalised over the k.
    logits [T][E] fp32 -> (ids int32 [T][k], gates float64 [T][k]).  The
    selection compares the double sigmoid of each fp32 logit, injective over
    logits in [-87, 16]; outside that range ties may appear."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    gates = np.empty((T, k), np.float64)
    _load().oq_router_topk(_p(logits), T, E, k, _p(ids), _p(gates))
    return ids, gates


def swiglu(a, b) -> np.ndarray:
    """h = a*sigmoid(a)*b in float64, rounded once to fp32."""
    a = _c(a, np.float64)
    b = _c(b, np.float64)
    assert a.shape == b.shape
    h = np.empty(a.shape, np.float32)
    _load().oq_swiglu(_p(a), _p(b), a.size, _p(h))
    return h


def rmsnorm(x, gamma, eps: float = 1e-5) -> np.ndarray:
    """RMSNorm of each row of x (fp32 [..., d]) with weight gamma [d], in
    double, rounded once to fp32 (TinyLLaMA guide 4.1)."""
    x = _c(x, np.float32)
    gamma = _c(gamma, np.float32)
    d = x.shape[-1]
    assert gamma.shape == (d,)
    rows = x.reshape(-1, d)
    out = np.empty_like(rows)
    for r in range(rows.shape[0]):
        row = np.ascontiguousarray(rows[r])
        o = np.empty(d, np.float32)
        _load().oq_rmsnorm(_p(row), _p(gamma), d, ctypes.c_double(eps), _p(o))
        out[r] = o
    return out.reshape(x.shape)


def moe_combine(z, gates) -> np.ndarray:
    """z [T][k][N] float64, gates [T][k] fp32 -> y [T][N] = sum_j g_j z_j (j ascending)."""
    z = _c(z, np.float64)
    gates = _c(gates, np.float32)
    T, k, N = z.shape
    y = np.empty((T, N), np.float64)
    _load().oq_moe_combine(_p(z), _p(gates), T, k, N, _p(y))
    return y


def moe_forward(experts_gate, experts_up, experts_down, ids, gates, qx, dx):
    """End-to-end oracle MoE layer for T tokens.

    experts_* : dict e -> (q, d) for every expert id used.  Gate/up are
    [F][H], down is [H][F].  qx/dx : Q8_0 of the token activations [T][H].
    Per slot j: a = W_gate x, b = W_up x (integer path), h = silu(a)*b -> fp32
    -> Q8_0, z_j = W_down h; then y = sum_j g_j z_j.  Returns (y [T][H], z, h).
    """
    T, k = ids.shape
    H = qx.shape[1]
    z = np.zeros((T, k, H), np.float64)
    hs = []
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            a, _ = matmul_int(*experts_gate[e], qx[t], dx[t])
            b, _ = matmul_int(*experts_up[e], qx[t], dx[t])
            h = swiglu(a[0], b[0])
            hq, hd = quantize_q8_0(h[None])
            zz, _ = matmul_int(*experts_down[e], hq, hd)
            z[t, j] = zz[0]
            hs.append(h)
    return moe_combine(z, gates), z, np.stack(hs).reshape(T, k, -1)
