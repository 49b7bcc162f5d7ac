"""Shared helpers of the GPU parity tests: the fp32 tolerance, conversions
between torch device tensors and the oracle's numpy arrays."""
import numpy as np
import torch

from oracle import oracle as O

QK = 32


def lib():
    from block_quantized_int4_gb300 import _build
    _build.build()
    from block_quantized_int4_gb300 import qmm
    return qmm


def u16(t: torch.Tensor) -> np.ndarray:
    """fp16 bit patterns held in an int16 tensor -> numpy uint16."""
    return t.detach().cpu().numpy().view(np.uint16)


def assert_close(y_gpu, y_ref, S, what=""):
    """|y_gpu - y_ref| <= 1e-5 * S + 1e-6 elementwise, S = sum_b |d_w d_x dot_b|."""
    y = y_gpu.detach().cpu().numpy().astype(np.float64) if isinstance(y_gpu, torch.Tensor) else y_gpu
    err = np.abs(y - y_ref)
    bound = 1e-5 * S + 1e-6
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outputs off tolerance; worst at {i}: "
                             f"gpu {y[i]!r} oracle {y_ref[i]!r} err {err[i]:.3g} bound {bound[i]:.3g}")
    return float(err.max()) if err.size else 0.0


def oracle_weights(w_cpu):
    """Oracle Q4_0 of fp32 weights (numpy) -> (signed q, d bits)."""
    return O.quantize_q4_0(np.ascontiguousarray(w_cpu, dtype=np.float32))


def planes_from_oracle(q, d):
    """Oracle signed codes -> the device plane bytes (as numpy), for comparing
    with what the GPU quantizer wrote: qs [N][K/2] bytes, d [N][B] uint16."""
    blocks = O.pack_q4_0_blocks(q, d)  # [N][B][18]
    N = q.shape[0]
    qs = np.ascontiguousarray(blocks[..., 2:]).reshape(N, -1)
    return qs, d
