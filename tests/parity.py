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


def planes_to_oracle(qs, d, N, K):
    """Device Q4_0 planes (qs [N][K/2] uint8, d [N][K/32] fp16 bits) -> the
    oracle's (signed codes [N][K] int8, d [N][K/32] uint16), through the
    page's 18-byte block format."""
    blocks = np.zeros((N, K // QK, 18), np.uint8)
    blocks[..., :2] = u16(d).reshape(N, K // QK, 1).view(np.uint8)
    blocks[..., 2:] = qs.detach().cpu().numpy().reshape(N, K // QK, 16)
    return O.unpack_q4_0_blocks(blocks, N, K)


def check_rmsnorm_q8_0(x, gamma, eps, gq, gd, what=""):
    """The fused RMSNorm -> Q8_0 staging (TinyLLaMA guide 4.1) against the
    definition: the codes must equal, bit for bit, the oracle's Q8_0 codes of
    z = fl(x * gamma) (a block's codes do not change when the block is scaled
    by a positive factor, here 1/rms); each block scale must be within one
    fp16 step of fp16(d32_z / rms), d32_z = fl(max|z_block| / 127), rms in
    float64 from the definition sqrt(mean(x^2) + eps)."""
    x = np.asarray(x, np.float32).reshape(-1)
    gamma = np.asarray(gamma, np.float32).reshape(-1)
    z = x * gamma  # IEEE fp32 products
    qz, _ = O.quantize_q8_0(z[None])
    gq = np.asarray(gq).reshape(-1)
    if not np.array_equal(gq, qz[0]):
        i = int(np.nonzero(gq != qz[0])[0][0])
        raise AssertionError(f"{what}: Q8_0 code {i} is {gq[i]}, the oracle's code of x*gamma is {qz[0][i]}")
    amax = np.abs(z.reshape(-1, QK)).max(axis=1)
    d32z = (amax / np.float32(127.0)).astype(np.float32)
    rms = np.sqrt(np.mean(x.astype(np.float64) ** 2) + eps)
    ref = (d32z.astype(np.float64) / rms).astype(np.float16).view(np.uint16).astype(np.int64)
    got = np.asarray(gd).reshape(-1).astype(np.int64)  # positive fp16 bit patterns
    off = np.abs(got - ref)
    assert (off <= 1).all(), f"{what}: block scale off by {off.max()} fp16 steps at block {int(off.argmax())}"
    return int((off == 1).sum())
