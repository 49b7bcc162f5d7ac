"""Weight-format variants against the oracle: the per-row-scale int4 / int2
container (Colibri page, "Arquitectura del Sistema") -- quantizer bit-exact,
GEMV with Q8_0 activations within the fp32 tolerance -- and the Q4_0 x fp32
dequantize-then-FMA GEMV (TinyLLaMA guide 6.2) within the same tolerance,
S = sum_k |d_w q_w x| for the latter."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import workloads
from parity import lib, u16, assert_close, oracle_weights, planes_from_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _weights(N, K, seed, sigma=0.02, outliers=True):
    w = workloads.weights(N, K, sigma=sigma, seed=seed, index=500)
    if outliers and N > 3:
        w[1] = 0.0                     # a zero row
        w[2, K // 3] = 0.5             # an outlier
    return w


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("N,K", [(37, 128), (5, 64), (300, 2048), (4096, 8192)])
def test_quantize_rowwise_bit_exact(bits, N, K):
    qmm = lib()
    w = _weights(N, K, seed=N + K)
    q, s = qmm.quantize_rowwise(w.to(DEV), bits)
    rq, rs = O.quantize_rowwise(w.numpy(), bits)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), O.pack_rowwise(rq, bits))


def _rowwise_case(qmm, bits, N, K, seed, random_codes=False):
    if random_codes:  # every code value, including -2^(bits-1), which the quantizer never writes
        g = torch.Generator().manual_seed(seed)
        q = torch.randint(0, 256, (N, K * bits // 8), generator=g, dtype=torch.uint8)
        s = torch.rand(N, generator=g) * 0.05 + 1e-3
        q, s = q.to(DEV), s.to(DEV)
    else:
        q, s = qmm.quantize_rowwise(_weights(N, K, seed=seed).to(DEV), bits)
    x = workloads.activations(1, K, seed=seed + 1)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    y = torch.full((N,), float("nan"), device=DEV)
    qmm.qmm_gemv_rowwise_q8_0(q, s, bits, N, K, xq, xd, y)
    codes = O.unpack_rowwise(q.cpu().numpy(), K, bits)
    return y, codes, s.cpu().numpy(), xq.cpu().numpy(), u16(xd)


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("N,K", [(1, 64), (7, 128), (130, 1024 + 64), (1001, 2048), (333, 8192), (64, 28672)])
def test_gemv_rowwise_matches_oracle(bits, N, K):
    """All rows, ragged N (not a multiple of the 4-row warp pass or of the
    grid), K not a multiple of one warp step."""
    qmm = lib()
    y, codes, s, xq, xd = _rowwise_case(qmm, bits, N, K, seed=3 * N + bits)
    ref, S = O.matmul_rowwise_int(codes, s, xq, xd)
    assert_close(y[None], ref, S, f"int{bits} rowwise {N}x{K}")


@pytest.mark.parametrize("bits", [4, 2])
def test_gemv_rowwise_every_code(bits):
    qmm = lib()
    N, K = 203, 4096
    y, codes, s, xq, xd = _rowwise_case(qmm, bits, N, K, seed=11, random_codes=True)
    assert set(np.unique(codes)) == set(range(-(2 ** (bits - 1)), 2 ** (bits - 1)))
    ref, S = O.matmul_rowwise_int(codes, s, xq, xd)
    assert_close(y[None], ref, S, f"int{bits} every code")


@pytest.mark.parametrize("bits", [4, 2])
def test_gemv_rowwise_full_size_sampled_rows(bits):
    """Large dense gate shape, 28672 x 8192: sampled rows against the oracle,
    every output finite."""
    qmm = lib()
    N, K = 28672, 8192
    w = workloads.weights(N, K, sigma=0.01, seed=0, index=501, device=DEV)
    q, s = qmm.quantize_rowwise(w, bits)
    x = workloads.activations(1, K, seed=5)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    y = torch.empty(N, device=DEV)
    qmm.qmm_gemv_rowwise_q8_0(q, s, bits, N, K, xq, xd, y)
    assert torch.isfinite(y).all()
    rows = np.array([0, 1, 4095, 4096, 17777, N - 5, N - 1])
    ri = torch.from_numpy(rows).to(DEV)
    codes = O.unpack_rowwise(q[ri].cpu().numpy(), K, bits)
    ref, S = O.matmul_rowwise_int(codes, s.cpu().numpy()[rows], xq.cpu().numpy(), u16(xd))
    assert_close(y[ri][None], ref, S, f"int{bits} full size")


def _fma_case(qmm, N, K, seed, random_codes=False):
    if random_codes:
        g = torch.Generator().manual_seed(seed)
        qs = torch.randint(0, 256, (N, K // 2), generator=g, dtype=torch.uint8)
        d = (torch.rand(N, K // 32, generator=g) * 0.02).half().view(torch.int16)
        qs, d = qs.to(DEV), d.to(DEV)
        q = O.unpack_q4_0_blocks(_blocks(qs, d, N, K), N, K)[0]
        dn = u16(d)
    else:
        w = _weights(N, K, seed=seed)
        q, dn = oracle_weights(w.numpy())
        qs_np, _ = planes_from_oracle(q, dn)
        qs = torch.from_numpy(qs_np).to(DEV)
        d = torch.from_numpy(dn.view(np.int16)).to(DEV)
    x = workloads.activations(1, K, seed=seed + 1)[0]
    y = torch.full((N,), float("nan"), device=DEV)
    qmm.qmm_gemv_q4_0_f32_fma(qs, d, N, K, x.to(DEV), y)
    return y, q, dn, x.numpy()


def _blocks(qs, d, N, K):
    blocks = np.zeros((N, K // 32, 18), np.uint8)
    blocks[..., :2] = u16(d).reshape(N, K // 32, 1).view(np.uint8)
    blocks[..., 2:] = qs.cpu().numpy().reshape(N, K // 32, 16)
    return blocks


@pytest.mark.parametrize("N,K", [(1, 32), (6, 96), (131, 1024 + 32), (1001, 2048), (200, 8192), (40, 28672),
                                 (9, 49152)])
def test_gemv_f32_fma_matches_oracle(N, K):
    qmm = lib()
    y, q, d, x = _fma_case(qmm, N, K, seed=N + 7)
    ref, S = O.matmul_q4_0_f32(q, d, x)
    assert_close(y[None], ref, S, f"f32 fma {N}x{K}")


def test_gemv_f32_fma_every_code_and_full_size():
    qmm = lib()
    y, q, d, x = _fma_case(qmm, 257, 4096, seed=21, random_codes=True)
    assert set(np.unique(q)) == set(range(-8, 8))
    ref, S = O.matmul_q4_0_f32(q, d, x)
    assert_close(y[None], ref, S, "f32 fma every code")
    # the large dense down shape, 8192 x 28672, sampled rows
    N, K = 8192, 28672
    w = workloads.weights(N, K, sigma=0.01, seed=0, index=502, device=DEV)
    qs, dd = qmm.quantize_q4_0(w)
    xx = workloads.activations(1, K, seed=6)[0]
    yy = torch.empty(N, device=DEV)
    qmm.qmm_gemv_q4_0_f32_fma(qs, dd, N, K, xx.to(DEV), yy)
    assert torch.isfinite(yy).all()
    ri = torch.tensor([0, 3, 4, 5000, N - 1], device=DEV)
    qr = O.unpack_q4_0_blocks(_blocks(qs[ri], dd[ri], len(ri), K), len(ri), K)[0]
    ref, S = O.matmul_q4_0_f32(qr, u16(dd[ri]), xx.numpy())
    assert_close(yy[ri][None], ref, S, "f32 fma full size")
