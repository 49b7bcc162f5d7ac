"""GPU quantizers against the CPU oracle, bit-exact: Q8_0 activations, Q4_0
weights, the page-format repack, SwiGLU + Q8_0."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import workloads
from parity import lib, u16, planes_from_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _adversarial(M, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g)
    x[0, :32] = 0  # zero block
    for lane in range(min(32, K // 32)):  # amax at every lane
        x[0, 32 * lane + lane] = 9.0 * (-1) ** lane
    if M > 1:
        x[1, :32] = torch.arange(32) - 16.0  # exact .5 ties
        x[1, 32:64] = torch.arange(32) - 16.5
        x[1, 32] = 127.0
    return x


@pytest.mark.parametrize("M,K", [(1, 2048), (3, 96), (7, 5632), (16, 8192), (64, 2048)])
def test_q8_0_bit_exact(M, K):
    qmm = lib()
    x = workloads.activations(M, K, seed=M)
    if M > 1:
        x[:2] = _adversarial(2, K, 5)
    q, d = qmm.quantize_q8_0(x.to(DEV))
    qo, do = O.quantize_q8_0(x.numpy())
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(u16(d), do)


def test_q8_0_row_stride_and_tail():
    qmm = lib()
    M, K, ld = 5, 160, 200
    xs = workloads.activations(M, ld, seed=3)
    x = xs.to(DEV)
    q = torch.full((M, K), 99, dtype=torch.int8, device=DEV)
    d = torch.zeros(M, K // 32, dtype=torch.int16, device=DEV)
    qmm.qmm_quantize_q8_0(x, M, K, ld, q, d)
    qo, do = O.quantize_q8_0(xs[:, :K].contiguous().numpy())
    assert np.array_equal(q.cpu().numpy(), qo) and np.array_equal(u16(d), do)


@pytest.mark.parametrize("N,K", [(1, 32), (37, 2048), (2560, 2048), (64, 5632)])
def test_q4_0_bit_exact(N, K):
    qmm = lib()
    w = workloads.weights(N, K, seed=1, index=N)
    w[0, :32] = 0
    if K >= 64:
        w[0, 32:64] = torch.tensor([0.07, -0.035, 0.005, -0.0049, 0.015, -0.015, 0, 0.064] + [0] * 24)
    qs, d = qmm.quantize_q4_0(w.to(DEV))
    q, do = O.quantize_q4_0(w.numpy())
    qs_ref, d_ref = planes_from_oracle(q, do)
    assert np.array_equal(qs.cpu().numpy(), qs_ref)
    assert np.array_equal(u16(d), d_ref)


def test_repack_from_page_blocks():
    """Page-format 18-byte blocks (from the oracle's packer) -> device planes."""
    qmm = lib()
    N, K = 33, 256
    rng = np.random.default_rng(0)
    q = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    d = rng.integers(0, 0x7C00, size=(N, K // 32)).astype(np.uint16)
    blocks = torch.from_numpy(O.pack_q4_0_blocks(q, d).reshape(-1).copy()).to(DEV)
    qs, dd = qmm.q4_0_planes(N, K)
    qmm.qmm_repack_q4_0(blocks, N, K, qs, dd)
    qs_ref, d_ref = planes_from_oracle(q, d)
    assert np.array_equal(qs.cpu().numpy(), qs_ref) and np.array_equal(u16(dd), d_ref)


@pytest.mark.parametrize("rows,K", [(1, 5632), (16, 2048), (3, 96)])
def test_swiglu_quantize(rows, K):
    """h within a few fp32 ulp of the oracle's double SwiGLU; Q8_0 of the GPU's
    own h bit-exact against the oracle quantizer."""
    qmm = lib()
    g = workloads.activations(rows, K, seed=11) * 3
    u = workloads.activations(rows, K, seed=12)
    q = torch.empty(rows, K, dtype=torch.int8, device=DEV)
    d = torch.empty(rows, K // 32, dtype=torch.int16, device=DEV)
    h = torch.empty(rows, K, dtype=torch.float32, device=DEV)
    qmm.qmm_swiglu_quantize_q8_0(g.to(DEV), u.to(DEV), rows, K, K, q, d, h)
    h_ref = O.swiglu(g.numpy().astype(np.float64), u.numpy().astype(np.float64))
    hg = h.cpu().numpy()
    # fp32 expf (<= 2 ulp), add, divide, multiply, each rounded: 8 ulp of h is a safe
    # bound; the absolute 1e-30 covers gate < -88, where expf(-gate) overflows to inf
    # and the GPU's h is 0 while the true value is below 1e-36.
    ulp = np.spacing(np.abs(h_ref).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(hg.astype(np.float64) - h_ref) <= 8 * ulp + 1e-30)
    qo, do = O.quantize_q8_0(hg)
    assert np.array_equal(q.cpu().numpy(), qo) and np.array_equal(u16(d), do)


def test_q8_0_bit_exact_across_scales():
    """Blocks whose magnitudes span 1e-30 .. 1e30 (scale of each block drawn
    log-uniformly), plus exact .5 ties at many scales: the GPU quantizer's
    division must agree with the oracle's IEEE division everywhere."""
    qmm = lib()
    g = torch.Generator().manual_seed(21)
    M, K = 64, 8192
    x = torch.randn(M, K, generator=g)
    scale = torch.pow(10.0, torch.empty(M, K // 32).uniform_(-30, 30, generator=g))
    x = (x.view(M, K // 32, 32) * scale[..., None]).view(M, K)
    ties = (torch.arange(32) - 16 + 0.5)
    for b in range(0, K // 32, 7):
        s = float(2.0 ** ((b % 61) - 30))
        x[0, 32 * b:32 * b + 32] = ties * s
        x[0, 32 * b] = 127 * s
    q, d = qmm.quantize_q8_0(x.to(DEV))
    qo, do = O.quantize_q8_0(x.numpy())
    assert np.array_equal(u16(d), do)
    assert np.array_equal(q.cpu().numpy(), qo)
