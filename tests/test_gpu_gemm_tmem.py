"""The tcgen05 small-batch GEMM (weight operand in tensor memory) against the
CPU oracle and against the warp-MMA GEMM on the same inputs.

Shapes are chosen for the kernel's row plan on a 152-SM GB300: one partial
MMA tile (rows not a multiple of 32), two tiles per super-tile, several
super-tiles per CTA with a short last CTA, K of one and of several 8-block
chunks, 2..16 tokens.  fp32 outputs: |y - y_ref| <= 1e-5*S + 1e-6; with unit
scales every output is an exact integer and must match bit for bit.  Also
here: the dp4a streaming kernel forced through the same selector
(qmm_debug_gemm_kernel) against the oracle."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity import lib, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture
def qmm():
    q = lib()
    prev = q.qmm_debug_gemm_kernel(q.GEMM_KERNEL_TMEM)
    yield q
    q.qmm_debug_gemm_kernel(prev)


def _rand_codes(N, M, K, seed):
    rng = np.random.default_rng(seed)
    qw = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    dw = rng.integers(0x1000, 0x2C00, size=(N, K // 32)).astype(np.uint16)
    qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    dx = rng.integers(0x1000, 0x3C00, size=(M, K // 32)).astype(np.uint16)
    return qw, dw, qx, dx


def _planes(q, qw, dw):
    N, K = qw.shape
    blocks = torch.from_numpy(O.pack_q4_0_blocks(qw, dw).reshape(-1).copy()).to(DEV)
    qs, d = q.q4_0_planes(N, K)
    q.qmm_repack_q4_0(blocks, N, K, qs, d)
    return qs, d


def _q8(qx, dx):
    return torch.from_numpy(qx).to(DEV), torch.from_numpy(dx.view(np.int16)).to(DEV)


@pytest.mark.parametrize("N,M,K", [(300, 16, 2048), (4100, 2, 256), (40000, 7, 512)])
def test_tmem_gemm_integer_grid_exact(qmm, N, M, K):
    """Unit scales: y is the exact integer product W x, so a wrong TMEM or
    shared-memory operand layout, a K-slot permutation that differs between
    A and B, or any loss in the MMA's fp32 sums shows as an inequality.
    Every nibble value (-8 included) and the full int8 range occur."""
    rng = np.random.default_rng(N + M)
    qw = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    qw[:7, :32] = -8
    qw[7:14, :32] = 7
    qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    qx[0, :32] = -127
    qx[-1, 32:64] = 127
    one = np.uint16(0x3C00)
    qs, d = _planes(qmm, qw, np.full((N, K // 32), one, np.uint16))
    xq, xd = _q8(qx, np.full((M, K // 32), one, np.uint16))
    y = qmm.gemm(qs, d, xq, xd)
    exact = (qx.astype(np.int64) @ qw.astype(np.int64).T).astype(np.float32)
    assert np.array_equal(y.cpu().numpy(), exact)
    assert qmm.qmm_last_device_error() == 0


@pytest.mark.parametrize("N,M,K", [(1, 2, 256), (13, 16, 768), (129, 5, 256), (2200, 16, 2048),
                                   (20000, 3, 768), (40000, 16, 512), (45600, 9, 256)])
def test_tmem_gemm_vs_oracle(qmm, N, M, K):
    """Random codes and scales, every output row against the oracle."""
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=N * 7 + M)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    y = qmm.gemm(qs, d, xq, xd)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y, ref, S, f"tmem gemm {N}x{K} M={M}")
    assert qmm.qmm_last_device_error() == 0


@pytest.mark.parametrize("M", [2, 16])
def test_tmem_and_warp_mma_kernels_agree(qmm, M):
    """The two GEMM kernels on the same inputs: both within the tolerance of
    each other (they differ only in the order of the fp32 block sums)."""
    N, K = 30000, 1024
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=M)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    y_tm = qmm.gemm(qs, d, xq, xd)
    qmm.qmm_debug_gemm_kernel(qmm.GEMM_KERNEL_MMA)
    y_mma = qmm.gemm(qs, d, xq, xd)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y_tm, ref, S, "tmem")
    assert_close(y_mma, ref, S, "warp mma")
    assert_close(y_tm, y_mma.cpu().numpy().astype(np.float64), 2 * S, "tmem vs warp mma")


def test_tmem_gemm_ldy(qmm):
    """Output row stride above N: the columns past N keep their contents."""
    N, K, M, ldy = 1000, 512, 16, 1040
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=3)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    y = torch.full((M, ldy), 7.0, device=DEV)
    qmm.qmm_gemm_q4_0_q8_0(qs, d, N, K, M, xq, xd, y, ldy)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y[:, :N], ref, S, "tmem ldy")
    assert torch.all(y[:, N:] == 7.0)


def test_tmem_gemm_rejects_what_it_cannot_take(qmm):
    """Forced onto the tensor-memory kernel, 17 tokens or K % 256 != 0 is a
    shape error and nothing is written; the selector rejects an unknown kernel."""
    N, K = 64, 512
    qw, dw, qx, dx = _rand_codes(N, 17, K, seed=5)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    y = torch.full((17, N), 7.0, device=DEV)
    with pytest.raises(qmm.QmmError) as ei:
        qmm.qmm_gemm_q4_0_q8_0(qs, d, N, K, 17, xq, xd, y, N)
    assert ei.value.status == 2
    qw2, dw2, qx2, dx2 = _rand_codes(N, 4, 96, seed=6)
    qs2, d2 = _planes(qmm, qw2, dw2)
    xq2, xd2 = _q8(qx2, dx2)
    y2 = torch.full((4, N), 7.0, device=DEV)
    with pytest.raises(qmm.QmmError) as ei:
        qmm.qmm_gemm_q4_0_q8_0(qs2, d2, N, 96, 4, xq2, xd2, y2, N)
    assert ei.value.status == 2
    assert torch.all(y == 7.0) and torch.all(y2 == 7.0)
    with pytest.raises(qmm.QmmError):
        qmm.qmm_debug_gemm_kernel(5)


@pytest.mark.parametrize("N,K,M", [(517, 2048, 2), (20000, 8192, 3), (300, 512, 5), (129, 256, 9)])
def test_streaming_kernel_selected_vs_oracle(N, K, M):
    """The dp4a streaming path forced for 2..9 tokens (one or two passes of
    up to 8 tokens over the weights) against the oracle."""
    q = lib()
    prev = q.qmm_debug_gemm_kernel(q.GEMM_KERNEL_STREAM)
    try:
        qw, dw, qx, dx = _rand_codes(N, M, K, seed=N + M)
        qs, d = _planes(q, qw, dw)
        xq, xd = _q8(qx, dx)
        y = q.gemm(qs, d, xq, xd)
        ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
        assert_close(y, ref, S, f"stream gemm {N}x{K} M={M}")
        assert q.qmm_last_device_error() == 0
    finally:
        q.qmm_debug_gemm_kernel(prev)
