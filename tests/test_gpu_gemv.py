"""GPU GEMV / small-batch GEMM / block dots against the CPU oracle.

Block dots: bit-exact.  fp32 outputs: |y_gpu - y_ref| <= 1e-5*S + 1e-6 with
S = sum_b |d_w d_x dot_b| (the oracle computes y and S in float64)."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import workloads
from parity import lib, u16, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rand_codes(N, M, K, seed):
    """Random codes using every nibble value (including -8) and random scales."""
    rng = np.random.default_rng(seed)
    qw = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    dw = rng.integers(0x1000, 0x2C00, size=(N, K // 32)).astype(np.uint16)
    qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    dx = rng.integers(0x1000, 0x3C00, size=(M, K // 32)).astype(np.uint16)
    return qw, dw, qx, dx


def _to_device_planes(qmm, qw, dw):
    N, K = qw.shape
    blocks = torch.from_numpy(O.pack_q4_0_blocks(qw, dw).reshape(-1).copy()).to(DEV)
    qs, d = qmm.q4_0_planes(N, K)
    qmm.qmm_repack_q4_0(blocks, N, K, qs, d)
    return qs, d


def _dev_q8(qx, dx):
    return torch.from_numpy(qx).to(DEV), torch.from_numpy(dx.view(np.int16)).to(DEV)


@pytest.mark.parametrize("N,M,K", [(1, 1, 32), (13, 3, 96), (70, 2, 2048), (9, 5, 5632)])
def test_block_dots_bit_exact(N, M, K):
    qmm = lib()
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=N + K)
    qs, d = _to_device_planes(qmm, qw, dw)
    xq, _ = _dev_q8(qx, dx)
    dots = torch.empty(M, N, K // 32, dtype=torch.int32, device=DEV)
    qmm.qmm_debug_block_dots(qs, N, K, M, xq, dots)
    assert np.array_equal(dots.cpu().numpy(), O.block_dots(qw, qx))


@pytest.mark.parametrize("N,K", [(1, 32), (7, 64), (257, 96), (1000, 2048), (2048, 2048), (33, 5632), (100, 28672)])
def test_gemv_random_codes(N, K):
    """Random nibbles incl. -8; rows not a multiple of the 8-row tile; K from one block to 896."""
    qmm = lib()
    qw, dw, qx, dx = _rand_codes(N, 1, K, seed=7 * N + K)
    qs, d = _to_device_planes(qmm, qw, dw)
    xq, xd = _dev_q8(qx, dx)
    y = qmm.gemv(qs, d, xq[0], xd[0])
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y[None], ref, S, f"gemv {N}x{K}")


def test_gemv_integer_grid_exact():
    """d = 1 on both sides: the GEMV is the exact integer product."""
    qmm = lib()
    rng = np.random.default_rng(3)
    N, K = 300, 2048
    w = rng.integers(-7, 8, size=(N, K)).astype(np.float32)
    w[:, ::32] = 7
    x = rng.integers(-127, 128, size=(1, K)).astype(np.float32)
    x[:, 3::32] = 127
    qs, d = qmm.quantize_q4_0(torch.from_numpy(w).to(DEV))
    xq, xd = qmm.quantize_q8_0(torch.from_numpy(x).to(DEV))
    y = qmm.gemv(qs, d, xq[0], xd[0])
    exact = (w.astype(np.int64) @ x[0].astype(np.int64)).astype(np.float32)
    assert np.array_equal(y.cpu().numpy(), exact)


def test_single_gemv_2048_seeded():
    """The 2048 x 2048 single GEMV: W ~ N(0, 0.02), x ~ N(0,1) with 1% x20 outliers, seed 0."""
    qmm = lib()
    c = workloads.SINGLE_GEMV
    w = workloads.weights(c["N"], c["K"], sigma=c["sigma"], seed=0, index=0)
    x = workloads.activations(1, c["K"], seed=0)
    qs, d = qmm.quantize_q4_0(w.to(DEV))
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    y = qmm.gemv(qs, d, xq[0], xd[0])
    qw, dw = O.quantize_q4_0(w.numpy())
    qx, dx = O.quantize_q8_0(x.numpy())
    assert np.array_equal(xq.cpu().numpy(), qx) and np.array_equal(u16(xd), dx)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y[None], ref, S, "single gemv")


@pytest.mark.parametrize("gate_up", [0, 1])
@pytest.mark.parametrize("N,K", [(2560, 2048), (2048, 5632), (31, 96), (32000, 2048), (3, 8192), (300, 28672)])
def test_fused_f32_gemv(gate_up, N, K):
    """fp32 activation quantized inside the GEMV launch: the Q8_0 it writes is
    bit-exact with the oracle quantizer (of SwiGLU(gate, up) in gate_up mode,
    fed the GPU's own h), and y is within tolerance."""
    qmm = lib()
    w = workloads.weights(N, K, seed=2, index=N)
    xin = workloads.activations(1, K * (2 if gate_up else 1), seed=4)[0]
    qs, d = qmm.quantize_q4_0(w.to(DEV))
    y = torch.empty(N, dtype=torch.float32, device=DEV)
    xq = torch.empty(K, dtype=torch.int8, device=DEV)
    xd = torch.empty(K // 32, dtype=torch.int16, device=DEV)
    xdev = xin.to(DEV)
    qmm.qmm_gemv_q4_0_f32(qs, d, N, K, xdev, None, y, xq, xd, flags=qmm.X_SWIGLU if gate_up else 0)
    if gate_up:
        hq = torch.empty(1, K, dtype=torch.int8, device=DEV)
        hd = torch.empty(1, K // 32, dtype=torch.int16, device=DEV)
        h = torch.empty(1, K, dtype=torch.float32, device=DEV)
        qmm.qmm_swiglu_quantize_q8_0(xdev[:K], xdev[K:], 1, K, K, hq, hd, h)
        qx, dx = O.quantize_q8_0(h.cpu().numpy())
    else:
        qx, dx = O.quantize_q8_0(xin.numpy()[None])
    assert np.array_equal(xq.cpu().numpy(), qx[0]) and np.array_equal(u16(xd), dx[0])
    qw, dw = O.quantize_q4_0(w.numpy())
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y[None], ref, S, "fused gemv")


def test_chained_gemv_launches():
    """Back-to-back dependent GEMVs launched with programmatic dependent launch:
    each reads the previous one's output."""
    qmm = lib()
    K = 2048
    ws = [workloads.weights(K, K, seed=9, index=i) for i in range(3)]
    planes = [qmm.quantize_q4_0(w.to(DEV)) for w in ws]
    x0 = workloads.activations(1, K, seed=9)[0].to(DEV)
    bufs = [x0] + [torch.empty(K, dtype=torch.float32, device=DEV) for _ in ws]
    qouts = [(torch.empty(K, dtype=torch.int8, device=DEV), torch.empty(K // 32, dtype=torch.int16, device=DEV))
             for _ in ws]
    for i, (qs, d) in enumerate(planes):
        qmm.qmm_gemv_q4_0_f32(qs, d, K, K, bufs[i], None, bufs[i + 1], qouts[i][0], qouts[i][1], flags=qmm.CHAIN)
    torch.cuda.synchronize()
    for i, w in enumerate(ws):
        qx, dx = O.quantize_q8_0(bufs[i].cpu().numpy()[None])
        assert np.array_equal(qouts[i][0].cpu().numpy(), qx[0])
        qw, dw = O.quantize_q4_0(w.numpy())
        ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
        assert_close(bufs[i + 1][None], ref, S, f"chain step {i}")


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 16, 33, 64])
def test_gemm_small_batch(M):
    qmm = lib()
    N, K = 517, 2048
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=M)
    qs, d = _to_device_planes(qmm, qw, dw)
    xq, xd = _dev_q8(qx, dx)
    y = qmm.gemm(qs, d, xq, xd)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y, ref, S, f"gemm M={M}")


@pytest.mark.parametrize("K", [256, 768])
@pytest.mark.parametrize("M", [2, 17, 40])
def test_gemm_row_groups_and_ragged_edges(M, K):
    """Enough rows that a CTA walks a full group of 128 rows and a remainder
    group whose row tiles split K across warps; K ends inside a unit (some
    8-block columns absent); the last token tile is ragged.  All rows
    against the oracle."""
    qmm = lib()
    N = 20000
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=M + K)
    qs, d = _to_device_planes(qmm, qw, dw)
    xq, xd = _dev_q8(qx, dx)
    y = qmm.gemm(qs, d, xq, xd)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y, ref, S, f"gemm {N}x{K} M={M}")
    assert qmm.qmm_last_device_error() == 0


@pytest.mark.parametrize("K", [26368, 39168, 39424])
def test_two_tokens_long_k(K):
    """Two tokens with a K whose two-token activation tile is above the
    streaming kernel's two-CTA cap: just above it (824 blocks) and at the
    one-CTA cap (1224 blocks: one CTA per SM), and just past that (1232
    blocks: the row kernel).  All rows against the oracle."""
    qmm = lib()
    N, M = 1000, 2
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=K)
    qs, d = _to_device_planes(qmm, qw, dw)
    xq, xd = _dev_q8(qx, dx)
    y = qmm.gemm(qs, d, xq, xd)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y, ref, S, f"gemm {N}x{K} M={M}")
    assert qmm.qmm_last_device_error() == 0


def test_gemm_ldy_and_chunked_k():
    """Output row stride > N, and K too long to stage for 8 tokens at once."""
    qmm = lib()
    N, K, M, ldy = 40, 28672, 8, 64
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=1)
    qs, d = _to_device_planes(qmm, qw, dw)
    xq, xd = _dev_q8(qx, dx)
    y = torch.full((M, ldy), 7.0, device=DEV)
    qmm.qmm_gemm_q4_0_q8_0(qs, d, N, K, M, xq, xd, y, ldy)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y[:, :N], ref, S, "gemm chunked")
    assert torch.all(y[:, N:] == 7.0)


@pytest.mark.parametrize("N,K", [(5632, 2048), (2048, 5632)])
def test_batched_decode_shapes_full(N, K):
    """Batched-decode shapes, M = 16, all rows against the oracle."""
    qmm = lib()
    M = 16
    w = workloads.weights(N, K, seed=0, index=N)
    x = workloads.activations(M, K, seed=0)
    qs, d = qmm.quantize_q4_0(w.to(DEV))
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    y = qmm.gemm(qs, d, xq, xd)
    qw, dw = O.quantize_q4_0(w.numpy())
    qx, dx = O.quantize_q8_0(x.numpy())
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y, ref, S, f"batched {N}x{K}")


def _sampled_rows(N, n, seed):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, n)]))
    return rows


@pytest.mark.parametrize("name,N,K,M", [("tinyllama.qkv", 2560, 2048, 1), ("tinyllama.down", 2048, 5632, 1),
                                        ("tinyllama.lm_head", 32000, 2048, 1),
                                        ("dense.gate", 28672, 8192, 1), ("dense.down", 8192, 28672, 16),
                                        ("dense.lm_head", 128256, 8192, 1), ("dense.gate", 28672, 8192, 16),
                                        ("dense.lm_head", 128256, 8192, 16), ("dense.up", 28672, 8192, 64),
                                        ("batched.gate", 5632, 2048, 64),
                                        # 2 tokens: the streaming kernel, at one CTA per SM for the long-K
                                        # down projection (an activation tile above the two-CTA cap)
                                        ("dense.gate", 28672, 8192, 2), ("dense.down", 8192, 28672, 2),
                                        ("dense.up", 28672, 8192, 4)])
def test_full_size_sampled_rows(name, N, K, M):
    """Full-size matrices on the GPU (weights drawn on the device), sampled
    rows recomputed by the oracle from the same fp32 rows."""
    qmm = lib()
    sigma = 0.01 if name.startswith("dense") else 0.02
    w = workloads.weights(N, K, sigma=sigma, seed=0, index=N + K, device=DEV)
    x = workloads.activations(M, K, seed=0, device=DEV)
    qs, d = qmm.quantize_q4_0(w)
    xq, xd = qmm.quantize_q8_0(x)
    y = qmm.gemm(qs, d, xq, xd) if M > 1 else qmm.gemv(qs, d, xq[0], xd[0])[None]
    rows = _sampled_rows(N, 64, N)
    wr = w[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    qw, dw = O.quantize_q4_0(wr)
    qx, dx = O.quantize_q8_0(x.cpu().numpy())
    assert np.array_equal(xq.cpu().numpy(), qx)
    # the sampled rows' device planes equal the oracle's quantization of the same rows
    assert np.array_equal(u16(d[torch.from_numpy(rows).to(DEV)]), dw)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y[:, rows], ref, S, name)


def test_fused_gemv_residual():
    """y = residual + W x (residual add in the epilogue)."""
    qmm = lib()
    N, K = 2048, 5632
    w = workloads.weights(N, K, seed=5, index=1)
    gu = workloads.activations(1, 2 * K, seed=5)[0]
    r = workloads.activations(1, N, seed=6)[0]
    qs, d = qmm.quantize_q4_0(w.to(DEV))
    y = torch.empty(N, device=DEV)
    y0 = torch.empty(N, device=DEV)
    g = gu.to(DEV)
    qmm.qmm_gemv_q4_0_f32(qs, d, N, K, g, r.to(DEV), y, flags=qmm.X_SWIGLU)
    qmm.qmm_gemv_q4_0_f32(qs, d, N, K, g, None, y0, flags=qmm.X_SWIGLU)
    diff = (y - y0).cpu().numpy().astype(np.float64)
    assert np.all(np.abs(diff - r.numpy()) <= np.spacing(np.abs(y.cpu().numpy())) + 1e-30)


@pytest.mark.parametrize("F,K", [(5632, 2048), (40, 256), (2048, 6144)])
def test_swiglu_pairs_epilogue(F, K):
    """Interleaved gate/up rows: y[i] = Swish(g_i) * u_i from the row pair
    (2i, 2i+1).  Checked against the oracle's float64 g, u and SwiGLU with the
    GEMV tolerance carried through: |dh| <= 1.1 |u| tol_g + |Swish(g)| tol_u
    (|Swish'| <= 1.1) plus 8 fp32 ulp of h."""
    qmm = lib()
    wg = workloads.weights(F, K, seed=7, index=1)
    wu = workloads.weights(F, K, seed=7, index=2)
    x = workloads.activations(1, K, seed=7)[0]
    w = torch.stack([wg, wu], dim=1).reshape(2 * F, K)  # rows g0, u0, g1, u1, ...
    qs, d = qmm.quantize_q4_0(w.to(DEV))
    h = torch.empty(F, device=DEV)
    qmm.qmm_gemv_q4_0_f32(qs, d, 2 * F, K, x.to(DEV), None, h, flags=qmm.Y_SWIGLU_PAIRS)
    qx, dx = O.quantize_q8_0(x.numpy()[None])
    g, Sg = O.matmul_int(*O.quantize_q4_0(wg.numpy()), qx, dx, nthreads=8)
    u, Su = O.matmul_int(*O.quantize_q4_0(wu.numpy()), qx, dx, nthreads=8)
    h_ref = O.swiglu(g[0], u[0]).astype(np.float64)
    sw = g[0] / (1 + np.exp(-g[0]))
    tol = 1.1 * np.abs(u[0]) * (1e-5 * Sg[0] + 1e-6) + np.abs(sw) * (1e-5 * Su[0] + 1e-6)
    tol += 8 * np.spacing(np.abs(h_ref).astype(np.float32)).astype(np.float64)
    err = np.abs(h.cpu().numpy().astype(np.float64) - h_ref)
    assert np.all(err <= tol), float((err - tol).max())


def test_stream_and_fallback_paths_agree_on_odd_k():
    """K % 256 != 0 takes the per-row kernel; results stay within tolerance."""
    qmm = lib()
    N, K = 130, 2080
    w = workloads.weights(N, K, seed=8)
    x = workloads.activations(1, K, seed=8)[0]
    qs, d = qmm.quantize_q4_0(w.to(DEV))
    y = torch.empty(N, device=DEV)
    qmm.qmm_gemv_q4_0_f32(qs, d, N, K, x.to(DEV), None, y)
    qx, dx = O.quantize_q8_0(x.numpy()[None])
    ref, S = O.matmul_int(*O.quantize_q4_0(w.numpy()), qx, dx, nthreads=8)
    assert_close(y[None], ref, S, "odd K")


@pytest.mark.parametrize("M,K", [(48, 2048), (49, 2048), (64, 2048), (32, 28672)])
def test_gemm_mma_integer_grid_exact(M, K):
    """The warp-MMA GEMM with d = 1 on both sides: every output is an exact
    integer (32..64 tokens, a ragged last row tile, full-magnitude codes), so
    any loss in the MMA's fp32 sums of the offset codes (or a wrong operand
    layout) shows as an inequality."""
    qmm = lib()
    rng = np.random.default_rng(M)
    N = 4100
    w = rng.integers(-7, 8, size=(N, K)).astype(np.float32)
    w[:, ::32] = 7
    w[:5, :64] = np.array([7, -7] * 32, dtype=np.float32)  # both signs, whole blocks
    x = rng.integers(-127, 128, size=(M, K)).astype(np.float32)
    x[:, 3::32] = 127
    x[0, :32] = 127  # largest |sum q_x| in a block
    qs, d = qmm.quantize_q4_0(torch.from_numpy(w).to(DEV))
    xq, xd = qmm.quantize_q8_0(torch.from_numpy(x).to(DEV))
    y = qmm.gemm(qs, d, xq, xd)
    exact = (x.astype(np.int64) @ w.astype(np.int64).T).astype(np.float32)
    assert np.array_equal(y.cpu().numpy(), exact)
    assert qmm.qmm_last_device_error() == 0


@pytest.mark.parametrize("case", ["f32_in_plain", "q8_in_pairs", "q8_in_residual", "f32_in_swiglu_x"])
def test_gemv_fused_q8_outputs(case):
    """qmm_gemv_fused: fp32 or Q8_0 activation in; fp32 y within tolerance of
    the oracle; the Q8_0 output is bit-identical to qmm_quantize_q8_0 applied
    to that y (the standalone quantizer is itself bit-exact against the
    oracle), i.e. the epilogue quantizes exactly like the quantizer."""
    qmm = lib()
    if case == "f32_in_plain":
        N, K, flags = 2560, 2048, 0
    elif case == "q8_in_pairs":
        N, K, flags = 2 * 5632, 2048, qmm.Y_SWIGLU_PAIRS
    elif case == "q8_in_residual":
        N, K, flags = 2048, 5632, 0
    else:
        N, K, flags = 2048, 5632, qmm.X_SWIGLU
    w = workloads.weights(N, K, seed=3, index=N + K)
    qs, d = qmm.quantize_q4_0(w.to(DEV))
    xin = workloads.activations(1, K * (2 if flags & qmm.X_SWIGLU else 1), seed=3)[0]
    xdev = xin.to(DEV)
    nout = N // 2 if flags & qmm.Y_SWIGLU_PAIRS else N
    y = torch.full((nout,), float("nan"), device=DEV)
    yq = torch.zeros(nout, dtype=torch.int8, device=DEV)
    yd = torch.zeros(nout // 32, dtype=torch.int16, device=DEV)
    res = workloads.activations(1, N, seed=4)[0] if case == "q8_in_residual" else None
    if case.startswith("q8_in"):
        xq, xd = qmm.quantize_q8_0(xdev)
        qmm.qmm_gemv_fused(qs, d, N, K, None, xq, xd, None if res is None else res.to(DEV), y, yq, yd, flags=flags)
        qx, dx = O.quantize_q8_0(xin.numpy()[None])
        assert np.array_equal(xq.cpu().numpy(), qx)
    else:
        qmm.qmm_gemv_fused(qs, d, N, K, xdev, None, None, None, y, yq, yd, flags=flags)
        if flags & qmm.X_SWIGLU:
            h = torch.empty(1, K, device=DEV)
            hq = torch.empty(1, K, dtype=torch.int8, device=DEV)
            hd = torch.empty(1, K // 32, dtype=torch.int16, device=DEV)
            qmm.qmm_swiglu_quantize_q8_0(xdev[:K], xdev[K:], 1, K, K, hq, hd, h)
            qx, dx = O.quantize_q8_0(h.cpu().numpy())
        else:
            qx, dx = O.quantize_q8_0(xin.numpy()[None])
    qw, dw = O.quantize_q4_0(w.numpy())
    if flags & qmm.Y_SWIGLU_PAIRS:
        ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
        g, u = ref[0, 0::2], ref[0, 1::2]
        h_ref = O.swiglu(g, u).astype(np.float64)
        sw = g / (1 + np.exp(-g))
        tol = 1.1 * np.abs(u) * (1e-5 * S[0, 0::2] + 1e-6) + np.abs(sw) * (1e-5 * S[0, 1::2] + 1e-6)
        tol += 8 * np.spacing(np.abs(h_ref).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - h_ref) <= tol)
    else:
        ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
        if res is not None:
            ref = ref + res.numpy().astype(np.float64)[None]
            # the fp32 add of the residual rounds once more: 2e-7 |y| > 1 ulp
            S = S + 0.02 * np.abs(ref)
        assert_close(y[None], ref, S, case)
    yq2, yd2 = qmm.quantize_q8_0(y)
    assert np.array_equal(yq.cpu().numpy(), yq2.cpu().numpy()[0])
    assert np.array_equal(u16(yd), u16(yd2)[0])


def test_gemv_fused_chain_of_q8_outputs():
    """Four chained launches (programmatic dependent launch), each reading the
    previous launch's Q8_0 output.  The oracle runs its own chain from the
    same fp32 input: the first step matches element by element; later steps
    can differ where a tiny fp32 difference moves an activation code at a
    rounding boundary, so they are held to a relative L2 bound of 1e-3.
    Every Q8_0 output equals qmm_quantize_q8_0 of the launch's own y."""
    qmm = lib()
    K = 2048
    ws = [workloads.weights(K, K, seed=12, index=i) for i in range(4)]
    planes = [qmm.quantize_q4_0(w.to(DEV)) for w in ws]
    x0 = workloads.activations(1, K, seed=12)[0]
    ys = [torch.empty(K, device=DEV) for _ in ws]
    qs_ = [(torch.empty(K, dtype=torch.int8, device=DEV), torch.empty(K // 32, dtype=torch.int16, device=DEV))
           for _ in ws]
    for i, (qs, d) in enumerate(planes):
        if i == 0:
            qmm.qmm_gemv_fused(qs, d, K, K, x0.to(DEV), None, None, None, ys[i], *qs_[i], flags=qmm.CHAIN)
        else:
            qmm.qmm_gemv_fused(qs, d, K, K, None, *qs_[i - 1], None, ys[i], *qs_[i], flags=qmm.CHAIN)
    torch.cuda.synchronize()
    x_ref = x0.numpy().astype(np.float32)[None]
    for i, w in enumerate(ws):
        ref, S = O.matmul_int(*O.quantize_q4_0(w.numpy()), *O.quantize_q8_0(x_ref), nthreads=8)
        if i == 0:
            assert_close(ys[i][None], ref, S, "chain step 0")
        yg = ys[i].cpu().numpy().astype(np.float64)
        assert np.linalg.norm(yg - ref[0]) <= 1e-3 * np.linalg.norm(ref[0]), i
        yq2, yd2 = qmm.quantize_q8_0(ys[i])
        assert np.array_equal(qs_[i][0].cpu().numpy(), yq2.cpu().numpy()[0])
        assert np.array_equal(u16(qs_[i][1]), u16(yd2)[0])
        x_ref = ref.astype(np.float32)
