"""The 16-warp layout of the warp-MMA small-batch GEMM (up to 16 tokens,
taken where its row plan qualifies) against the oracle and against the
row-group kernel on the same inputs.

Shapes are chosen for the row plan on a 152-SM GB300 (rows per CTA =
ceil(N / 152) rounded up to the 64-row granule, else the 32-row one): two or
three 64-row sets per CTA and three 32-row sets, each with a short last CTA
(and two shapes whose plans stay on the row-group kernel); K of half a unit (8 blocks), one and a half units, four units and
many units (the stage ring wraps several times); 2..16 tokens with ragged
token tiles.  fp32 outputs: |y - y_ref| <= 1e-5*S + 1e-6; with unit scales
every output is an exact integer and must match bit for bit."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity import lib, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"

# N -> (rows per CTA, granule) on 152 SMs: the three plans of the 16-warp
# layout (two or three row tiles per warp), then two that stay on the
# row-group kernel (one row tile per warp would be the wide plan)
ROW_PLANS = {18000: (128, 64), 27000: (192, 64), 13000: (96, 32), 7400: (64, 64), 3000: (32, 32)}


@pytest.fixture
def qmm():
    q = lib()
    prev = q.qmm_debug_gemm_kernel(q.GEMM_KERNEL_MMA)  # 2..4 tokens too, not the streaming kernel
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


def test_row_plans_are_the_intended_ones():
    """The shapes below exercise the granules named in ROW_PLANS only on a
    152-SM part; elsewhere they still run (other plans), so this is a note."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip(f"{sms} SMs: the row plans differ from the ones the shapes were chosen for")
    for N, (rpc, g) in ROW_PLANS.items():
        need = -(-N // sms)
        assert -(-need // g) * g == rpc


@pytest.mark.parametrize("N", sorted(ROW_PLANS))
@pytest.mark.parametrize("K,M", [(256, 16), (768, 9), (2048, 2), (2048, 8), (2048, 13)])
# (the 96-row plan, N = 13000, takes 9..16 tokens; 2 and 8 run on the row-group kernel there)
def test_wide_vs_oracle(qmm, N, K, M):
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=N + K + M)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    y = qmm.gemm(qs, d, xq, xd)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y, ref, S, f"wide gemm {N}x{K} M={M}")
    assert qmm.qmm_last_device_error() == 0


@pytest.mark.parametrize("N,K,M", [(28672, 8192, 16), (8192, 28672, 16), (13000, 8192, 5)])
def test_wide_large_k_sampled_rows(qmm, N, K, M):
    """Full-size FFN products: about 1500 sampled rows (both ends included)
    against the oracle and against the row-group kernel (same exact block
    dots, fp32 sums in another order)."""
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=N + M)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    y = qmm.gemm(qs, d, xq, xd)
    rng = np.random.default_rng(K)
    rows = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N), rng.integers(0, N, 1372)]))
    ref, S = O.matmul_int(qw, dw, qx, dx, rows=rows, nthreads=8)
    assert_close(y[:, torch.from_numpy(rows).to(DEV)], ref, S, f"wide gemm {N}x{K} M={M} sampled")
    qmm.qmm_debug_gemm_kernel(qmm.GEMM_KERNEL_MMA_GROUPS)
    y2 = qmm.gemm(qs, d, xq, xd)
    qmm.qmm_debug_gemm_kernel(qmm.GEMM_KERNEL_MMA)
    sel = torch.from_numpy(rows).to(DEV)
    diff = (y - y2).abs()[:, sel].double().cpu().numpy()
    assert np.all(diff <= 2e-5 * S + 2e-6)
    assert torch.isfinite(y).all() and qmm.qmm_last_device_error() == 0


@pytest.mark.parametrize("N,K,M", [(27000, 8192, 16), (7400, 2048, 11), (13000, 768, 16)])
def test_wide_integer_grid_exact(qmm, N, K, M):
    """d = 1 on both sides, full-magnitude codes: every output is an exact
    integer and must be equal (a wrong fragment, swizzle or block pairing
    changes some of them)."""
    rng = np.random.default_rng(N + M)
    w = rng.integers(-7, 8, size=(N, K)).astype(np.float32)
    w[:, ::32] = 7
    x = rng.integers(-127, 128, size=(M, K)).astype(np.float32)
    x[:, 5::32] = 127
    qs, d = qmm.quantize_q4_0(torch.from_numpy(w).to(DEV))
    xq, xd = qmm.quantize_q8_0(torch.from_numpy(x).to(DEV))
    y = qmm.gemm(qs, d, xq, xd)
    exact = (x.astype(np.float64) @ w.astype(np.float64).T).astype(np.float32)
    assert np.array_equal(y.cpu().numpy(), exact)
    assert qmm.qmm_last_device_error() == 0


# N -> (chunk rows, chunks per CTA) on 152 SMs for the plans that walk several
# row chunks per CTA; each has a last CTA with fewer chunks and a last chunk
# with fewer rows
MULTI_PLANS = {58000: (192, 2), 110000: (192, 4), 128256: (128, 7)}


@pytest.mark.parametrize("N", sorted(MULTI_PLANS))
@pytest.mark.parametrize("K,M", [(768, 16), (2048, 4), (2048, 9)])
def test_wide_several_chunks_per_cta(qmm, N, K, M):
    """Rows at every chunk and CTA boundary (and 2000 more) against the oracle."""
    rpc, nchunk = MULTI_PLANS[N]
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=N + K + M)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    y = qmm.gemm(qs, d, xq, xd)
    rng = np.random.default_rng(N + M)
    edges = np.arange(0, N, rpc)
    rows = np.unique(np.clip(np.concatenate([edges, edges - 1, edges + 15, edges + rpc - 1, rng.integers(0, N, 2000),
                                             np.arange(N - 40, N)]), 0, N - 1))
    ref, S = O.matmul_int(qw, dw, qx, dx, rows=rows, nthreads=8)
    assert_close(y[:, torch.from_numpy(rows).to(DEV)], ref, S, f"wide gemm {N}x{K} M={M} chunks")
    assert torch.isfinite(y).all() and qmm.qmm_last_device_error() == 0


def test_multi_chunk_plans_are_the_intended_ones():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip(f"{sms} SMs: the row plans differ from the ones the shapes were chosen for")
    for N, (rpc, nchunk) in MULTI_PLANS.items():
        need = -(-N // sms)
        per = {r: -(-(-(-N // r)) // sms) for r in (128, 192)}
        pick = 192 if per[192] * 192 <= per[128] * 128 else 128
        assert (pick, per[pick]) == (rpc, nchunk)
        assert pick * per[pick] * 100 <= -(-need // 16) * 16 * 108


# N, K -> (chunk rows, CTAs per cluster splitting K) on 152 SMs: 192-row
# chunks where the busiest CTA's rows x units, counted at 0.9, are fewer;
# clusters of at most 4
SPLIT_PLANS = {(8192, 28672): (192, 3), (8000, 16640): (192, 3), (4096, 14336): (128, 4), (2048, 28672): (128, 4),
               (5000, 16640): (128, 3)}


@pytest.mark.parametrize("N,K", sorted(SPLIT_PLANS))
@pytest.mark.parametrize("M", [16, 5])
def test_wide_split_k_clusters(qmm, N, K, M):
    """K shared by the CTAs of a cluster (uneven shares and a last half unit
    for K = 16640): sampled rows, both ends and every chunk edge, against the
    oracle; the same call twice gives the same bits (the ranks' sums are
    added in a fixed order)."""
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=N + K + M)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    y = qmm.gemm(qs, d, xq, xd)
    y2 = qmm.gemm(qs, d, xq, xd)
    assert torch.equal(y, y2)
    rng = np.random.default_rng(N + M)
    rpc = SPLIT_PLANS[(N, K)][0]
    edges = np.arange(0, N, rpc)
    rows = np.unique(np.clip(np.concatenate([edges, edges - 1, edges + rpc - 1, rng.integers(0, N, 600),
                                             np.arange(N - 20, N)]), 0, N - 1))
    ref, S = O.matmul_int(qw, dw, qx, dx, rows=rows, nthreads=8)
    assert_close(y[:, torch.from_numpy(rows).to(DEV)], ref, S, f"split-K gemm {N}x{K} M={M}")
    assert torch.isfinite(y).all() and qmm.qmm_last_device_error() == 0


def test_split_plans_are_the_intended_ones():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip(f"{sms} SMs: the row plans differ from the ones the shapes were chosen for")
    for (N, K), plan in SPLIT_PLANS.items():
        assert -(-N // sms) <= 64
        units = -(-(K // 32) // 16)
        costs = {}
        for rpc in (192, 128):
            ns = min(4, sms // -(-N // rpc))
            if ns >= 2 and units >= 6 * ns:
                costs[(rpc, ns)] = rpc * -(-units // ns) * (9 if rpc == 192 else 10)
        assert min(costs, key=costs.get) == plan


def test_wide_ldy(qmm):
    """Output row stride > N: the columns past N stay untouched."""
    N, K, M, ldy = 27000, 1024, 16, 27008
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=9)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    y = torch.full((M, ldy), 7.0, device=DEV)
    qmm.qmm_gemm_q4_0_q8_0(qs, d, N, K, M, xq, xd, y, ldy)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y[:, :N], ref, S, "wide ldy")
    assert torch.all(y[:, N:] == 7.0)


# (N, K, M) through the 16-warp plans both entries take (one chunk of 96 / 128
# / 192 rows per CTA, clusters splitting 128-row chunks' K); large N, where
# the workspace entry cuts the product evenly over the SMs instead, is
# test_workspace_even_cut, and the shapes whose K the plain entry splits over
# 192-row chunks are test_workspace_split_plans'
WS_CASES = [(27000, 2048, 16), (27000, 768, 9), (18000, 2048, 5), (13000, 2048, 12), (5000, 16640, 9),
            (2048, 28672, 3)]


@pytest.mark.parametrize("N,K,M", WS_CASES)
def test_workspace_path_matches_staged_path(qmm, N, K, M):
    """qmm_gemm_q4_0_q8_0_ws (the activation's MMA operand formed once into
    the workspace, which starts out full of junk) gives the staged path's
    results bit for bit; sampled rows also against the oracle."""
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=N + 3 * K + M)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    y0 = qmm.gemm(qs, d, xq, xd)
    nbytes = qmm.qmm_gemm_workspace_size(K, M)
    ws = torch.full((max(nbytes, 1),), 0xAB, dtype=torch.uint8, device=DEV)
    y1 = qmm.gemm(qs, d, xq, xd, workspace=ws)
    assert torch.equal(y0, y1)
    rng = np.random.default_rng(N)
    rows = np.unique(np.concatenate([np.arange(40), np.arange(N - 40, N), rng.integers(0, N, 400)]))
    ref, S = O.matmul_int(qw, dw, qx, dx, rows=rows, nthreads=8)
    assert_close(y1[:, torch.from_numpy(rows).to(DEV)], ref, S, f"workspace gemm {N}x{K} M={M}")
    assert qmm.qmm_last_device_error() == 0


@pytest.mark.parametrize("N,K,M", [(8192, 28672, 16), (8000, 16640, 9), (8192, 28672, 4)])
def test_workspace_split_plans(qmm, N, K, M):
    """Where the plain entry splits K over clusters sharing 192-row chunks,
    the workspace entry splits 128-row chunks (2- or 3-CTA clusters): sampled
    rows at both chunk sizes' edges against the oracle, and the same bits on
    a second call."""
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=N + 7 * K + M)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    ws = torch.full((qmm.qmm_gemm_workspace_size(K, M),), 0x3C, dtype=torch.uint8, device=DEV)
    y = qmm.gemm(qs, d, xq, xd, workspace=ws)
    y2 = qmm.gemm(qs, d, xq, xd, workspace=ws)
    assert torch.equal(y, y2)
    rng = np.random.default_rng(N + M)
    edges = np.concatenate([np.arange(0, N, 128), np.arange(0, N, 192)])
    rows = np.unique(np.clip(np.concatenate([edges, edges - 1, rng.integers(0, N, 400), np.arange(N - 20, N)]),
                             0, N - 1))
    ref, S = O.matmul_int(qw, dw, qx, dx, rows=rows, nthreads=8)
    assert_close(y[:, torch.from_numpy(rows).to(DEV)], ref, S, f"workspace split plan {N}x{K} M={M}")
    assert qmm.qmm_last_device_error() == 0


def test_workspace_path_integer_grid_exact(qmm):
    """d = 1 on both sides through the workspace path: exact integers."""
    N, K, M = 27000, 8192, 16
    rng = np.random.default_rng(7)
    w = rng.integers(-7, 8, size=(N, K)).astype(np.float32)
    w[:, 3::32] = -7  # every block's max |w| is 7: d = 1
    x = rng.integers(-127, 128, size=(M, K)).astype(np.float32)
    x[:, 9::32] = -127
    qs, d = qmm.quantize_q4_0(torch.from_numpy(w).to(DEV))
    xq, xd = qmm.quantize_q8_0(torch.from_numpy(x).to(DEV))
    ws = torch.empty(qmm.qmm_gemm_workspace_size(K, M), dtype=torch.uint8, device=DEV)
    y = qmm.gemm(qs, d, xq, xd, workspace=ws)
    exact = (x.astype(np.float64) @ w.astype(np.float64).T).astype(np.float32)
    assert np.array_equal(y.cpu().numpy(), exact)
    assert qmm.qmm_last_device_error() == 0


def test_workspace_entry_edges(qmm):
    """The workspace entry with ldy > N (columns past N untouched); with 17
    tokens (no workspace needed: the plain entry's path); with xd only 2-byte
    aligned (the 16-warp layout does not apply: same results as the plain
    entry); and one workspace reused by back-to-back calls of different K on
    one stream (each call's preparation waits for the call before)."""
    N, K = 27000, 1024
    # ldy > N
    qw, dw, qx, dx = _rand_codes(N, 16, K, seed=21)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    ws = torch.empty(qmm.qmm_gemm_workspace_size(K, 16), dtype=torch.uint8, device=DEV)
    ldy = N + 40
    y = torch.full((16, ldy), 7.0, device=DEV)
    qmm.qmm_gemm_q4_0_q8_0_ws(qs, d, N, K, 16, xq, xd, y, ldy, ws, ws.numel())
    assert torch.equal(y[:, :N], qmm.gemm(qs, d, xq, xd)) and torch.all(y[:, N:] == 7.0)
    # 17 tokens: no workspace
    assert qmm.qmm_gemm_workspace_size(K, 17) == 0
    qw7, dw7, qx7, dx7 = _rand_codes(N, 17, K, seed=22)
    xq7, xd7 = _q8(qx7, dx7)
    y7 = torch.empty(17, N, device=DEV)
    qmm.qmm_gemm_q4_0_q8_0_ws(qs, d, N, K, 17, xq7, xd7, y7, N, None, 0)
    assert torch.equal(y7, qmm.gemm(qs, d, xq7, xd7))
    # xd 2-byte aligned only
    xd_buf = torch.zeros(16 * (K // 32) + 8, dtype=torch.int16, device=DEV)
    xd_odd = xd_buf[1:1 + 16 * (K // 32)].view(16, K // 32)
    xd_odd.copy_(xd)
    assert xd_odd.data_ptr() % 16 == 2
    y2 = torch.empty(16, N, device=DEV)
    qmm.qmm_gemm_q4_0_q8_0_ws(qs, d, N, K, 16, xq, xd_odd, y2, N, ws, ws.numel())
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y2, ref, S, "workspace entry, xd 2-byte aligned")
    # one workspace, calls of different K back to back
    K2 = 4096
    qw2, dw2, qx2, dx2 = _rand_codes(N, 16, K2, seed=23)
    qs2, d2 = _planes(qmm, qw2, dw2)
    xq2, xd2 = _q8(qx2, dx2)
    big = torch.empty(qmm.qmm_gemm_workspace_size(K2, 16), dtype=torch.uint8, device=DEV)
    ya = torch.empty(16, N, device=DEV)
    yb = torch.empty(16, N, device=DEV)
    qmm.qmm_gemm_q4_0_q8_0_ws(qs2, d2, N, K2, 16, xq2, xd2, ya, N, big, big.numel())
    qmm.qmm_gemm_q4_0_q8_0_ws(qs, d, N, K, 16, xq, xd, yb, N, big, big.numel())
    assert torch.equal(ya, qmm.gemm(qs2, d2, xq2, xd2)) and torch.equal(yb, qmm.gemm(qs, d, xq, xd))
    assert qmm.qmm_last_device_error() == 0


@pytest.mark.parametrize("N,K,M", [(5632, 2048, 16), (2048, 5632, 9), (2560, 2048, 8), (1000, 8192, 5),
                                   (300, 28672, 12), (4096, 14336, 7), (3000, 2048, 16)])
def test_workspace_small_products(qmm, N, K, M):
    """Small products through the workspace entry (the 16-warp layout does not
    apply to most of them: the entry falls back to the plain one, which must
    then ignore the workspace; the two long-K shapes split K over clusters)
    against the oracle, all rows."""
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=N + K + M + 1)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    ws = torch.full((qmm.qmm_gemm_workspace_size(K, M),), 0x5A, dtype=torch.uint8, device=DEV)
    y = qmm.gemm(qs, d, xq, xd, workspace=ws)
    ref, S = O.matmul_int(qw, dw, qx, dx, nthreads=8)
    assert_close(y, ref, S, f"workspace gemm small N {N}x{K} M={M}")
    y2 = qmm.gemm(qs, d, xq, xd, workspace=ws)
    assert torch.equal(y, y2)
    assert qmm.qmm_last_device_error() == 0


@pytest.mark.parametrize("N,K,M", [(128256, 768, 16), (58000, 2048, 9), (110000, 512, 4), (40000, 1024, 16),
                                   (110000, 768, 16), (128256, 512, 4), (128256, 2048, 7)])
def test_workspace_even_cut(qmm, N, K, M):
    """Large N through the workspace entry: where it pays (lm_head-sized N),
    the product's (chunk, unit) sequence cut evenly over the SMs, chunks cut
    between two CTAs finished through y and a flag; elsewhere several chunks
    per CTA.  Rows at every 192-row chunk edge (and more) against the oracle,
    and the same bits on a second call."""
    qw, dw, qx, dx = _rand_codes(N, M, K, seed=N + 5 * K + M)
    qs, d = _planes(qmm, qw, dw)
    xq, xd = _q8(qx, dx)
    ws = torch.full((qmm.qmm_gemm_workspace_size(K, M),), 0x77, dtype=torch.uint8, device=DEV)
    y = qmm.gemm(qs, d, xq, xd, workspace=ws)
    y2 = qmm.gemm(qs, d, xq, xd, workspace=ws)
    assert torch.equal(y, y2)
    rng = np.random.default_rng(N)
    edges = np.arange(0, N, 192)
    rows = np.unique(np.clip(np.concatenate([edges, edges - 1, edges + 100, rng.integers(0, N, 1500),
                                             np.arange(N - 30, N)]), 0, N - 1))
    ref, S = O.matmul_int(qw, dw, qx, dx, rows=rows, nthreads=8)
    assert_close(y[:, torch.from_numpy(rows).to(DEV)], ref, S, f"workspace even cut {N}x{K} M={M}")
    assert qmm.qmm_last_device_error() == 0
