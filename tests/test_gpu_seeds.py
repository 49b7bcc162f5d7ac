"""Seed sweep {0, 1, 2} on the workload shapes, with the input recipe of
each configuration: the single 2048 x 2048 GEMV end to end (GPU Q4_0 and
Q8_0 quantizers bit-exact against the oracle's, the product within the fp32
tolerance), the batched 5632 x 2048 GEMM at 16 and 64 tokens on sampled rows,
and the GLM-scale router (ids equal, gates within 1e-6)."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import workloads
from parity import lib, u16, assert_close, planes_from_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
SEEDS = [0, 1, 2]


def _quantized(qmm, N, K, sigma, seed, index=0):
    w = workloads.weights(N, K, sigma=sigma, seed=seed, index=index)
    qs, d = qmm.quantize_q4_0(w.to(DEV))
    q, dn = O.quantize_q4_0(w.numpy())
    ref_qs, _ = planes_from_oracle(q, dn)
    assert np.array_equal(qs.cpu().numpy(), ref_qs) and np.array_equal(u16(d), dn)
    return qs, d, q, dn


@pytest.mark.parametrize("seed", SEEDS)
def test_single_gemv_end_to_end(seed):
    qmm = lib()
    c = workloads.SINGLE_GEMV
    N, K = c["N"], c["K"]
    qs, d, q, dn = _quantized(qmm, N, K, c["sigma"], seed)
    x = workloads.activations(1, K, seed=seed)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    rq, rd = O.quantize_q8_0(x.numpy())
    assert np.array_equal(xq.cpu().numpy(), rq) and np.array_equal(u16(xd), rd)
    y = qmm.gemv(qs, d, xq[0], xd[0])
    ref, S = O.matmul_int(q, dn, rq, rd, nthreads=8)
    assert_close(y[None], ref, S, f"config 0 seed {seed}")


@pytest.mark.parametrize("seed", SEEDS)
@pytest.mark.parametrize("M", [16, 64])
def test_batched_gemm_sampled_rows(seed, M):
    qmm = lib()
    c = workloads.BATCHED
    N, K = 5632, 2048
    qs, d, q, dn = _quantized(qmm, N, K, c["sigma"], seed, index=1)
    x = workloads.activations(M, K, seed=seed)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    y = qmm.gemm(qs, d, xq, xd)
    rows = np.array([0, 1, 63, 64, 2047, 4000, N - 2, N - 1])
    ref, S = O.matmul_int(q, dn, xq.cpu().numpy(), u16(xd), rows=rows, nthreads=8)
    assert_close(y[:, torch.from_numpy(rows).to(DEV)], ref, S, f"config 2 M={M} seed {seed}")


@pytest.mark.parametrize("seed", SEEDS)
def test_router_seed_sweep(seed):
    qmm = lib()
    c = workloads.MOE
    T, E, k = 16, c["experts"], c["top_k"]
    logits = workloads.router_logits(T, E, seed=seed)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    gates = torch.empty(T, k, device=DEV)
    qmm.qmm_moe_router_topk(logits.to(DEV), T, E, k, ids, gates)
    ref_ids, ref_g = O.router_topk(logits.numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.all(np.abs(gates.cpu().numpy().astype(np.float64) - ref_g) <= 1e-6)
