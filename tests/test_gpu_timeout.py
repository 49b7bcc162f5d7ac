"""Failure handling of the streaming GEMV kernel without a GPU fault: every
wait on the device is bounded.  With the test hook qmm_debug_stream_wait the
bound is cut to 1 ms and each CTA's producer never issues its last weight
copy (a completion that nothing signals), so the consumers' waits run out:
the launch returns, the device error word reads QMM_ERR_TIMEOUT, and the
next normal launch on the same context matches the oracle within the fp32
tolerance |y - y_ref| <= 1e-5 * S + 1e-6."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import workloads
from parity import lib, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT = 6  # QMM_ERR_TIMEOUT


def _gemv_case(qmm, N, K, seed):
    w = workloads.weights(N, K, sigma=0.02, seed=seed, index=0)
    x = workloads.activations(1, K, seed=seed, index=1)
    qs, d = qmm.quantize_q4_0(w.to(DEV))
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    ref, S = O.matmul_int(*O.quantize_q4_0(w.numpy()), *O.quantize_q8_0(x.numpy()), nthreads=8)
    return qs, d, xq, xd, ref, S


# 2048 x 2048: one weight unit per CTA; 2048 x 28672: 14 units per CTA through
# an 8-stage ring (stages reused before the withheld last unit)
@pytest.mark.parametrize("N,K", [(2048, 2048), (2048, 28672)])
def test_withheld_copy_times_out_and_the_context_stays_usable(N, K):
    qmm = lib()
    qs, d, xq, xd, ref, S = _gemv_case(qmm, N, K, seed=21)
    y = torch.zeros(N, device=DEV)
    assert qmm.qmm_last_device_error() == 0
    prev = qmm.qmm_debug_stream_wait(1_000_000, withhold_last_copy=True)
    try:
        assert prev == 2_000_000_000
        qmm.qmm_gemv_q4_0_q8_0(qs, d, N, K, xq[0], xd[0], y)
        assert qmm.qmm_last_device_error() == TIMEOUT
        assert qmm.qmm_last_device_error() == 0  # read once, then clear
    finally:
        qmm.qmm_debug_stream_wait(prev, withhold_last_copy=False)
    qmm.qmm_gemv_q4_0_q8_0(qs, d, N, K, xq[0], xd[0], y)
    assert qmm.qmm_last_device_error() == 0
    assert_close(y[None], ref, S, f"GEMV {N}x{K} after a timed-out launch")


def test_fused_rmsnorm_launch_times_out_then_recovers():
    """The decode step's fused launch form (RMSNorm-ed fp32 input, Q8_0 and
    fp32 outputs) under the same withheld copy."""
    qmm = lib()
    N, K = 2560, 2048
    w = workloads.weights(N, K, sigma=0.02, seed=22, index=0)
    x = workloads.activations(1, K, seed=22, index=1).to(DEV)[0].contiguous()
    gamma = workloads.norm_weights(K, seed=22, index=2, device=DEV)
    qs, d = qmm.quantize_q4_0(w.to(DEV))
    y = torch.zeros(N, device=DEV)
    yq = torch.zeros(N, dtype=torch.int8, device=DEV)
    yd = torch.zeros(N // 32, dtype=torch.int16, device=DEV)
    op = qmm.gemv_op(qs, d, N, K, x=x, norm_w=gamma, norm_eps=1e-5, y=y, yq=yq, yd=yd)
    prev = qmm.qmm_debug_stream_wait(1_000_000, withhold_last_copy=True)
    try:
        qmm.qmm_gemv_fused_op(op)
        assert qmm.qmm_last_device_error() == TIMEOUT
    finally:
        qmm.qmm_debug_stream_wait(prev, withhold_last_copy=False)
    qmm.qmm_gemv_fused_op(op)
    assert qmm.qmm_last_device_error() == 0
    y_first = y.clone()
    qmm.qmm_gemv_fused_op(op)
    assert qmm.qmm_last_device_error() == 0
    assert torch.equal(y, y_first) and torch.isfinite(y).all()
