"""The headline decode step (TinyLLaMA-1.1B shapes, hidden 2048) against the
oracle at its real size, stage by stage: layer 0's four projections and the
lm_head of bench.TinyLlamaDecode, launched with the step's own partitions,
each fed the previous stage's GPU output (TinyLLaMA guide 5.2 layer graph:
RMSNorm, QKV, O + residual, RMSNorm, gate/up with SwiGLU (4.4), down +
residual; final RMSNorm (4.1) and lm_head).

Checks per stage:
- RMSNorm -> Q8_0 staging (QKV, gate/up, lm_head): codes bit-exact against
  the oracle's Q8_0 of fl(x * gamma), scales within one fp16 step of
  fp16(d32_z / rms) (parity.check_rmsnorm_q8_0);
- each product: |y - y_ref| <= 1e-5 * S + 1e-6 against the oracle's integer
  path on the GPU's own staged activation;
- residual adds (O, down): that bound plus one fp32 rounding of the sum,
  2^-24 * |y|;
- SwiGLU of gate/up: the product bounds carried through SwiGLU, which is
  1.1-Lipschitz in the gate (max |d silu/dg| < 1.1) and |silu(g)|-Lipschitz
  in up, plus 8 fp32 roundings of the GPU's own fp32 SwiGLU;
- every Q8_0 output: bit-exact against the oracle's quantizer applied to the
  GPU's own fp32 output."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity import lib, u16, assert_close, planes_to_oracle, check_rmsnorm_q8_0

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS32 = 2.0 ** -24


def _np(t):
    return t.detach().cpu().numpy()


def _q8_equal(gq, gd, y, what):
    """The GPU's Q8_0 output equals the oracle quantizer on the GPU's fp32 y."""
    q, d = O.quantize_q8_0(np.asarray(y, np.float32)[None])
    assert np.array_equal(_np(gq), q[0]), f"{what}: Q8_0 codes"
    assert np.array_equal(u16(gd), d[0]), f"{what}: Q8_0 scales"


def _swiglu_bound(g, u, Sg, Su, h_ref):
    tg, tu = 1e-5 * Sg + 1e-6, 1e-5 * Su + 1e-6
    silu = g / (1.0 + np.exp(-g))
    return 1.1 * (np.abs(u) + tu) * tg + (np.abs(silu) + 1.1 * tg) * tu + 8 * EPS32 * np.abs(h_ref) + 1e-30


def test_decode_step_layer0_and_lm_head_against_oracle():
    qmm = lib()
    import bench
    dec = bench.TinyLlamaDecode(qmm, torch, seed=0)
    H, F, Q, V = dec.H, dec.F, dec.Q, dec.V
    ops = [dec.op_list[i] for i in (0, 1, 2, 3, len(dec.op_list) - 1)]
    # extra outputs only (they change no launch partition): the staged Q8_0
    # activation of each RMSNorm launch, and fp32 copies of QKV and gate/up
    z8 = lambda n: (torch.zeros(n, dtype=torch.int8, device=DEV),  # noqa: E731
                    torch.zeros(n // 32, dtype=torch.int16, device=DEV))
    st_qkv, st_gu, st_lm = z8(H), z8(H), z8(H)
    y_qkv = torch.zeros(Q, device=DEV)
    h_gu = torch.zeros(F, device=DEV)
    lay = [qmm.GemvOp.from_buffer_copy(o) for o in ops]
    for o, st in ((lay[0], st_qkv), (lay[2], st_gu), (lay[4], st_lm)):
        o.xq, o.xd = st[0].data_ptr(), st[1].data_ptr()
    lay[0].y = y_qkv.data_ptr()
    lay[2].y = h_gu.data_ptr()
    # layer 0's output feeds the lm_head directly
    lay[4].x = ops[3].y
    for o in lay:
        qmm.qmm_gemv_fused_op(o)
    assert qmm.qmm_last_device_error() == 0

    L0 = dec.layers[0]
    g_attn, g_ffn = dec.norms[0]
    x_in = _np(dec.x_in)
    # QKV on RMSNorm(x)
    check_rmsnorm_q8_0(x_in, _np(g_attn), dec.eps, _np(st_qkv[0]), u16(st_qkv[1]), "QKV staging")
    W = planes_to_oracle(*L0["qkv"], Q, H)
    y_ref, S = O.matmul_int(*W, _np(st_qkv[0]), u16(st_qkv[1]), nthreads=16)
    assert_close(y_qkv[None], y_ref, S, "QKV")
    _q8_equal(dec.qkv_q[0], dec.qkv_q[1], _np(y_qkv), "QKV Q8_0 output")
    # O on the first H outputs, + x
    W = planes_to_oracle(*L0["o"], H, H)
    y_ref, S = O.matmul_int(*W, _np(dec.qkv_q[0])[:H], u16(dec.qkv_q[1])[:H // 32], nthreads=16)
    hmid = _np(dec.hmid).astype(np.float64)
    ref = y_ref[0] + x_in
    bound = 1e-5 * S[0] + 1e-6 + EPS32 * np.abs(hmid)
    assert (np.abs(hmid - ref) <= bound).all(), "O + residual"
    # gate/up on RMSNorm(hmid), SwiGLU of the row pairs
    check_rmsnorm_q8_0(_np(dec.hmid), _np(g_ffn), dec.eps, _np(st_gu[0]), u16(st_gu[1]), "gate/up staging")
    qw, dw = planes_to_oracle(*L0["gu"], 2 * F, H)
    sq, sd = _np(st_gu[0]), u16(st_gu[1])
    g_ref, Sg = O.matmul_int(qw[0::2], dw[0::2], sq, sd, nthreads=16)
    u_ref, Su = O.matmul_int(qw[1::2], dw[1::2], sq, sd, nthreads=16)
    h_ref = O.swiglu(g_ref[0], u_ref[0]).astype(np.float64)
    h = _np(h_gu).astype(np.float64)
    bound = _swiglu_bound(g_ref[0], u_ref[0], Sg[0], Su[0], h_ref)
    bad = np.abs(h - h_ref) > bound
    assert not bad.any(), f"SwiGLU of gate/up: {int(bad.sum())} outputs off"
    _q8_equal(dec.ffn_q[0], dec.ffn_q[1], _np(h_gu), "gate/up Q8_0 output")
    # down, + hmid
    W = planes_to_oracle(*L0["down"], H, F)
    y_ref, S = O.matmul_int(*W, _np(dec.ffn_q[0]), u16(dec.ffn_q[1]), nthreads=16)
    h1 = _np(dec.h[0]).astype(np.float64)
    bound = 1e-5 * S[0] + 1e-6 + EPS32 * np.abs(h1)
    assert (np.abs(h1 - (y_ref[0] + hmid)) <= bound).all(), "down + residual"
    # lm_head on RMSNorm(h1)
    check_rmsnorm_q8_0(_np(dec.h[0]), _np(dec.norm_final), dec.eps, _np(st_lm[0]), u16(st_lm[1]), "lm_head staging")
    W = planes_to_oracle(*dec.lm_head, V, H)
    y_ref, S = O.matmul_int(*W, _np(st_lm[0]), u16(st_lm[1]), nthreads=16)
    assert_close(dec.logits[None], y_ref, S, "lm_head")


@pytest.mark.parametrize("K", [512, 2048, 4096])
def test_fused_rmsnorm_staging_bit_exact(K):
    """The fused RMSNorm -> Q8_0 staging alone at hidden 512, 2048 and 4096
    (the longest row of its one-pass form): codes bit-exact, scales within
    one fp16 step, over several seeds and a row with large outliers."""
    qmm = lib()
    import workloads
    N = 256
    w = workloads.weights(N, K, seed=31, index=0, device=DEV)
    qs, d = qmm.quantize_q4_0(w)
    for seed in range(4):
        x = workloads.activations(1, K, seed=40 + seed, device=DEV)[0].contiguous()
        if seed == 3:
            x[::97] *= 1000.0
        gamma = workloads.norm_weights(K, seed=40 + seed, index=3, device=DEV)
        y = torch.zeros(N, device=DEV)
        xq = torch.zeros(K, dtype=torch.int8, device=DEV)
        xd = torch.zeros(K // 32, dtype=torch.int16, device=DEV)
        qmm.qmm_gemv_fused_op(qmm.gemv_op(qs, d, N, K, x=x, norm_w=gamma, norm_eps=1e-5, xq=xq, xd=xd, y=y))
        assert qmm.qmm_last_device_error() == 0
        check_rmsnorm_q8_0(_np(x), _np(gamma), 1e-5, _np(xq), u16(xd), f"K={K} seed {seed}")
        y_ref, S = O.matmul_int(*planes_to_oracle(qs, d, N, K), _np(xq), u16(xd))
        assert_close(y[None], y_ref, S, f"K={K} seed {seed}")
