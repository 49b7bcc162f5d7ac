"""A small decoder stack run as the decode step's fused GEMV launches
(qmm_gemv_fused_op): the first op against the oracle (bit-exact RMSNorm ->
Q8_0 codes, fp32 tolerance on the product), the whole stack against the
oracle's own stack within a relative L2 of 1e-3, and the same result from a
replayed CUDA graph of the chained (programmatic dependent launch) form."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import workloads
from parity import lib, u16, assert_close, check_rmsnorm_q8_0

pytestmark = pytest.mark.gpu
DEV = "cuda"


class MiniDecode:
    """Decoder layers shaped like the bench's TinyLLaMA step, small dims: QKV on
    RMSNorm(h) -> Q8_0; O on the q slice + h -> h1; gate/up on RMSNorm(h1)
    with SwiGLU pairs -> Q8_0; down + h1 -> h; lm_head on RMSNorm(h)."""

    def __init__(self, qmm, H=512, Q=640, F=1024, V=1000, L=2, seed=7):
        self.qmm, self.H, self.Q, self.F, self.V, self.L = qmm, H, Q, F, V, L
        idx = [0]

        def planes(N, K):
            w = workloads.weights(N, K, sigma=0.02, seed=seed, index=idx[0], device=DEV)
            idx[0] += 1
            return qmm.quantize_q4_0(w)

        self.layers = []
        for li in range(L):
            qkv, o = planes(Q, H), planes(H, H)
            g, u = planes(F, H), planes(F, H)
            gu = (torch.stack([g[0], u[0]], 1).reshape(2 * F, -1).contiguous(),
                  torch.stack([g[1], u[1]], 1).reshape(2 * F, -1).contiguous())
            norms = (workloads.norm_weights(H, seed=seed, index=2 * li, device=DEV),
                     workloads.norm_weights(H, seed=seed, index=2 * li + 1, device=DEV))
            self.layers.append((qkv, o, gu, planes(H, F), norms))
        self.lm = planes(V, H)
        self.norm_final = workloads.norm_weights(H, seed=seed, index=99, device=DEV)
        z = lambda n, dt=torch.float32: torch.zeros(n, dtype=dt, device=DEV)  # noqa: E731
        q8 = lambda n: (z(n, torch.int8), z(n // 32, torch.int16))  # noqa: E731
        self.x = workloads.activations(1, H, seed=seed, device=DEV)[0].contiguous()
        self.h = [z(H), z(H)]
        self.hmid = z(H)
        self.qkv_q, self.ffn_q = q8(Q), q8(F)
        self.a0 = q8(H)  # the staged (normalized, quantized) activation of op 0
        self.logits = z(V)

    def ops(self):
        m, H, Q, F, V = self.qmm, self.H, self.Q, self.F, self.V
        ops, h_in = [], self.x
        for li, (qkv, o, gu, down, (ga, gf)) in enumerate(self.layers):
            h_out = self.h[li % 2]
            extra = dict(xq=self.a0[0], xd=self.a0[1]) if li == 0 else {}
            ops.append(m.gemv_op(*qkv, Q, H, x=h_in, norm_w=ga, yq=self.qkv_q[0], yd=self.qkv_q[1], **extra))
            ops.append(m.gemv_op(*o, H, H, xq=self.qkv_q[0], xd=self.qkv_q[1], residual=h_in, y=self.hmid))
            ops.append(m.gemv_op(*gu, 2 * F, H, x=self.hmid, norm_w=gf, yq=self.ffn_q[0], yd=self.ffn_q[1],
                                 flags=m.Y_SWIGLU_PAIRS))
            ops.append(m.gemv_op(*down, H, F, xq=self.ffn_q[0], xd=self.ffn_q[1], residual=self.hmid, y=h_out))
            h_in = h_out
        ops.append(m.gemv_op(*self.lm, V, H, x=h_in, norm_w=self.norm_final, y=self.logits))
        return ops

    def buffers(self):
        return (self.logits, self.h[0], self.h[1], self.hmid, *self.qkv_q, *self.ffn_q, *self.a0)

    def run_one_by_one(self):
        for op in self.ops():
            self.qmm.qmm_gemv_fused_op(op)

    def snapshot(self):
        return [t.clone() for t in self.buffers()]

    def reset_outputs(self):
        for t in self.buffers():
            t.fill_(0)


def test_chained_launches_from_a_graph_equal_plain_launches():
    """The ops launched with programmatic dependent launch from a replayed
    CUDA graph give exactly the outputs of plain launches, replay after
    replay."""
    qmm = lib()
    qmm.qmm_last_device_error()
    dec = MiniDecode(qmm)
    dec.run_one_by_one()
    torch.cuda.synchronize()
    ref = dec.snapshot()
    ops = dec.ops()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for op in ops:
            qmm.qmm_gemv_fused_op(op, qmm.CHAIN, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for op in ops:
            qmm.qmm_gemv_fused_op(op, qmm.CHAIN, stream=torch.cuda.current_stream())
    for rep in range(3):
        dec.reset_outputs()
        g.replay()
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(dec.snapshot(), ref)):
            assert torch.equal(a, b), f"output {i} differs from the plain launches (replay {rep})"
    assert qmm.qmm_last_device_error() == 0


def test_op_chain_entry_equals_plain_launches():
    """qmm_gemv_fused_ops (the whole op list in one call, chained and plain)
    gives exactly the outputs of one qmm_gemv_fused_op call per op."""
    qmm = lib()
    qmm.qmm_last_device_error()
    dec = MiniDecode(qmm)
    dec.run_one_by_one()
    torch.cuda.synchronize()
    ref = dec.snapshot()
    ops = dec.ops()
    arr = qmm.gemv_op_array(ops)
    for flags in (0, qmm.CHAIN):
        dec.reset_outputs()
        qmm.qmm_gemv_fused_ops(arr, len(ops), flags)
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(dec.snapshot(), ref)):
            assert torch.equal(a, b), f"output {i} differs from one call per op (flags {flags})"
    # a bad last op: its status, and nothing of the chain launched
    bad = qmm.gemv_op(ops[0].w_qs, ops[0].w_d, 64, 288, xq=dec.a0[0], xd=dec.a0[1], y=dec.logits)
    arr_bad = qmm.gemv_op_array(ops + [bad])
    dec.reset_outputs()
    torch.cuda.synchronize()
    with pytest.raises(qmm.QmmError) as ei:
        qmm.qmm_gemv_fused_ops(arr_bad, len(ops) + 1, qmm.CHAIN)
    assert ei.value.status == 2
    torch.cuda.synchronize()
    assert all(torch.count_nonzero(t) == 0 for t in dec.buffers())
    assert qmm.qmm_last_device_error() == 0


def _planes_to_oracle(qs, d, N, K):
    blocks = np.zeros((N, K // 32, 18), np.uint8)
    blocks[..., :2] = u16(d).reshape(N, K // 32, 1).view(np.uint8)
    blocks[..., 2:] = qs.cpu().numpy().reshape(N, K // 32, 16)
    return O.unpack_q4_0_blocks(blocks, N, K)


def test_first_op_and_end_to_end_against_oracle():
    """Op 0: the GPU's Q8_0 of RMSNorm(x): codes bit-exact against the
    oracle's Q8_0 of fl(x * gamma), scales within one fp16 step of
    fp16(d32_z / rms); its output against the oracle's product of the GPU's
    own codes.  Then the oracle runs the whole chain on its own
    (RMSNorm, Q8_0 of each intermediate) and the logits agree to a relative
    L2 of 1e-3."""
    qmm = lib()
    dec = MiniDecode(qmm, L=1)
    dec.run_one_by_one()
    assert qmm.qmm_last_device_error() == 0
    H, Q, F, V = dec.H, dec.Q, dec.F, dec.V
    (qkv, o, gu, down, (ga, gf)) = dec.layers[0]
    x = dec.x.cpu().numpy()[None]
    a_ref = O.rmsnorm(x, ga.cpu().numpy(), eps=1e-5)
    qa, da = O.quantize_q8_0(a_ref)
    gqa, gda = dec.a0[0].cpu().numpy()[None], u16(dec.a0[1])[None]
    check_rmsnorm_q8_0(x[0], ga.cpu().numpy(), 1e-5, gqa[0], gda[0], "op 0 staging")
    # QKV of the GPU's own codes: the Q8_0 output within one step of the oracle's
    yq_ref, S = O.matmul_int(*_planes_to_oracle(*qkv, Q, H), gqa, gda)
    qy, dy = O.quantize_q8_0(yq_ref.astype(np.float32))
    assert (np.abs(dec.qkv_q[0].cpu().numpy().astype(int) - qy[0].astype(int)) <= 1).all()
    # the oracle's own chain
    qx, dx = qa, da
    t, _ = O.matmul_int(*_planes_to_oracle(*qkv, Q, H), qx, dx)
    q1, d1 = O.quantize_q8_0(t.astype(np.float32))
    t, _ = O.matmul_int(*_planes_to_oracle(*o, H, H), q1[:, :H], d1[:, :H // 32])
    h1 = (t + x).astype(np.float32)
    b = O.rmsnorm(h1, gf.cpu().numpy(), eps=1e-5)
    qb, db = O.quantize_q8_0(b)
    g_u, _ = O.matmul_int(*_planes_to_oracle(*gu, 2 * F, H), qb, db)
    hm = O.swiglu(g_u[:, 0::2], g_u[:, 1::2])
    qm, dm = O.quantize_q8_0(hm)
    t, _ = O.matmul_int(*_planes_to_oracle(*down, H, F), qm, dm)
    h2 = (t + h1).astype(np.float32)
    c = O.rmsnorm(h2, dec.norm_final.cpu().numpy(), eps=1e-5)
    qc, dc = O.quantize_q8_0(c)
    logits, _ = O.matmul_int(*_planes_to_oracle(*dec.lm, V, H), qc, dc)
    g = dec.logits.cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all()
    rel = np.linalg.norm(g - logits[0]) / np.linalg.norm(logits[0])
    assert rel < 1e-3, rel
