"""qmm_decode_chain: the decode step as one launch with flagged hand-over
between its ops gives bit-identical outputs to the same ops launched one by
one through qmm_gemv_fused_op (same per-row arithmetic, Q8_0 rule and
RMSNorm reduction order), call after call on one workspace and from a
replayed CUDA graph; at the TinyLLaMA-1.1B size (22 layers, hidden 2048)
its logits equal those of the 89-launch step."""
import pytest
import torch

import workloads
from parity import lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


class Mini:
    """A few decoder layers at small sizes, as both op lists."""

    def __init__(self, qmm, H=512, Q=640, F=1024, V=1000, L=3, seed=9):
        self.qmm, self.H, self.Q, self.F, self.V, self.L = qmm, H, Q, F, V, L
        idx = [0]

        def planes(N, K):
            w = workloads.weights(N, K, sigma=0.02, seed=seed, index=idx[0], device=DEV)
            idx[0] += 1
            return qmm.quantize_q4_0(w)

        self.layers = []
        for li in range(L):
            g, u = planes(F, H), planes(F, H)
            gu = (torch.stack([g[0], u[0]], 1).reshape(2 * F, -1).contiguous(),
                  torch.stack([g[1], u[1]], 1).reshape(2 * F, -1).contiguous())
            self.layers.append(dict(qkv=planes(Q, H), o=planes(H, H), gu=gu, down=planes(H, F),
                                    ga=workloads.norm_weights(H, seed=seed, index=2 * li, device=DEV),
                                    gf=workloads.norm_weights(H, seed=seed, index=2 * li + 1, device=DEV)))
        self.lm = planes(V, H)
        self.gfin = workloads.norm_weights(H, seed=seed, index=99, device=DEV)
        z = lambda n, dt=torch.float32: torch.zeros(n, dtype=dt, device=DEV)  # noqa: E731
        q8 = lambda n: (z(n, torch.int8), z(n // 32, torch.int16))  # noqa: E731
        self.x = workloads.activations(1, H, seed=seed, device=DEV)[0].contiguous()
        self.ref_h = [z(H) for _ in range(L)]
        self.ref_hmid = [z(H) for _ in range(L)]
        self.qkv_q, self.ffn_q = q8(Q), q8(F)
        self.ref_logits = z(V)
        self.ref_a0 = q8(H)
        self.h = [z(H) for _ in range(L)]
        self.hmid = [z(H) for _ in range(L)]
        self.logits = z(V)
        self.a0 = q8(H)

    def per_op(self):
        m, H, Q, F, V = self.qmm, self.H, self.Q, self.F, self.V
        h_in = self.x
        for li, Lw in enumerate(self.layers):
            extra = dict(xq=self.ref_a0[0], xd=self.ref_a0[1]) if li == 0 else {}
            m.qmm_gemv_fused_op(m.gemv_op(*Lw["qkv"], Q, H, x=h_in, norm_w=Lw["ga"], yq=self.qkv_q[0],
                                          yd=self.qkv_q[1], **extra))
            m.qmm_gemv_fused_op(m.gemv_op(*Lw["o"], H, H, xq=self.qkv_q[0], xd=self.qkv_q[1], residual=h_in,
                                          y=self.ref_hmid[li]))
            m.qmm_gemv_fused_op(m.gemv_op(*Lw["gu"], 2 * F, H, x=self.ref_hmid[li], norm_w=Lw["gf"],
                                          yq=self.ffn_q[0], yd=self.ffn_q[1], flags=m.Y_SWIGLU_PAIRS))
            m.qmm_gemv_fused_op(m.gemv_op(*Lw["down"], H, F, xq=self.ffn_q[0], xd=self.ffn_q[1],
                                          residual=self.ref_hmid[li], y=self.ref_h[li]))
            h_in = self.ref_h[li]
        m.qmm_gemv_fused_op(m.gemv_op(*self.lm, V, H, x=h_in, norm_w=self.gfin, y=self.ref_logits))

    def chain(self):
        m, H, Q, F, V = self.qmm, self.H, self.Q, self.F, self.V
        ops = []
        for li, Lw in enumerate(self.layers):
            b, first = 4 * li, li == 0
            extra = dict(xq=self.a0[0], xd=self.a0[1]) if first else {}
            ops.append(m.chain_op(*Lw["qkv"], Q, H, src=-1 if first else b - 1, x=self.x if first else None,
                                  norm_w=Lw["ga"], **extra))
            ops.append(m.chain_op(*Lw["o"], H, H, src=b, residual=-2 if first else b - 1,
                                  x=self.x if first else None, y=self.hmid[li]))
            ops.append(m.chain_op(*Lw["gu"], 2 * F, H, src=b + 1, norm_w=Lw["gf"], flags=m.Y_SWIGLU_PAIRS))
            ops.append(m.chain_op(*Lw["down"], H, F, src=b + 2, residual=b + 1, y=self.h[li]))
        ops.append(m.chain_op(*self.lm, V, H, src=4 * self.L - 1, norm_w=self.gfin, y=self.logits))
        return ops

    def outputs(self):
        return [self.logits, *self.h, *self.hmid, *self.a0]

    def refs(self):
        return [self.ref_logits, *self.ref_h, *self.ref_hmid, *self.ref_a0]


def test_decode_chain_equals_per_op_launches_call_after_call():
    qmm = lib()
    qmm.qmm_last_device_error()
    m = Mini(qmm)
    m.per_op()
    ops = m.chain()
    wsb = qmm.qmm_decode_chain_workspace_size(ops)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    for call in range(3):  # the workspace carries the call counter: no clearing in between
        for t in m.outputs():
            t.fill_(0)
        qmm.qmm_decode_chain(ops, ws, wsb)
        assert qmm.qmm_last_device_error() == 0
        for i, (a, b) in enumerate(zip(m.outputs(), m.refs())):
            assert torch.equal(a, b), f"output {i} differs from the per-op launches (call {call})"
    assert int(ws[:4].view(torch.int32).item()) == 3  # three calls counted


def test_decode_chain_from_a_replayed_graph():
    qmm = lib()
    m = Mini(qmm, L=2, seed=10)
    m.per_op()
    ops = m.chain()
    wsb = qmm.qmm_decode_chain_workspace_size(ops)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        qmm.qmm_decode_chain(ops, ws, wsb, stream=s)  # first call outside capture (one-time set-up)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        qmm.qmm_decode_chain(ops, ws, wsb, stream=torch.cuda.current_stream())
    for _ in range(4):
        m.logits.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(m.logits, m.ref_logits)
    assert qmm.qmm_last_device_error() == 0


def test_decode_chain_full_tinyllama_step_equals_per_op_step():
    qmm = lib()
    import bench
    dec = bench.TinyLlamaDecode(qmm, torch, seed=4)
    dec.step()
    torch.cuda.synchronize()
    ref = dec.logits.clone()
    href = [h.clone() for h in dec.h]
    hmid = dec.hmid.clone()
    ops = (qmm.ChainOp * dec.n_ops)(*dec.decode_ops(intermediates=True))
    for call in range(2):
        dec.logits.fill_(0)
        for h in dec.h:
            h.fill_(0)
        qmm.qmm_decode_chain(ops, dec.dws, dec.dws_bytes)
        assert qmm.qmm_last_device_error() == 0
        assert torch.isfinite(ref).all()
        assert torch.equal(dec.logits, ref), f"logits differ (call {call})"
        assert all(torch.equal(a, b) for a, b in zip(dec.h, href))
        assert torch.equal(dec.hmid, hmid)
