"""Sigmoid top-k router on the GPU (Colibri page, "Arquitectura del Sistema")
against the oracle's router: expert ids identical (the selection is an
integer decision on exact fp32 logits), gates within 1e-6 (fp32 expf and
division against double); the expert grouping it builds in the same launch
against the counting definition; the expert GEMV on that grouping equal,
bit for bit, to qmm_moe_gemv on the same ids; and a MoE layer run from router
logits end to end against the oracle layer."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import workloads
from parity import lib, assert_close
from test_gpu_moe import Experts

pytestmark = pytest.mark.gpu
DEV = "cuda"
GATE_TOL = 1e-6


def _route(qmm, logits, k, group):
    T, E = logits.shape
    ids = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    gates = torch.full((T, k), float("nan"), device=DEV)
    ws, wsb = None, 0
    if group:
        wsb = qmm.qmm_moe_workspace_size(E, T, k)
        ws = torch.full((wsb,), 0xAB, dtype=torch.uint8, device=DEV)  # need not start zeroed
    qmm.qmm_moe_router_topk(logits.to(DEV).contiguous(), T, E, k, ids, gates, ws, wsb)
    assert qmm.qmm_last_device_error() == 0
    return ids.cpu().numpy(), gates.cpu().numpy(), ws


def _check_router(ids, gates, logits, k):
    ref_ids, ref_g = O.router_topk(logits.numpy(), k)
    assert np.array_equal(ids, ref_ids)
    assert np.all(np.abs(gates.astype(np.float64) - ref_g) <= GATE_TOL)


def _check_grouping(ws, ids, E):
    """Tables (int32 words): counts[E] | offsets[E+1] | cursor[E] | active[E]
    | n_active | slots[T*k]: counts per expert, exclusive offsets, active
    experts in ascending order with the start of each one's slots, each
    expert's slot span holding exactly the slots routed to it (in any
    order)."""
    w = ws.view(torch.int32).cpu().numpy()
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    active = np.nonzero(counts)[0]
    assert np.array_equal(w[:E], counts)
    assert np.array_equal(w[E:2 * E + 1], offsets)
    a0 = 3 * E + 1
    n_active = w[4 * E + 1]
    assert n_active == len(active)
    assert np.array_equal(w[a0:a0 + n_active], active)
    c0 = 2 * E + 1  # cursor[i]: the start of the i-th active expert's slots
    assert np.array_equal(w[c0:c0 + n_active], offsets[active])
    slots = w[4 * E + 2:4 * E + 2 + flat.size]
    for e in active:
        span = slots[offsets[e]:offsets[e + 1]]
        assert sorted(span.tolist()) == np.nonzero(flat == e)[0].tolist(), e


@pytest.mark.parametrize("T,E,k", [(16, 256, 8), (1, 256, 8), (7, 40, 5), (3, 1024, 64), (2, 1, 1), (4, 33, 33),
                                   (300, 256, 8)])
@pytest.mark.parametrize("group", [False, True])
def test_router_matches_oracle(T, E, k, group):
    logits = workloads.router_logits(T, E, seed=T + E)
    ids, gates, ws = _route(lib(), logits, k, group)
    _check_router(ids, gates, logits, k)
    if group:
        _check_grouping(ws, ids, E)


def test_router_ties_and_domain_ends():
    """Integer-valued logits (ties everywhere: lower expert index first),
    equal logits, and logits at both ends of the domain [-87, 16]."""
    qmm = lib()
    g = torch.Generator().manual_seed(4)
    cases = [torch.randint(-3, 4, (50, 96), generator=g).float(),
             torch.full((4, 64), 0.5),
             torch.empty(20, 512).uniform_(-87, 16, generator=g),
             torch.tensor([[16.0, 15.999999, -87.0, 16.0, -86.99999, 0.0]])]
    for L in cases:
        for k in (1, 3, min(32, L.shape[1])):
            ids, gates, ws = _route(qmm, L, k, group=True)
            _check_router(ids, gates, L, k)
            _check_grouping(ws, ids, L.shape[1])


def test_router_many_tokens_one_cta_and_grid_agree():
    """The grouping launch routes every token in one CTA; the plain launch
    spreads tokens over many CTAs: same ids and bit-identical gates."""
    qmm = lib()
    logits = workloads.router_logits(2000, 256, seed=9)
    a_ids, a_g, ws = _route(qmm, logits, 8, group=True)
    b_ids, b_g, _ = _route(qmm, logits, 8, group=False)
    assert np.array_equal(a_ids, b_ids) and np.array_equal(a_g, b_g)
    _check_router(a_ids, a_g, logits, 8)
    _check_grouping(ws, a_ids, 256)


@pytest.mark.parametrize("E,N,K,x_per_slot", [(64, 300, 512, 0), (64, 300, 512, 1), (16, 40, 96, 0)])
def test_pregrouped_gemv_equals_gemv_on_same_ids(E, N, K, x_per_slot):
    """Streaming kernel (K multiple of 256) and the fallback kernel (K = 96)."""
    qmm = lib()
    T, k = 16, 4
    logits = workloads.router_logits(T, E, seed=3)
    ids, gates, ws = _route(qmm, logits, k, group=True)
    ex = Experts(qmm, E, N, K, ids.reshape(-1), seed=2)
    x = workloads.activations(T * k if x_per_slot else T, K, seed=5)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    wsb = ws.numel()
    y_pre = torch.full((T * k, N), float("nan"), device=DEV)
    qmm.qmm_moe_gemv_pregrouped(ex.qs, ex.d, E, N, K, T, k, xq, xd, x_per_slot, y_pre, ws, wsb)
    y_ref = torch.full((T * k, N), float("nan"), device=DEV)
    ws2 = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    qmm.qmm_moe_gemv(ex.qs, ex.d, E, N, K, torch.from_numpy(ids).to(DEV), T, k, xq, xd, x_per_slot, y_ref, ws2, wsb)
    assert qmm.qmm_last_device_error() == 0
    assert torch.equal(y_pre, y_ref)
    qx, dx = O.quantize_q8_0(x.numpy())
    for s in (0, 9, T * k - 1):
        row = s if x_per_slot else s // k
        ref, S = O.matmul_int(*ex.oracle[int(ids.reshape(-1)[s])], qx[row], dx[row])
        assert_close(y_pre[s][None], ref, S, f"slot {s}")


def test_moe_layer_from_router_logits_end_to_end():
    """A small MoE layer entirely on the GPU from router logits (route + group,
    gate, up, SwiGLU + Q8_0, down, combine) against the oracle's layer with
    the oracle's router: same experts, relative L2 of the output <= 1e-4 (the
    fp32 gates and SwiGLU may move an activation code at a rounding
    boundary)."""
    qmm = lib()
    T, E, k, H, F = 4, 32, 4, 512, 256
    logits = workloads.router_logits(T, E, seed=12)
    ids_ref, gates_ref = O.router_topk(logits.numpy(), k)
    used = np.unique(ids_ref)
    gate = Experts(qmm, E, F, H, used, seed=7, base_index=0)
    up = Experts(qmm, E, F, H, used, seed=7, base_index=1000)
    down = Experts(qmm, E, H, F, used, seed=7, base_index=2000)
    x = workloads.activations(T, H, seed=13)
    wsb = qmm.qmm_moe_workspace_size(E, T, k)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    gts = torch.empty(T, k, device=DEV)
    qmm.qmm_moe_router_topk(logits.to(DEV), T, E, k, ids, gts, ws, wsb)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    yg = torch.empty(T * k, F, device=DEV)
    yu = torch.empty(T * k, F, device=DEV)
    qmm.qmm_moe_gemv_pregrouped(gate.qs, gate.d, E, F, H, T, k, xq, xd, 0, yg, ws, wsb)
    qmm.qmm_moe_gemv_pregrouped(up.qs, up.d, E, F, H, T, k, xq, xd, 0, yu, ws, wsb)
    hq = torch.empty(T * k, F, dtype=torch.int8, device=DEV)
    hd = torch.empty(T * k, F // 32, dtype=torch.int16, device=DEV)
    qmm.qmm_swiglu_quantize_q8_0(yg, yu, T * k, F, F, hq, hd)
    z = torch.empty(T * k, H, device=DEV)
    qmm.qmm_moe_gemv_pregrouped(down.qs, down.d, E, H, F, T, k, hq, hd, 1, z, ws, wsb)
    y = torch.empty(T, H, device=DEV)
    qmm.qmm_moe_combine(z, gts, T, k, H, y)
    assert qmm.qmm_last_device_error() == 0
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    qx, dx = O.quantize_q8_0(x.numpy())
    y_ref, _, _ = O.moe_forward(gate.oracle, up.oracle, down.oracle, ids_ref, gates_ref.astype(np.float32), qx, dx)
    rel = np.linalg.norm(y.cpu().numpy() - y_ref) / np.linalg.norm(y_ref)
    assert rel <= 1e-4, rel


@pytest.mark.parametrize("T,E,k,H,F", [(1, 256, 8, 512, 256), (3, 8, 8, 256, 512), (16, 64, 8, 512, 256)])
def test_moe_layer_entry_equals_its_four_calls(T, E, k, H, F):
    """qmm_moe_layer_f32 (router, gate/up + SwiGLU, down, combine as one call,
    the down launch reading the grouping and streaming weights before the
    gate/up launch ends) gives ids, gates, h, z and y of the four separate
    calls bit for bit, for two layers back to back on different routings
    (one slot per weight pass, every expert routed, four slots per pass),
    called directly and replayed from a CUDA graph; and the layer against
    the oracle's (relative L2 <= 1e-4, as the layer test above)."""
    qmm = lib()
    gate = Experts(qmm, E, F, H, np.arange(E), seed=17, base_index=0, oracle_ids=[])
    up = Experts(qmm, E, F, H, np.arange(E), seed=17, base_index=1000, oracle_ids=[])
    down = Experts(qmm, E, H, F, np.arange(E), seed=17, base_index=2000, oracle_ids=[])
    gu_qs = torch.stack([gate.qs, up.qs], dim=2).reshape(E, 2 * F, H // 2).contiguous()
    gu_d = torch.stack([gate.d, up.d], dim=2).reshape(E, 2 * F, H // 32).contiguous()
    wsb = qmm.qmm_moe_workspace_size(E, T, k)
    logits = [workloads.router_logits(T, E, seed=40 + r).to(DEV).contiguous() for r in range(2)]
    xs = [workloads.activations(T, H, seed=50 + r).to(DEV).contiguous() for r in range(2)]

    def bufs():
        return dict(ids=torch.full((T, k), -7, dtype=torch.int32, device=DEV),
                    gates=torch.full((T, k), float("nan"), device=DEV),
                    h=torch.full((T * k, F), float("nan"), device=DEV),
                    z=torch.full((T * k, H), float("nan"), device=DEV),
                    y=torch.full((T, H), float("nan"), device=DEV),
                    ws=torch.full((wsb,), 0x3A, dtype=torch.uint8, device=DEV))

    sep = [bufs() for _ in range(2)]
    for r, b in enumerate(sep):
        qmm.qmm_moe_router_topk(logits[r], T, E, k, b["ids"], b["gates"], b["ws"], wsb)
        qmm.qmm_moe_gemv_gate_up(gu_qs, gu_d, E, 2 * F, H, T, k, xs[r], None, None, 0, b["h"], b["ws"], wsb)
        qmm.qmm_moe_gemv_pregrouped_f32(down.qs, down.d, E, H, F, T, k, b["h"], 1, b["z"], b["ws"], wsb)
        qmm.qmm_moe_combine(b["z"], b["gates"], T, k, H, b["y"])
    one = [bufs() for _ in range(2)]
    for r, b in enumerate(one):  # back to back on the stream
        qmm.qmm_moe_layer_f32(logits[r], T, E, k, gu_qs, gu_d, down.qs, down.d, H, F, xs[r], b["ids"], b["gates"],
                              b["h"], b["z"], b["y"], b["ws"], wsb)
    assert qmm.qmm_last_device_error() == 0
    for a, b in zip(sep, one):
        for key in ("ids", "gates", "h", "z", "y"):
            assert torch.equal(a[key], b[key]), key
        assert not torch.isnan(b["y"]).any()
    # the same two layers captured in a CUDA graph and replayed twice (the
    # launches keep their programmatic dependencies as graph edges)
    gph = [bufs() for _ in range(2)]

    def run():
        for r, b in enumerate(gph):
            qmm.qmm_moe_layer_f32(logits[r], T, E, k, gu_qs, gu_d, down.qs, down.d, H, F, xs[r], b["ids"],
                                  b["gates"], b["h"], b["z"], b["y"], b["ws"], wsb)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for b in gph:
        b["y"].fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert qmm.qmm_last_device_error() == 0
    for a, b in zip(sep, gph):
        for key in ("ids", "gates", "h", "z", "y"):
            assert torch.equal(a[key], b[key]), key
    # the layer against the oracle's layer (the fp32 activations quantized as qmm_quantize_q8_0 does)
    ids_ref, gates_ref = O.router_topk(logits[0].cpu().numpy(), k)
    assert np.array_equal(one[0]["ids"].cpu().numpy(), ids_ref)
    gate.oracle_from_planes(ids_ref.reshape(-1))
    up.oracle_from_planes(ids_ref.reshape(-1))
    down.oracle_from_planes(ids_ref.reshape(-1))
    qx, dx = O.quantize_q8_0(xs[0].cpu().numpy())
    y_ref, _, _ = O.moe_forward(gate.oracle, up.oracle, down.oracle, ids_ref, gates_ref.astype(np.float32), qx, dx)
    rel = np.linalg.norm(one[0]["y"].cpu().numpy() - y_ref) / np.linalg.norm(y_ref)
    assert rel <= 1e-4, rel
