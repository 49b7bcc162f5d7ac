"""qmm_moe_gemv_gate_up -- the gate and up expert GEMVs and SwiGLU (TinyLLaMA
guide section 4.4) in one launch over interleaved gate/up rows -- against the
unfused path on the same grouping: every output bit-identical to
qmm_swiglu_quantize_q8_0's h_out of the two separate qmm_moe_gemv_pregrouped
outputs (one slot per weight pass and four), and against the oracle's fp64
SwiGLU of its own gate and up products with the tolerance propagated through
the SwiGLU."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import workloads
from parity import lib
from test_gpu_moe import Experts

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _interleave(a, b):
    """Rows of a and b alternated (g0, u0, g1, u1, ...) per expert."""
    return torch.stack([a, b], dim=2).reshape(a.shape[0], 2 * a.shape[1], a.shape[2]).contiguous()


def _layer_inputs(qmm, T, E, k, F, H, x_per_slot, seed):
    logits = workloads.router_logits(T, E, seed=seed)
    wsb = qmm.qmm_moe_workspace_size(E, T, k)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    gts = torch.empty(T, k, device=DEV)
    qmm.qmm_moe_router_topk(logits.to(DEV), T, E, k, ids, gts, ws, wsb)
    used = np.unique(ids.cpu().numpy())
    gate = Experts(qmm, E, F, H, used, seed=seed, base_index=0)
    up = Experts(qmm, E, F, H, used, seed=seed, base_index=1000)
    x = workloads.activations(T * k if x_per_slot else T, H, seed=seed + 1)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    return ids.cpu().numpy(), ws, wsb, gate, up, x, xq, xd


@pytest.mark.parametrize("T,E,k,F,H,x_per_slot", [(1, 64, 8, 300, 512, 0), (16, 64, 8, 300, 512, 0),
                                                  (16, 32, 4, 256, 1024, 1), (3, 8, 8, 40, 256, 0)])
def test_gate_up_equals_separate_gemvs_and_swiglu(T, E, k, F, H, x_per_slot):
    """Bit-identical to gate and up as two pregrouped launches plus the SwiGLU
    kernel; 16 tokens x top-8 of 64 experts takes the four-slots-per-pass
    kernel, one token the one-slot kernel; F not a multiple of the 32-row
    group leaves ragged pairs at each expert's end; 8 experts x top-8 routes
    every expert."""
    qmm = lib()
    ids, ws, wsb, gate, up, x, xq, xd = _layer_inputs(qmm, T, E, k, F, H, x_per_slot, seed=T + E)
    gu_qs, gu_d = _interleave(gate.qs, up.qs), _interleave(gate.d, up.d)
    h = torch.full((T * k, F), float("nan"), device=DEV)
    qmm.qmm_moe_gemv_gate_up(gu_qs, gu_d, E, 2 * F, H, T, k, None, xq, xd, x_per_slot, h, ws, wsb)
    yg = torch.empty(T * k, F, device=DEV)
    yu = torch.empty(T * k, F, device=DEV)
    qmm.qmm_moe_gemv_pregrouped(gate.qs, gate.d, E, F, H, T, k, xq, xd, x_per_slot, yg, ws, wsb)
    qmm.qmm_moe_gemv_pregrouped(up.qs, up.d, E, F, H, T, k, xq, xd, x_per_slot, yu, ws, wsb)
    hq = torch.empty(T * k, F, dtype=torch.int8, device=DEV)
    hd = torch.empty(T * k, F // 32, dtype=torch.int16, device=DEV)
    h_ref = torch.empty(T * k, F, device=DEV)
    if F % 32 == 0:
        qmm.qmm_swiglu_quantize_q8_0(yg, yu, T * k, F, F, hq, hd, h_ref)
    else:  # the SwiGLU kernel takes whole 32-blocks: pad the rows to the next block
        Fp = (F + 31) // 32 * 32
        pad = lambda t: torch.nn.functional.pad(t, (0, Fp - F)).contiguous()  # noqa: E731
        hp = torch.empty(T * k, Fp, device=DEV)
        qmm.qmm_swiglu_quantize_q8_0(pad(yg), pad(yu), T * k, Fp, Fp, torch.empty(T * k, Fp, dtype=torch.int8,
                                     device=DEV), torch.empty(T * k, Fp // 32, dtype=torch.int16, device=DEV), hp)
        h_ref = hp[:, :F].contiguous()
    assert qmm.qmm_last_device_error() == 0
    assert not torch.isnan(h).any()
    assert torch.equal(h, h_ref)


def test_gate_up_vs_oracle_swiglu():
    """h against SwiGLU of the oracle's fp64 gate and up products: |h - h_ref|
    <= 1.1 tol_g |u| + |silu(g)| tol_u + 2^-23 |h_ref| + 1e-7, with tol = 1e-5 S +
    1e-6 the product tolerance and 1.1 >= max |silu'|."""
    qmm = lib()
    T, E, k, F, H = 4, 32, 4, 256, 1024
    ids, ws, wsb, gate, up, x, xq, xd = _layer_inputs(qmm, T, E, k, F, H, 0, seed=21)
    h = torch.empty(T * k, F, device=DEV)
    qmm.qmm_moe_gemv_gate_up(_interleave(gate.qs, up.qs), _interleave(gate.d, up.d), E, 2 * F, H, T, k, None, xq, xd, 0,
                             h, ws, wsb)
    assert qmm.qmm_last_device_error() == 0
    qx, dx = O.quantize_q8_0(x.numpy())
    flat = ids.reshape(-1)
    for s in range(T * k):
        g, Sg = O.matmul_int(*gate.oracle[int(flat[s])], qx[s // k], dx[s // k])
        u, Su = O.matmul_int(*up.oracle[int(flat[s])], qx[s // k], dx[s // k])
        g, u, Sg, Su = g[0], u[0], Sg[0], Su[0]
        sg = g / (1.0 + np.exp(-g))
        ref = sg * u
        bound = 1.1 * (1e-5 * Sg + 1e-6) * np.abs(u) + np.abs(sg) * (1e-5 * Su + 1e-6) + 2.0 ** -23 * np.abs(ref) + 1e-7
        err = np.abs(h[s].cpu().numpy().astype(np.float64) - ref)
        assert np.all(err <= bound), (s, float(np.max(err - bound)))


def test_gate_up_shape_errors():
    """Odd N (rows that do not pair) and K off the streaming kernel's 256
    multiple are shape errors; nothing is written."""
    qmm = lib()
    T, E, k = 2, 8, 2
    wsb = qmm.qmm_moe_workspace_size(E, T, k)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    qs = torch.zeros(E, 64, 256, dtype=torch.uint8, device=DEV)
    d = torch.zeros(E, 64, 16, dtype=torch.int16, device=DEV)
    xq = torch.zeros(T, 512, dtype=torch.int8, device=DEV)
    xd = torch.zeros(T, 16, dtype=torch.int16, device=DEV)
    h = torch.full((T * k, 32), 7.0, device=DEV)
    with pytest.raises(qmm.QmmError) as ei:
        qmm.qmm_moe_gemv_gate_up(qs, d, E, 63, 512, T, k, None, xq, xd, 0, h, ws, wsb)
    assert ei.value.status == 2
    with pytest.raises(qmm.QmmError) as ei:
        qmm.qmm_moe_gemv_gate_up(qs, d, E, 64, 96, T, k, None, xq[:, :96].contiguous(), xd[:, :3].contiguous(), 0, h, ws,
                                 wsb)
    assert ei.value.status == 2
    assert torch.all(h == 7.0)


@pytest.mark.parametrize("T,E,k,F,H", [(1, 64, 8, 256, 512), (16, 64, 8, 512, 1024)])
def test_fp32_activations_equal_quantize_then_gemv(T, E, k, F, H):
    """fp32 activations quantized inside the launch: qmm_moe_gemv_gate_up with
    x equals it with qmm_quantize_q8_0(x), and qmm_moe_gemv_pregrouped_f32 on
    the fp32 SwiGLU output equals qmm_moe_gemv_pregrouped on its Q8_0, bit for
    bit (one slot per weight pass and four)."""
    qmm = lib()
    ids, ws, wsb, gate, up, x, xq, xd = _layer_inputs(qmm, T, E, k, F, H, 0, seed=31 + T)
    gu_qs, gu_d = _interleave(gate.qs, up.qs), _interleave(gate.d, up.d)
    xf = x.to(DEV).contiguous()
    h_q8 = torch.full((T * k, F), float("nan"), device=DEV)
    qmm.qmm_moe_gemv_gate_up(gu_qs, gu_d, E, 2 * F, H, T, k, None, xq, xd, 0, h_q8, ws, wsb)
    h_f32 = torch.full((T * k, F), float("nan"), device=DEV)
    qmm.qmm_moe_gemv_gate_up(gu_qs, gu_d, E, 2 * F, H, T, k, xf, None, None, 0, h_f32, ws, wsb)
    assert torch.equal(h_f32, h_q8)
    down = Experts(qmm, E, H, F, np.unique(ids), seed=31 + T, base_index=2000)
    hq, hd = qmm.quantize_q8_0(h_f32)
    z_q8 = torch.full((T * k, H), float("nan"), device=DEV)
    qmm.qmm_moe_gemv_pregrouped(down.qs, down.d, E, H, F, T, k, hq, hd, 1, z_q8, ws, wsb)
    z_f32 = torch.full((T * k, H), float("nan"), device=DEV)
    qmm.qmm_moe_gemv_pregrouped_f32(down.qs, down.d, E, H, F, T, k, h_f32, 1, z_f32, ws, wsb)
    assert qmm.qmm_last_device_error() == 0
    assert not torch.isnan(z_f32).any()
    assert torch.equal(z_f32, z_q8)


def test_fp32_activation_entry_errors():
    """The fp32 entry needs a 16-byte aligned x and the streaming kernel (K a
    multiple of 256)."""
    qmm = lib()
    T, E, k = 2, 8, 2
    wsb = qmm.qmm_moe_workspace_size(E, T, k)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    qs = torch.zeros(E, 64, 48, dtype=torch.uint8, device=DEV)
    d = torch.zeros(E, 64, 3, dtype=torch.int16, device=DEV)
    x = torch.zeros(T, 100, device=DEV)
    y = torch.full((T * k, 64), 7.0, device=DEV)
    with pytest.raises(qmm.QmmError) as ei:
        qmm.qmm_moe_gemv_pregrouped_f32(qs, d, E, 64, 96, T, k, x, 0, y, ws, wsb)
    assert ei.value.status == 2
    with pytest.raises(qmm.QmmError) as ei:
        qmm.qmm_moe_gemv_pregrouped_f32(qs, d, E, 64, 96, T, k, x[:, 1:], 0, y, ws, wsb)
    assert ei.value.status == 3
    assert torch.all(y == 7.0)


@pytest.mark.parametrize("T", [1, 16])
def test_glm_layer_recipe_full_size(T):
    """The GLM-scale layer as bench.py runs it (router + grouping; gate/up
    with SwiGLU in one launch; down; combine; at one token the fp32
    activations are quantized inside the expert GEMVs, at 16 tokens by
    standalone launches) equals, bit for bit at every stage, the same layer
    with separate gate and up launches, the SwiGLU kernel and Q8_0 launches;
    at one token the output is also within relative L2 1e-4 of the oracle
    layer (SwiGLU in fp32 vs float64 may move an activation code by one)."""
    qmm = lib()
    c = workloads.MOE
    H, F, E, k = c["hidden"], c["expert_ffn"], c["experts"], c["top_k"]
    logits = workloads.router_logits(T, E, seed=3)
    wsb = qmm.qmm_moe_workspace_size(E, T, k)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    gts = torch.empty(T, k, device=DEV)
    qmm.qmm_moe_router_topk(logits.to(DEV), T, E, k, ids, gts, ws, wsb)
    used = np.unique(ids.cpu().numpy())
    keep = used if T == 1 else []
    gate = Experts(qmm, E, F, H, used, seed=3, base_index=0, device_gen=DEV, oracle_ids=keep)
    up = Experts(qmm, E, F, H, used, seed=3, base_index=1000, device_gen=DEV, oracle_ids=keep)
    down = Experts(qmm, E, H, F, used, seed=3, base_index=2000, device_gen=DEV, oracle_ids=keep)
    gu_qs, gu_d = _interleave(gate.qs, up.qs), _interleave(gate.d, up.d)
    x = workloads.activations(T, H, seed=4)
    xf = x.to(DEV).contiguous()
    xq, xd = qmm.quantize_q8_0(xf)

    # the bench recipe
    h = torch.empty(T * k, F, device=DEV)
    z = torch.empty(T * k, H, device=DEV)
    y = torch.empty(T, H, device=DEV)
    if T * k * 4 <= E:
        qmm.qmm_moe_gemv_gate_up(gu_qs, gu_d, E, 2 * F, H, T, k, xf, None, None, 0, h, ws, wsb)
        qmm.qmm_moe_gemv_pregrouped_f32(down.qs, down.d, E, H, F, T, k, h, 1, z, ws, wsb)
    else:
        qmm.qmm_moe_gemv_gate_up(gu_qs, gu_d, E, 2 * F, H, T, k, None, xq, xd, 0, h, ws, wsb)
        hq, hd = qmm.quantize_q8_0(h)
        qmm.qmm_moe_gemv_pregrouped(down.qs, down.d, E, H, F, T, k, hq, hd, 1, z, ws, wsb)
    qmm.qmm_moe_combine(z, gts, T, k, H, y)

    # the unfused layer
    yg = torch.empty(T * k, F, device=DEV)
    yu = torch.empty(T * k, F, device=DEV)
    qmm.qmm_moe_gemv_pregrouped(gate.qs, gate.d, E, F, H, T, k, xq, xd, 0, yg, ws, wsb)
    qmm.qmm_moe_gemv_pregrouped(up.qs, up.d, E, F, H, T, k, xq, xd, 0, yu, ws, wsb)
    h2 = torch.empty(T * k, F, device=DEV)
    h2q = torch.empty(T * k, F, dtype=torch.int8, device=DEV)
    h2d = torch.empty(T * k, F // 32, dtype=torch.int16, device=DEV)
    qmm.qmm_swiglu_quantize_q8_0(yg, yu, T * k, F, F, h2q, h2d, h2)
    z2 = torch.empty(T * k, H, device=DEV)
    qmm.qmm_moe_gemv_pregrouped(down.qs, down.d, E, H, F, T, k, h2q, h2d, 1, z2, ws, wsb)
    y2 = torch.empty(T, H, device=DEV)
    qmm.qmm_moe_combine(z2, gts, T, k, H, y2)
    assert qmm.qmm_last_device_error() == 0
    assert torch.equal(h, h2)
    assert torch.equal(z, z2)
    assert torch.equal(y, y2)

    if T == 1:
        qx, dx = O.quantize_q8_0(x.numpy())
        ref_ids, ref_g = O.router_topk(logits.numpy(), k)
        assert np.array_equal(ids.cpu().numpy(), ref_ids)
        y_ref, _, _ = O.moe_forward(gate.oracle, up.oracle, down.oracle, ref_ids, ref_g.astype(np.float32), qx, dx)
        rel = np.linalg.norm(y.cpu().numpy() - y_ref) / np.linalg.norm(y_ref)
        assert rel <= 1e-4, rel


@pytest.mark.parametrize("T,E,k", [(1, 64, 8), (16, 256, 8), (5, 33, 4)])
def test_group_ids_tables_and_gate_up_on_them(T, E, k):
    """qmm_moe_group_ids on ids that are not the router's (random, with
    duplicates inside a token): the tables equal the counting definition; and
    on the router's own ids the fused gate/up over these tables equals, bit
    for bit, the same launch over the router's grouping."""
    from test_gpu_router import _check_grouping
    qmm = lib()
    rng = np.random.default_rng(T * 100 + E)
    ids_any = rng.integers(0, E, size=(T, k)).astype(np.int32)
    ids_any[0, :2] = 0  # a duplicate expert inside one token
    wsb = qmm.qmm_moe_workspace_size(E, T, k)
    ws = torch.full((wsb,), 0xCD, dtype=torch.uint8, device=DEV)  # need not start initialised
    qmm.qmm_moe_group_ids(torch.from_numpy(ids_any).to(DEV), T, k, E, ws, wsb)
    assert qmm.qmm_last_device_error() == 0
    _check_grouping(ws, ids_any, E)

    F, H = 256, 512
    ids, ws_r, _, gate, up, x, xq, xd = _layer_inputs(qmm, T, E, k, F, H, 0, seed=T + 7)
    gu_qs, gu_d = _interleave(gate.qs, up.qs), _interleave(gate.d, up.d)
    h_r = torch.full((T * k, F), float("nan"), device=DEV)
    qmm.qmm_moe_gemv_gate_up(gu_qs, gu_d, E, 2 * F, H, T, k, None, xq, xd, 0, h_r, ws_r, wsb)
    ws_g = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    qmm.qmm_moe_group_ids(torch.from_numpy(ids).to(DEV), T, k, E, ws_g, wsb)
    h_g = torch.full((T * k, F), float("nan"), device=DEV)
    qmm.qmm_moe_gemv_gate_up(gu_qs, gu_d, E, 2 * F, H, T, k, None, xq, xd, 0, h_g, ws_g, wsb)
    assert qmm.qmm_last_device_error() == 0
    assert torch.equal(h_g, h_r)


def test_group_ids_reports_an_id_out_of_range():
    """An id outside [0, E) is left out of the tables and reported through
    the device error word; the other slots are grouped."""
    qmm = lib()
    T, E, k = 2, 8, 2
    ids = np.array([[1, 9], [3, 1]], np.int32)
    wsb = qmm.qmm_moe_workspace_size(E, T, k)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    qmm.qmm_last_device_error()
    qmm.qmm_moe_group_ids(torch.from_numpy(ids).to(DEV), T, k, E, ws, wsb)
    assert qmm.qmm_last_device_error() == 7
    w = ws.view(torch.int32).cpu().numpy()
    assert w[1] == 2 and w[3] == 1 and w[4 * E + 1] == 2  # counts of experts 1 and 3; two active
