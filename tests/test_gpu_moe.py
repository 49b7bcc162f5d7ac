"""MoE expert-grouped GEMV against the CPU oracle, stage by stage (every
stage fed generator inputs, never another GPU stage's output), then the whole
layer end to end with a propagated tolerance."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import workloads
from parity import lib, u16, assert_close, planes_to_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


class Experts:
    """E experts of one matrix kind (N x K each), stored back to back as planes;
    fp32 rows kept on the host only for the experts the test routes to."""

    def __init__(self, qmm, E, N, K, used, sigma=0.02, seed=0, base_index=0, device_gen="cpu", oracle_ids=None):
        self.E, self.N, self.K = E, N, K
        self.qs = torch.zeros(E, N, K // 2, dtype=torch.uint8, device=DEV)
        self.d = torch.zeros(E, N, K // 32, dtype=torch.int16, device=DEV)
        self.oracle = {}
        keep = set(int(v) for v in (used if oracle_ids is None else oracle_ids))
        for e in sorted(set(int(v) for v in used)):
            w = workloads.weights(N, K, sigma=sigma, seed=seed, index=base_index + e, device=device_gen)
            qmm.qmm_quantize_q4_0(w.to(DEV), N, K, K, self.qs[e], self.d[e])
            if e in keep:
                self.oracle[e] = O.quantize_q4_0(w.cpu().numpy())

    def oracle_from_planes(self, ids):
        """Oracle copies of experts `ids` read back from the device planes
        (the GPU quantizer is bit-exact against the oracle's)."""
        for e in sorted(set(int(v) for v in ids) - set(self.oracle)):
            self.oracle[e] = planes_to_oracle(self.qs[e], self.d[e], self.N, self.K)


def _ids_gates(T, E, k, seed):
    logits = workloads.router_logits(T, E, seed=seed).numpy()
    ids, gates = O.router_topk(logits, k)
    return ids, gates.astype(np.float32)


def _moe_gemv(qmm, ex, ids, T, k, xq, xd, x_per_slot):
    ws_bytes = qmm.qmm_moe_workspace_size(ex.E, T, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    y = torch.full((T * k, ex.N), float("nan"), device=DEV)
    qmm.qmm_moe_gemv(ex.qs, ex.d, ex.E, ex.N, ex.K, ids, T, k, xq, xd, x_per_slot, y, ws, ws_bytes)
    return y


@pytest.mark.parametrize("T,E,k,N,K", [(1, 8, 2, 64, 96), (16, 64, 8, 300, 512), (5, 4, 4, 17, 2048),
                                         (5, 33, 4, 64, 512), (16, 33, 8, 40, 256)])
def test_moe_gemv_shared_x(T, E, k, N, K):
    qmm = lib()
    ids, _ = _ids_gates(T, E, k, seed=T)
    ex = Experts(qmm, E, N, K, ids.reshape(-1), seed=1)
    x = workloads.activations(T, K, seed=2)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    y = _moe_gemv(qmm, ex, torch.from_numpy(ids).to(DEV), T, k, xq, xd, 0)
    assert qmm.qmm_last_device_error() == 0
    qx, dx = O.quantize_q8_0(x.numpy())
    for t in range(T):
        for j in range(k):
            ref, S = O.matmul_int(*ex.oracle[int(ids[t, j])], qx[t], dx[t])
            assert_close(y[t * k + j][None], ref, S, f"slot ({t},{j})")


def test_moe_gemv_per_slot_x_duplicates_and_empty_experts():
    """x per slot (the down projection), duplicate ids inside a token, most
    experts without tokens, one expert with many tokens (> one token group)."""
    qmm = lib()
    T, E, k, N, K = 6, 32, 4, 130, 256
    ids = np.array([[3, 3, 7, 31]] * 3 + [[7, 7, 7, 7], [0, 3, 31, 7], [3, 0, 0, 3]], np.int32)
    ex = Experts(qmm, E, N, K, ids.reshape(-1), seed=3)
    x = workloads.activations(T * k, K, seed=4)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    y = _moe_gemv(qmm, ex, torch.from_numpy(ids).to(DEV), T, k, xq, xd, 1)
    qx, dx = O.quantize_q8_0(x.numpy())
    for s in range(T * k):
        ref, S = O.matmul_int(*ex.oracle[int(ids.reshape(-1)[s])], qx[s], dx[s])
        assert_close(y[s][None], ref, S, f"slot {s}")


def test_moe_bad_expert_id_is_skipped_and_reported():
    qmm = lib()
    T, E, k, N, K = 2, 8, 2, 40, 64
    ids = np.array([[1, 9], [-1, 2]], np.int32)  # 9 and -1 are out of range
    ex = Experts(qmm, E, N, K, [1, 2], seed=5)
    x = workloads.activations(T, K, seed=6)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    y = _moe_gemv(qmm, ex, torch.from_numpy(ids).to(DEV), T, k, xq, xd, 0)
    assert qmm.qmm_last_device_error() == 7
    assert qmm.qmm_last_device_error() == 0  # the word is cleared once read
    yc = y.cpu()
    assert torch.isnan(yc[1]).all() and torch.isnan(yc[2]).all()  # skipped slots untouched
    qx, dx = O.quantize_q8_0(x.numpy())
    for s, (t, e) in {0: (0, 1), 3: (1, 2)}.items():
        ref, S = O.matmul_int(*ex.oracle[e], qx[t], dx[t])
        assert_close(y[s][None], ref, S, f"slot {s}")


def test_moe_combine():
    qmm = lib()
    T, k, N = 16, 8, 6144
    g = torch.Generator().manual_seed(3)
    z = torch.randn(T, k, N, generator=g)
    _, gates = _ids_gates(T, 256, k, seed=3)
    y = torch.empty(T, N, device=DEV)
    qmm.qmm_moe_combine(z.to(DEV), torch.from_numpy(gates).to(DEV), T, k, N, y)
    ref = O.moe_combine(z.numpy().astype(np.float64), gates)
    mag = O.moe_combine(np.abs(z.numpy()).astype(np.float64), np.abs(gates))
    assert np.all(np.abs(y.cpu().numpy() - ref) <= 1e-6 * mag + 1e-30)


@pytest.mark.parametrize("T", [1, 16])
def test_glm_moe_layer_full_size(T):
    """GLM-scale layer: hidden 6144, 256 experts of 2048 x 6144 gate/up and
    6144 x 2048 down, sigmoid top-8 router, SwiGLU between.

    Stage checks (each against the oracle on generator inputs): gate/up for
    every routed slot (T = 1) or sampled slots (T = 16); the down projection
    on a generator activation per slot.  End to end, at 1 and 16 tokens (128
    slots, every one in the oracle layer): the full GPU layer against the
    oracle layer, relative L2 error <= 1e-4 -- SwiGLU in fp32 on
    the GPU vs float64 in the oracle may move an activation code by one at a
    rounding boundary, so this stage is bounded, not bit-matched."""
    qmm = lib()
    c = workloads.MOE
    H, F, E, k = c["hidden"], c["expert_ffn"], c["experts"], c["top_k"]
    ids, gates = _ids_gates(T, E, k, seed=0)
    used = ids.reshape(-1)
    slots = list(range(T * k)) if T == 1 else [0, 5, 17, 63, 64, 100, 127]
    checked = used[slots]
    gate = Experts(qmm, E, F, H, used, seed=0, base_index=0, device_gen=DEV, oracle_ids=checked)
    up = Experts(qmm, E, F, H, used, seed=0, base_index=1000, device_gen=DEV, oracle_ids=checked)
    down = Experts(qmm, E, H, F, used, seed=0, base_index=2000, device_gen=DEV, oracle_ids=checked)
    x = workloads.activations(T, H, seed=0)
    ids_d = torch.from_numpy(ids).to(DEV)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    qx, dx = O.quantize_q8_0(x.numpy())
    assert np.array_equal(xq.cpu().numpy(), qx)

    yg = _moe_gemv(qmm, gate, ids_d, T, k, xq, xd, 0)
    yu = _moe_gemv(qmm, up, ids_d, T, k, xq, xd, 0)
    for s in slots:
        t, e = s // k, int(used[s])
        for ex, yy in ((gate, yg), (up, yu)):
            ref, S = O.matmul_int(*ex.oracle[e], qx[t], dx[t])
            assert_close(yy[s][None], ref, S, f"gate/up slot {s}")

    # down projection on a generator activation per slot
    hx = workloads.activations(T * k, F, seed=1)
    hq, hd = qmm.quantize_q8_0(hx.to(DEV))
    yd = _moe_gemv(qmm, down, ids_d, T, k, hq, hd, 1)
    qh, dh = O.quantize_q8_0(hx.numpy())
    for s in slots:
        ref, S = O.matmul_int(*down.oracle[int(used[s])], qh[s], dh[s])
        assert_close(yd[s][None], ref, S, f"down slot {s}")

    # end to end, every routed slot (the oracle's copies of the routed
    # experts not yet held are read from the device planes)
    h_q = torch.empty(T * k, F, dtype=torch.int8, device=DEV)
    h_d = torch.empty(T * k, F // 32, dtype=torch.int16, device=DEV)
    qmm.qmm_swiglu_quantize_q8_0(yg, yu, T * k, F, F, h_q, h_d)
    z = _moe_gemv(qmm, down, ids_d, T, k, h_q, h_d, 1)
    y = torch.empty(T, H, device=DEV)
    qmm.qmm_moe_combine(z, torch.from_numpy(gates).to(DEV), T, k, H, y)
    for ex in (gate, up, down):
        ex.oracle_from_planes(used)
    y_ref, _, _ = O.moe_forward(gate.oracle, up.oracle, down.oracle, ids, gates, qx, dx)
    rel = np.linalg.norm(y.cpu().numpy() - y_ref) / np.linalg.norm(y_ref)
    assert rel <= 1e-4, rel
