"""qmm_moe_gemv_static -- the MoE expert GEMV whose routing tables live in the
library's fixed device scratch (no workspace, no allocation) -- called through
the C ABI twice in a row with different routings, each output checked
against qmm_moe_gemv with a caller workspace and against the oracle, within
the fp32 tolerance |y - y_ref| <= 1e-5 * S + 1e-6; the second call is
watched for device allocations (torch's allocator and the driver's free
memory).  Collected last so it also runs after every other GPU test has used
the device."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import workloads
from parity import lib, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _experts(qmm, E, N, K, used, seed):
    qs = torch.zeros(E, N, K // 2, dtype=torch.uint8, device=DEV)
    d = torch.zeros(E, N, K // 32, dtype=torch.int16, device=DEV)
    ref = {}
    for e in sorted(set(int(v) for v in used)):
        w = workloads.weights(N, K, sigma=0.02, seed=seed, index=e)
        qmm.qmm_quantize_q4_0(w.to(DEV), N, K, K, qs[e], d[e])
        ref[e] = O.quantize_q4_0(w.numpy())
    return qs, d, ref


def _with_workspace(qmm, qs, d, E, N, K, ids, T, k, xq, xd, per_slot):
    ws_bytes = qmm.qmm_moe_workspace_size(E, T, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    y = torch.full((T * k, N), float("nan"), device=DEV)
    qmm.qmm_moe_gemv(qs, d, E, N, K, ids, T, k, xq, xd, per_slot, y, ws, ws_bytes)
    return y


def test_static_scratch_moe_matches_workspace_entry_twice():
    qmm = lib()
    qmm.qmm_last_device_error()  # start from a clear device error word
    E, N, K = 64, 300, 512
    # call 1: 16 tokens, top-8 by the sigmoid router, activation shared per token
    T1, k1 = 16, 8
    ids1, _ = O.router_topk(workloads.router_logits(T1, E, seed=11).numpy(), k1)
    # call 2: other routing, one activation row per slot, duplicates, fewer tokens
    T2, k2 = 5, 4
    ids2 = np.array([[3, 3, 60, 1], [7, 7, 7, 7], [0, 63, 3, 12], [12, 12, 0, 5], [1, 2, 3, 4]], np.int32)
    qs, d, ref = _experts(qmm, E, N, K, np.concatenate([ids1.reshape(-1), ids2.reshape(-1)]), seed=12)

    x1 = workloads.activations(T1, K, seed=13)
    x2 = workloads.activations(T2 * k2, K, seed=14)
    cases = [(ids1, T1, k1, x1, 0), (ids2, T2, k2, x2, 1)]
    # every input and output exists before the first call, so the two calls
    # below run back to back and the second one can be watched for allocations
    outs = []
    for ids, T, k, x, per_slot in cases:
        xq, xd = qmm.quantize_q8_0(x.to(DEV))
        ids_d = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(DEV)
        y = torch.full((T * k, N), float("nan"), device=DEV)
        outs.append((y, xq, xd, ids_d))
    torch.cuda.synchronize()
    mem = []
    for (ids, T, k, x, per_slot), (y, xq, xd, ids_d) in zip(cases, outs):  # two static calls in a row
        qmm.qmm_moe_gemv_static(qs, d, E, N, K, ids_d, T, k, xq, xd, per_slot, y)
        torch.cuda.synchronize()
        mem.append((torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]))
    # the second call (the device already set up by the first) allocated
    # nothing: neither through torch's allocator nor from the driver
    assert mem[1] == mem[0], mem
    for (ids, T, k, x, per_slot), (y_static, xq, xd, ids_d) in zip(cases, outs):
        y_ws = _with_workspace(qmm, qs, d, E, N, K, ids_d, T, k, xq, xd, per_slot)
        qx, dx = O.quantize_q8_0(x.numpy())
        flat = ids.reshape(-1)
        for s in range(T * k):
            row = s if per_slot else s // k
            y_ref, S = O.matmul_int(*ref[int(flat[s])], qx[row], dx[row])
            y_ws_s = y_ws[s].cpu().numpy().astype(np.float64)
            assert_close(y_static[s][None], y_ws_s[None], S, f"vs workspace, slot {s}")
            assert_close(y_static[s][None], y_ref, S, f"vs oracle, slot {s}")
    assert qmm.qmm_last_device_error() == 0


def test_static_scratch_rejects_sizes_beyond_its_limit():
    qmm = lib()
    E, k = 256, 8
    # (4E + 2 + T*k) int32 words: T = 8064 needs 262,152 B > 256 KiB
    assert qmm.qmm_moe_workspace_size(E, 8063, k) <= 256 * 1024 < qmm.qmm_moe_workspace_size(E, 8064, k)
    small = torch.zeros(64, dtype=torch.uint8, device=DEV)
    y = torch.full((4,), float("nan"), device=DEV)
    with pytest.raises(qmm.QmmError) as ei:
        qmm.qmm_moe_gemv_static(small, small, E, 64, 64, small, 8064, k, small, small, 0, y)
    assert ei.value.status == 9
    assert torch.isnan(y.cpu()).all()  # nothing launched
    assert qmm.qmm_last_device_error() == 0
