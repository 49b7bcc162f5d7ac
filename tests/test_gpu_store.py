"""Expert hot-store on the device: over a sequence of routed decode steps
with evictions (and experts loaded again after one), a separate copy stream
and prefetch of the next step's experts, the expert GEMV on the slot arena
(ids remapped by the store) matches the oracle's product with each slot's
routed expert within |y - y_ref| <= 1e-5 * S + 1e-6, and is bit-identical to
the same GEMV on all experts resident; the store's hit and
miss counts follow the host policy; an expert that is not resident maps to
-1 and is reported."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import workloads
from parity import lib, u16, assert_close, planes_to_oracle
from test_store_lru import RefLru

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _experts(qmm, E, N, K, seed):
    qs = torch.empty(E, N, K // 2, dtype=torch.uint8, device=DEV)
    d = torch.empty(E, N, K // 32, dtype=torch.int16, device=DEV)
    for e in range(E):
        w = workloads.weights(N, K, sigma=0.02, seed=seed, index=e, device=DEV)
        qmm.qmm_quantize_q4_0(w, N, K, K, qs[e], d[e])
    return qs, d


@pytest.mark.parametrize("separate_copy_stream,prefetch", [(False, False), (True, False), (True, True)])
def test_store_gemv_equals_all_resident(separate_copy_stream, prefetch):
    qmm = lib()
    E, S, N, K, T, k = 48, 10, 256, 512, 2, 4
    qs, d = _experts(qmm, E, N, K, seed=5)
    host = (qs.cpu().pin_memory(), d.cpu().pin_memory())
    arena = (torch.zeros(S, N, K // 2, dtype=torch.uint8, device=DEV),
             torch.zeros(S, N, K // 32, dtype=torch.int16, device=DEV))
    slot_of = torch.empty(E, dtype=torch.int32, device=DEV)
    store = qmm.ExpertStore(E, S, [(host[0], arena[0]), (host[1], arena[1])], slot_of)
    ref = RefLru(E, S)
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream() if separate_copy_stream else compute
    wsb = qmm.qmm_moe_workspace_size(max(E, S), T, k)
    ws1 = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ws2 = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    # skewed routing: a fixed per-expert bias on the router logits
    bias = torch.randn(E, generator=torch.Generator().manual_seed(1)) * 1.5
    steps = [O.router_topk((workloads.router_logits(T, E, seed=100 + i) + bias).numpy(), k)[0] for i in range(25)]
    x = workloads.activations(T, K, seed=3)
    xq, xd = qmm.quantize_q8_0(x.to(DEV))
    outs, refs = [], []
    seen, reloaded = set(), set()  # experts loaded before; experts loaded again after an eviction
    for i, ids in enumerate(steps):
        flat = ids.reshape(-1).tolist()
        reloaded |= {e for e in flat if e in seen and e not in ref.res}
        store.request(flat, compute, copy)
        ref.request(flat, use=True)
        seen |= set(flat)
        ids_d = torch.from_numpy(ids).to(DEV)
        slot_ids = torch.empty_like(ids_d)
        store.map_ids(ids_d, slot_ids)
        y = torch.empty(T * k, N, device=DEV)
        qmm.qmm_moe_gemv(arena[0], arena[1], S, N, K, slot_ids, T, k, xq, xd, 0, y, ws1, wsb)
        store.release(compute)
        if prefetch and i + 1 < len(steps):
            nxt = steps[i + 1].reshape(-1).tolist()
            reloaded |= {e for e in nxt if e in seen and e not in ref.res}
            store.prefetch(nxt, copy)
            ref.request(nxt, use=False)
        y_ref = torch.empty(T * k, N, device=DEV)
        qmm.qmm_moe_gemv(qs, d, E, N, K, ids_d, T, k, xq, xd, 0, y_ref, ws2, wsb)
        outs.append(y)
        refs.append(y_ref)
    assert qmm.qmm_last_device_error() == 0
    for i, (a, b) in enumerate(zip(outs, refs)):
        assert torch.equal(a, b), f"step {i}"
    # every slot of every step against the oracle's product with the routed
    # expert (read from the all-resident planes), including experts that
    # were evicted and loaded again
    assert reloaded, "the routing never brought an evicted expert back"
    qx, dx = xq.cpu().numpy(), u16(xd)
    Wo = {}
    for i, ids in enumerate(steps):
        for s_, e in enumerate(ids.reshape(-1).tolist()):
            if e not in Wo:
                Wo[e] = planes_to_oracle(qs[e], d[e], N, K)
            y_ref, S = O.matmul_int(*Wo[e], qx[s_ // k], dx[s_ // k])
            assert_close(outs[i][s_][None], y_ref, S, f"step {i} slot {s_} (expert {e})")
    st = store.stats()
    assert {k_: st[k_] for k_ in ("hits", "misses", "evictions", "prefetched")} == ref.stats
    assert st["misses"] > 0 and st["evictions"] > 0 and st["hits"] > 0
    assert st["bytes_copied"] == (st["misses"] + st["prefetched"]) * (N * K // 2 + N * K // 32 * 2)
    assert all(int(slot_of[e]) == ref.res.get(e, -1) for e in range(E))


def test_store_map_of_absent_expert_is_reported():
    qmm = lib()
    E, S, N, K = 8, 2, 64, 64
    qs, d = _experts(qmm, E, N, K, seed=6)
    host = (qs.cpu().pin_memory(), d.cpu().pin_memory())
    arena = (torch.zeros(S, N, K // 2, dtype=torch.uint8, device=DEV),
             torch.zeros(S, N, K // 32, dtype=torch.int16, device=DEV))
    slot_of = torch.empty(E, dtype=torch.int32, device=DEV)
    store = qmm.ExpertStore(E, S, [(host[0], arena[0]), (host[1], arena[1])], slot_of)
    qmm.qmm_last_device_error()
    store.request([3, 5])
    ids = torch.tensor([3, 5, 6], dtype=torch.int32, device=DEV)
    out = torch.empty_like(ids)
    store.map_ids(ids, out)
    assert out.tolist() == [0, 1, -1]
    assert qmm.qmm_last_device_error() == 7  # QMM_ERR_BAD_EXPERT_ID
    with pytest.raises(qmm.QmmError):
        store.request([0, 1, 2])  # three distinct experts, two slots
    assert torch.equal(arena[0][0], qs[3]) and torch.equal(arena[1][1], d[5])
