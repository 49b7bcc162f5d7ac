#!/usr/bin/env python
"""Benchmark of the Q4_0 x Q8_0 decode path on GB300.

Headline (the JSON line's `value`): batch-1 GEMV weight GB/s over a
TinyLLaMA-1.1B-shaped decode step -- 22 layers of fused QKV 2048->2560,
O 2048->2048, gate/up 2048->2x5632 (one launch over interleaved rows, SwiGLU
in its epilogue), down 5632->2048 (residual add in its epilogue), then
lm_head 2048->32000: 89 dependent GEMVs per step.  The residual stream stays
fp32 and is RMSNorm-ed and quantized to Q8_0 inside the GEMV that reads it;
QKV and gate/up hand the next GEMV a Q8_0 output; O and down add the
residual.  The step runs as 89 launches chained with programmatic dependent
launch (qmm_gemv_fused_op), replayed from a CUDA graph.  581,861,376 weight
bytes per step (> L2, so no flush).

Also reported on the same line (`also`): batch-16 GEMM TOPS on the large
dense FFN + lm_head shapes, and the GLM-scale MoE layer.

`--impl reference` times the CPU oracle on a bounded row sample of the same
decode step (the reference arm: a deliberately plain program, for context).
"""
from __future__ import annotations

import argparse
import concurrent.futures
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
# DRAM traffic per launch of the decode step's kernel from an ncu capture, and
# the sources it was taken from (a JSON record beside the ncu summaries)
DECODE_TRAFFIC = os.path.join(ROOT, "profiles", "decode_step_traffic.json")


def _sources_digest(paths):
    h = hashlib.sha256()
    for path in paths:
        with open(os.path.join(ROOT, path), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _profiled_traffic():
    """DRAM bytes per launch of the decode kernel from the committed capture
    record, or None once the kernel sources differ from the captured ones."""
    try:
        with open(DECODE_TRAFFIC) as f:
            rec = json.load(f)
        digest = _sources_digest(rec["sources"])
    except Exception:
        return None
    return int(rec["traffic_bytes_per_launch"]) if digest.startswith(rec["sources_sha256"]) else None


def max_over_ranks(torch, times, device):
    """Each rank's timed-region lengths -> the maximum over ranks of each (one
    all-reduce; any backend: `device` is where the backend keeps tensors),
    followed by a barrier."""
    tt = torch.tensor([float(v) for v in times], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.barrier()
    return tt.tolist()


def whole_job_gbs(world_size, bytes_per_step_per_rank, steps, seconds):
    """Weak-scaling whole-job throughput: every rank streams the same
    weights each step, so the job moves world_size times the bytes in the
    slowest rank's time."""
    return world_size * bytes_per_step_per_rank * steps / seconds / 1e9


def _peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------- dist
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- decode step
class TinyLlamaDecode:
    """Weights and buffers of the TinyLLaMA-shaped decode step, and the step itself."""

    def __init__(self, qmm, torch, seed=0, dev="cuda"):
        c = workloads.TINYLLAMA
        self.qmm, self.torch, self.dev = qmm, torch, dev
        self.H, self.F, self.Q, self.V, self.L = c["hidden"], c["ffn"], c["qkv"], c["vocab"], c["layers"]
        sigma = c["sigma"]
        self.layers = []
        idx = 0

        def planes(N, K):
            nonlocal idx
            w = workloads.weights(N, K, sigma=sigma, seed=seed, index=idx, device=dev)
            idx += 1
            qs, d = qmm.quantize_q4_0(w)
            del w
            return qs, d

        for _ in range(self.L):
            qkv = planes(self.Q, self.H)
            o = planes(self.H, self.H)
            g = planes(self.F, self.H)
            u = planes(self.F, self.H)
            # gate and up rows interleaved (g0, u0, g1, u1, ...): one launch
            # computes both and writes SwiGLU(g, u) from each row pair
            gu = (torch.stack([g[0], u[0]], 1).reshape(2 * self.F, -1).contiguous(),
                  torch.stack([g[1], u[1]], 1).reshape(2 * self.F, -1).contiguous())
            down = planes(self.H, self.F)
            self.layers.append({"qkv": qkv, "o": o, "gu": gu, "down": down})
        self.lm_head = planes(self.V, self.H)
        self.weight_bytes = sum(workloads.q4_0_bytes(N, K) for _, N, K in workloads.tinyllama_matrices())
        f32 = lambda n: torch.zeros(n, dtype=torch.float32, device=dev)  # noqa: E731
        q8 = lambda n: (torch.zeros(n, dtype=torch.int8, device=dev),  # noqa: E731
                        torch.zeros(n // 32, dtype=torch.int16, device=dev))
        # RMSNorm weights ahead of attention and FFN in every layer, and the final one
        self.norms = [(workloads.norm_weights(self.H, seed=seed, index=2000 + 2 * li, device=dev),
                       workloads.norm_weights(self.H, seed=seed, index=2001 + 2 * li, device=dev))
                      for li in range(self.L)]
        self.norm_final = workloads.norm_weights(self.H, seed=seed, index=1999, device=dev)
        self.eps = 1e-5
        self.x_in = workloads.activations(1, self.H, seed=seed, device=dev)[0].contiguous()
        self.h = [f32(self.H), f32(self.H)]       # fp32 residual stream after each layer (ping-pong)
        self.hmid = f32(self.H)                   # ... after the attention half of a layer
        self.qkv_q, self.ffn_q = q8(self.Q), q8(self.F)
        self.logits = f32(self.V)
        self.launches_per_step = 4 * self.L + 1  # step(): one launch per GEMV
        # algorithmic bytes per step: weights + activations and norm weights
        # read + outputs written (Q8_0: 34 bytes per 32 values; fp32: 4)
        q8b = lambda n: n // 32 * 34  # noqa: E731
        H4 = 4 * self.H
        act = 0
        for _ in range(self.L):
            act += H4 + H4 + q8b(self.Q)              # QKV: RMSNorm(h) -> Q8_0 out
            act += q8b(self.H) + H4 + H4              # O: q slice in, residual in, fp32 out
            act += H4 + H4 + q8b(self.F)              # gate/up: RMSNorm(h1), SwiGLU pairs -> Q8_0 out
            act += q8b(self.F) + H4 + H4              # down: residual in, fp32 out
        act += H4 + H4 + 4 * self.V                   # lm_head: RMSNorm(h) -> logits
        self.algo_bytes = self.weight_bytes + act

        self.op_list = self._ops()
        self.n_ops = len(self.op_list)
        self.op_array = qmm.gemv_op_array(self.op_list)

    def _ops(self):
        """The decode step as qmm_gemv_op descriptors, in order.  Per layer
        (TinyLLaMA guide 5.2 graph; attention itself is outside this path):
        QKV on RMSNorm(h) -> Q8_0; O on the q slice, + h -> h1 (fp32); gate/up
        on RMSNorm(h1) with SwiGLU of row pairs -> Q8_0; down, + h1 -> next h.
        Then the lm_head on RMSNorm(h)."""
        q, H, F = self.qmm, self.H, self.F
        op, eps = q.gemv_op, self.eps
        ops, h_in = [], self.x_in
        for li, Lw in enumerate(self.layers):
            g_attn, g_ffn = self.norms[li]
            h_out = self.h[li % 2]
            ops.append(op(*Lw["qkv"], self.Q, H, x=h_in, norm_w=g_attn, norm_eps=eps, yq=self.qkv_q[0],
                          yd=self.qkv_q[1]))
            ops.append(op(*Lw["o"], H, H, xq=self.qkv_q[0], xd=self.qkv_q[1], residual=h_in, y=self.hmid))
            ops.append(op(*Lw["gu"], 2 * F, H, x=self.hmid, norm_w=g_ffn, norm_eps=eps, yq=self.ffn_q[0],
                          yd=self.ffn_q[1], flags=q.Y_SWIGLU_PAIRS))
            ops.append(op(*Lw["down"], H, F, xq=self.ffn_q[0], xd=self.ffn_q[1], residual=self.hmid, y=h_out))
            h_in = h_out
        ops.append(op(*self.lm_head, self.V, H, x=h_in, norm_w=self.norm_final, norm_eps=eps, y=self.logits))
        return ops

    def step(self, stream=None):
        """The step as 89 GEMV launches chained with programmatic dependent launch."""
        for o in self.op_list:
            self.qmm.qmm_gemv_fused_op(o, self.qmm.CHAIN, stream=stream)

    def step_chain(self, stream=None):
        """The same 89 launches from one qmm_gemv_fused_ops call."""
        self.qmm.qmm_gemv_fused_ops(self.op_array, self.n_ops, self.qmm.CHAIN, stream=stream)

def _graph(torch, fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm: lazy attribute set-up happens outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _time_graph(torch, g, steps, warmup):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3  # seconds


def _flush_l2(torch, buf):
    buf.add_(1.0)


# ---------------------------------------------------------------------------- extras
def bench_gemm_b16(qmm, torch, reps=20, dev="cuda", M=16):
    """Batch-M GEMM (16 by default; 2 = a one-draft speculative verify) on the
    large dense FFN + lm_head shapes (TOPS = 2*M*N*K per second), through
    qmm_gemm_q4_0_q8_0_ws."""
    mats = workloads.large_dense_matrices()
    sigma = workloads.LARGE_DENSE["sigma"]
    ws, xs, ys, ops, wbytes = [], [], [], 0, 0
    # one workspace for the set: the calls run one after another on one stream
    wsb = max(max(1, qmm.qmm_gemm_workspace_size(K, M)) for _, N, K in mats)
    work = torch.empty(wsb, dtype=torch.uint8, device=dev)
    for i, (_, N, K) in enumerate(mats):
        w = workloads.weights(N, K, sigma=sigma, seed=0, index=100 + i, device=dev)
        ws.append((qmm.quantize_q4_0(w), N, K))
        del w
        x = workloads.activations(M, K, seed=0, index=600 + i, device=dev)
        xs.append(qmm.quantize_q8_0(x))
        ys.append(torch.empty(M, N, device=dev))
        ops += 2 * M * N * K
        wbytes += workloads.q4_0_bytes(N, K)

    def run():
        for ((qs, d), N, K), (xq, xd), y in zip(ws, xs, ys):
            qmm.qmm_gemm_q4_0_q8_0_ws(qs, d, N, K, M, xq, xd, y, N, work, wsb)

    g = _graph(torch, run)
    t = _time_graph(torch, g, reps, 3)
    per = t / reps
    return {"metric": f"batch-{M} Q4_0xQ8_0 GEMM TOPS", "value": round(ops / per / 1e12, 2), "unit": "TOPS",
            "ms_per_step": round(per * 1e3, 4), "weight_GBps": round(wbytes / per / 1e9, 1),
            "config": {"workload": workloads.LARGE_DENSE["name"] + f", batch {M}", "M": M,
                       "shapes": [[N, K] for _, N, K in mats], "l2": "inputs larger than L2 (987 MB weights)"}}


def bench_moe(qmm, torch, T=16, reps=10, dev="cuda"):
    """GLM-scale MoE layer, T tokens, from router logits on the device:
    sigmoid top-k router + slot grouping; gate and up expert GEMVs with
    SwiGLU in one launch (interleaved gate/up rows); down expert GEMV;
    combine.  With few routed slots (T*k*4 <= E: the expert GEMV takes one
    slot per weight pass) the two GEMVs quantize their fp32 activations
    while staging them (four launches: 1 token 49.9 -> 49.1 us); with more,
    each CTA would requantize four activation rows per expert segment, and
    standalone Q8_0 launches of x and h are faster (six launches: 16 tokens
    477.8 -> 469.3 us).  One graph replay runs the layer on three routings
    in turn (back to back, as consecutive layers run), so no layer finds its
    experts' weights in L2 from the layer before; the time is per layer."""
    import numpy as np
    c = workloads.MOE
    H, F, E, k = c["hidden"], c["expert_ffn"], c["experts"], c["top_k"]
    sigma = c["sigma"]

    def experts(N, K, base):
        qs = torch.empty(E, N, K // 2, dtype=torch.uint8, device=dev)
        d = torch.empty(E, N, K // 32, dtype=torch.int16, device=dev)
        for e in range(E):
            w = workloads.weights(N, K, sigma=sigma, seed=0, index=base + e, device=dev)
            qmm.qmm_quantize_q4_0(w, N, K, K, qs[e], d[e])
        return qs, d

    gate, up, down = experts(F, H, 0), experts(F, H, 1000), experts(H, F, 2000)
    # gate and up rows interleaved per expert (g0, u0, g1, u1, ...)
    gu = tuple(torch.stack([g, u], dim=2).reshape(E, 2 * F, g.shape[2]).contiguous() for g, u in zip(gate, up))
    del gate, up
    # R routings (router logits of seeds 0..R-1): one graph replay runs the
    # layer once on each, so consecutive layers read different experts and no
    # expert's weights are still in L2 from the layer before
    R = 3
    logits = [workloads.router_logits(T, E, seed=r).to(dev) for r in range(R)]
    ids = [torch.empty(T, k, dtype=torch.int32, device=dev) for _ in range(R)]
    gts = [torch.empty(T, k, dtype=torch.float32, device=dev) for _ in range(R)]
    x = workloads.activations(T, H, seed=0, device=dev)
    h = torch.empty(T * k, F, device=dev)
    in_launch = T * k * 4 <= E
    xq = torch.empty(T, H, dtype=torch.int8, device=dev)
    xd = torch.empty(T, H // 32, dtype=torch.int16, device=dev)
    hq = torch.empty(T * k, F, dtype=torch.int8, device=dev)
    hd = torch.empty(T * k, F // 32, dtype=torch.int16, device=dev)
    z = torch.empty(T * k, H, device=dev)
    y = torch.empty(T, H, device=dev)
    wsb = qmm.qmm_moe_workspace_size(E, T, k)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)

    def layer(r):
        if in_launch:
            # the layer entry: router + grouping, gate/up + SwiGLU, down, combine;
            # the down launch streams its weights before the gate/up launch ends
            qmm.qmm_moe_layer_f32(logits[r], T, E, k, *gu, *down, H, F, x, ids[r], gts[r], h, z, y, ws, wsb)
            return
        # the router (sigmoid top-k) groups the slots by expert in the same
        # launch; the expert GEMVs reuse that grouping
        qmm.qmm_moe_router_topk(logits[r], T, E, k, ids[r], gts[r], ws, wsb)
        qmm.qmm_quantize_q8_0(x, T, H, H, xq, xd)
        qmm.qmm_moe_gemv_gate_up(*gu, E, 2 * F, H, T, k, None, xq, xd, 0, h, ws, wsb)
        qmm.qmm_quantize_q8_0(h, T * k, F, F, hq, hd)
        qmm.qmm_moe_gemv_pregrouped(*down, E, H, F, T, k, hq, hd, 1, z, ws, wsb)
        qmm.qmm_moe_combine(z, gts[r], T, k, H, y)

    def run():
        for r in range(R):
            layer(r)

    g = _graph(torch, run)
    # bookkeeping for the byte count, outside the timed region
    uniq = [len(np.unique(i.cpu().numpy())) for i in ids]
    t = _time_graph(torch, g, reps, 3)
    per = t / (reps * R)  # one layer
    wbytes = sum(uniq) / R * 3 * workloads.q4_0_bytes(F, H)
    return {"metric": "MoE layer expert-weight GB/s", "value": round(wbytes / per / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(per * 1e3, 4), "tokens_per_s": round(T / per, 1), "unique_experts": uniq,
            "config": {"workload": c["name"], "T": T, "experts": E, "top_k": k, "hidden": H, "expert_ffn": F,
                       "launches": 4 if in_launch else 6, "routings": R,
                       "l2": "each replay runs the layer on 3 routings in turn (router logits of seeds 0, 1, 2)"}}


def bench_moe_store(qmm, torch, T=1, dev="cuda"):
    """GLM-scale MoE layer with an expert store: all 256 experts (interleaved
    gate/up planes and down planes; 21.2 MB each) in pinned host memory, 64
    of them resident in a slot arena in HBM.  Each decode step: router on the
    device, its expert ids to the host, store request (copies of missing
    experts on a copy stream), ids remapped to slots and grouped, the layer on
    the arena (gate/up with SwiGLU in one launch, down, combine), release.
    Routing is skewed by a fixed per-expert bias.  Timed end to end (the host
    reads each step's ids), after as many warm-up steps as timed ones."""
    import numpy as np
    c = workloads.MOE
    H, F, E, k = c["hidden"], c["expert_ffn"], c["experts"], c["top_k"]
    S, steps = c["store_slots"], c["store_steps"]
    # gate/up: rows interleaved per expert (g0, u0, g1, u1, ...), 2F x H
    shapes = {"gate_up": (2 * F, H, (0, 1)), "down": (H, F, (2,))}
    host, arena = {}, {}
    for name, (N, K, kinds) in shapes.items():
        hq = torch.empty(E, N, K // 2, dtype=torch.uint8, pin_memory=True)
        hd = torch.empty(E, N, K // 32, dtype=torch.int16, pin_memory=True)
        rows = N // len(kinds)
        tq = [torch.empty(rows, K // 2, dtype=torch.uint8, device=dev) for _ in kinds]
        td = [torch.empty(rows, K // 32, dtype=torch.int16, device=dev) for _ in kinds]
        for e in range(E):
            for j, kind in enumerate(kinds):
                w = workloads.weights(rows, K, sigma=c["sigma"], seed=0, index=1000 * kind + e, device=dev)
                qmm.qmm_quantize_q4_0(w, rows, K, K, tq[j], td[j])
            hq[e].copy_(torch.stack(tq, dim=1).reshape(N, K // 2))
            hd[e].copy_(torch.stack(td, dim=1).reshape(N, K // 32))
        host[name] = (hq, hd)
        arena[name] = (torch.empty(S, N, K // 2, dtype=torch.uint8, device=dev),
                       torch.empty(S, N, K // 32, dtype=torch.int16, device=dev))
    slot_of = torch.empty(E, dtype=torch.int32, device=dev)
    planes = [(host[n][i], arena[n][i]) for n in shapes for i in (0, 1)]
    store = qmm.ExpertStore(E, S, planes, slot_of)
    bias = workloads.expert_bias(E, scale=c["store_skew"])
    logits = [(workloads.router_logits(T, E, seed=10 + i) + bias).to(dev) for i in range(2 * steps)]
    x = workloads.activations(T, H, seed=0, device=dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    slot_ids = torch.empty_like(ids)
    gts = torch.empty(T, k, device=dev)
    h = torch.empty(T * k, F, device=dev)
    z, y = torch.empty(T * k, H, device=dev), torch.empty(T, H, device=dev)
    wsb = qmm.qmm_moe_workspace_size(E, T, k)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ids_host = torch.empty(T, k, dtype=torch.int32, pin_memory=True)
    compute, copy = torch.cuda.current_stream(), torch.cuda.Stream()

    def step(lg):
        qmm.qmm_moe_router_topk(lg, T, E, k, ids, gts)
        ids_host.copy_(ids, non_blocking=True)
        torch.cuda.current_stream().synchronize()  # the host needs the ids to drive the copies
        store.request(ids_host.view(-1).tolist(), compute, copy)
        store.map_ids(ids, slot_ids)
        qmm.qmm_moe_group_ids(slot_ids, T, k, S, ws, wsb)
        agu, ad = arena["gate_up"], arena["down"]
        # fp32 activations quantized inside the expert GEMVs (few routed slots per pass)
        qmm.qmm_moe_gemv_gate_up(agu[0], agu[1], S, 2 * F, H, T, k, x, None, None, 0, h, ws, wsb)
        qmm.qmm_moe_gemv_pregrouped_f32(ad[0], ad[1], S, H, F, T, k, h, 1, z, ws, wsb)
        qmm.qmm_moe_combine(z, gts, T, k, H, y)
        store.release(compute)

    for i in range(steps):  # warm the store
        step(logits[i])
    torch.cuda.synchronize()
    s0 = store.stats()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    for i in range(steps, 2 * steps):
        step(logits[i])
    e1.record(compute)
    torch.cuda.synchronize()
    per = e0.elapsed_time(e1) / 1e3 / steps
    s1 = store.stats()
    hits, misses = s1["hits"] - s0["hits"], s1["misses"] - s0["misses"]
    copied = s1["bytes_copied"] - s0["bytes_copied"]
    assert qmm.qmm_last_device_error() == 0
    return {"metric": "MoE layer with expert store, ms per decode step", "value": round(per * 1e3, 4), "unit": "ms",
            "tokens_per_s": round(T / per, 1), "hit_rate": round(hits / max(1, hits + misses), 3),
            "h2d_bytes_per_step": int(copied / steps), "h2d_GBps_avg": round(copied / steps / per / 1e9, 1),
            "config": {"workload": c["name"] + ", expert store", "T": T, "experts": E, "top_k": k,
                       "slots_in_hbm": S, "expert_bytes": 3 * workloads.q4_0_bytes(F, H), "routing_skew": c["store_skew"],
                       "steps": steps}}


# ---------------------------------------------------------------------------- single-kernel cases
def run_case(qmm, torch, name, calls, dev="cuda"):
    """One kernel of the path on one workload shape, called `calls` times
    with CUDA-event timing of each call (no flush: every case reads more than
    L2 per call except decode_gateup, 13 MB, which is what one launch of the
    decode step reads).  For profiler captures (`ncu -k ... -s 3 -c 1`)."""
    M, flags = 1, 0
    if name in ("decode_gateup", "decode_qkv_norm"):  # one launch of the TinyLLaMA decode step
        c = workloads.TINYLLAMA
        N, K, sigma = (2 * c["ffn"], c["hidden"], c["sigma"]) if name == "decode_gateup" else \
            (c["qkv"], c["hidden"], c["sigma"])
    elif name == "lm_head_8192":
        N, K, sigma = workloads.LARGE_DENSE["vocab"], workloads.LARGE_DENSE["hidden"], workloads.LARGE_DENSE["sigma"]
    elif name in ("gemm_b16", "gemm_b64", "gemm_b16_ws"):
        N, K, sigma = workloads.LARGE_DENSE["ffn"], workloads.LARGE_DENSE["hidden"], workloads.LARGE_DENSE["sigma"]
        M = 64 if name == "gemm_b64" else 16
    elif name == "gemm_b16_dense":  # the batch-16 set of the default line: gate, up, down, lm_head
        return {"case": name, **bench_gemm_b16(qmm, torch, reps=max(calls, 3))}
    elif name == "moe_T16":
        return _moe_case(qmm, torch, calls, dev)
    elif name in ("moe_layer_T1", "moe_layer_T16"):  # the whole MoE layer of the default line
        return {"case": name, **bench_moe(qmm, torch, T=1 if name == "moe_layer_T1" else 16, reps=max(calls, 3))}
    elif name == "moe_store":
        return {"case": name, **bench_moe_store(qmm, torch, T=1)}
    elif name == "decode_pdl":  # the whole TinyLLaMA-shaped decode step
        dec = TinyLlamaDecode(qmm, torch)
        ts = _time_calls(torch, dec.step, calls)
        return {"case": name, "us_per_call": [round(t * 1e6, 2) for t in ts],
                "weight_GBps_best": round(dec.weight_bytes / min(ts) / 1e9, 1)}
    else:
        raise SystemExit(f"unknown case {name}")
    w = workloads.weights(N, K, sigma=sigma, seed=0, index=0, device=dev)
    qs, d = qmm.quantize_q4_0(w)
    del w
    xq, xd = qmm.quantize_q8_0(workloads.activations(M, K, seed=0, device=dev))
    y = torch.empty(M, N, device=dev)
    if name == "decode_gateup":  # gate/up: interleaved rows, SwiGLU pairs, Q8_0 in and out
        yq = torch.empty(N // 2, dtype=torch.int8, device=dev)
        yd = torch.empty(N // 64, dtype=torch.int16, device=dev)
        op = lambda: qmm.qmm_gemv_fused(qs, d, N, K, None, xq, xd, None, None, yq, yd,  # noqa: E731
                                        flags=qmm.CHAIN | qmm.Y_SWIGLU_PAIRS)
    elif name == "decode_qkv_norm":  # QKV: fp32 residual stream in, RMSNorm + Q8_0 in the launch, Q8_0 out
        yq = torch.empty(N, dtype=torch.int8, device=dev)
        yd = torch.empty(N // 32, dtype=torch.int16, device=dev)
        h = workloads.activations(1, K, seed=0, device=dev)[0].contiguous()
        g = workloads.norm_weights(K, seed=0, device=dev)
        o1 = qmm.gemv_op(qs, d, N, K, x=h, norm_w=g, yq=yq, yd=yd)
        op = lambda: qmm.qmm_gemv_fused_op(o1, qmm.CHAIN)  # noqa: E731
    elif M == 1:
        op = lambda: qmm.qmm_gemv_q4_0_q8_0(qs, d, N, K, xq, xd, y)  # noqa: E731
    elif name == "gemm_b16_ws":  # the workspace entry: activation operand prepared once per call
        work = torch.empty(qmm.qmm_gemm_workspace_size(K, M), dtype=torch.uint8, device=dev)
        op = lambda: qmm.qmm_gemm_q4_0_q8_0_ws(qs, d, N, K, M, xq, xd, y, N, work, work.numel())  # noqa: E731
    else:
        op = lambda: qmm.qmm_gemm_q4_0_q8_0(qs, d, N, K, M, xq, xd, y, N)  # noqa: E731
    ts = _time_calls(torch, op, calls)
    wbytes = workloads.q4_0_bytes(N, K)
    return {"case": name, "N": N, "K": K, "M": M, "us_per_call": [round(t * 1e6, 2) for t in ts],
            "weight_GBps_best": round(wbytes / min(ts) / 1e9, 1), "TOPS_best": round(2 * M * N * K / min(ts) / 1e12, 2)}


def _time_calls(torch, op, calls):
    st = torch.cuda.current_stream()
    ts = []
    for _ in range(calls):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        op()
        e1.record(st)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    return ts


def _moe_case(qmm, torch, calls, dev):
    """The gate-projection expert GEMV of the GLM-scale MoE layer at 16 tokens
    (256 experts resident, top-8 of a seeded sigmoid router)."""
    import numpy as np
    c = workloads.MOE
    H, F, E, k, T = c["hidden"], c["expert_ffn"], c["experts"], c["top_k"], 16
    qs = torch.empty(E, F, H // 2, dtype=torch.uint8, device=dev)
    d = torch.empty(E, F, H // 32, dtype=torch.int16, device=dev)
    for e in range(E):
        w = workloads.weights(F, H, sigma=c["sigma"], seed=0, index=e, device=dev)
        qmm.qmm_quantize_q4_0(w, F, H, H, qs[e], d[e])
    top = torch.topk(torch.sigmoid(workloads.router_logits(T, E, seed=0).double()), k, dim=1, sorted=True)
    ids = top.indices.to(torch.int32).to(dev)
    uniq = len(np.unique(top.indices.numpy()))
    xq, xd = qmm.quantize_q8_0(workloads.activations(T, H, seed=0, device=dev))
    y = torch.empty(T * k, F, device=dev)
    wsb = qmm.qmm_moe_workspace_size(E, T, k)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ts = _time_calls(torch, lambda: qmm.qmm_moe_gemv(qs, d, E, F, H, ids, T, k, xq, xd, 0, y, ws, wsb), calls)
    wbytes = uniq * workloads.q4_0_bytes(F, H)
    return {"case": "moe_T16", "E": E, "N": F, "K": H, "T": T, "unique_experts": uniq,
            "us_per_call": [round(t * 1e6, 2) for t in ts], "weight_GBps_best": round(wbytes / min(ts) / 1e9, 1)}


# ---------------------------------------------------------------------------- every config
L2_BYTES = 129 << 20


def _rotated_us(torch, make_op, nbytes, calls_min=24):
    """Device time per call of an op over `copies` distinct weight copies
    (together at least 3x the L2), launched back to back from a CUDA graph,
    so every call reads its weights from HBM."""
    copies = int(max(2, min(128, -(-3 * L2_BYTES // max(nbytes, 1)))))
    ops = [make_op() for _ in range(copies)]
    reps = max(1, -(-calls_min // copies))

    def run():
        for _ in range(reps):
            for op in ops:
                op()

    g = _graph(torch, run)
    per_call = _replay_stats(torch, g, reps * copies)
    _LAST_STATS.clear()
    _LAST_STATS.update(per_call)
    return per_call["mean"]


_LAST_STATS = {}
NOMINAL_HBM_GBS = 8000.0  # the nominal HBM3e figure the target is quoted against


def _replay_stats(torch, g, calls, replays=20, warmup=3):
    """Per-call device time (us) of a graph of `calls` calls: each of
    `replays` replays timed on its own with CUDA events; mean, median, p10,
    p90 of the per-call averages."""
    import numpy as np
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(replays + 1)]
    ev[0].record(st)
    for i in range(replays):
        g.replay()
        ev[i + 1].record(st)
    torch.cuda.synchronize()
    t = np.array([ev[i].elapsed_time(ev[i + 1]) * 1e3 / calls for i in range(replays)])
    return {"mean": float(t.mean()), "median": float(np.median(t)), "p10": float(np.percentile(t, 10)),
            "p90": float(np.percentile(t, 90)), "replays": replays, "calls_per_replay": calls}


def _stats_keys(stats):
    return {"us_median": round(stats["median"], 2), "us_p10": round(stats["p10"], 2),
            "us_p90": round(stats["p90"], 2), "timed_replays": stats["replays"],
            "calls_per_replay": stats["calls_per_replay"]}


def product_us(qmm, torch, N, K, M, sigma, fused_f32=False, dev="cuda"):
    """Device time per call (us) of one Q4_0 x Q8_0 product of M tokens with
    its weights cold in HBM (rotated over copies larger than L2): the batch-1
    GEMV (M = 1), the small-batch GEMM, or the fused GEMV on an fp32 input."""
    w = workloads.weights(N, K, sigma=sigma, seed=0, index=0, device=dev)
    qs, d = qmm.quantize_q4_0(w)
    del w
    x = workloads.activations(M, K, seed=0, device=dev)
    xq, xd = qmm.quantize_q8_0(x)
    y = torch.empty(M, N, device=dev)
    # the small-batch GEMM through its workspace entry (the activation operand
    # formed once per call where the 16-warp layout applies)
    ws = torch.empty(max(1, qmm.qmm_gemm_workspace_size(K, M)), dtype=torch.uint8, device=dev)

    def make():
        q2, d2 = qs.clone(), d.clone()
        if fused_f32:
            return lambda: qmm.qmm_gemv_fused(q2, d2, N, K, x[0], None, None, None, y[0], None, None)
        if M == 1:
            return lambda: qmm.qmm_gemv_q4_0_q8_0(q2, d2, N, K, xq[0], xd[0], y[0])
        return lambda: qmm.qmm_gemm_q4_0_q8_0_ws(q2, d2, N, K, M, xq, xd, y, N, ws, ws.numel())

    us = _rotated_us(torch, make, workloads.q4_0_bytes(N, K))
    del qs, d
    torch.cuda.empty_cache()
    return us


def bench_gemv_set(qmm, torch, name, mats, sigma, dev="cuda"):
    """Batch-1 GEMVs (qmm_gemv_q4_0_q8_0, Q8_0 activation in) of a set of
    matrices, each timed alone with its weights cold in HBM: per matrix and
    for the set, weight GB/s and the fraction of the measured copy peak."""
    peak, peak_kind = _peaks()
    rows, tot_us, tot_b = [], 0.0, 0
    for mname, N, K in mats:
        us = product_us(qmm, torch, N, K, 1, sigma, dev=dev)
        wb = workloads.q4_0_bytes(N, K)
        tot_us += us
        tot_b += wb
        rows.append({"matrix": mname, "N": N, "K": K, "us_per_call": round(us, 2), "us_median": round(
            _LAST_STATS["median"], 2), "weight_GBps": round(wb / us / 1e3, 1),
            "frac_of_hbm_peak": round(wb / us / 1e3 / peak, 4)})
    return {"metric": "batch-1 Q4_0xQ8_0 GEMV weight GB/s", "value": round(tot_b / tot_us / 1e3, 1),
            "unit": "GB/s", "frac_of_hbm_peak": round(tot_b / tot_us / 1e3 / peak, 4), "peak_kind": peak_kind,
            "us_per_set": round(tot_us, 2), "weight_bytes": tot_b, "matrices": rows,
            "config": {"workload": name, "M": 1,
                       "l2": "each matrix rotated over weight copies at least 3x the L2 (129 MB) in size"}}


def run_configs(qmm, torch, dev="cuda"):
    """One JSON line per workload of the five configurations: kernel-only
    device time per call with weights cold in HBM, weight GB/s (and % of the
    measured copy peak), TOPS."""
    peak, peak_kind = _peaks()
    out = []

    def line(cfg, name, N, K, M, us, extra=None):
        wb = workloads.q4_0_bytes(N, K)
        d = {"config": cfg, "workload": name, "N": N, "K": K, "M": M, "us_per_call": round(us, 2),
             "weight_GBps": round(wb / us / 1e3, 1), "pct_of_hbm_peak": round(100 * wb / us / 1e3 / peak, 1),
             "pct_of_nominal_8TBps": round(100 * wb / us / 1e3 / NOMINAL_HBM_GBS, 1),
             "TOPS": round(2 * M * N * K / us / 1e6, 2),
             "tokens_per_s": round(M / us * 1e6, 1),  # tokens through this one product per second
             "peak_kind": peak_kind, **_stats_keys(_LAST_STATS)}
        if extra:
            d.update(extra)
        print(json.dumps(d), flush=True)
        out.append(d)

    def product(N, K, M, sigma, fused_f32=False):
        return product_us(qmm, torch, N, K, M, sigma, fused_f32, dev)

    # read-only stream reference: a 4 GiB fp32 sum (library reduction), the
    # third denominator beside the copy peak and the nominal 8 TB/s
    buf = torch.ones(1 << 30, dtype=torch.float32, device=dev)
    g = _graph(torch, lambda: buf.sum())
    rs = _replay_stats(torch, g, 1, replays=10)
    ro = {"config": "reference", "workload": "read-only stream probe: sum of 4 GiB fp32 (torch)",
          "us_per_call": round(rs["mean"], 1), "read_GBps": round(buf.numel() * 4 / rs["mean"] / 1e3, 1),
          "copy_peak_GBps": peak, "peak_kind": peak_kind, "nominal_GBps": NOMINAL_HBM_GBS}
    print(json.dumps(ro), flush=True)
    out.append(ro)
    del buf, g
    torch.cuda.empty_cache()
    c = workloads.SINGLE_GEMV
    line(0, c["name"] + " (Q8_0 activation in)", c["N"], c["K"], 1, product(c["N"], c["K"], 1, c["sigma"]))
    line(0, c["name"] + " (fp32 activation in, quantized in the launch)", c["N"], c["K"], 1,
         product(c["N"], c["K"], 1, c["sigma"], fused_f32=True))
    dec = TinyLlamaDecode(qmm, torch)
    for path, fn in (("89 launches chained with PDL (qmm_gemv_fused_op)", dec.step),):
        g = _graph(torch, fn)
        stats = _replay_stats(torch, g, 1, replays=100)
        per = stats["mean"] * 1e-6
        d1 = {"config": 1, "workload": workloads.TINYLLAMA["name"] + ": whole decode step, " + path,
              "M": 1, "us_per_call": round(per * 1e6, 2), **_stats_keys(stats), "weight_bytes": dec.weight_bytes,
              "weight_GBps": round(dec.weight_bytes / per / 1e9, 1),
              "pct_of_hbm_peak": round(100 * dec.weight_bytes / per / 1e9 / peak, 1),
              "TOPS": round(2 * dec.weight_bytes / 0.5625 / per / 1e12, 3), "tokens_per_s": round(1 / per, 1),
              "peak_kind": peak_kind}
        print(json.dumps(d1), flush=True)
        out.append(d1)
        del g
    del dec
    torch.cuda.empty_cache()
    for N, K in workloads.BATCHED["shapes"]:
        for M in workloads.BATCHED["M"]:
            line(2, f"batched decode GEMM {N}x{K}", N, K, M, product(N, K, M, workloads.BATCHED["sigma"]))
    for name, N, K in workloads.large_dense_matrices():
        for M in workloads.LARGE_DENSE["M"]:
            line(3, f"large dense {name} {N}x{K}", N, K, M, product(N, K, M, workloads.LARGE_DENSE["sigma"]))
    for name, N, K in (("gate", 28672, 8192), ("down", 8192, 28672), ("TinyLLaMA gate/up", 11264, 2048)):
        for variant in ("int4 per-row x Q8_0", "int2 per-row x Q8_0", "Q4_0 x fp32 (dequantize-then-FMA)"):
            us, wb = format_variant_us(qmm, torch, variant, N, K)
            d = {"config": 3, "workload": f"format variant, {variant}, {name} {N}x{K}", "N": N, "K": K, "M": 1,
                 "us_per_call": round(us, 2), "weight_bytes": wb, "weight_GBps": round(wb / us / 1e3, 1),
                 "pct_of_hbm_peak": round(100 * wb / us / 1e3 / peak, 1),
                 "pct_of_nominal_8TBps": round(100 * wb / us / 1e3 / NOMINAL_HBM_GBS, 1), "peak_kind": peak_kind,
                 **_stats_keys(_LAST_STATS)}
            print(json.dumps(d), flush=True)
            out.append(d)
    for T in workloads.MOE["T"]:
        r = bench_moe(qmm, torch, T=T)
        print(json.dumps({"config": 4, **r}), flush=True)
        out.append(r)
    r = bench_moe_store(qmm, torch, T=1)
    print(json.dumps({"config": 4, **r}), flush=True)
    out.append(r)
    return out


def format_variant_us(qmm, torch, variant, N, K, dev="cuda"):
    """Device time per batch-1 call of a weight-format variant (weights
    rotated over copies larger than L2) and its weight bytes."""
    w = workloads.weights(N, K, sigma=0.01, seed=0, index=0, device=dev)
    if variant.startswith("int"):
        bits = 4 if variant.startswith("int4") else 2
        q, sc = qmm.quantize_rowwise(w, bits)
        xq, xd = qmm.quantize_q8_0(workloads.activations(1, K, seed=0, device=dev))
        wb = N * K * bits // 8 + 4 * N

        def make():
            q2, s2 = q.clone(), sc.clone()
            y = torch.empty(N, device=dev)
            return lambda: qmm.qmm_gemv_rowwise_q8_0(q2, s2, bits, N, K, xq, xd, y)
    else:
        q, sc = qmm.quantize_q4_0(w)
        x = workloads.activations(1, K, seed=0, device=dev)[0].contiguous()
        wb = workloads.q4_0_bytes(N, K)

        def make():
            q2, s2 = q.clone(), sc.clone()
            y = torch.empty(N, device=dev)
            return lambda: qmm.qmm_gemv_q4_0_f32_fma(q2, s2, N, K, x, y)
    del w
    us = _rotated_us(torch, make, wb)
    del q, sc
    torch.cuda.empty_cache()
    return us, wb


# ---------------------------------------------------------------------------- CPU oracle baseline
def oracle_decode_sample(torch, rows=256):
    """Oracle inputs for a row sample of every matrix of the decode step: the
    first `rows` rows of each (weights drawn with the same recipe on the CPU
    and quantized by the oracle) and the Q8_0 activation of each width."""
    from oracle import oracle as O
    mats = workloads.tinyllama_matrices()
    sigma = workloads.TINYLLAMA["sigma"]
    xs, out = {}, []
    for i, (_, N, K) in enumerate(mats):
        g = torch.Generator().manual_seed(i)
        w = (torch.randn(min(rows, N), K, generator=g) * sigma).numpy()
        if K not in xs:
            xs[K] = O.quantize_q8_0(workloads.activations(1, K, seed=0).numpy())
        out.append(O.quantize_q4_0(w) + xs[K])
    return out, f"first {rows} rows of each of the {len(mats)} decode matrices"


def oracle_pass(prep, threads):
    """One pass of the oracle's integer path over the sample; returns weight
    bytes.  With several threads the matrices run concurrently, one thread
    each (the oracle's C code runs outside the interpreter lock); splitting a
    256-row sample matrix over many threads would time thread start-up."""
    from oracle import oracle as O
    if threads <= 1:
        for qw, dw, qx, dx in prep:
            O.matmul_int(qw, dw, qx, dx, nthreads=1)
    else:
        with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda p: O.matmul_int(*p, nthreads=1), prep))
    return sum(workloads.q4_0_bytes(*p[0].shape) for p in prep)


def cpu_oracle_sample(torch, target_s=12.0, threads=None):
    """Time the oracle on the row sample, repeated for about `target_s`
    seconds of CPU work.  Returns (weight GB/s, seconds, threads, description)."""
    threads = threads or os.cpu_count() or 1
    prep, desc = oracle_decode_sample(torch)
    t0 = time.perf_counter()
    nbytes, passes = 0, 0
    while True:
        nbytes += oracle_pass(prep, threads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= target_s:
            break
    return nbytes / dt / 1e9, dt, threads, f"{desc}, {passes} passes"


def cpu_dequant_config0(torch, repeats=3):
    """The oracle's float64 dequantize-then-multiply path on the single
    2048 x 2048 GEMV (weight GB/s, seconds per product)."""
    from oracle import oracle as O
    c = workloads.SINGLE_GEMV
    qw, dw = O.quantize_q4_0(workloads.weights(c["N"], c["K"], sigma=c["sigma"], seed=0, index=0).numpy())
    qx, dx = O.quantize_q8_0(workloads.activations(1, c["K"], seed=0).numpy())
    t0 = time.perf_counter()
    for _ in range(repeats):
        O.matmul_dequant(qw, dw, qx, dx)
    dt = (time.perf_counter() - t0) / repeats
    return workloads.q4_0_bytes(c["N"], c["K"]) / dt / 1e9, dt


# ---------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="qmm", choices=["qmm", "reference"])
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=256, help="rows per matrix per reference-arm step")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU work of the cpu_baseline sample")
    ap.add_argument("--configs", action="store_true",
                    help="time every workload of the five configurations instead (one JSON line each)")
    ap.add_argument("--case", default=None,
                    help="time one kernel instead: decode_gateup, decode_qkv_norm, decode_pdl, lm_head_8192, "
                         "gemm_b16, gemm_b16_ws, gemm_b16_dense, "
                         "gemm_b64, moe_T16, moe_layer_T1, moe_layer_T16, moe_store")
    ap.add_argument("--gemm-kernel", default="auto", choices=["auto", "mma", "tmem", "stream"],
                    help="small-batch GEMM kernel (qmm_debug_gemm_kernel): automatic choice, warp MMA, tcgen05 or "
                         "dp4a streaming")
    args = ap.parse_args()
    ws, rank, local = _dist()

    import torch

    if args.configs:
        torch.cuda.set_device(local)
        from block_quantized_int4_gb300 import _build
        _build.build()
        from block_quantized_int4_gb300 import qmm
        run_configs(qmm, torch)
        return
    if args.case:
        torch.cuda.set_device(local)
        from block_quantized_int4_gb300 import _build
        _build.build()
        from block_quantized_int4_gb300 import qmm
        qmm.qmm_debug_gemm_kernel({"auto": 0, "mma": 1, "tmem": 2, "stream": 3}[args.gemm_kernel])
        print(json.dumps(run_case(qmm, torch, args.case, max(args.steps, 1))), flush=True)
        return

    if args.impl == "reference":
        return main_reference(args, torch, ws, rank)

    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from block_quantized_int4_gb300 import _build
    if rank == 0 or ws == 1:
        _build.build()
    if ws > 1:
        torch.distributed.barrier()
    from block_quantized_int4_gb300 import qmm

    dec = TinyLlamaDecode(qmm, torch)
    g = _graph(torch, dec.step)

    # e2e through the C ABI with host buffers: pinned x in, logits out, every step
    x_host = dec.x_in.cpu().pin_memory()
    logits_host = torch.empty(dec.V, dtype=torch.float32).pin_memory()

    def e2e_step():
        dec.x_in.copy_(x_host, non_blocking=True)
        g.replay()
        logits_host.copy_(dec.logits, non_blocking=True)

    # the same with the step's launches issued every step through the C ABI,
    # no graph: one qmm_gemv_fused_ops call (the library's own loop over the
    # 89 ops; host-side checks and launch cost included)
    def e2e_eager_step():
        dec.x_in.copy_(x_host, non_blocking=True)
        dec.step_chain()
        logits_host.copy_(dec.logits, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        t = _time_graph(torch, g, args.steps, 0)
        # e2e leg
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(args.steps):
            e2e_step()
        e1.record(st)
        torch.cuda.synchronize()
        t_e2e = e0.elapsed_time(e1) / 1e3
        # eager e2e leg
        for _ in range(3):
            e2e_eager_step()
        torch.cuda.synchronize()
        e0.record(st)
        for _ in range(args.steps):
            e2e_eager_step()
        e1.record(st)
        torch.cuda.synchronize()
        t_eager = e0.elapsed_time(e1) / 1e3
    if ws > 1:
        t, t_e2e, t_eager = max_over_ranks(torch, [t, t_e2e, t_eager], "cuda")

    per = t / args.steps
    value = whole_job_gbs(ws, dec.weight_bytes, args.steps, t)
    e2e_value = whole_job_gbs(ws, dec.weight_bytes, args.steps, t_e2e)
    eager_value = whole_job_gbs(ws, dec.weight_bytes, args.steps, t_eager)
    peak, peak_kind = _peaks()
    achieved = dec.algo_bytes / per / 1e9
    extras = {}
    if not args.no_extras and rank == 0:
        c0 = workloads.SINGLE_GEMV
        extras["gemv_config0"] = bench_gemv_set(qmm, torch, c0["name"], [("W", c0["N"], c0["K"])], c0["sigma"])
        extras["gemv_large_dense_batch1"] = bench_gemv_set(
            qmm, torch, workloads.LARGE_DENSE["name"] + ", batch 1", workloads.large_dense_matrices(),
            workloads.LARGE_DENSE["sigma"])
        extras["gemm_batch16"] = bench_gemm_b16(qmm, torch)
        extras["gemm_batch2"] = bench_gemm_b16(qmm, torch, M=2)
        extras["moe_T16"] = bench_moe(qmm, torch, T=16)
        extras["moe_T1"] = bench_moe(qmm, torch, T=1)
    cpu = None
    if rank == 0 and ws >= 1:
        gbs, dt, thr, desc = cpu_oracle_sample(torch, target_s=args.cpu_seconds)
        gbs1, dt1, _, desc1 = cpu_oracle_sample(torch, target_s=max(0.5, args.cpu_seconds / 4), threads=1)
        dq_gbs, dq_s = cpu_dequant_config0(torch)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": thr, "kind": "oracle",
               "sample": desc + f" ({dt:.1f} s of CPU work)",
               "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                                 "sample": desc1 + f" ({dt1:.1f} s)"},
               "dequantize_path_config0": {"value": round(dq_gbs, 4), "unit": "GB/s", "cores": 1,
                                           "seconds_per_product": round(dq_s, 4),
                                           "sample": "float64 dequantize-then-multiply, 2048 x 2048 GEMV"}}
    if rank == 0:
        line = {
            "metric": "batch-1 Q4_0xQ8_0 GEMV weight GB/s (TinyLLaMA-1.1B-shaped decode step)",
            "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int4xint8->fp32", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) activations with 1% x20 outliers)",
            "config": {"workload": workloads.TINYLLAMA["name"], "layers": dec.L, "hidden": dec.H, "ffn": dec.F,
                       "qkv": dec.Q, "vocab": dec.V, "batch": 1, "weight_bytes_per_step": dec.weight_bytes,
                       "launches_per_step": dec.launches_per_step, "parallelism": f"replicas x{ws}",
                       "l2": "inputs larger than L2 (582 MB of weights per step, each read once)",
                       "pct_of_hbm_peak": round(100 * value / ws / peak, 1)},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": _profiled_traffic(),
                         "kernel": "stream_rows_kernel<1,*,*,*> (all 89 launches of the step)",
                         "algorithmic_bytes_per_launch": round(dec.algo_bytes / dec.launches_per_step),
                         "avg_launch_us": round(per / dec.launches_per_step * 1e6, 3),
                         "peak_kind": peak_kind, "frac_of": peak_kind + " HBM copy bandwidth"},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": dec.H * 4,
                    "d2h_bytes_per_step": dec.V * 4},
            "e2e_eager": {"value": round(eager_value, 1), "unit": "GB/s", "ms_per_step": round(t_eager / args.steps * 1e3, 4),
                          "h2d_bytes_per_step": dec.H * 4, "d2h_bytes_per_step": dec.V * 4,
                          "how": "one qmm_gemv_fused_ops call per step (89 launches from the library's loop), no graph"},
            "gpu_launches": dec.launches_per_step * args.steps,
            "clocks": clk.summary(),
            "also": extras,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main_reference(args, torch, ws, rank):
    """The oracle on the host cores, same metric and config, bounded sample per step."""
    if ws > 1 and rank != 0:
        return
    from oracle import oracle as O
    O.build()
    threads = os.cpu_count() or 1
    prep, desc = oracle_decode_sample(torch, rows=args.cpu_rows)
    desc += " per step"
    for _ in range(args.warmup):
        oracle_pass(prep, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        nbytes = oracle_pass(prep, threads)
    dt = time.perf_counter() - t0
    value = nbytes * args.steps / dt / 1e9
    line = {"impl": "reference", "metric": "batch-1 Q4_0xQ8_0 GEMV weight GB/s (TinyLLaMA-1.1B-shaped decode step)",
            "value": round(value, 4), "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int4xint8->f64", "data": "synthetic",
            "config": {"workload": workloads.TINYLLAMA["name"], "batch": 1, "sample": desc},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
