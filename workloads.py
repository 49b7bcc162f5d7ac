"""Seeded synthetic inputs and workload shapes.

This module is shared by the tests, the bench and the smoke check.  It holds
none of the quantization arithmetic: it only draws fp32 weights,
activations and router logits, and lists the matrix shapes of the workloads.

Recipe (one sub-seed per tensor, ``seed*1000 + index``, so results do not
depend on generation order):

* weights  W[N][K] ~ N(0, sigma), fp32 (sigma 0.02; 0.01 for the large dense
  model);
* activations x[M][K] ~ N(0, 1), fp32, with round(1% of M*K) entries, chosen
  uniformly without replacement, multiplied by 20 (outliers);
* router logits [T][E] ~ N(0, 1), fp32;
* RMSNorm weights gamma[K] = 1 + 0.1 * N(0, 1), fp32 (the decode step's
  normalizations; a trained gamma stays near 1).

Generation runs on the requested device with torch's generator for that
device (CPU: mt19937; CUDA: Philox), so one seed gives
different tensors on CPU and on GPU; a test that compares two sides always
hands both the same tensor.
"""
from __future__ import annotations

import torch

QK = 32


def _gen(seed: int, index: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000 + int(index))
    return g


def weights(N: int, K: int, sigma: float = 0.02, seed: int = 0, index: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed, index, device)
    return torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * sigma


def activations(M: int, K: int, seed: int = 0, index: int = 500, outlier_frac: float = 0.01,
                outlier_scale: float = 20.0, device="cpu") -> torch.Tensor:
    g = _gen(seed, index, device)
    x = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    n = x.numel()
    n_out = int(round(outlier_frac * n))
    if n_out:
        idx = torch.randperm(n, generator=g, device=device)[:n_out]
        x.view(-1)[idx] *= outlier_scale
    return x


def router_logits(T: int, E: int, seed: int = 0, index: int = 900, device="cpu") -> torch.Tensor:
    g = _gen(seed, index, device)
    return torch.randn(T, E, generator=g, device=device, dtype=torch.float32)


def expert_bias(E: int, scale: float = 1.5, seed: int = 0, index: int = 901, device="cpu") -> torch.Tensor:
    """A fixed per-expert offset of the router logits, scale * N(0, 1): some
    experts are routed to much more often than others, which is what gives an
    expert cache its hits (the pages give no routing statistics; this skew is
    a synthetic stand-in)."""
    g = _gen(seed, index, device)
    return scale * torch.randn(E, generator=g, device=device, dtype=torch.float32)


def norm_weights(K: int, seed: int = 0, index: int = 700, device="cpu") -> torch.Tensor:
    g = _gen(seed, index, device)
    return 1.0 + 0.1 * torch.randn(K, generator=g, device=device, dtype=torch.float32)


# --------------------------------------------------------------------------
# Workload shapes.  (N, K) = (output rows, reduction length); y = W x.
# --------------------------------------------------------------------------

SINGLE_GEMV = {"name": "single Q4_0xQ8_0 GEMV 2048x2048, batch 1", "N": 2048, "K": 2048, "sigma": 0.02}

# TinyLLaMA-1.1B-shaped decode: hidden 2048, 32 q-heads / 4 kv-heads of 64
# (fused QKV 2048 -> 2560), O 2048 -> 2048, gate/up 2048 -> 5632,
# down 5632 -> 2048, 22 layers, lm_head 2048 -> 32000.
TINYLLAMA = {
    "name": "TinyLLaMA-1.1B-shaped decode GEMVs, batch 1",
    "hidden": 2048, "ffn": 5632, "qkv": 2560, "vocab": 32000, "layers": 22, "sigma": 0.02,
}

# Batched decode / speculative verify.
BATCHED = {"name": "batched decode GEMM", "shapes": [(5632, 2048), (2048, 5632)],
           "M": [1, 2, 4, 8, 16, 32, 64], "sigma": 0.02}

# Large dense decode: hidden 8192, FFN 28672, vocab 128256.
LARGE_DENSE = {"name": "large dense decode (hidden 8192, FFN 28672, vocab 128256)",
               "hidden": 8192, "ffn": 28672, "vocab": 128256, "M": [1, 16], "sigma": 0.01}

# GLM-scale MoE layer: hidden 6144, 256 experts of gate/up 6144 -> 2048 and
# down 2048 -> 6144, sigmoid router, top-8.
MOE = {"name": "GLM-scale MoE expert layer", "hidden": 6144, "expert_ffn": 2048, "experts": 256,
       "top_k": 8, "T": [1, 16], "sigma": 0.02,
       # expert store: slots in HBM, decode steps timed, skew of the routing
       "store_slots": 64, "store_steps": 64, "store_skew": 1.5}


def tinyllama_matrices():
    """Per-step matrix sequence [(name, N, K)] of the TinyLLaMA-shaped decode."""
    c = TINYLLAMA
    h, f = c["hidden"], c["ffn"]
    seq = []
    for layer in range(c["layers"]):
        seq += [(f"L{layer}.qkv", c["qkv"], h), (f"L{layer}.o", h, h),
                (f"L{layer}.gate", f, h), (f"L{layer}.up", f, h), (f"L{layer}.down", h, f)]
    seq.append(("lm_head", c["vocab"], h))
    return seq


def large_dense_matrices():
    c = LARGE_DENSE
    h, f = c["hidden"], c["ffn"]
    return [("gate", f, h), ("up", f, h), ("down", h, f), ("lm_head", c["vocab"], h)]


def q4_0_bytes(N: int, K: int) -> int:
    """Bytes of the Q4_0 encoding of an N x K matrix (18 bytes per 32 values)."""
    return N * (K // QK) * 18
