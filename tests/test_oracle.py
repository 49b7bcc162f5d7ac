"""Pins for the CPU oracle, checked against things other than the oracle itself:
worked blocks from the pages' definitions (tests/golden), library routines
(torch and numpy IEEE fp16 conversion, numpy float64 matmul), closed forms
(integer-grid inputs), invariants of the quantizers and brute force on tiny
inputs.  No GPU."""
import os

import numpy as np
import pytest

from oracle import oracle as O
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.split()
    return out


# ----------------------------------------------------------------- fp16
def test_f16_decode_exhaustive_vs_numpy():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_encode_exhaustive_vs_torch():
    """All 2^32 fp32 bit patterns against torch's CPU round-to-nearest-even .half()."""
    import torch
    chunk = 1 << 24
    base = np.arange(chunk, dtype=np.uint32)
    for start in range(0, 1 << 32, chunk):
        bits = base + np.uint32(start)
        f = bits.view(np.float32)
        ours = O.f32_to_f16_bits(f)
        ref = torch.from_numpy(f).half().view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(f)
        if nan.any():
            # NaN in -> NaN out (payload not specified)
            assert np.all((ours[nan] & 0x7C00) == 0x7C00) and np.all((ours[nan] & 0x3FF) != 0)
            ok = (ours == ref) | nan
        else:
            ok = ours == ref
        if not ok.all():
            i = int(np.nonzero(~ok)[0][0])
            raise AssertionError(f"fp32 bits {bits[i]:#x}: ours {ours[i]:#x}, torch {ref[i]:#x}")


def test_f16_encode_rounding_boundaries_vs_torch():
    """Every exponent x mantissa-top x the rounding-critical low bits, against torch CPU .half()."""
    import torch
    hi = np.arange(1 << 19, dtype=np.uint32) << 13  # sign, exponent, top 10 mantissa bits
    lows = np.array([0, 1, 0x0FFF, 0x1000, 0x1001, 0x1FFF], dtype=np.uint32)
    bits = (hi[:, None] | lows[None, :]).reshape(-1)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]  # no inf/NaN
    f = bits.view(np.float32)
    ours = O.f32_to_f16_bits(f)
    ref = torch.from_numpy(f.copy()).half().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ----------------------------------------------------------------- quantizers
def test_q8_0_worked_block():
    g = _golden("q8_0_ramp_block.txt")
    x = np.array([float(v) for v in g["x"]], np.float32)
    q, d = O.quantize_q8_0(x[None])
    assert d[0, 0] == int(g["d16"][0], 16)
    assert q[0].tolist() == [int(v) for v in g["q"]]


def test_q4_0_worked_block():
    g = _golden("q4_0_small_block.txt")
    w = np.array([float(v) for v in g["w"]], np.float32)
    q, d = O.quantize_q4_0(w[None])
    assert d[0, 0] == int(g["d16"][0], 16)
    assert q[0].tolist() == [int(v) for v in g["q"]]


def test_q4_0_block_format_sizes():
    g = _golden("q4_0_block_format.txt")
    assert int(g["values_per_block"][0]) == O.QK
    rng = np.random.default_rng(1)
    q = rng.integers(-8, 8, size=(3, 64)).astype(np.int8)
    d = rng.integers(0, 0x7C00, size=(3, 2)).astype(np.uint16)
    blocks = O.pack_q4_0_blocks(q, d)
    assert blocks.shape[-1] == int(g["block_bytes"][0]) == int(g["scale_bytes"][0]) + int(g["nibble_bytes"][0])
    # scale is the first 2 bytes, little endian
    assert np.array_equal(blocks[..., 0].astype(np.uint16) | (blocks[..., 1].astype(np.uint16) << 8), d)
    # 32 four-bit values in 16 bytes: element j low nibble, j+16 high nibble, offset 8
    assert np.array_equal((blocks[0, 0, 2:] & 0xF).astype(np.int8) - 8, q[0, :16])
    assert np.array_equal((blocks[0, 0, 2:] >> 4).astype(np.int8) - 8, q[0, 16:32])
    q2, d2 = O.unpack_q4_0_blocks(blocks, 3, 64)
    assert np.array_equal(q2, q) and np.array_equal(d2, d)
    total = sum(workloads.q4_0_bytes(N, K) for _, N, K in workloads.tinyllama_matrices())
    assert total == 581_861_376
    assert abs(total / 1e6 - float(g["tinyllama_4bit_mb_approx"][0])) / 600 < 0.05


def _numpy_quantize(v, qmax, qmin):
    """Independent restatement with numpy fp32 ops (division, |.|, floor)."""
    v = v.astype(np.float32).reshape(-1, 32)
    amax = np.abs(v).max(axis=1)
    d32 = (amax / np.float32(qmax)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (v / d32[:, None]).astype(np.float32)
    a = np.floor(np.abs(r).astype(np.float64) + 0.5) * np.sign(r)
    a = np.where(amax[:, None] == 0, 0, a)
    q = np.clip(a, qmin, qmax).astype(np.int8)
    return q, d32


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_q8_0_matches_numpy_restatement(seed):
    x = workloads.activations(4, 2048, seed=seed).numpy()
    q, d = O.quantize_q8_0(x)
    qn, d32 = _numpy_quantize(x, 127, -127)
    assert np.array_equal(q.reshape(-1, 32), qn)
    assert np.array_equal(d.reshape(-1), d32.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("seed", [0, 1])
def test_q4_0_matches_numpy_restatement(seed):
    w = workloads.weights(64, 2048, seed=seed).numpy()
    q, d = O.quantize_q4_0(w)
    qn, d32 = _numpy_quantize(w, 7, -8)
    assert np.array_equal(q.reshape(-1, 32), qn)
    assert np.array_equal(d.reshape(-1), d32.astype(np.float16).view(np.uint16))


def _adversarial_blocks(rng, n):
    """Random blocks plus zero blocks, amax at every lane, exact .5 ties."""
    x = rng.standard_normal((n, 32)).astype(np.float32)
    x[0] = 0
    for lane in range(32):
        x[1 + lane] = rng.uniform(-1, 1, 32).astype(np.float32)
        x[1 + lane, lane] = 4.0 * (-1) ** lane
    # ties: amax 127 -> d32 = 1, values k + 0.5 are exact ties
    x[40] = (np.arange(32) - 16 + 0.5).astype(np.float32)
    x[40, 0] = 127
    x[41] = -x[40]
    return x


def test_q8_0_invariants():
    rng = np.random.default_rng(7)
    x = _adversarial_blocks(rng, 256)
    q, d = O.quantize_q8_0(x.reshape(1, -1))
    q = q.reshape(-1, 32)
    d = d.reshape(-1)
    # zero block
    assert d[0] == 0 and not q[0].any()
    # every nonzero block reaches |q| = 127
    nz = np.abs(x).max(axis=1) > 0
    assert np.all(np.abs(q[nz]).max(axis=1) == 127)
    assert q.min() >= -127 and q.max() <= 127
    # ties round half away from zero (x = k + 0.5 with d32 = 1)
    assert q[40, 1:].tolist() == [int(np.sign(v) * np.floor(abs(v) + 0.5)) for v in x[40, 1:]]
    # sign symmetry
    qn, dn = O.quantize_q8_0(-x.reshape(1, -1))
    assert np.array_equal(qn.reshape(-1, 32), -q) and np.array_equal(dn.reshape(-1), d)
    # power-of-two scaling leaves q unchanged and scales d exactly
    q2, d2 = O.quantize_q8_0((x * np.float32(4)).reshape(1, -1))
    assert np.array_equal(q2.reshape(-1, 32), q)
    f = O.f16_bits_to_f32(d)
    f2 = O.f16_bits_to_f32(d2.reshape(-1))
    assert np.array_equal(f2, f * 4)
    # round-trip bound |x - d32*q| <= d32/2 (+ 1 ulp of the product)
    amax = np.abs(x).max(axis=1)
    d32 = (amax / np.float32(127)).astype(np.float32)
    err = np.abs(x.astype(np.float64) - d32[:, None].astype(np.float64) * q)
    bound = d32[:, None].astype(np.float64) / 2 * (1 + 1e-6) + np.spacing(np.abs(x)).astype(np.float64)
    assert np.all(err <= bound)


def test_q4_0_invariants():
    rng = np.random.default_rng(8)
    w = _adversarial_blocks(rng, 256) * np.float32(0.01)
    q, d = O.quantize_q4_0(w.reshape(1, -1))
    q = q.reshape(-1, 32)
    nz = np.abs(w).max(axis=1) > 0
    assert np.all(np.abs(q[nz]).max(axis=1) == 7)
    assert q.min() >= -7 and q.max() <= 7  # Delta = amax/7 never reaches -8
    assert not q[0].any() and d.reshape(-1)[0] == 0
    qn, dn = O.quantize_q4_0(-w.reshape(1, -1))
    assert np.array_equal(qn.reshape(-1, 32), -q) and np.array_equal(dn, d)


# ----------------------------------------------------------------- products
def _rand_q(rng, N, M, K):
    qw = rng.integers(-8, 8, size=(N, K)).astype(np.int8)  # all 16 nibble values incl. -8
    qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    dw = rng.integers(0x1000, 0x2C00, size=(N, K // 32)).astype(np.uint16)
    dx = rng.integers(0x1000, 0x3C00, size=(M, K // 32)).astype(np.uint16)
    return qw, dw, qx, dx


def test_single_product_table_exhaustive():
    """All 16 weight values x all 255 activation values through the block dot."""
    qw = np.repeat(np.arange(-8, 8, dtype=np.int8)[:, None], 32, axis=1)
    qx = np.repeat(np.arange(-127, 128, dtype=np.int8)[:, None], 32, axis=1)
    dots = O.block_dots(qw, qx)[:, :, 0]
    assert np.array_equal(dots, 32 * np.outer(np.arange(-127, 128), np.arange(-8, 8)))


def test_integer_grid_closed_form():
    """With d = 1 on both sides, y is exactly the integer product W x."""
    rng = np.random.default_rng(3)
    N, M, K = 37, 5, 256
    w = rng.integers(-7, 8, size=(N, K)).astype(np.float32)
    w[:, ::32] = 7  # every block holds a 7 -> Delta = 1
    x = rng.integers(-127, 128, size=(M, K)).astype(np.float32)
    x[:, 5::32] = -127  # every block holds a -127 -> d = 1
    qw, dw = O.quantize_q4_0(w)
    qx, dx = O.quantize_q8_0(x)
    assert np.all(dw == 0x3C00) and np.all(dx == 0x3C00)
    y, _ = O.matmul_int(qw, dw, qx, dx)
    exact = x.astype(np.int64) @ w.astype(np.int64).T
    assert np.array_equal(y, exact.astype(np.float64))
    yd = O.matmul_dequant(qw, dw, qx, dx)
    assert np.array_equal(yd, exact.astype(np.float64))


@pytest.mark.parametrize("N,M,K", [(1, 1, 32), (8, 3, 64), (5, 2, 96), (3, 4, 160)])
def test_brute_force_dequantized_matmul(N, M, K):
    rng = np.random.default_rng(N * 100 + K)
    qw, dw, qx, dx = _rand_q(rng, N, M, K)
    W = np.repeat(dw.view(np.float16).astype(np.float64), 32, axis=1) * qw
    X = np.repeat(dx.view(np.float16).astype(np.float64), 32, axis=1) * qx
    ref = X @ W.T
    y, S = O.matmul_int(qw, dw, qx, dx)
    yd = O.matmul_dequant(qw, dw, qx, dx)
    scale = np.abs(X) @ np.abs(W).T + 1e-300
    assert np.all(np.abs(y - ref) <= 1e-13 * scale)
    assert np.all(np.abs(yd - ref) <= 1e-13 * scale)
    # S bounds |y| and is what the fp32 tolerance is built on
    assert np.all(np.abs(y) <= S * (1 + 1e-15))
    dots = O.block_dots(qw, qx)
    manual = np.einsum("nbi,mbi->mnb", qw.reshape(N, -1, 32).astype(np.int64),
                       qx.reshape(M, -1, 32).astype(np.int64))
    assert np.array_equal(dots, manual)


def test_int_and_dequant_paths_agree_realistic():
    w = workloads.weights(96, 2048, seed=0).numpy()
    x = workloads.activations(2, 2048, seed=0).numpy()
    qw, dw = O.quantize_q4_0(w)
    qx, dx = O.quantize_q8_0(x)
    y, S = O.matmul_int(qw, dw, qx, dx)
    yd = O.matmul_dequant(qw, dw, qx, dx)
    assert np.all(np.abs(y - yd) <= 1e-12 * S + 1e-300)
    # and the quantized product approximates the fp32 product
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    rel = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert rel < 0.1


def test_row_subset_and_threads():
    rng = np.random.default_rng(11)
    qw, dw, qx, dx = _rand_q(rng, 50, 3, 128)
    y, S = O.matmul_int(qw, dw, qx, dx)
    rows = np.array([49, 0, 7, 7, 31])
    ys, Ss = O.matmul_int(qw, dw, qx, dx, rows=rows, nthreads=3)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(Ss, S[:, rows])
    y4, _ = O.matmul_int(qw, dw, qx, dx, nthreads=4)
    assert np.array_equal(y4, y)


# ----------------------------------------------------------------- MoE pieces
def test_router_topk_order_ties_and_normalisation():
    logits = np.array([[0.0, 2.0, 2.0, -1.0, 5.0, 2.0]], np.float32)
    ids, g = O.router_topk(logits, 3)
    assert ids[0].tolist() == [4, 1, 2]  # ties -> lower index first
    s = 1 / (1 + np.exp(-logits[0, [4, 1, 2]].astype(np.float64)))
    assert np.allclose(g[0], s / s.sum(), rtol=1e-15)
    assert abs(g.sum() - 1) < 1e-15
    L = workloads.router_logits(16, 256).numpy()
    ids, g = O.router_topk(L, 8)
    for t in range(16):
        assert len(set(ids[t].tolist())) == 8
        assert ids[t].tolist() == np.argsort(-L[t], kind="stable")[:8].tolist()  # sigmoid is monotone


def test_router_topk_against_stable_argsort_and_expit():
    """The router's selection is the top-k of sigmoid scores; sigmoid is
    strictly increasing (and injective in double over fp32 logits in
    [-87, 16]), so it must equal numpy's stable argsort of -logits (ties to
    the lower index).  Gates: scipy's expit of the chosen logits, normalised
    over the k."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(21)
    cases = [
        rng.standard_normal((64, 256)).astype(np.float32),           # the GLM-scale router
        rng.integers(-3, 4, (64, 40)).astype(np.float32),             # heavy ties, E not a multiple of 32
        rng.uniform(-87, 16, (8, 1024)).astype(np.float32),           # the domain's ends
        np.zeros((3, 17), np.float32),                                # all equal
    ]
    for L in cases:
        T, E = L.shape
        for k in sorted({1, 2, 8, min(E, 32), E}):
            if k > E:
                continue
            ids, g = O.router_topk(L, k)
            want = np.argsort(-L.astype(np.float64), axis=1, kind="stable")[:, :k]
            assert np.array_equal(ids, want), (L.shape, k)
            s = special.expit(np.take_along_axis(L, want, 1).astype(np.float64))
            assert np.allclose(g, s / s.sum(1, keepdims=True), rtol=1e-14, atol=0)
            assert np.allclose(g.sum(1), 1.0, rtol=1e-14)
    # all-equal logits: the k lowest indices, each gate exactly 1/k
    ids, g = O.router_topk(np.full((2, 10), 0.25, np.float32), 4)
    assert ids.tolist() == [[0, 1, 2, 3]] * 2 and (g == 0.25).all()
    # two candidates: gates sigma(a)/(sigma(a)+sigma(b)), larger logit first
    ids, g = O.router_topk(np.array([[-1.0, 3.0]], np.float32), 2)
    sa, sb = 1 / (1 + np.exp(1.0)), 1 / (1 + np.exp(-3.0))
    assert ids.tolist() == [[1, 0]] and np.allclose(g[0], [sb / (sa + sb), sa / (sa + sb)], rtol=1e-15)


def test_swiglu_identities():
    a = np.array([0.0, 1.0, -1.0, 30.0, -30.0, 0.5], np.float64)
    b = np.ones_like(a)
    h = O.swiglu(a, b)
    assert h[0] == 0.0
    # silu(a) - silu(-a) = a
    assert abs((float(h[1]) - float(h[2])) - 1.0) < 1e-7
    assert abs(float(h[3]) - 30.0) < 1e-6 and abs(float(h[4])) < 1e-10
    h2 = O.swiglu(a, 2 * b)
    assert np.array_equal(h2, (2 * h.astype(np.float64)).astype(np.float32))


def test_moe_combine_linear():
    rng = np.random.default_rng(5)
    z = rng.standard_normal((2, 3, 4))
    g = np.array([[1, 0, 0], [0.25, 0.5, 0.25]], np.float32)
    y = O.moe_combine(z, g)
    assert np.array_equal(y[0], z[0, 0])
    assert np.allclose(y[1], 0.25 * z[1, 0] + 0.5 * z[1, 1] + 0.25 * z[1, 2], rtol=0, atol=1e-15)


# ---------------------------------------------------------------- RMSNorm (TinyLLaMA guide 4.1)
def _golden_kv(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        if line.startswith("#") or not line.strip():
            continue
        k, *v = line.split()
        out[k] = [float(t) for t in v]
    return out


def test_rmsnorm_worked_example():
    g = _golden_kv("rmsnorm_small.txt")
    y = O.rmsnorm(np.array(g["x"], np.float32), np.array(g["gamma"], np.float32), eps=g["eps"][0])
    assert np.array_equal(y, np.array(g["y"], np.float32))


def test_rmsnorm_closed_forms_and_invariants():
    rng = np.random.default_rng(5)
    d = 96
    gamma = rng.normal(1.0, 0.1, d).astype(np.float32)
    # a constant vector c: every element becomes c / sqrt(c^2 + eps) * gamma_i
    for c, eps in [(3.0, 0.0), (-0.5, 1e-5), (1e-3, 1e-5)]:
        y = O.rmsnorm(np.full(d, c, np.float32), gamma, eps=eps)
        want = (np.float64(np.float32(c)) / np.sqrt(np.float64(np.float32(c)) ** 2 + eps) * gamma).astype(np.float32)
        assert np.array_equal(y, want)
    # scale invariance (eps = 0): powers of two change nothing; sign flips the output
    x = rng.standard_normal((3, d)).astype(np.float32)
    y = O.rmsnorm(x, gamma, eps=0.0)
    assert np.array_equal(O.rmsnorm(x * 8, gamma, eps=0.0), y)
    assert np.array_equal(O.rmsnorm(-x, gamma, eps=0.0), -y)
    # unit gamma: the output's mean square is 1 (up to the fp32 rounding of each element)
    y1 = O.rmsnorm(x, np.ones(d, np.float32), eps=0.0).astype(np.float64)
    assert np.allclose((y1 ** 2).mean(axis=1), 1.0, rtol=1e-6)
    # eps > 0 shrinks the output towards zero
    assert (np.abs(O.rmsnorm(x, gamma, eps=1.0)) <= np.abs(y)).all()


# ----------------------------------------------------------------- per-row int4 / int2 containers
def test_rowwise_worked_example():
    g = _golden_kv("rowwise_small.txt")
    w = np.tile(np.array(g["w"], np.float32), 4)[None]
    for bits in (4, 2):
        q, s = O.quantize_rowwise(w, bits)
        assert s[0] == np.float32(g[f"s{bits}"][0])
        assert q[0].tolist() == [int(v) for v in g[f"q{bits}"]] * 4
        packed = O.pack_rowwise(q, bits)
        per_pattern = len(g[f"p{bits}"])
        assert packed[0].tolist() == [int(v) for v in g[f"p{bits}"]] * (packed.shape[1] // per_pattern)
        assert np.array_equal(O.unpack_rowwise(packed, 32, bits), q)


def test_rowwise_quantizer_invariants():
    rng = np.random.default_rng(31)
    w = (rng.standard_normal((40, 96)) * 0.02).astype(np.float32)
    w[3] = 0.0  # a zero row
    w[5, 7] = 1.0  # an outlier
    for bits in (4, 2):
        qmax, qmin = 2 ** (bits - 1) - 1, -(2 ** (bits - 1))
        q, s = O.quantize_rowwise(w, bits)
        assert q.min() >= qmin and q.max() <= qmax
        assert s[3] == 0 and (q[3] == 0).all()
        nz = np.abs(w).max(1) > 0
        # the scale is amax / qmax in fp32, and the row's largest value reaches +-qmax
        assert np.array_equal(s, (np.abs(w).max(1) / np.float32(qmax)).astype(np.float32))
        assert (np.abs(q[nz]).max(1) == qmax).all()
        # round trip: |w - s q| <= s/2 (up to the fp32 rounding of w/s)
        err = np.abs(w.astype(np.float64) - s[:, None].astype(np.float64) * q)
        assert (err <= s[:, None] * (0.5 + 1e-6)).all()
        # sign symmetry and power-of-two scaling
        qn, sn = O.quantize_rowwise(-w, bits)
        assert np.array_equal(qn, -q) and np.array_equal(sn, s)
        q2, s2 = O.quantize_rowwise(w * 4, bits)
        assert np.array_equal(q2, q) and np.array_equal(s2, s * 4)
    # int2 codes are ternary: -2 is never produced (amax/1 maps the extreme to +-1)
    q, _ = O.quantize_rowwise(w, 2)
    assert set(np.unique(q)) <= {-1, 0, 1}


def test_rowwise_packing_against_bit_loops():
    rng = np.random.default_rng(32)
    for bits in (4, 2):
        per, off = 8 // bits, 2 ** (bits - 1)
        q = rng.integers(-off, off, (3, 64)).astype(np.int8)  # every code, including -2^(bits-1)
        packed = O.pack_rowwise(q, bits)
        for n in range(3):
            for j in range(64 // per):
                byte = 0
                for i in range(per):
                    byte += (int(q[n, j * per + i]) + off) * (2 ** (bits * i))
                assert packed[n, j] == byte
        assert np.array_equal(O.unpack_rowwise(packed, 64, bits), q)


def test_matmul_rowwise_int_brute_force_and_q4_0_equivalence():
    rng = np.random.default_rng(33)
    N, K, M = 7, 96, 3
    for bits in (4, 2):
        off = 2 ** (bits - 1)
        qw = rng.integers(-off, off, (N, K)).astype(np.int8)
        s = rng.uniform(0.001, 0.1, N).astype(np.float32)
        qx = rng.integers(-127, 128, (M, K)).astype(np.int8)
        dx = O.f32_to_f16_bits(rng.uniform(0.001, 0.1, (M, K // 32)).astype(np.float32))
        y, S = O.matmul_rowwise_int(qw, s, qx, dx)
        dxf = np.float16(0) + dx.view(np.float16).astype(np.float64)
        for m in range(M):
            for n in range(N):
                want, mag = 0.0, 0.0
                for b in range(K // 32):
                    dot = sum(int(qw[n, 32 * b + i]) * int(qx[m, 32 * b + i]) for i in range(32))
                    want += float(s[n]) * dxf[m, b] * dot
                    mag += abs(float(s[n]) * dxf[m, b] * dot)
                assert abs(y[m, n] - want) <= 1e-12 * mag and abs(S[m, n] - mag) <= 1e-12 * mag
    # with every row scale an fp16 value, the per-row product equals the Q4_0
    # product whose block scales all carry that value (same codes)
    qw = rng.integers(-8, 8, (N, K)).astype(np.int8)
    s = (2.0 ** rng.integers(-8, -2, N)).astype(np.float32)
    dw = np.repeat(O.f32_to_f16_bits(s)[:, None], K // 32, 1)
    y1, S1 = O.matmul_rowwise_int(qw, s, qx, dx)
    y2, S2 = O.matmul_int(qw, dw, qx, dx)
    assert np.array_equal(y1, y2) and np.array_equal(S1, S2)


def test_matmul_q4_0_f32_against_numpy_and_brute_force():
    rng = np.random.default_rng(34)
    N, K, M = 9, 128, 2
    qw = rng.integers(-8, 8, (N, K)).astype(np.int8)
    dw = O.f32_to_f16_bits(rng.uniform(0.001, 0.05, (N, K // 32)).astype(np.float32))
    x = rng.standard_normal((M, K)).astype(np.float32)
    y, S = O.matmul_q4_0_f32(qw, dw, x)
    wf = np.repeat(dw.view(np.float16).astype(np.float64), 32, 1) * qw
    want = x.astype(np.float64) @ wf.T
    mag = np.abs(x.astype(np.float64)) @ np.abs(wf).T
    assert np.all(np.abs(y - want) <= 1e-13 * mag)
    assert np.allclose(S, mag, rtol=1e-13)
    # one (m, n) by a plain loop
    acc = 0.0
    for k in range(K):
        acc += float(np.float16(dw[4, k // 32].view(np.float16))) * int(qw[4, k]) * float(x[1, k])
    assert abs(y[1, 4] - acc) <= 1e-13 * mag[1, 4]
    # x = the dequantized Q8_0 of an activation: equals the Q4_0 x Q8_0 integer path
    xq, xd = O.quantize_q8_0(x)
    xdeq = (xq.astype(np.float64) * np.repeat(xd.view(np.float16).astype(np.float64), 32, 1)).astype(np.float32)
    y3, _ = O.matmul_q4_0_f32(qw, dw, xdeq)
    y4, S4 = O.matmul_int(qw, dw, xq, xd)
    assert np.all(np.abs(y3 - y4) <= 1e-13 * S4)


# ---------------------------------------------------------------- MoE layer (Colibri page, system architecture)
def test_moe_forward_integer_grid_closed_form():
    """moe_forward on an integer grid where every stage is exact, so the
    layer has a closed form computed here with plain integer arithmetic.

    Per slot j of token t (Colibri page's flow: experts compute, results are
    combined by the gates; SwiGLU of the TinyLLaMA guide 4.4, silu(gate)*up):
    - all scales are 1.0, and token t's activation codes are 127 at column
      2t and 1 at column 2t + 1 (so its Q8_0 block has d = 1);
    - gate rows hold 0 or 1 at column 2t and 0 at 2t + 1, so a = W_gate x is
      0 or 127; sigmoid(127) is 1.0 in double, so silu(a) is 0 or 127 exactly;
    - up rows hold m * s at column 2t + 1 (s in {-1, 0, 1}, m a power of two
      per expert) and 0 at column 2t, so b = W_up x = m * s;
    - h = silu(a) * b is 127 * m * s or 0; its Q8_0 block has d = m and codes
      127 * s (or 0) exactly;
    - z = W_down h_q = m * (integer dot), and y = sum_j g_j z_j with gates
      that are exact binary fractions.
    Ids repeat an expert inside token 1 (each slot is computed on its own), and
    the experts differ, so a gate/up swap (silu(b) * a is not an integer), a
    slot-to-expert index slip, or a combine over the wrong axis all change y."""
    H = F = 32
    E, T, k = 3, 2, 2
    ids = np.array([[2, 0], [1, 1]], np.int32)
    gates = np.array([[0.75, 0.25], [0.625, 0.375]], np.float32)
    m_of = {0: 1, 1: 2, 2: 4}
    one = np.uint16(0x3C00)  # fp16 1.0
    fill = lambda f, e: ((f * 7 + e * 3) % 16) - 8  # noqa: E731  (columns the activations never touch)
    gate, up, down = {}, {}, {}
    for e in range(E):
        g = np.zeros((F, H), np.int8)
        u = np.zeros((F, H), np.int8)
        for f in range(F):
            g[f, 4:] = fill(f, e)
            u[f, 4:] = fill(f + 1, e)
            g[f, 0] = 1 if (f + e) % 3 else 0          # token 0's gate column
            g[f, 2] = 1 if (f + 2 * e) % 4 else 0      # token 1's gate column
            u[f, 1] = m_of[e] * (((f * 5 + e) % 3) - 1)   # token 0's up column
            u[f, 3] = m_of[e] * (((f * 3 + 2 * e) % 3) - 1)  # token 1's up column
        dn = np.array([[((n * 3 + f * 5 + e * 7) % 16) - 8 for f in range(F)] for n in range(H)], np.int8)
        gate[e] = (g, np.full((F, 1), one))
        up[e] = (u, np.full((F, 1), one))
        down[e] = (dn, np.full((H, 1), one))
    qx = np.zeros((T, H), np.int8)
    qx[0, 0], qx[0, 1], qx[1, 2], qx[1, 3] = 127, 1, 127, 1
    dx = np.full((T, 1), one)

    y, z, h = O.moe_forward(gate, up, down, ids, gates, qx, dx)

    # the closed form, in integers
    z_ref = np.zeros((T, k, H), np.int64)
    for t in range(T):
        for j in range(k):
            e, m = int(ids[t, j]), m_of[int(ids[t, j])]
            a = gate[e][0].astype(np.int64) @ qx[t].astype(np.int64)
            b = up[e][0].astype(np.int64) @ qx[t].astype(np.int64)
            assert set(np.unique(a)) <= {0, 127} and (a == 127).any()
            assert set(np.unique(b)) <= {-m, 0, m}
            h_int = np.where(a == 127, 127 * b, 0)
            assert np.abs(h_int).max() == 127 * m  # so the block scale is m and the codes h / m
            assert np.array_equal(h[t, j], h_int.astype(np.float32))
            z_ref[t, j] = m * (down[e][0].astype(np.int64) @ (h_int // m))
    assert np.array_equal(z, z_ref.astype(np.float64))
    y_ref = (gates[:, :, None].astype(np.float64) * z_ref).sum(axis=1)
    assert np.array_equal(y, y_ref)
    # two values worked out by hand as spot checks of the integer closed form
    assert z_ref[0, 0, 0] == 4 * 127 * int(
        sum(down[2][0][0, f] * np.sign(up[2][0][f, 1]) for f in range(F) if gate[2][0][f, 0]))
    assert y[1, 5] == 0.625 * z_ref[1, 0, 5] + 0.375 * z_ref[1, 1, 5]
