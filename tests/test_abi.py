"""The C-ABI library: it builds, loads, exports every entry point that
include/qmm.h declares, and rejects bad arguments on the host (status codes,
nothing launched).  No GPU needed: every call here fails validation before
any CUDA call, or reports that no sm_103 device is present."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qmm():
    from block_quantized_int4_gb300 import _build
    _build.build()
    from block_quantized_int4_gb300 import qmm as m
    return m


def _header_functions():
    text = open(os.path.join(ROOT, "include", "qmm.h")).read()
    return re.findall(r"^QMM_API\s+[\w\s\*]+?\b(qmm_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_entry_points():
    names = set(_header_functions())
    for n in ["qmm_quantize_q8_0", "qmm_gemv_q4_0_q8_0", "qmm_gemm_q4_0_q8_0", "qmm_moe_gemv",
              "qmm_quantize_q4_0", "qmm_repack_q4_0", "qmm_swiglu_quantize_q8_0", "qmm_debug_block_dots",
              "qmm_last_device_error", "qmm_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(qmm):
    lib = ctypes.CDLL(qmm.LIB_PATH)
    for name in _header_functions():
        assert hasattr(lib, name), f"{name} declared in qmm.h but not exported"
    assert set(qmm.SIGNATURES) <= set(_header_functions())


def test_status_strings_and_version(qmm):
    assert qmm.abi_version() == 2
    for code, name in qmm.STATUS.items():
        assert qmm.status_string(code).startswith(name)
    assert "UNKNOWN" in qmm.status_string(99)


def _call(qmm, name, *args):
    return getattr(qmm.library_handle(), name)(*args)


def test_shape_and_argument_errors_return_status(qmm):
    A16 = 0x10000  # a fake, 16-byte aligned address: never dereferenced
    # K not a multiple of 32
    assert _call(qmm, "qmm_gemv_q4_0_q8_0", A16, A16, 64, 48, A16, A16, A16, None) == 2
    assert _call(qmm, "qmm_quantize_q8_0", A16, 1, 33, 33, A16, A16, None) == 2
    # negative sizes / null pointers
    assert _call(qmm, "qmm_gemm_q4_0_q8_0", A16, A16, -1, 64, 1, A16, A16, A16, 64, None) == 1
    assert _call(qmm, "qmm_gemm_q4_0_q8_0", None, A16, 64, 64, 1, A16, A16, A16, 64, None) == 1
    assert _call(qmm, "qmm_quantize_q8_0", None, 1, 64, 64, A16, A16, None) == 1
    # ldy < N
    assert _call(qmm, "qmm_gemm_q4_0_q8_0", A16, A16, 64, 64, 2, A16, A16, A16, 32, None) == 1
    # empty products are shape errors, empty quantizations are no-ops
    assert _call(qmm, "qmm_gemm_q4_0_q8_0", A16, A16, 64, 64, 0, A16, A16, A16, 64, None) == 2
    assert _call(qmm, "qmm_quantize_q8_0", A16, 0, 64, 64, A16, A16, None) == 0
    assert _call(qmm, "qmm_moe_gemv", A16, A16, 4, 64, 64, A16, 0, 2, A16, A16, 0, A16, A16, 1 << 20, None) == 0


def test_alignment_errors(qmm):
    A16, ODD = 0x10000, 0x10001
    assert _call(qmm, "qmm_gemv_q4_0_q8_0", A16 + 8, A16, 64, 64, A16, A16, A16, None) == 3  # qs not 16-B
    assert _call(qmm, "qmm_gemv_q4_0_q8_0", A16, ODD, 64, 64, A16, A16, A16, None) == 3  # d not 2-B
    assert _call(qmm, "qmm_gemv_q4_0_q8_0", A16, A16, 64, 64, A16 + 4, A16, A16, None) == 3  # xq not 16-B
    assert _call(qmm, "qmm_quantize_q8_0", A16 + 4, 1, 64, 64, A16, A16, None) == 3
    assert _call(qmm, "qmm_quantize_q8_0", A16, 2, 64, 66, A16, A16, None) == 3  # ldx % 4


def test_workspace_rules(qmm):
    n = qmm.qmm_moe_workspace_size(256, 16, 8)
    assert n % 16 == 0 and n >= 4 * (256 * 4 + 2 + 128)
    A16 = 0x10000
    assert _call(qmm, "qmm_moe_gemv", A16, A16, 256, 64, 64, A16, 16, 8, A16, A16, 0, A16, A16, n - 16, None) == 8
    assert _call(qmm, "qmm_moe_gemv", A16, A16, 256, 64, 64, A16, 16, 8, A16, A16, 0, A16, None, n, None) == 8


def test_gemm_workspace_size_and_rules(qmm):
    """qmm_gemm_workspace_size: one record of 9216 * ceil(M / 8) bytes per 512
    columns of K (rounded up) and 16 KiB of flags for 1..16 tokens, 0
    otherwise; the workspace
    entry checks the product's arguments first (same statuses as the plain
    entry), then the workspace (NULL, too small, misaligned: QMM_ERR_WORKSPACE),
    all before any device call."""
    flags = 4096 * 4  # the even cut's flag words
    assert qmm.qmm_gemm_workspace_size(8192, 16) == 16 * 18432 + flags
    assert qmm.qmm_gemm_workspace_size(8192, 8) == 16 * 9216 + flags
    assert qmm.qmm_gemm_workspace_size(768, 9) == 2 * 18432 + flags    # a last half unit is a whole record
    assert qmm.qmm_gemm_workspace_size(2048, 17) == 0
    assert qmm.qmm_gemm_workspace_size(2048, 0) == 0
    out = ctypes.c_size_t(0)
    lib = qmm.library_handle()
    assert lib.qmm_gemm_workspace_size(48, 4, ctypes.byref(out)) == 2
    assert lib.qmm_gemm_workspace_size(64, -1, ctypes.byref(out)) == 1
    assert lib.qmm_gemm_workspace_size(64, 4, None) == 1
    A16 = 0x10000
    n = qmm.qmm_gemm_workspace_size(8192, 16)
    ws = lambda *a: _call(qmm, "qmm_gemm_q4_0_q8_0_ws", *a)  # noqa: E731
    assert ws(A16, A16, -1, 8192, 16, A16, A16, A16, 64, A16, n, None) == 1       # as the plain entry
    assert ws(A16, A16, 64, 48, 16, A16, A16, A16, 64, A16, n, None) == 2
    assert ws(A16, A16 + 1, 64, 8192, 16, A16, A16, A16, 64, A16, n, None) == 3
    assert ws(A16, A16, 64, 8192, 16, A16, A16, A16, 64, None, n, None) == 8      # no workspace
    assert ws(A16, A16, 64, 8192, 16, A16, A16, A16, 64, A16, n - 16, None) == 8  # too small
    assert ws(A16, A16, 64, 8192, 16, A16, A16, A16, 64, A16 + 64, n, None) == 8  # not 128-byte aligned


def test_static_scratch_limit_and_arguments(qmm):
    """qmm_moe_gemv_static checks its fixed scratch limit (256 KiB) on the
    host before touching a device."""
    A16 = 0x10000
    assert qmm.qmm_moe_workspace_size(256, 8064, 8) > 256 * 1024
    assert _call(qmm, "qmm_moe_gemv_static", A16, A16, 256, 64, 64, A16, 8064, 8, A16, A16, 0, A16, None) == 9
    assert _call(qmm, "qmm_moe_gemv_static", A16, A16, 0, 64, 64, A16, 1, 8, A16, A16, 0, A16, None) == 1
    assert _call(qmm, "qmm_moe_gemv_static", A16, A16, 8, 0, 64, A16, 1, 8, A16, A16, 0, A16, None) == 1
    assert _call(qmm, "qmm_moe_gemv_static", A16, A16, 8, 64, 48, A16, 1, 2, A16, A16, 0, A16, None) == 2
    assert _call(qmm, "qmm_moe_gemv_static", A16, A16, 8, 64, 64, A16, 0, 2, A16, A16, 0, A16, None) == 0
    assert _call(qmm, "qmm_moe_gemv_static", A16 + 2, A16, 8, 64, 64, A16, 1, 2, A16, A16, 0, A16, None) == 3
    assert _call(qmm, "qmm_moe_gemv_static", A16, A16, 8, 64, 64, None, 1, 2, A16, A16, 0, A16, None) == 1
    # ids are checked after the other pointers, as qmm_moe_gemv does: a null
    # ids with a misaligned weight plane is an alignment error in both
    ws = qmm.qmm_moe_workspace_size(8, 1, 2)
    assert _call(qmm, "qmm_moe_gemv", A16 + 2, A16, 8, 64, 64, None, 1, 2, A16, A16, 0, A16, A16, ws, None) == 3
    assert _call(qmm, "qmm_moe_gemv_static", A16 + 2, A16, 8, 64, 64, None, 1, 2, A16, A16, 0, A16, None) == 3
    assert _call(qmm, "qmm_moe_gemv_static", A16, A16, 8, 64, 64, A16 + 2, 1, 2, A16, A16, 0, A16, None) == 3


def test_fused_op_validation(qmm):
    """qmm_gemv_fused_op rejects bad descriptors before any launch."""
    A16 = 0x10000
    good = dict(w_qs=A16, w_d=A16, N=64, K=256, xq=A16, xd=A16, yq=A16, yd=A16)

    def run(o, flags=0):
        op = qmm.gemv_op(**o)
        return qmm.library_handle().qmm_gemv_fused_op(ctypes.byref(op), flags, None)

    assert run(good, flags=1) == 1                  # only QMM_CHAIN (4) as a call flag
    assert run(dict(good, K=288)) == 2             # K % 256 != 0
    assert run(dict(good, flags=4)) == 1           # only Y_SWIGLU_PAIRS as an op flag
    assert run(dict(good, N=48)) == 2              # Q8_0 output needs N % 32 == 0
    assert run(dict(good, w_d=A16 + 2)) == 3       # scale plane 16-byte aligned
    assert run(dict(good, yq=None, yd=None)) == 1  # no output at all
    assert run(dict(good, flags=2, residual=A16)) == 1  # pairs with a residual


def test_fused_ops_chain_validation(qmm):
    """qmm_gemv_fused_ops checks every op before launching any: the first bad
    op's status; bad counts, a NULL array and unknown flags are QMM_ERR_ARG;
    an empty chain is a no-op (a valid chain reaches the device check: the
    test below, run only where no GPU is present)."""
    A16 = 0x10000
    good = qmm.gemv_op(A16, A16, 64, 256, xq=A16, xd=A16, yq=A16, yd=A16)
    bad_k = qmm.gemv_op(A16, A16, 64, 288, xq=A16, xd=A16, yq=A16, yd=A16)
    bad_al = qmm.gemv_op(A16, A16 + 2, 64, 256, xq=A16, xd=A16, yq=A16, yd=A16)
    lib = qmm.library_handle()
    arr = qmm.gemv_op_array([good, good, bad_k, bad_al])
    assert lib.qmm_gemv_fused_ops(arr, 4, 0, None) == 2      # op 2 is the first bad one
    arr2 = qmm.gemv_op_array([good, bad_al, bad_k])
    assert lib.qmm_gemv_fused_ops(arr2, 3, 0, None) == 3
    assert lib.qmm_gemv_fused_ops(arr, -1, 0, None) == 1
    assert lib.qmm_gemv_fused_ops(None, 2, 0, None) == 1
    assert lib.qmm_gemv_fused_ops(arr, 2, 1, None) == 1      # only QMM_CHAIN as a call flag
    assert lib.qmm_gemv_fused_ops(None, 0, 0, None) == 0


def test_router_and_pregrouped_validation(qmm):
    """qmm_moe_router_topk: 1 <= k <= min(E, 64), E <= 1024, workspace size
    and alignment; qmm_moe_layer_f32: the checks of its four launches, all
    made before the first; qmm_moe_gemv_pregrouped: the workspace rules of
    qmm_moe_gemv.  All rejected on the host."""
    A16 = 0x10000
    r = lambda *a: _call(qmm, "qmm_moe_router_topk", *a)  # noqa: E731
    n = qmm.qmm_moe_workspace_size(256, 16, 8)
    assert r(A16, 16, 256, 0, A16, A16, None, 0, None) == 1          # k = 0
    assert r(A16, -1, 256, 8, A16, A16, None, 0, None) == 1          # T < 0
    assert r(A16, 16, 256, 65, A16, A16, None, 0, None) == 2         # k > QMM_ROUTER_MAX_K
    assert r(A16, 16, 4, 5, A16, A16, None, 0, None) == 2            # k > E
    assert r(A16, 16, 1025, 8, A16, A16, None, 0, None) == 2         # E > QMM_ROUTER_MAX_EXPERTS
    assert r(A16, 0, 256, 8, A16, A16, None, 0, None) == 0           # T = 0: no-op
    assert r(None, 16, 256, 8, A16, A16, None, 0, None) == 1         # null logits
    assert r(A16, 16, 256, 8, A16, A16, A16, n - 16, None) == 8      # workspace too small
    assert r(A16 + 2, 16, 256, 8, A16, A16, None, 0, None) == 3      # logits not 4-byte aligned
    assert r(A16, 16, 256, 8, A16, A16, A16 + 8, n, None) == 3       # workspace not 16-byte aligned
    ly = lambda T, k, H, F, ptrs, ws, wsb: _call(qmm, "qmm_moe_layer_f32", A16, T, 256, k, *ptrs[:4], H, F,  # noqa: E731
                                                  *ptrs[4:], ws, wsb, None)
    ok = [A16] * 10  # gu_qs, gu_d, down_qs, down_d, x, ids, gates, h, z, y
    assert ly(-1, 8, 512, 256, ok, A16, n) == 1                       # T < 0
    assert ly(16, 0, 512, 256, ok, A16, n) == 1                       # k = 0
    assert ly(16, 8, 500, 256, ok, A16, n) == 2                       # H % 32
    assert ly(0, 8, 512, 256, ok, A16, n) == 0                        # T = 0: no-op
    assert ly(16, 8, 512, 256, ok[:9] + [None], A16, n) == 1          # no y
    assert ly(16, 8, 512, 256, ok, A16, n - 16) == 8                  # workspace too small
    assert ly(16, 8, 512, 256, ok, None, n) == 8                      # workspace required
    assert ly(16, 8, 512, 256, ok[:4] + [A16 + 4] + ok[5:], A16, n) == 3  # x not 16-byte aligned
    assert ly(16, 8, 512, 256, [A16 + 8] + ok[1:], A16, n) == 3       # gate/up nibbles not 16-byte aligned
    assert ly(16, 8, 512, 96, ok, A16, n) == 2                        # F: no streaming path
    assert ly(16, 8, 512, 256, [A16, A16 + 2] + ok[2:], A16, n) == 2  # gate/up scales: no streaming path
    p = lambda *a: _call(qmm, "qmm_moe_gemv_pregrouped", *a)  # noqa: E731
    assert p(A16, A16, 256, 64, 64, 16, 8, A16, A16, 0, A16, A16, n - 16, None) == 8
    assert p(A16, A16, 256, 64, 64, 16, 8, A16, A16, 0, A16, None, n, None) == 8
    assert p(A16, A16, 256, 64, 48, 16, 8, A16, A16, 0, A16, A16, n, None) == 2
    assert p(A16, A16, 256, 64, 64, 0, 8, A16, A16, 0, A16, A16, n, None) == 0


def test_format_variant_validation(qmm):
    """Per-row int4/int2 quantizer and GEMV, Q4_0 x fp32 FMA GEMV: bits,
    K multiples, K limits, alignment, all rejected on the host."""
    A16 = 0x10000
    q = lambda *a: _call(qmm, "qmm_quantize_rowwise", *a)  # noqa: E731
    assert q(A16, 4, 64, 64, 3, A16, A16, None) == 1          # bits not 2 or 4
    assert q(A16, 4, 96, 96, 2, A16, A16, None) == 2          # int2 needs K % 64 == 0
    assert q(A16, 4, 48, 48, 4, A16, A16, None) == 2          # int4 needs K % 32 == 0
    assert q(A16, 4, 64, 32, 4, A16, A16, None) == 1          # ldw < K
    assert q(A16, 0, 64, 64, 4, A16, A16, None) == 0          # N = 0: no-op
    assert q(A16 + 2, 4, 64, 64, 4, A16, A16, None) == 3
    g = lambda *a: _call(qmm, "qmm_gemv_rowwise_q8_0", *a)  # noqa: E731
    assert g(A16, A16, 3, 8, 64, A16, A16, A16, None) == 1
    assert g(A16, A16, 2, 8, 96, A16, A16, A16, None) == 2
    assert g(A16, A16, 4, 8, 131072 + 32, A16, A16, A16, None) == 2   # above QMM_ROWWISE_MAX_K
    assert g(A16 + 8, A16, 4, 8, 64, A16, A16, A16, None) == 3        # codes not 16-byte aligned
    assert g(A16, A16, 4, 8, 64, A16 + 4, A16, A16, None) == 3        # xq not 16-byte aligned
    assert g(A16, A16, 4, 0, 64, A16, A16, A16, None) == 1
    f = lambda *a: _call(qmm, "qmm_gemv_q4_0_f32_fma", *a)  # noqa: E731
    assert f(A16, A16, 8, 48, A16, A16, None) == 2                    # K % 32
    assert f(A16, A16, 8, 49152 + 32, A16, A16, None) == 2            # above QMM_F32_FMA_MAX_K
    assert f(A16, A16, 8, 64, A16 + 4, A16, None) == 3                # x not 16-byte aligned
    assert f(None, A16, 8, 64, A16, A16, None) == 1


def test_valid_call_without_gpu_reports_device_error(qmm):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    A16 = 0x10000
    assert _call(qmm, "qmm_gemv_q4_0_q8_0", A16, A16, 64, 64, A16, A16, A16, None) == 4
    assert _call(qmm, "qmm_moe_gemv_static", A16, A16, 8, 64, 64, A16, 1, 2, A16, A16, 0, A16, None) == 4
    op = qmm.gemv_op(A16, A16, 64, 256, xq=A16, xd=A16, y=A16)
    assert qmm.library_handle().qmm_gemv_fused_op(ctypes.byref(op), 0, None) == 4
    assert _call(qmm, "qmm_moe_router_topk", A16, 16, 256, 8, A16, A16, None, 0, None) == 4
    assert _call(qmm, "qmm_gemv_rowwise_q8_0", A16, A16, 4, 8, 64, A16, A16, A16, None) == 4
    assert _call(qmm, "qmm_gemv_q4_0_f32_fma", A16, A16, 8, 64, A16, A16, None) == 4
    assert _call(qmm, "qmm_quantize_rowwise", A16, 4, 64, 64, 2, A16, A16, None) == 4
    assert _call(qmm, "qmm_last_device_error", None) == 4
    # a chain of valid ops; the workspace entry with 17 tokens (no workspace
    # needed: the plain entry's path)
    good = qmm.gemv_op(A16, A16, 64, 256, xq=A16, xd=A16, yq=A16, yd=A16)
    assert qmm.library_handle().qmm_gemv_fused_ops(qmm.gemv_op_array([good, good]), 2, 4, None) == 4
    assert _call(qmm, "qmm_gemm_q4_0_q8_0_ws", A16, A16, 64, 8192, 17, A16, A16, A16, 64, None, 0, None) == 4


def test_gemm_kernel_selector_and_moe_fp32_validation(qmm):
    """qmm_debug_gemm_kernel accepts the five documented kernels, returns the
    previous choice and rejects others; the fp32-activation and gate/up MoE
    entries reject bad shapes, workspaces and alignment on the host."""
    prev = ctypes.c_int(-1)
    lib = qmm._lib
    assert lib.qmm_debug_gemm_kernel(3, ctypes.byref(prev)) == 0
    start = prev.value
    assert lib.qmm_debug_gemm_kernel(4, ctypes.byref(prev)) == 0 and prev.value == 3
    assert lib.qmm_debug_gemm_kernel(2, ctypes.byref(prev)) == 0 and prev.value == 4
    assert lib.qmm_debug_gemm_kernel(5, None) == 1
    assert lib.qmm_debug_gemm_kernel(-1, None) == 1
    assert lib.qmm_debug_gemm_kernel(start, ctypes.byref(prev)) == 0 and prev.value == 2
    A16 = 0x10000
    n = qmm.qmm_moe_workspace_size(256, 16, 8)
    f = lambda *a: _call(qmm, "qmm_moe_gemv_pregrouped_f32", *a)  # noqa: E731
    assert f(A16, A16, 256, 64, 64, 16, 8, A16, 0, A16, A16, n - 16, None) == 8  # workspace too small
    assert f(A16, A16, 256, 64, 48, 16, 8, A16, 0, A16, A16, n, None) == 2       # K % 32
    assert f(A16, A16, 256, 64, 64, 16, 8, None, 0, A16, A16, n, None) == 1      # no activation
    assert f(A16, A16, 256, 64, 64, 16, 8, A16 + 4, 0, A16, A16, n, None) == 3   # x not 16-byte aligned
    assert f(A16, A16, 256, 64, 64, 0, 8, A16, 0, A16, A16, n, None) == 0        # T = 0: no-op
    g = lambda *a: _call(qmm, "qmm_moe_gemv_gate_up", *a)  # noqa: E731
    assert g(A16, A16, 256, 63, 256, 16, 8, None, A16, A16, 0, A16, A16, n, None) == 2  # N odd
    assert g(A16, A16, 256, 64, 256, 16, 8, A16 + 4, None, None, 0, A16, A16, n, None) == 3  # fp32 x misaligned
    assert g(A16, A16, 256, 64, 256, 16, 8, None, A16, A16, 0, A16, A16, n - 16, None) == 8  # workspace
    gi = lambda *a: _call(qmm, "qmm_moe_group_ids", *a)  # noqa: E731
    assert gi(A16, 16, 0, 256, A16, n, None) == 1            # k = 0
    assert gi(A16, 16, 8, 256, None, n, None) == 1           # no workspace
    assert gi(A16, 16, 8, 256, A16, n - 16, None) == 8       # workspace too small
    assert gi(A16 + 2, 16, 8, 256, A16, n, None) == 3        # ids misaligned
    assert gi(A16, 0, 8, 256, A16, n, None) == 0             # T = 0: no-op


def test_stream_wait_hook_arguments(qmm):
    """qmm_debug_stream_wait: bound in [1e3, 1e10] ns, withhold flag 0 or 1;
    returns the previous bound (two seconds by default)."""
    lib = qmm._lib
    prev = ctypes.c_uint64(0)
    assert lib.qmm_debug_stream_wait(999, 0, None) == 1
    assert lib.qmm_debug_stream_wait(10_000_000_001, 0, None) == 1
    assert lib.qmm_debug_stream_wait(1_000_000, 2, None) == 1
    assert lib.qmm_debug_stream_wait(1_000_000, 0, ctypes.byref(prev)) == 0 and prev.value == 2_000_000_000
    assert lib.qmm_debug_stream_wait(2_000_000_000, 0, ctypes.byref(prev)) == 0 and prev.value == 1_000_000
