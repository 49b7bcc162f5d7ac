"""The product path from plain C, with no Python in between: a C11 program
allocates device buffers with the CUDA runtime, uploads an integer-grid
problem (all scales 1.0, so every output is an exact integer), calls
qmm_quantize_q8_0 and qmm_gemv_q4_0_q8_0 on the default stream, and checks
the Q8_0 codes and the GEMV outputs bit for bit against the exact integer
product it computes itself."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = "/usr/local/cuda"

C_PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime.h>
#include "qmm.h"

enum { N = 96, K = 512, B = K / 32 };

static int wq(int n, int k) { return ((n * 7 + k * 13) % 16) - 8; }  /* codes in [-8, 7] */
static int xq(int k) { return k % 32 == 5 ? 127 : ((k * 29) % 255) - 127; }  /* in [-127, 127] */

int main(void) {
    uint8_t* h_qs = malloc((size_t)N * K / 2);
    uint16_t* h_wd = malloc((size_t)N * B * 2);
    float* h_x = malloc((size_t)K * 4);
    for (int n = 0; n < N; ++n)
        for (int b = 0; b < B; ++b) {
            h_wd[n * B + b] = 0x3C00; /* fp16 1.0 */
            for (int j = 0; j < 16; ++j) {
                const int lo = wq(n, 32 * b + j) + 8, hi = wq(n, 32 * b + j + 16) + 8;
                h_qs[(size_t)n * K / 2 + b * 16 + j] = (uint8_t)(lo | (hi << 4));
            }
        }
    /* every 32-block of x holds integers in [-127, 127] with a 127 in it, so
       its Q8_0 scale is 1.0 and its codes are the values themselves */
    for (int k = 0; k < K; ++k) h_x[k] = (float)xq(k);

    uint8_t* qs; uint16_t* wd; float* x; int8_t* q; uint16_t* d; float* y;
    if (cudaMalloc((void**)&qs, (size_t)N * K / 2) || cudaMalloc((void**)&wd, (size_t)N * B * 2) ||
        cudaMalloc((void**)&x, (size_t)K * 4) || cudaMalloc((void**)&q, K) || cudaMalloc((void**)&d, B * 2) ||
        cudaMalloc((void**)&y, (size_t)N * 4))
        return 20;
    if (cudaMemcpy(qs, h_qs, (size_t)N * K / 2, cudaMemcpyHostToDevice) ||
        cudaMemcpy(wd, h_wd, (size_t)N * B * 2, cudaMemcpyHostToDevice) ||
        cudaMemcpy(x, h_x, (size_t)K * 4, cudaMemcpyHostToDevice))
        return 21;
    if (qmm_quantize_q8_0(x, 1, K, K, q, d, NULL) != QMM_OK) return 22;
    if (qmm_gemv_q4_0_q8_0(qs, wd, N, K, q, d, y, NULL) != QMM_OK) return 23;
    if (qmm_last_device_error(NULL) != QMM_OK) return 24;
    int8_t h_q[K]; uint16_t h_d[B]; float h_y[N];
    if (cudaMemcpy(h_q, q, K, cudaMemcpyDeviceToHost) || cudaMemcpy(h_d, d, B * 2, cudaMemcpyDeviceToHost) ||
        cudaMemcpy(h_y, y, (size_t)N * 4, cudaMemcpyDeviceToHost))
        return 25;
    for (int b = 0; b < B; ++b) if (h_d[b] != 0x3C00) return 30;
    for (int k = 0; k < K; ++k) if (h_q[k] != (int)h_x[k]) return 31;
    for (int n = 0; n < N; ++n) {
        long s = 0;
        for (int k = 0; k < K; ++k) s += (long)wq(n, k) * (long)h_q[k];
        if (h_y[n] != (float)s) { fprintf(stderr, "row %d: %g vs %ld\n", n, h_y[n], s); return 32; }
    }
    cudaFree(qs); cudaFree(wd); cudaFree(x); cudaFree(q); cudaFree(d); cudaFree(y);
    free(h_qs); free(h_wd); free(h_x);
    printf("ok\n");
    return 0;
}
"""


def test_c_program_runs_the_gemv_on_device_buffers(tmp_path):
    from block_quantized_int4_gb300 import _build
    _build.build()
    from block_quantized_int4_gb300 import qmm
    libdir = os.path.dirname(qmm.LIB_PATH)
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "gemv_from_c.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "gemv_from_c"
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), str(src), "-o", str(exe), "-L", libdir, "-lqmm",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + libdir,
           "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
