"""The boundary from plain C: include/qmm.h compiles as C11 with warnings as
errors, a C program links libqmm.so and calls entries that need no GPU
(version, status strings, argument checks that fail before any device call,
the host-only LRU policy)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "qmm.h"

int main(void) {
    if (qmm_abi_version() != QMM_ABI_VERSION) return 10;
    if (strncmp(qmm_status_string(QMM_ERR_SHAPE), "QMM_ERR_SHAPE", 13) != 0) return 11;
    /* K not a multiple of 32: rejected before any device work */
    const uint8_t* qs = (const uint8_t*)0x10000;
    const uint16_t* d = (const uint16_t*)0x10000;
    if (qmm_gemv_q4_0_q8_0(qs, d, 64, 48, (const int8_t*)0x10000, d, (float*)0x10000, NULL) != QMM_ERR_SHAPE)
        return 12;
    size_t ws = 0;
    if (qmm_moe_workspace_size(256, 16, 8, &ws) != QMM_OK || ws == 0 || ws % 16 != 0) return 13;
    /* the expert-store policy runs on the host */
    qmm_lru* lru = NULL;
    if (qmm_lru_create(8, 2, &lru) != QMM_OK) return 14;
    int32_t keys[3] = {5, 6, 5}, slots[3], lk[3], ls[3], nl = 0;
    if (qmm_lru_request(lru, keys, 3, 1, slots, lk, ls, &nl) != QMM_OK) return 15;
    if (nl != 2 || slots[0] != 0 || slots[1] != 1 || slots[2] != 0) return 16;
    int64_t hits = -1, misses = -1;
    if (qmm_lru_stats(lru, &hits, &misses, NULL, NULL) != QMM_OK || hits != 0 || misses != 2) return 17;
    qmm_lru_destroy(lru);
    printf("ok\n");
    return 0;
}
"""


@pytest.fixture(scope="module")
def libdir():
    from block_quantized_int4_gb300 import _build
    _build.build()
    from block_quantized_int4_gb300 import qmm
    return os.path.dirname(qmm.LIB_PATH)


def test_header_is_c11_and_library_links(libdir, tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_qmm.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_qmm"
    inc = os.path.join(ROOT, "include")
    cuda_inc = "/usr/local/cuda/include"
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", inc, str(src), "-o", str(exe),
           "-L", libdir, "-lqmm", "-Wl,-rpath," + libdir]
    if os.path.isdir(cuda_inc):
        cmd[4:4] = ["-I", cuda_inc]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
