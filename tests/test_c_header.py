"""include/nvfp4.h is a C ABI: a plain C99 program must compile against it
(strict, warnings as errors), link libnvfp4.so and call it.  The calls made
here are the host-only ones (version, status strings, workspace sizes) and
argument checks that return before the library touches a GPU, so the test
runs without one.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

from gemm_nvfp4_gb300 import build

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "nvfp4.h"

static int expect(int got, int want, const char *what)
{
    if (got != want) {
        printf("%s: got %d, want %d\n", what, got, want);
        return 1;
    }
    return 0;
}

int main(void)
{
    int bad = 0;
    uint32_t code = 0;
    const uint16_t *x = NULL;
    /* a 16-byte-aligned address that is never dereferenced: the calls below
       return from their host-side checks */
    static uint16_t fake_buf[16];
    const uint16_t *fake16 = (const uint16_t *)(((uintptr_t)fake_buf + 15) & ~(uintptr_t)15);
    size_t ws;

    bad |= nvfp4_version() < 100;
    bad |= strncmp(nvfp4_status_string(NVFP4_ERR_DEVICE_TIMEOUT), "NVFP4_", 6) != 0;
    ws = nvfp4_workspace_bytes(NVFP4_OP_GEMV_SKINNY, 4, 4096, 4096);
    bad |= ws < NVFP4_STATUS_WORD_OFFSET + 4;
    bad |= nvfp4_workspace_bytes(NVFP4_OP_GEMV_SKINNY, 17, 4096, 4096) != 0;
    bad |= expect(nvfp4_gemv_skinny(x, 1, NULL, NULL, NULL, 64, 64, NULL, NVFP4_OUT_F32, NULL, 0, NULL),
                  NVFP4_ERR_INVALID_ARG, "skinny with null pointers");
    bad |= expect(nvfp4_gemm_prefill(x, 40, NULL, NULL, NULL, 64, 40, NULL, NVFP4_OUT_BF16, NULL, 0, NULL),
                  NVFP4_ERR_UNSUPPORTED_SHAPE, "prefill with K % 16 != 0");
    bad |= expect(nvfp4_quantize(NULL, 16, 16, NULL, NULL, NULL, NULL, 0, NULL), NVFP4_ERR_INVALID_ARG,
                  "quantize with null pointers");
    bad |= expect(nvfp4_device_status(NULL, 256, 1, &code, NULL), NVFP4_ERR_INVALID_ARG,
                  "device status without a workspace");
    /* a problem whose scratch exceeds the fixed array is refused before any CUDA call */
    bad |= nvfp4_workspace_bytes(NVFP4_OP_GEMV_SKINNY, 1, 64, (int64_t)1 << 20) <= NVFP4_NOALLOC_SCRATCH_BYTES;
    bad |= expect(nvfp4_gemv_skinny_noalloc(fake16, 1, (const uint8_t *)fake16, (const uint8_t *)fake16,
                                            (const float *)fake16, 64, (int64_t)1 << 20, (void *)fake16,
                                            NVFP4_OUT_F32, NULL),
                  NVFP4_ERR_WORKSPACE, "no-allocation call beyond its scratch");
    /* bad arguments are reported as by nvfp4_gemv_skinny, before the size limit */
    bad |= expect(nvfp4_gemv_skinny_noalloc(x, 1, NULL, NULL, NULL, 64, (int64_t)1 << 20, NULL, NVFP4_OUT_F32,
                                            NULL),
                  NVFP4_ERR_INVALID_ARG, "no-allocation call with null pointers");
    printf(bad ? "FAILED\n" : "ok\n");
    return bad;
}
"""


@pytest.fixture(scope="module")
def libdir():
    return os.path.dirname(build.build())


def test_header_compiles_as_c99_and_links(libdir, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler on this host")
    src = tmp_path / "prog.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "prog"
    include = os.path.dirname(build.HEADER)
    cmd = [cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", include, str(src), "-o", str(exe),
           "-L", libdir, "-lnvfp4", f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
