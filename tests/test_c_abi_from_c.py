"""The C ABI from plain C: a C99 program includes include/mxfp4moe.h, links against the
built libmxfp4moe.so and calls the entry points that need no GPU (version, status strings,
argument validation that rejects a call before any CUDA work)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mxfp4moe.h"

int main(void) {
    char buf[16];
    int bad;
    if (mx_version() < 100) return 1;
    if (strcmp(mx_status_string(MX_ERR_UNSUPPORTED), "MX_ERR_UNSUPPORTED") != 0) return 2;
    /* cols not a multiple of 32: rejected before any CUDA call, nothing dereferenced */
    bad = mxfp4_dequant((const uint8_t*)buf, (const uint8_t*)buf, buf, 4, 48, NULL);
    if (bad != MX_ERR_UNSUPPORTED) return 3;
    if (moe_mxfp4_workspace_size(16, 256, 128, 4, 2, 1) == 0) return 4;
    if (nvfp4_tiled_scales_bytes(300, 7168) != (size_t)3 * 112 * 512) return 5;
    printf("ok %d\n", mx_version());
    return 0;
}
"""


def test_c_program_uses_the_library(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from fp4_block_scaled_mxfp4_gb300 import build
    lib = build.build()
    src = tmp_path / "use_abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_abi"
    libdir = os.path.dirname(lib)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", str(src), "-I",
                        os.path.join(ROOT, "include"), "-L", libdir, "-l:libmxfp4moe.so", "-Wl,-rpath," + libdir,
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.strip().startswith("ok ")
